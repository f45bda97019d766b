"""Failure detection without a GPU fault: a bounded wait that nothing will
complete runs out, the kernel records it and returns, the host reads
ATTN_ERR_TIMEOUT, and the context keeps working afterwards."""
import pytest
import torch

import attention_attn_fwd_08_gb300 as A
from helpers import run_fwd_case

pytestmark = pytest.mark.gpu

ST_SELFTEST = 1 << 7


def test_bounded_wait_times_out_and_context_survives():
    st, _ = A.attn_get_device_status()  # clear anything left over
    A.attn_selftest_bounded_wait(50_000)  # 50 ms
    st, word = A.attn_get_device_status()
    assert st == A.ERR_TIMEOUT and word & ST_SELFTEST
    st, word = A.attn_get_device_status()  # reading clears the word
    assert st == A.OK and word == 0
    run_fwd_case("bf16", 1, 130, 130, 2, 1, 64, causal=True, seed=11)


def test_selftest_rejects_unbounded_limits():
    with pytest.raises(A.AttnError):
        A.attn_selftest_bounded_wait(0)
    with pytest.raises(A.AttnError):
        A.attn_selftest_bounded_wait(10_000_000)
