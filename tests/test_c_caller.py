"""The C ABI from a plain C99 program: include/attn.h compiles as C with every
warning an error, the program links against libattn_gb300.so, and calls that
need no GPU (version, status strings, workspace sizes, the decode plan and
argument rejection) behave as the header states."""
import os
import shutil
import subprocess

import pytest

import attention_attn_fwd_08_gb300 as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("failed: %s (line %d)\n", #c, __LINE__); ++fails; } } while (0)

int main(void)
{
    void* bad = (void*)0x1000;  /* never dereferenced: every call below fails validation first */
    int splits = 0, chunk = 0;
    CHECK(attn_abi_version() == 1);
    CHECK(strstr(attn_status_string(ATTN_ERR_INVALID_ARG), "invalid") != NULL);
    CHECK(attn_bwd_workspace_size(4, 2048, 32) == (size_t)2 * 4 * 2048 * 32 * 4);
    CHECK(attn_decode_workspace_size(1, 1, 100, 3, 2, 128) == 0);
    CHECK(attn_decode_plan(16, 1, 32768, 32, 8, &splits, &chunk) == ATTN_OK);
    CHECK(chunk % 64 == 0 && (long long)splits * chunk >= 32768 && (long long)(splits - 1) * chunk < 32768);
    CHECK(attn_decode_plan(1, 1, 16, 8, 3, &splits, &chunk) == ATTN_ERR_INVALID_ARG);
    /* H not a multiple of Hkv; an unsupported head size; a misaligned pointer */
    CHECK(attn_fwd(ATTN_BF16, bad, bad, bad, bad, NULL, 1, 4, 4, 3, 2, 64, 0.125f, 1, 0, 0.f, 0, NULL, 0, NULL)
          == ATTN_ERR_INVALID_ARG);
    CHECK(attn_fwd(ATTN_BF16, bad, bad, bad, bad, NULL, 1, 4, 4, 2, 1, 48, 0.125f, 1, 0, 0.f, 0, NULL, 0, NULL)
          == ATTN_ERR_UNSUPPORTED);
    CHECK(attn_fwd(ATTN_BF16, (void*)0x1001, bad, bad, bad, NULL, 1, 4, 4, 2, 1, 64, 0.125f, 1, 0, 0.f, 0, NULL, 0,
                   NULL) == ATTN_ERR_INVALID_ARG);
    /* an empty batch is a no-op */
    CHECK(attn_fwd(ATTN_BF16, bad, bad, bad, bad, NULL, 0, 4, 4, 2, 1, 64, 0.125f, 1, 0, 0.f, 0, NULL, 0, NULL)
          == ATTN_OK);
    printf("%s\n", fails ? "FAILED" : "ok");
    return fails != 0;
}
"""


def test_plain_c_program_uses_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    A.lib()  # builds the library if it is missing or stale
    lib = A.library_path()
    src = tmp_path / "caller.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
