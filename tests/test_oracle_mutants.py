"""The pins catch plausible mistakes in the oracle.

Each case copies oracle/ to a scratch directory, plants one mistake in the copy
(a flipped sign, a dropped term, an off-by-one bound, a wrong index or operand),
and runs every oracle pin against the copy in a child process: at least one pin
must fail.  An unmodified copy must pass them all, which shows that the child
really tests the copy.  Nothing here touches the oracle in place."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_ext_pins.py", "tests/test_oracle_varlen_pins.py",
        "tests/test_oracle_rope_pins.py"]

C, PY = "attn_oracle.c", "__init__.py"
WORKERS = min(8, os.cpu_count() or 2)
THREADS = max(1, (os.cpu_count() or 2) // WORKERS)  # per child, so the children share the cores
# (what the mistake breaks, file, text, planted text)
MUTANTS = [
    ("softcap derivative sign", C, "ds *= 1.0 - t * t;", "ds *= 1.0 + t * t;"),
    ("softcap derivative of the capped score", C, "double t = tanh(raw[j] / softcap);",
     "double t = tanh(raw[j] * tanh(raw[j] / softcap));"),
    ("dropped D term", C, "double ds = pij * (dpij - Di);", "double ds = pij * dpij;"),
    ("dK without the scale", C, "dkj[e] += scale * ds * qi[e];", "dkj[e] += ds * qi[e];"),
    ("dV from the wrong operand", C, "dvj[e] += pij * doi[e];", "dvj[e] += pij * qi[e];"),
    ("dQ from V instead of K", C, "dqi[e] += scale * ds * kj[e];", "dqi[e] += scale * ds * vj[e];"),
    ("GQA head map h mod Hkv", C, "const int kvh = h / G;", "const int kvh = h % d->Hkv;"),
    ("causal bound off by one", C, "if (d->causal && j > p) return 0;", "if (d->causal && j >= p) return 0;"),
    ("window bound off by one", C, "if (gap >= d->window) return 0;", "if (gap > d->window) return 0;"),
    ("query offset ignored", C, "const long long p = (long long)i + d->q_offset;", "const long long p = (long long)i;"),
    ("mask threshold", C, "b * d->mask_bstride + j] > 0.5)", "b * d->mask_bstride + j] >= 0.5)"),
    ("score scale dropped", C, "s *= d->scale;", "s *= 1.0;"),
    ("softcap outer factor dropped", C, "d->softcap * tanh(s / d->softcap)", "tanh(s / d->softcap)"),
    ("LSE in log2 units", C, "return m + log(l);", "return m + log2(l);"),
    ("P not normalised", C, "for (int j = 0; j < d->Tk; ++j) prob[j] /= l;", ""),
    ("fully masked row LSE", C, "        return -INFINITY;\n    }\n    double l = 0.0;",
     "        return 0.0;\n    }\n    double l = 0.0;"),
    ("right window side off by one", C, "if (d->wr >= 0 && j > p + d->wr) return 0;",
     "if (d->wr >= 0 && j > p + d->wr + 1) return 0;"),
    ("left window side off by one", C, "if (d->wl >= 0 && j < p - d->wl) return 0;",
     "if (d->wl >= 0 && j <= p - d->wl) return 0;"),
    ("bias ignored", C, "if (d->bias)\n", "if (0 && d->bias)\n"),
    ("bias rows and columns swapped", C, "(long long)i * d->bs[2] +\n                              (long long)j * d->bs[3]",
     "(long long)j * d->bs[2] +\n                              (long long)i * d->bs[3]"),
    ("packed sequences read the first sequence's keys", PY,
     "ob, lb = fwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1]",
     "ob, lb = fwd(q[None, q0:q1], k[None, 0:k1 - k0], v[None, 0:k1 - k0]"),
    ("rotary turn in the wrong direction", PY, "= a * c - b * sn", "= a * c + b * sn"),
    ("rotary frequency exponent", PY, "(-2.0 * i / hd)", "(-1.0 * i / hd)"),
    ("rotary position without the token index", PY, "p = float(pos + s)", "p = float(pos)"),
]


def run_pins(work, fname=None, old=None, new=None):
    """Copy oracle/ under `work`, plant the change, run the pins there; returns the
    child's (exit status, output tail)."""
    dst = os.path.join(work, "oracle")
    os.makedirs(dst)
    for f in (C, PY):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, f))
    if fname is not None:
        path = os.path.join(dst, fname)
        text = open(path).read()
        if text.count(old) != 1:
            return -1, "the text to change must occur once: %r" % old
        open(path, "w").write(text.replace(old, new))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([work, ROOT]), OMP_NUM_THREADS=str(THREADS),
               MKL_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    # run from the scratch directory, so that `import oracle` finds the copy first
    probe = "import oracle, sys; sys.exit(0 if oracle.__file__.startswith(%r) else 5)" % work
    if subprocess.run([sys.executable, "-c", probe], cwd=work, env=env).returncode != 0:
        return -2, "the child imported another oracle"
    pins = [os.path.join(ROOT, p) for p in PINS]
    r = subprocess.run([sys.executable, "-m", "pytest", *pins, "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=work, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, (r.stdout + r.stderr)[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every case at once (the children are independent processes)."""
    base = tmp_path_factory.mktemp("mutants")
    cases = [("unmodified", None, None, None)] + MUTANTS
    with ThreadPoolExecutor(max_workers=WORKERS) as ex:
        futs = {c[0]: ex.submit(run_pins, str(base / ("case%02d" % n)), *c[1:]) for n, c in enumerate(cases)}
        return {name: f.result() for name, f in futs.items()}


def test_unmodified_copy_passes_every_pin(outcomes):
    rc, out = outcomes["unmodified"]
    assert rc == 0, out


@pytest.mark.parametrize("what", [m[0] for m in MUTANTS], ids=[m[0].replace(" ", "-") for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, what):
    rc, out = outcomes[what]
    assert rc == 1, "no pin caught: %s (exit %d)\n%s" % (what, rc, out)
