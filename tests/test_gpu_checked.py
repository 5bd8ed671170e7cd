"""The bounds-checked build of the library on the affine path (see
tests/checked_run.py, which runs in a child process): parity unchanged, no
access outside a buffer, and the checker's own probe reported."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu


def test_checked_build_runs_the_affine_path_clean():
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "checked_run.py")], capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert '"checked_build": true' in r.stdout


def test_normal_build_ignores_the_probe():
    # the same probe through libdq.so: range tests compile away, nothing latches
    import test_gpu_affine as TA
    from quantized_decode_attention_gb300 import _lib
    w, S = TA.CASES["llama2-ragged"]
    cache, k, v, q, T, Qc = TA.run_case(w, S)
    assert os.path.basename(_lib.load()._name) == "libdq.so"
    assert _lib.load().dq_test_checked_probe(cache.ctx, None) == 0
    cache.check()
    cache.close()
