"""The affine path through the bounds-checked library (libdq_checked.so, built
with DQ_CHECKED): every global access on it tests its byte range against its
buffer and latches a status bit instead of going outside, which every
cache.check() below would report.  Runs in a process of its own, since a
process loads one build of the library.  The cases are the parity tests of
the normal build (bit-exact codes, attention against the oracle), so the
checks must neither fire nor change a result; then the checker's own probe
must be reported, and the context must keep working after it.

Prints one JSON line; exits non-zero on the first failure."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

from quantized_decode_attention_gb300 import build as B  # noqa: E402

B.build(checked=True)
from quantized_decode_attention_gb300 import _lib  # noqa: E402

_lib.use_checked_build()

import test_gpu_affine as TA  # noqa: E402
import test_gpu_step as TS  # noqa: E402
import test_zz_no_alloc as TN  # noqa: E402


def main():
    import torch
    done = []
    for name in ("llama2-ragged", "llama3-ragged", "llama4-ragged", "d64-bf16-2bit", "qwen-dense-clip", "llama2-quest",
                 "llama2-meta32"):
        TA.test_quantize_bit_exact(name)
        TA.test_attention_parity(name, "f32")
        done.append(name)
    for name in ("llama2", "dense-clip", "quest"):
        TS.test_decode_step_equals_append_then_attention(name)
        done.append("step-" + name)
    TN.test_noalloc_dense_transform_matches_context_and_oracle()
    done.append("noalloc-dense")
    assert os.path.basename(_lib.load()._name) == "libdq_checked.so", _lib.load()._name
    # the checker itself: a range one byte past a buffer is latched and reported
    w, S = TA.CASES["llama2-ragged"]
    cache, k, v, q, T, Qc = TA.run_case(w, S)
    lib = _lib.load()
    assert lib.dq_test_checked_probe(cache.ctx, None) == 0
    try:
        cache.check()
    except _lib.DQError as e:
        assert e.name == "DQ_EINVAL" and "outside its buffer" in str(e), str(e)
    else:
        raise AssertionError("the checked build did not report the probe")
    cache.check()  # reported once
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    cache.attention(TA.to_device(q, "f32"), out, S)
    cache.check()
    cache.close()
    print(json.dumps({"checked_build": True, "cases": done}))


if __name__ == "__main__":
    main()
