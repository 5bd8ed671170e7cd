"""Quantized KV cache and GQA decode attention for GB300 (sm_103a).

The compute lives in libdq.so (CUDA kernels behind the C ABI of include/dq.h);
this package is its Python binding.  Build it with ``build.build()``.
"""
from ._lib import (BUFFER_NAMES, Buffers, Config, DQError, KVCache, TensorCfg, kv_sizes, load,  # noqa: F401
                   make_config, symbol_probs)
