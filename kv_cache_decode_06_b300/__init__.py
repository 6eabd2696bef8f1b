"""GQA decode over a bf16 KV cache, and the K/V mean-pool conversion, for B300 (sm_103a).

The compute path is the CUDA library ``libgqa_b300.so`` (C ABI in
``include/gqa.h``); :mod:`kv_cache_decode_06_b300.gqa` is its Python binding.
:mod:`kv_cache_decode_06_b300.inputs` draws the seeded synthetic workloads.
"""
from .gqa import (  # noqa: F401
    GQAError, PATH_AUTO, PATH_SIMT, PATH_TCGEN05, FLAG_SEQ_LEN_CLAMPED, FLAG_WAIT_TIMEOUT,
    alloc_workspace, decode, load, meanpool_kv, meanpool_kv_strided, read_flags, select_path, workspace_size,
)
