"""GB300 (sm_103a) KV-cache decode step: in-place append + split-T decode attention.

The compute path is the C-ABI library ``libkvd.so`` (``include/kvd.h``), built
from ``csrc/`` by ``build.py``; ``kvd`` is its thin Python binding.  Importing
this package does not load the library; the first call does, and raises when
it is missing.
"""
from .kvd import (  # noqa: F401
    KVD_BF16, KVD_DEVERR_PAGE, KVD_DEVERR_PAST_LEN, KVD_DEVERR_TIMEOUT, KVD_ERR_CAPACITY, KVD_ERR_CUDA,
    KVD_ERR_INVALID_ARG, KVD_ERR_UNSUPPORTED, KVD_ERR_WORKSPACE, KVD_F16, KVD_F32, KVD_OK, KvdError,
    KVD_STEP_HISTORY_STABLE, alloc_host_inputs, alloc_host_staging, kvd_decode_step_host, kvd_decode_step_host_packed,
    kvd_host_staging_bytes,
    alloc_workspace, kvd_append, kvd_cache_bytes, kvd_decode_attention, kvd_decode_attention_noalloc,
    kvd_decode_plan, kvd_decode_step, kvd_decode_workspace_bytes, kvd_paged_append,
    kvd_paged_decode_attention, kvd_paged_decode_step, KVD_E4M3, kvd_append_e4m3,
    kvd_decode_attention_e4m3, kvd_decode_step_e4m3,
    kvd_status_string, kvd_workspace_init, library_path, load, raw,
)
