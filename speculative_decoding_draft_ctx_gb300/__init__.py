"""GB300 (sm_103a) DSpark fused context-KV write.

One kernel launch norms (Gemma RMSNorm), ropes (partial NeoX) and stores the
context K/V of every draft layer into its paged KV cache, as bf16 or fp8
e4m3; a second launch does the draft tokens' fused QK-norm / RoPE with their
K/V insert.  The compute runs in ``libdspark_ctx_kv.so`` (C ABI declared in
``include/dspark_ctx_kv.h``); this package is its ctypes binding.
"""

from ._binding import (  # noqa: F401
    CACHE_ROW, EXPORTS, FLAG_COUNTER, FLAG_POS_RANGE, FLAG_SLOT_RANGE, FLAG_TIMEOUT, HEAD_DIM, KV_BF16, KV_FP8_E4M3, STATUS,
    STATUS_CODE, CacheDesc, DSparkError, Tables, cache_desc, check, dspark_ctx_kv_last_error,
    dspark_ctx_kv_rotary_dims_supported, dspark_ctx_kv_status_string, dspark_ctx_kv_validate_layers,
    dspark_ctx_kv_write, dspark_ctx_kv_write_ex, dspark_qknorm_rope_kv_insert, dspark_ctx_kv_project,
    dspark_ctx_kv_project_write, dspark_gemma_rms_norm, dspark_ctx_kv_write_layer_slots, kv_dtype_code, lib,
    library_path, dspark_ctx_kv_write_general, dspark_ctx_kv_general_supported,
    dspark_ctx_kv_validate_layers_general, dspark_ctx_kv_write_sched, dspark_ctx_kv_write_noalloc,
)
from .writer import (  # noqa: F401
    ContextKVWriter, gemma_rms_norm, general_layout_supported, project_context_kv, qknorm_rope_kv_insert,
    rotary_dims_supported,
)
