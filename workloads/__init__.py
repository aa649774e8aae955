"""Seeded synthetic inputs shared by the oracle-side tests, the CUDA path's
tests and the benchmark.  Holds no arithmetic of the write itself."""

from .synth import (  # noqa: F401
    HEAD_DIM, ROW_ELEMS, PREFILL_BYTE, KV_BF16, KV_FP8, Workload, WORKLOADS,
    WORKLOADS_BY_NAME, Inputs, generate, make_caches, take_tokens,
    rope_cos_sin_cache, compulsory_bytes, describe, layer_slot_mappings, GENERAL_WORKLOADS,
    GENERAL_WORKLOADS_BY_NAME, pages_layout,
)
from .qk_insert import (  # noqa: F401
    QUERY_ROWS_PER_REQUEST, QkWorkload, QK_WORKLOADS, QK_WORKLOADS_BY_NAME, QkInputs, generate_qk,
    make_qk_cache, qk_compulsory_bytes, describe_qk,
)
from .proj import (  # noqa: F401
    ProjWorkload, PROJ_WORKLOADS, PROJ_WORKLOADS_BY_NAME, ProjInputs, generate_proj, proj_flops, with_all_kv,
)
from .hidden_norm import (  # noqa: F401
    NormWorkload, NORM_WORKLOADS, NORM_WORKLOADS_BY_NAME, generate_norm, norm_bytes,
)
