"""The user-facing writer object, shaped like the pages' DSparkContextKVWriter.

vLLM DSpark context-KV writer page: ``DSparkContextKVWriter(attn_layers)``
validates the layers' cache layout, ``supported(attn_layers)`` reports
whether the fused write can serve them, and calling the writer with
``(all_kv, k_norm_weight, eps, positions, cos_sin_cache, rotary_dim,
slot_mapping)`` stores every layer's context K/V.  Here the layers are given
as their cache tensors and fp32 scale tensors; the layout check, the offset /
pointer tables and the write all run in the C library.
"""

from __future__ import annotations

from ._binding import (
    HEAD_DIM, DSparkError, Tables, cache_desc, dspark_ctx_kv_general_supported, dspark_ctx_kv_rotary_dims_supported,
    dspark_ctx_kv_project, dspark_ctx_kv_project_write, dspark_ctx_kv_validate_layers,
    dspark_ctx_kv_validate_layers_general, dspark_ctx_kv_write, dspark_ctx_kv_write_ex, dspark_ctx_kv_write_general,
    dspark_ctx_kv_write_layer_slots, dspark_gemma_rms_norm, dspark_qknorm_rope_kv_insert, kv_dtype_code,
)


def rotary_dims_supported(rotary_dim: int, head_dim: int) -> bool:
    """The kernel rotates the leading 16, 32 or 64 dims of a 128-dim head."""
    return dspark_ctx_kv_rotary_dims_supported(rotary_dim, head_dim)


def general_layout_supported(head_dim: int, rotary_dim: int, block_size: int) -> bool:
    """The general write's rule: head_dim 64, 128 or 256, rotary_dim even in
    [2, head_dim], any block size >= 1."""
    return dspark_ctx_kv_general_supported(head_dim, rotary_dim, block_size)


class ContextKVWriter:
    """Writes precomputed context K/V into every draft layer's paged cache.

    ``kv_caches[l]``: ``[num_blocks, nkv, block_size, 256]`` bf16 (``"auto"``)
    or uint8 (``"fp8"``); ``k_scales[l]``, ``v_scales[l]``: fp32 CUDA tensors.
    The offset tables are rebuilt only when a cache or scale moves, and never
    while the current stream is capturing a CUDA graph.

    ``general=True`` also takes the layouts the pages' writer refuses: caches
    ``[num_blocks, nkv, block_size, 2 * head_dim]`` with head_dim 64, 128 or
    256, any block size, and any even rotary_dim up to the head dim (the
    general write; the pages' layouts still run on their own kernels).
    """

    def __init__(self, kv_caches, k_scales, v_scales, kv_cache_dtype="auto", general=False):
        self.kv_caches = list(kv_caches)
        self.k_scales = list(k_scales)
        self.v_scales = list(v_scales)
        self.kv_cache_dtype = kv_cache_dtype
        self.general = bool(general)
        (dspark_ctx_kv_validate_layers_general if self.general else dspark_ctx_kv_validate_layers)(self._descs())
        c0 = self.kv_caches[0]
        self.num_layers = len(self.kv_caches)
        self.num_blocks, self.num_kv_heads, self.block_size = (int(s) for s in c0.shape[:3])
        self.head_dim = int(c0.shape[3]) // 2
        self._dtype = kv_dtype_code(kv_cache_dtype)
        self._tables = Tables(self.num_layers)

    def _descs(self):
        return [cache_desc(c, self.kv_cache_dtype, k, v)
                for c, k, v in zip(self.kv_caches, self.k_scales, self.v_scales)]

    @staticmethod
    def supported(kv_caches, k_scales, v_scales, kv_cache_dtype="auto", general=False) -> bool:
        check = dspark_ctx_kv_validate_layers_general if general else dspark_ctx_kv_validate_layers
        try:
            check([cache_desc(c, kv_cache_dtype, k, v) for c, k, v in zip(kv_caches, k_scales, v_scales)])
        except DSparkError:
            return False
        return len(kv_caches) > 0

    @property
    def tables(self) -> Tables:
        return self._tables

    def ensure_tables(self, stream=None):
        self._tables.update(self.kv_caches, self.k_scales, self.v_scales, stream)

    def __call__(self, all_kv, k_norm_weight, eps, positions, cos_sin_cache, rotary_dim, slot_mapping,
                 stream=None, error_flags=None):
        """``slot_mapping``: one int64 tensor shared by every layer, or a list
        of one per layer (the same tensor everywhere counts as shared, like
        the pages' _shared_slot_mapping; otherwise each layer's rows go to
        its own slots)."""
        num_ctx, L, two, nkv, hd = all_kv.shape
        if L != self.num_layers or nkv != self.num_kv_heads or two != 2 or hd != self.head_dim:
            raise DSparkError(1, f"all_kv shape {tuple(all_kv.shape)} does not match the layers")
        if num_ctx == 0:
            return
        per_layer = None
        if isinstance(slot_mapping, (list, tuple)):
            if len(slot_mapping) != L or any(s is None for s in slot_mapping):
                raise DSparkError(1, "one slot mapping per layer expected")
            if all(s.data_ptr() == slot_mapping[0].data_ptr() for s in slot_mapping):
                slot_mapping = slot_mapping[0]
            else:
                per_layer = slot_mapping
        self.ensure_tables(stream)
        t = self._tables
        if per_layer is not None:
            t.update_slots(per_layer, stream)
        if self.general:
            dspark_ctx_kv_write_general(all_kv, k_norm_weight, positions,
                                        slot_mapping if per_layer is None else None,
                                        t.layer_slots if per_layer is not None else None, num_ctx, cos_sin_cache,
                                        cos_sin_cache.shape[0], self.kv_caches[0], self.num_blocks, t.cache_offsets,
                                        t.k_scales, t.v_scales, L, nkv, self.head_dim, self.block_size, rotary_dim,
                                        eps, self._dtype, error_flags, stream)
            return
        if per_layer is not None:
            dspark_ctx_kv_write_layer_slots(all_kv, k_norm_weight, positions, t.layer_slots, num_ctx,
                                            cos_sin_cache, cos_sin_cache.shape[0], self.kv_caches[0],
                                            self.num_blocks, t.cache_offsets, t.k_scales, t.v_scales, L, nkv,
                                            self.block_size, rotary_dim, eps, self._dtype, error_flags, stream)
            return
        args = (all_kv, k_norm_weight, positions, slot_mapping, num_ctx, cos_sin_cache,
                cos_sin_cache.shape[0], self.kv_caches[0], self.num_blocks, t.cache_offsets,
                t.k_scales, t.v_scales, L, nkv, self.block_size, rotary_dim, eps, self._dtype)
        if error_flags is None:
            dspark_ctx_kv_write(*args, stream=stream)
        else:
            dspark_ctx_kv_write_ex(*args, error_flags, stream=stream)

    def project_and_write(self, context_states, w_kv, k_norm_weight, eps, positions, cos_sin_cache, rotary_dim,
                          slot_mapping, stream=None, error_flags=None):
        """Project the (normed) context states with the stacked K/V weights
        ``w_kv`` ``[L * 2 * nkv * 128, hidden]`` and write every layer's
        context K/V in the same launch: all_kv never reaches device memory."""
        num_ctx, hidden = context_states.shape
        if w_kv.shape[0] != self.num_layers * 2 * self.num_kv_heads * HEAD_DIM or w_kv.shape[1] != hidden:
            raise DSparkError(1, f"w_kv shape {tuple(w_kv.shape)} does not match the layers and hidden {hidden}")
        if num_ctx == 0:
            return
        self.ensure_tables(stream)
        t = self._tables
        dspark_ctx_kv_project_write(context_states, w_kv, num_ctx, hidden, k_norm_weight, positions, slot_mapping,
                                    cos_sin_cache, cos_sin_cache.shape[0], self.kv_caches[0], self.num_blocks,
                                    t.cache_offsets, t.k_scales, t.v_scales, self.num_layers, self.num_kv_heads,
                                    self.block_size, rotary_dim, eps, self._dtype, error_flags, stream)


def qknorm_rope_kv_insert(qkv, q_norm_weight, k_norm_weight, cos_sin_cache, positions, num_heads,
                          num_kv_heads, rotary_dim, eps, slot_mapping=None, kv_cache=None,
                          k_scale=None, v_scale=None, q_fp8_out=None, q_fp8_scale=1.0,
                          error_flags=None, stream=None):
    """The draft tokens' fused QK-norm / RoPE on ``qkv`` (in place), also
    storing their K/V (DSpark draft model page, dspark_qknorm_rope_kv_insert).

    ``qkv``: bf16 ``[T, (num_heads + 2 num_kv_heads) * 128]``.  With
    ``slot_mapping`` and ``kv_cache`` (``[num_blocks, num_kv_heads,
    block_size, 256]``, bf16 or uint8 for fp8 e4m3 with the fp32 CUDA scalars
    ``k_scale`` / ``v_scale``) every token with a slot has its K'|V rows
    inserted; ``q_fp8_out`` (uint8 ``[T, num_heads * 128]``) receives
    e4m3(q' / q_fp8_scale).  The block size and the cache dtype are read from
    ``kv_cache``.
    """
    import torch

    T = qkv.shape[0]
    if qkv.dim() != 2 or qkv.shape[1] != (num_heads + 2 * num_kv_heads) * HEAD_DIM:
        raise DSparkError(1, f"qkv shape {tuple(qkv.shape)} does not match {num_heads}+2x{num_kv_heads} heads")
    if (slot_mapping is None) != (kv_cache is None):
        raise DSparkError(1, "slot_mapping and kv_cache go together")
    num_blocks = block_size = 0
    dtype = "auto"
    if kv_cache is not None:
        num_blocks, nkv, block_size = (int(x) for x in kv_cache.shape[:3])
        if nkv != num_kv_heads or kv_cache.shape[3] != 2 * HEAD_DIM:
            raise DSparkError(1, f"kv_cache shape {tuple(kv_cache.shape)} does not match {num_kv_heads} KV heads")
        dtype = "fp8" if kv_cache.dtype == torch.uint8 else "auto"
    dspark_qknorm_rope_kv_insert(qkv, q_norm_weight, k_norm_weight, cos_sin_cache, cos_sin_cache.shape[0],
                                 positions, T, num_heads, num_kv_heads, rotary_dim, eps, slot_mapping,
                                 kv_cache, num_blocks, block_size, dtype, k_scale, v_scale, q_fp8_out,
                                 q_fp8_scale, error_flags, stream)


def project_context_kv(context_states, w_kv, num_layers, num_kv_heads, out=None, stream=None):
    """all_kv = bf16(context_states @ w_kv^T) as ``[num_ctx, L, 2, nkv, 128]``
    on the tensor cores (the fused projection the context-KV writer reads)."""
    import torch

    num_ctx, hidden = context_states.shape
    if out is None:
        out = torch.empty((num_ctx, num_layers, 2, num_kv_heads, HEAD_DIM), dtype=torch.bfloat16,
                          device=context_states.device)
    dspark_ctx_kv_project(context_states, w_kv, out, num_ctx, hidden, num_layers, num_kv_heads, stream)
    return out


def gemma_rms_norm(x, weight, eps, out=None, stream=None):
    """The hidden-state Gemma RMSNorm of the context states (the draft model's
    hidden_norm): ``bf16(x * rsqrt(mean(x^2) + eps) * (1 + weight))`` per row
    of ``x`` (bf16 ``[rows, hidden]``); ``out=x`` works in place."""
    import torch

    rows, hidden = x.shape
    if out is None:
        out = torch.empty_like(x)
    dspark_gemma_rms_norm(x, weight, out, rows, hidden, eps, stream)
    return out
