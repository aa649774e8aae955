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
    dspark_ctx_kv_validate_layers_general, dspark_ctx_kv_write_general, dspark_ctx_kv_write_sched,
    dspark_gemma_rms_norm, dspark_qknorm_rope_kv_insert, kv_dtype_code,
)
from ._binding import _stream as _stream_handle


def _need(cond, message: str):
    if not cond:
        raise DSparkError(1, message)


def _check_tensor(name, x, dtype, device, shape=None, ndim=None):
    """A tensor argument as the kernels read it: of ``dtype``, on ``device``,
    contiguous (the library receives only its address), and of ``shape``
    (``None`` in a shape entry: any extent) or ``ndim`` when given."""
    import torch

    _need(isinstance(x, torch.Tensor), f"{name} must be a tensor, got {type(x).__name__}")
    _need(x.dtype == dtype, f"{name} must be {dtype}, got {x.dtype}")
    _need(x.device == device, f"{name} is on {x.device}, expected {device}")
    _need(x.is_contiguous(), f"{name} must be contiguous")
    if ndim is not None:
        _need(x.dim() == ndim, f"{name} must have {ndim} dims, got shape {tuple(x.shape)}")
    if shape is not None:
        _need(x.dim() == len(shape) and all(e is None or int(a) == e for a, e in zip(x.shape, shape)),
              f"{name} must have shape {tuple('*' if e is None else e for e in shape)}, got {tuple(x.shape)}")


def _check_index(name, x, device, count):
    """positions / slot mappings: int64, contiguous, at least ``count``
    entries (the kernels read entries 0 .. count - 1)."""
    import torch

    _check_tensor(name, x, torch.int64, device, ndim=1)
    _need(x.numel() >= count, f"{name} has {x.numel()} entries, {count} tokens")


def _check_cos_sin(x, rotary_dim, device):
    import torch

    _check_tensor("cos_sin_cache", x, torch.bfloat16, device, ndim=2)
    _need(int(x.shape[1]) == int(rotary_dim),
          f"cos_sin_cache rows hold {int(x.shape[1])} values, rotary_dim is {rotary_dim}")
    _need(x.shape[0] > 0, "cos_sin_cache is empty")


def _check_flags(error_flags, device):
    import torch

    if error_flags is not None:
        _check_tensor("error_flags", error_flags, torch.int32, device)
        _need(error_flags.numel() >= 1, "error_flags must hold one int32 word")


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
        # the writer's own error word: every launch reports into it unless the
        # caller passes one (see error_flags())
        import torch

        self._flags = torch.zeros(1, dtype=torch.int32, device=c0.device)
        # work counters of the dynamic tail, one per stream the writer has
        # launched on outside capture: calls on one stream run in order and
        # share a counter, calls on different streams may overlap and must not
        self._work = {}

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

    def error_flags(self, clear: bool = True) -> int:
        """The bits the kernels raised in the writer's own error word since it
        was last cleared (calls that passed their own ``error_flags`` report
        there instead): FLAG_SLOT_RANGE / FLAG_POS_RANGE for rows skipped as
        out of range, FLAG_TIMEOUT when a launch gave up on a bounded wait and
        left rows unwritten, FLAG_COUNTER when a work counter was found not
        zero (rows of the tail unwritten).  Reading it synchronises with the
        device."""
        v = int(self._flags.item())
        if clear and v:
            self._flags.zero_()
        return v

    def ensure_tables(self, stream=None):
        self._tables.update(self.kv_caches, self.k_scales, self.v_scales, stream)

    def __call__(self, all_kv, k_norm_weight, eps, positions, cos_sin_cache, rotary_dim, slot_mapping,
                 stream=None, error_flags=None):
        """``slot_mapping``: one int64 tensor shared by every layer, or a list
        of one per layer (the same tensor everywhere counts as shared, like
        the pages' _shared_slot_mapping; otherwise each layer's rows go to
        its own slots)."""
        import torch

        dev = self.kv_caches[0].device
        _check_tensor("all_kv", all_kv, torch.bfloat16, dev, ndim=5)
        num_ctx, L, two, nkv, hd = all_kv.shape
        if L != self.num_layers or nkv != self.num_kv_heads or two != 2 or hd != self.head_dim:
            raise DSparkError(1, f"all_kv shape {tuple(all_kv.shape)} does not match the layers")
        _check_tensor("k_norm_weight", k_norm_weight, torch.bfloat16, dev, shape=(L, self.head_dim))
        _check_index("positions", positions, dev, num_ctx)
        _check_cos_sin(cos_sin_cache, rotary_dim, dev)
        _check_flags(error_flags, dev)
        per_layer = None
        if isinstance(slot_mapping, (list, tuple)):
            if len(slot_mapping) != L or any(s is None for s in slot_mapping):
                raise DSparkError(1, "one slot mapping per layer expected")
            for l, s in enumerate(slot_mapping):
                _check_index(f"slot_mapping[{l}]", s, dev, num_ctx)
            if all(s.data_ptr() == slot_mapping[0].data_ptr() for s in slot_mapping):
                slot_mapping = slot_mapping[0]
            else:
                per_layer = slot_mapping
        else:
            _check_index("slot_mapping", slot_mapping, dev, num_ctx)
        if num_ctx == 0:
            return
        if error_flags is None:
            error_flags = self._flags
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
        dspark_ctx_kv_write_sched(all_kv, k_norm_weight, positions, slot_mapping if per_layer is None else None,
                                  t.layer_slots if per_layer is not None else None, num_ctx, cos_sin_cache,
                                  cos_sin_cache.shape[0], self.kv_caches[0], self.num_blocks, t.cache_offsets,
                                  t.k_scales, t.v_scales, L, nkv, self.block_size, rotary_dim, eps, self._dtype,
                                  error_flags, self._work_counter(stream), stream)

    def _work_counter(self, stream):
        """The dynamic tail's counter of ``stream`` (None: the fixed split).
        Counters are made and zeroed outside capture only, so a call captured
        on a stream the writer has not launched on before takes the fixed
        split, and a captured call uses its stream's counter: a graph replay
        must then not overlap the writer's other calls on that stream."""
        import torch

        h = _stream_handle(stream)
        c = self._work.get(h)
        if c is None and not torch.cuda.is_current_stream_capturing():
            dev = self.kv_caches[0].device
            c = torch.zeros(2, dtype=torch.int64, device=dev)
            # zeroed on the current stream: land before a launch on another
            torch.cuda.current_stream(dev).synchronize()
            self._work[h] = c
        return c

    def project_and_write(self, context_states, w_kv, k_norm_weight, eps, positions, cos_sin_cache, rotary_dim,
                          slot_mapping, stream=None, error_flags=None):
        """Project the (normed) context states with the stacked K/V weights
        ``w_kv`` ``[L * 2 * nkv * 128, hidden]`` and write every layer's
        context K/V in the same launch: all_kv never reaches device memory."""
        import torch

        dev = self.kv_caches[0].device
        _need(self.head_dim == HEAD_DIM, "the fused projection takes head_dim 128")
        _check_tensor("context_states", context_states, torch.bfloat16, dev, ndim=2)
        num_ctx, hidden = context_states.shape
        _check_tensor("w_kv", w_kv, torch.bfloat16, dev, ndim=2)
        if w_kv.shape[0] != self.num_layers * 2 * self.num_kv_heads * HEAD_DIM or w_kv.shape[1] != hidden:
            raise DSparkError(1, f"w_kv shape {tuple(w_kv.shape)} does not match the layers and hidden {hidden}")
        _check_tensor("k_norm_weight", k_norm_weight, torch.bfloat16, dev, shape=(self.num_layers, HEAD_DIM))
        _check_index("positions", positions, dev, num_ctx)
        _check_index("slot_mapping", slot_mapping, dev, num_ctx)
        _check_cos_sin(cos_sin_cache, rotary_dim, dev)
        _check_flags(error_flags, dev)
        if num_ctx == 0:
            return
        if error_flags is None:
            error_flags = self._flags
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

    _need(isinstance(qkv, torch.Tensor), "qkv must be a tensor")
    dev = qkv.device
    _check_tensor("qkv", qkv, torch.bfloat16, dev, ndim=2)
    T = qkv.shape[0]
    if qkv.shape[1] != (num_heads + 2 * num_kv_heads) * HEAD_DIM:
        raise DSparkError(1, f"qkv shape {tuple(qkv.shape)} does not match {num_heads}+2x{num_kv_heads} heads")
    _check_tensor("q_norm_weight", q_norm_weight, torch.bfloat16, dev, shape=(HEAD_DIM,))
    _check_tensor("k_norm_weight", k_norm_weight, torch.bfloat16, dev, shape=(HEAD_DIM,))
    _check_cos_sin(cos_sin_cache, rotary_dim, dev)
    _check_index("positions", positions, dev, T)
    _check_flags(error_flags, dev)
    if (slot_mapping is None) != (kv_cache is None):
        raise DSparkError(1, "slot_mapping and kv_cache go together")
    num_blocks = block_size = 0
    dtype = "auto"
    if kv_cache is not None:
        _check_index("slot_mapping", slot_mapping, dev, T)
        _need(isinstance(kv_cache, torch.Tensor) and kv_cache.dtype in (torch.bfloat16, torch.uint8),
              "kv_cache must be a bf16 or uint8 (fp8 e4m3) tensor")
        _check_tensor("kv_cache", kv_cache, kv_cache.dtype, dev, ndim=4)
        num_blocks, nkv, block_size = (int(x) for x in kv_cache.shape[:3])
        if nkv != num_kv_heads or kv_cache.shape[3] != 2 * HEAD_DIM:
            raise DSparkError(1, f"kv_cache shape {tuple(kv_cache.shape)} does not match {num_kv_heads} KV heads")
        dtype = "fp8" if kv_cache.dtype == torch.uint8 else "auto"
        for name, sc in (("k_scale", k_scale), ("v_scale", v_scale)):
            if sc is not None:
                _check_tensor(name, sc, torch.float32, dev)
                _need(sc.numel() >= 1, f"{name} must hold one fp32 value")
    if q_fp8_out is not None:
        _check_tensor("q_fp8_out", q_fp8_out, torch.uint8, dev, shape=(T, num_heads * HEAD_DIM))
    dspark_qknorm_rope_kv_insert(qkv, q_norm_weight, k_norm_weight, cos_sin_cache, cos_sin_cache.shape[0],
                                 positions, T, num_heads, num_kv_heads, rotary_dim, eps, slot_mapping,
                                 kv_cache, num_blocks, block_size, dtype, k_scale, v_scale, q_fp8_out,
                                 q_fp8_scale, error_flags, stream)


def project_context_kv(context_states, w_kv, num_layers, num_kv_heads, out=None, stream=None):
    """all_kv = bf16(context_states @ w_kv^T) as ``[num_ctx, L, 2, nkv, 128]``
    on the tensor cores (the fused projection the context-KV writer reads)."""
    import torch

    _need(isinstance(context_states, torch.Tensor), "context_states must be a tensor")
    dev = context_states.device
    _check_tensor("context_states", context_states, torch.bfloat16, dev, ndim=2)
    num_ctx, hidden = context_states.shape
    _check_tensor("w_kv", w_kv, torch.bfloat16, dev, shape=(num_layers * 2 * num_kv_heads * HEAD_DIM, hidden))
    if out is None:
        out = torch.empty((num_ctx, num_layers, 2, num_kv_heads, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    _check_tensor("out", out, torch.bfloat16, dev)
    _need(out.numel() == num_ctx * num_layers * 2 * num_kv_heads * HEAD_DIM,
          f"out has {out.numel()} elements, the projection {num_ctx} x {num_layers * 2 * num_kv_heads * HEAD_DIM}")
    dspark_ctx_kv_project(context_states, w_kv, out, num_ctx, hidden, num_layers, num_kv_heads, stream)
    return out


def gemma_rms_norm(x, weight, eps, out=None, stream=None):
    """The hidden-state Gemma RMSNorm of the context states (the draft model's
    hidden_norm): ``bf16(x * rsqrt(mean(x^2) + eps) * (1 + weight))`` per row
    of ``x`` (bf16 ``[rows, hidden]``); ``out=x`` works in place."""
    import torch

    _need(isinstance(x, torch.Tensor), "x must be a tensor")
    _check_tensor("x", x, torch.bfloat16, x.device, ndim=2)
    rows, hidden = x.shape
    _check_tensor("weight", weight, torch.bfloat16, x.device, shape=(hidden,))
    if out is None:
        out = torch.empty_like(x)
    _check_tensor("out", out, torch.bfloat16, x.device, shape=(rows, hidden))
    dspark_gemma_rms_norm(x, weight, out, rows, hidden, eps, stream)
    return out
