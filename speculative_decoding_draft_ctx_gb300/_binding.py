"""ctypes binding of libdspark_ctx_kv.so (include/dspark_ctx_kv.h).

Argument marshalling only: tensors become device addresses and sizes, the
current torch stream becomes the cudaStream_t, and a non-zero status becomes
a DSparkError.  Every step of the write runs in the library's kernel; there
is no other implementation to fall back to, so a missing or unloadable
library raises at first use.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KV_BF16 = 0
KV_FP8_E4M3 = 1
HEAD_DIM = 128
CACHE_ROW = 256

STATUS = {
    0: "DSPARK_OK", 1: "DSPARK_ERR_INVALID_ARG", 2: "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM",
    3: "DSPARK_ERR_BLOCK_SIZE", 4: "DSPARK_ERR_ALIGNMENT", 5: "DSPARK_ERR_DTYPE",
    6: "DSPARK_ERR_CAPTURING", 7: "DSPARK_ERR_CUDA",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}
FLAG_SLOT_RANGE = 0x1
FLAG_POS_RANGE = 0x2
FLAG_TIMEOUT = 0x4
FLAG_COUNTER = 0x8

# every function the header declares
EXPORTS = (
    "dspark_ctx_kv_write", "dspark_ctx_kv_write_ex", "dspark_ctx_kv_rotary_dims_supported",
    "dspark_ctx_kv_validate_layers", "dspark_ctx_kv_tables_create", "dspark_ctx_kv_tables_update",
    "dspark_ctx_kv_tables_cache_offsets", "dspark_ctx_kv_tables_k_scales",
    "dspark_ctx_kv_tables_v_scales", "dspark_ctx_kv_tables_builds", "dspark_ctx_kv_tables_destroy",
    "dspark_ctx_kv_last_error", "dspark_ctx_kv_status_string", "dspark_qknorm_rope_kv_insert",
    "dspark_ctx_kv_project", "dspark_ctx_kv_project_write", "dspark_gemma_rms_norm",
    "dspark_ctx_kv_write_layer_slots", "dspark_ctx_kv_tables_update_slots", "dspark_ctx_kv_tables_layer_slots",
    "dspark_ctx_kv_write_general", "dspark_ctx_kv_general_supported", "dspark_ctx_kv_validate_layers_general",
    "dspark_ctx_kv_write_sched", "dspark_ctx_kv_write_noalloc",
)


class DSparkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


class CacheDesc(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p), ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4),
        ("ndim", ctypes.c_int32), ("elem_size", ctypes.c_int32), ("cache_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("scales_ok", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (speculative_decoding_draft_ctx_gb300.build.build())")
        L = ctypes.CDLL(path)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        write_args = [P, P, P, P, I64, P, I64, P, I64, P, P, P, I, I, I, I, ctypes.c_float, I]
        L.dspark_ctx_kv_write.argtypes = write_args + [P]
        L.dspark_ctx_kv_write.restype = I
        L.dspark_ctx_kv_write_ex.argtypes = write_args + [P, P]
        L.dspark_ctx_kv_write_ex.restype = I
        L.dspark_ctx_kv_rotary_dims_supported.argtypes = [I, I]
        L.dspark_ctx_kv_rotary_dims_supported.restype = I
        L.dspark_ctx_kv_validate_layers.argtypes = [I, ctypes.POINTER(CacheDesc)]
        L.dspark_ctx_kv_validate_layers.restype = I
        L.dspark_ctx_kv_tables_create.argtypes = [I, ctypes.POINTER(P)]
        L.dspark_ctx_kv_tables_create.restype = I
        L.dspark_ctx_kv_tables_update.argtypes = [P, P, ctypes.c_size_t, P, P, P]
        L.dspark_ctx_kv_tables_update.restype = I
        for n in ("dspark_ctx_kv_tables_cache_offsets", "dspark_ctx_kv_tables_k_scales",
                  "dspark_ctx_kv_tables_v_scales"):
            getattr(L, n).argtypes = [P]
            getattr(L, n).restype = P
        L.dspark_ctx_kv_tables_builds.argtypes = [P]
        L.dspark_ctx_kv_tables_builds.restype = I64
        L.dspark_ctx_kv_tables_destroy.argtypes = [P]
        L.dspark_ctx_kv_tables_destroy.restype = None
        L.dspark_ctx_kv_last_error.argtypes = []
        L.dspark_ctx_kv_last_error.restype = ctypes.c_char_p
        L.dspark_ctx_kv_status_string.argtypes = [I]
        L.dspark_ctx_kv_status_string.restype = ctypes.c_char_p
        L.dspark_qknorm_rope_kv_insert.argtypes = [P, P, P, P, I64, P, I64, I, I, I, ctypes.c_float, P, P, I64,
                                                   I, I, P, P, P, ctypes.c_float, P, P]
        L.dspark_qknorm_rope_kv_insert.restype = I
        L.dspark_ctx_kv_project.argtypes = [P, P, P, I64, I, I, I, P]
        L.dspark_ctx_kv_project.restype = I
        L.dspark_ctx_kv_project_write.argtypes = [P, P, I64, I, P, P, P, P, I64, P, I64, P, P, P, I, I, I, I,
                                                  ctypes.c_float, I, P, P]
        L.dspark_ctx_kv_project_write.restype = I
        L.dspark_gemma_rms_norm.argtypes = [P, P, P, I64, I, ctypes.c_float, P]
        L.dspark_gemma_rms_norm.restype = I
        L.dspark_ctx_kv_write_layer_slots.argtypes = write_args[:3] + [P] + write_args[4:] + [P, P]
        L.dspark_ctx_kv_write_layer_slots.restype = I
        L.dspark_ctx_kv_write_sched.argtypes = write_args[:4] + [P] + write_args[4:] + [P, P, P]
        L.dspark_ctx_kv_write_sched.restype = I
        L.dspark_ctx_kv_write_noalloc.argtypes = write_args[:4] + [P] + write_args[4:] + [P, P]
        L.dspark_ctx_kv_write_noalloc.restype = I
        L.dspark_ctx_kv_tables_update_slots.argtypes = [P, P, P]
        L.dspark_ctx_kv_tables_update_slots.restype = I
        L.dspark_ctx_kv_tables_layer_slots.argtypes = [P]
        L.dspark_ctx_kv_tables_layer_slots.restype = P
        L.dspark_ctx_kv_write_general.argtypes = [P, P, P, P, P, I64, P, I64, P, I64, P, P, P, I, I, I, I, I,
                                                  ctypes.c_float, I, P, P]
        L.dspark_ctx_kv_write_general.restype = I
        L.dspark_ctx_kv_general_supported.argtypes = [I, I, I]
        L.dspark_ctx_kv_general_supported.restype = I
        L.dspark_ctx_kv_validate_layers_general.argtypes = [I, ctypes.POINTER(CacheDesc)]
        L.dspark_ctx_kv_validate_layers_general.restype = I
        _lib = L
        return L


def check(status: int):
    if status != 0:
        raise DSparkError(status, lib().dspark_ctx_kv_last_error().decode())


def _addr(x) -> int:
    """Device address of a tensor, or an int address as is (0 = NULL)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kv_dtype_code(kv_dtype) -> int:
    if kv_dtype in (KV_BF16, "bf16", "auto", "bfloat16"):
        return KV_BF16
    if kv_dtype in (KV_FP8_E4M3, "fp8", "fp8_e4m3"):
        return KV_FP8_E4M3
    return -1


def dspark_ctx_kv_write(all_kv, knorm_w, positions, slot_mapping, num_ctx, cos_sin, max_pos,
                        layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                        block_size, rotary_dim, eps, kv_dtype, stream=None):
    """``dspark_ctx_kv_write`` of the C ABI: tensors (or int addresses) in,
    DSparkError on a non-OK status."""
    check(lib().dspark_ctx_kv_write(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(slot_mapping), int(num_ctx),
        _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets),
        _addr(k_scales), _addr(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim),
        float(eps), kv_dtype_code(kv_dtype), _stream(stream)))


def dspark_ctx_kv_write_ex(all_kv, knorm_w, positions, slot_mapping, num_ctx, cos_sin, max_pos,
                           layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                           block_size, rotary_dim, eps, kv_dtype, error_flags, stream=None):
    """``dspark_ctx_kv_write_ex``: as dspark_ctx_kv_write, plus the device
    error word (an int32 tensor of one element, or an address)."""
    check(lib().dspark_ctx_kv_write_ex(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(slot_mapping), int(num_ctx),
        _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets),
        _addr(k_scales), _addr(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim),
        float(eps), kv_dtype_code(kv_dtype), _addr(error_flags), _stream(stream)))


def dspark_ctx_kv_write_sched(all_kv, knorm_w, positions, slot_mapping, layer_slot_mappings, num_ctx, cos_sin,
                              max_pos, layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                              block_size, rotary_dim, eps, kv_dtype, error_flags, work_counter, stream=None):
    """``dspark_ctx_kv_write_sched``: the write with a shared ``slot_mapping``
    or a per-layer ``layer_slot_mappings`` table (exactly one given), the
    error word, and ``work_counter`` (two zeroed int64 words on the device,
    or ``None`` for the fixed split)."""
    check(lib().dspark_ctx_kv_write_sched(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(slot_mapping), _addr(layer_slot_mappings),
        int(num_ctx), _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets),
        _addr(k_scales), _addr(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim), float(eps),
        kv_dtype_code(kv_dtype), _addr(error_flags), _addr(work_counter), _stream(stream)))


def dspark_ctx_kv_write_noalloc(all_kv, knorm_w, positions, slot_mapping, layer_slot_mappings, num_ctx, cos_sin,
                                max_pos, layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                                block_size, rotary_dim, eps, kv_dtype, error_flags=None, stream=None):
    """``dspark_ctx_kv_write_noalloc``: the per-layer tables as Python
    sequences (host memory): ``cache_offsets`` L ints (element offsets from
    ``layer0_cache``), ``k_scales`` / ``v_scales`` L device scalars (or
    ``None`` for bf16), ``layer_slot_mappings`` L int64 device tensors (or
    ``None`` with ``slot_mapping``)."""
    def ptrs(xs):
        return None if xs is None else (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])

    offs = (ctypes.c_int64 * len(cache_offsets))(*[int(o) for o in cache_offsets])
    check(lib().dspark_ctx_kv_write_noalloc(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(slot_mapping), ptrs(layer_slot_mappings),
        int(num_ctx), _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), offs, ptrs(k_scales),
        ptrs(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim), float(eps), kv_dtype_code(kv_dtype),
        _addr(error_flags), _stream(stream)))


def dspark_qknorm_rope_kv_insert(qkv, q_norm_w, k_norm_w, cos_sin, max_pos, positions, num_tokens,
                                 num_heads, num_kv_heads, rotary_dim, eps, slot_mapping, kv_cache,
                                 num_blocks, block_size, kv_dtype, k_scale, v_scale, q_fp8_out,
                                 q_fp8_scale, error_flags=None, stream=None):
    """``dspark_qknorm_rope_kv_insert`` of the C ABI: tensors (or int
    addresses, None = NULL) in, DSparkError on a non-OK status."""
    check(lib().dspark_qknorm_rope_kv_insert(
        _addr(qkv), _addr(q_norm_w), _addr(k_norm_w), _addr(cos_sin), int(max_pos), _addr(positions),
        int(num_tokens), int(num_heads), int(num_kv_heads), int(rotary_dim), float(eps),
        _addr(slot_mapping), _addr(kv_cache), int(num_blocks), int(block_size), kv_dtype_code(kv_dtype),
        _addr(k_scale), _addr(v_scale), _addr(q_fp8_out), float(q_fp8_scale), _addr(error_flags),
        _stream(stream)))


def dspark_gemma_rms_norm(x, w, out, rows, hidden, eps, stream=None):
    """``dspark_gemma_rms_norm`` of the C ABI."""
    check(lib().dspark_gemma_rms_norm(_addr(x), _addr(w), _addr(out), int(rows), int(hidden), float(eps),
                                      _stream(stream)))


def dspark_ctx_kv_project(x, w_kv, all_kv_out, num_ctx, hidden, L, nkv, stream=None):
    """``dspark_ctx_kv_project`` of the C ABI."""
    check(lib().dspark_ctx_kv_project(_addr(x), _addr(w_kv), _addr(all_kv_out), int(num_ctx), int(hidden),
                                      int(L), int(nkv), _stream(stream)))


def dspark_ctx_kv_project_write(x, w_kv, num_ctx, hidden, knorm_w, positions, slot_mapping, cos_sin, max_pos,
                                layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv, block_size,
                                rotary_dim, eps, kv_dtype, error_flags=None, stream=None):
    """``dspark_ctx_kv_project_write`` of the C ABI."""
    check(lib().dspark_ctx_kv_project_write(
        _addr(x), _addr(w_kv), int(num_ctx), int(hidden), _addr(knorm_w), _addr(positions), _addr(slot_mapping),
        _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets), _addr(k_scales),
        _addr(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim), float(eps), kv_dtype_code(kv_dtype),
        _addr(error_flags), _stream(stream)))


def dspark_ctx_kv_write_layer_slots(all_kv, knorm_w, positions, layer_slot_mappings, num_ctx, cos_sin, max_pos,
                                    layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                                    block_size, rotary_dim, eps, kv_dtype, error_flags=None, stream=None):
    """``dspark_ctx_kv_write_layer_slots``: per-layer slot mappings given as a
    device pointer table (an address)."""
    check(lib().dspark_ctx_kv_write_layer_slots(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(layer_slot_mappings), int(num_ctx),
        _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets),
        _addr(k_scales), _addr(v_scales), int(L), int(nkv), int(block_size), int(rotary_dim),
        float(eps), kv_dtype_code(kv_dtype), _addr(error_flags), _stream(stream)))


def dspark_ctx_kv_write_general(all_kv, knorm_w, positions, slot_mapping, layer_slot_mappings, num_ctx, cos_sin,
                                max_pos, layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                                head_dim, block_size, rotary_dim, eps, kv_dtype, error_flags=None, stream=None):
    """``dspark_ctx_kv_write_general``: head dims 64 / 128 / 256, any even
    rotary_dim up to the head dim, any block size; a shared ``slot_mapping``
    or a per-layer ``layer_slot_mappings`` pointer table (an address), the
    other None."""
    check(lib().dspark_ctx_kv_write_general(
        _addr(all_kv), _addr(knorm_w), _addr(positions), _addr(slot_mapping), _addr(layer_slot_mappings),
        int(num_ctx), _addr(cos_sin), int(max_pos), _addr(layer0_cache), int(num_blocks), _addr(cache_offsets),
        _addr(k_scales), _addr(v_scales), int(L), int(nkv), int(head_dim), int(block_size), int(rotary_dim),
        float(eps), kv_dtype_code(kv_dtype), _addr(error_flags), _stream(stream)))


def dspark_ctx_kv_general_supported(head_dim: int, rotary_dim: int, block_size: int) -> bool:
    return bool(lib().dspark_ctx_kv_general_supported(int(head_dim), int(rotary_dim), int(block_size)))


def dspark_ctx_kv_rotary_dims_supported(rotary_dim: int, head_dim: int) -> bool:
    return bool(lib().dspark_ctx_kv_rotary_dims_supported(int(rotary_dim), int(head_dim)))


def dspark_ctx_kv_status_string(status: int) -> str:
    return lib().dspark_ctx_kv_status_string(int(status)).decode()


def dspark_ctx_kv_last_error() -> str:
    return lib().dspark_ctx_kv_last_error().decode()


def cache_desc(cache, kv_cache_dtype, k_scale, v_scale) -> CacheDesc:
    """Describe one layer's cache tensor and scales for the layout check."""
    import torch

    d = CacheDesc()
    bound = isinstance(cache, torch.Tensor) and cache.numel() > 0
    d.data = cache.data_ptr() if bound else 0
    nd = cache.dim() if isinstance(cache, torch.Tensor) else 0
    d.ndim = nd
    for i in range(min(nd, 4)):
        d.shape[i] = cache.shape[i]
        d.stride[i] = cache.stride(i)
    if isinstance(cache, torch.Tensor):
        d.elem_size = cache.element_size()
        d.cache_dtype = {torch.bfloat16: KV_BF16, torch.uint8: KV_FP8_E4M3}.get(cache.dtype, -1)
    d.kv_dtype = kv_dtype_code(kv_cache_dtype)

    def fp32_cuda(s):
        return isinstance(s, torch.Tensor) and s.dtype == torch.float32 and s.is_cuda

    d.scales_ok = int(fp32_cuda(k_scale) and fp32_cuda(v_scale))
    d.k_scale = k_scale.data_ptr() if isinstance(k_scale, torch.Tensor) else 0
    d.v_scale = v_scale.data_ptr() if isinstance(v_scale, torch.Tensor) else 0
    return d


def dspark_ctx_kv_validate_layers(descs) -> None:
    arr = (CacheDesc * len(descs))(*descs)
    check(lib().dspark_ctx_kv_validate_layers(len(descs), arr))


def dspark_ctx_kv_validate_layers_general(descs) -> None:
    arr = (CacheDesc * len(descs))(*descs)
    check(lib().dspark_ctx_kv_validate_layers_general(len(descs), arr))


class Tables:
    """Owner of one dspark_ctx_kv_tables object."""

    def __init__(self, L: int):
        h = ctypes.c_void_p()
        check(lib().dspark_ctx_kv_tables_create(int(L), ctypes.byref(h)))
        self._h = h
        self.L = int(L)

    def update(self, caches, k_scales, v_scales, stream=None):
        L = self.L
        cp = (ctypes.c_void_p * L)(*[_addr(c) for c in caches])
        kp = (ctypes.c_void_p * L)(*[_addr(s) for s in k_scales]) if k_scales is not None else None
        vp = (ctypes.c_void_p * L)(*[_addr(s) for s in v_scales]) if v_scales is not None else None
        esize = caches[0].element_size() if hasattr(caches[0], "element_size") else 2
        check(lib().dspark_ctx_kv_tables_update(self._h, cp, esize, kp, vp, _stream(stream)))

    def update_slots(self, slot_mappings, stream=None):
        """Per-layer slot mappings (one int64 CUDA tensor per layer)."""
        sp = (ctypes.c_void_p * self.L)(*[_addr(s) for s in slot_mappings])
        check(lib().dspark_ctx_kv_tables_update_slots(self._h, sp, _stream(stream)))

    @property
    def layer_slots(self) -> int:
        return lib().dspark_ctx_kv_tables_layer_slots(self._h) or 0

    @property
    def cache_offsets(self) -> int:
        return lib().dspark_ctx_kv_tables_cache_offsets(self._h) or 0

    @property
    def k_scales(self) -> int:
        return lib().dspark_ctx_kv_tables_k_scales(self._h) or 0

    @property
    def v_scales(self) -> int:
        return lib().dspark_ctx_kv_tables_v_scales(self._h) or 0

    @property
    def builds(self) -> int:
        return int(lib().dspark_ctx_kv_tables_builds(self._h))

    def close(self):
        if self._h is not None and self._h.value:
            lib().dspark_ctx_kv_tables_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
