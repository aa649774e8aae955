"""CPU oracle of the DSpark fused context-KV write (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product path never imports this
package, and this package imports nothing from the product path.

The arithmetic lives in ``ctx_kv_oracle.c`` (plain C, fp64, one row at a
time); this module only marshals numpy arrays into it with ctypes.  See that
file's header for the definition it follows (vLLM DSpark context-KV writer
page, module docstring; DSpark draft model page,
``precompute_and_store_context_kv``).

Parity status: pinned.  ``tests/test_oracle_pins.py`` ties every step to
closed forms, invariants, brute force over the fp8 code space and special
cases that reduce to library routines.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ctx_kv_oracle.c")
_SRC_QK = os.path.join(_HERE, "qk_insert_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libctx_kv_oracle.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
HEAD_DIM = 128          # the pages' head dim
ROW = 256
MAX_HEAD_DIM = 256      # the general write's largest head dim

ERRORS = {
    0: "ok", -1: "bad argument", -2: "slot beyond the cache", -3: "duplicate valid slot",
    -4: "position beyond the cos|sin table", -5: "fp8 scale not positive and finite",
    -6: "alternate buffer too small", -7: "out of memory",
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C11, no FMA contraction, so x86-64 and
    aarch64 hosts evaluate every expression identically)."""
    with _lock:
        stale = not os.path.exists(_LIB_PATH) or any(
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(src) for src in (_SRC, _SRC_QK))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                   "-Wall", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, _SRC_QK, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleInputs(ctypes.Structure):
    _fields_ = [
        ("all_kv", ctypes.c_void_p), ("knorm_w", ctypes.c_void_p),
        ("positions", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
        ("cos_sin", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("num_ctx", ctypes.c_int64), ("max_pos", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("eps", ctypes.c_float), ("layer_slots", ctypes.c_void_p),
        ("head_dim", ctypes.c_int32),
    ]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        L.dspark_oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        L.dspark_oracle_bf16_decode.restype = ctypes.c_double
        L.dspark_oracle_bf16_rne.argtypes = [ctypes.c_double]
        L.dspark_oracle_bf16_rne.restype = ctypes.c_uint16
        L.dspark_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.dspark_oracle_e4m3_decode.restype = ctypes.c_double
        L.dspark_oracle_e4m3_rne_sat.argtypes = [ctypes.c_float]
        L.dspark_oracle_e4m3_rne_sat.restype = ctypes.c_uint8
        L.dspark_oracle_gemma_knorm.argtypes = [P, P, ctypes.c_float, P, P]
        L.dspark_oracle_gemma_knorm.restype = ctypes.c_int
        L.dspark_oracle_gemma_knorm_n.argtypes = [P, P, ctypes.c_int, ctypes.c_float, P, P]
        L.dspark_oracle_gemma_knorm_n.restype = ctypes.c_int
        L.dspark_oracle_rope_pair.argtypes = [ctypes.c_uint16] * 4 + [P, P]
        L.dspark_oracle_rope_pair.restype = None
        L.dspark_oracle_row.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P, P, P]
        L.dspark_oracle_row.restype = ctypes.c_int
        L.dspark_oracle_dest_row.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int64]
        L.dspark_oracle_dest_row.restype = ctypes.c_int64
        L.dspark_oracle_check_inputs.argtypes = [P]
        L.dspark_oracle_check_inputs.restype = ctypes.c_int
        L.dspark_oracle_write.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, P, P, P,
                                          ctypes.c_int64, P]
        L.dspark_oracle_write.restype = ctypes.c_int
        L.dspark_oracle_write_threads.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
        L.dspark_oracle_write_threads.restype = ctypes.c_int
        L.dspark_oracle_rows.argtypes = [P, P, ctypes.c_int64, P, P, P, P, ctypes.c_int64, P]
        L.dspark_oracle_rows.restype = ctypes.c_int
        L.dspark_oracle_gemma_norm_rows.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, P, P]
        L.dspark_oracle_gemma_norm_rows.restype = ctypes.c_int64
        L.dspark_oracle_bf16_rne_array.argtypes = [P, P, ctypes.c_int64]
        L.dspark_oracle_bf16_rne_array.restype = None
        L.dspark_oracle_qk_check.argtypes = [P, ctypes.c_int, ctypes.c_int]
        L.dspark_oracle_qk_check.restype = ctypes.c_int
        L.dspark_oracle_qk_insert.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P, P,
                                              ctypes.c_int64, P]
        L.dspark_oracle_qk_insert.restype = ctypes.c_int
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int):
    if rc != 0:
        raise OracleError(f"oracle: {ERRORS.get(rc, rc)}")


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- scalars

def bf16_decode(bits: int) -> float:
    return lib().dspark_oracle_bf16_decode(int(bits))


def bf16_rne(x: float) -> int:
    return int(lib().dspark_oracle_bf16_rne(float(x)))


def e4m3_decode(code: int) -> float:
    return lib().dspark_oracle_e4m3_decode(int(code))


def e4m3_rne_sat(x: float) -> int:
    """Code of the fp32 value nearest to ``x`` (``x`` is first rounded to fp32)."""
    return int(lib().dspark_oracle_e4m3_rne_sat(float(np.float32(x))))


# ---------------------------------------------------------------- steps

def gemma_norm_rows(x_bits: np.ndarray, w_bits: np.ndarray, eps: float):
    """The hidden-state Gemma RMSNorm of every row of x ([rows, n] bf16 codes)
    with weight w ([n]): (y, y_alt) bf16 codes, y_alt the admissible other
    neighbour where the exact value is within 2^-18 of a midpoint."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, n = x.shape
    w = np.ascontiguousarray(w_bits, dtype=np.uint16).reshape(n)
    y = np.empty_like(x)
    ya = np.empty_like(x)
    lib().dspark_oracle_gemma_norm_rows(_ptr(x), _ptr(w), rows, n, ctypes.c_float(eps), _ptr(y), _ptr(ya))
    return y, ya


def bf16_rne_array(x: np.ndarray) -> np.ndarray:
    """bf16 codes (RNE) of fp64 values, elementwise."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, np.uint16)
    lib().dspark_oracle_bf16_rne_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 values of bf16 codes (a bf16 code is the top half of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def project_context_kv(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """The fused context-KV projection: all_kv[t, n] = bf16(sum_k x[t, k] w[n, k]),
    the sum exact up to fp64 rounding (an fp64 matmul), one rounding to bf16.
    x_bits: [T, hidden], w_bits: [N, hidden] (bf16 codes); returns [T, N] codes."""
    x = bf16_values(x_bits)
    w = bf16_values(w_bits)
    return bf16_rne_array(x @ w.T)


def gemma_knorm(k_bits: np.ndarray, w_bits: np.ndarray, eps: float):
    """Step 2 on one K row (bf16 bits; 128 elements through the pages' entry
    point, any other length through the head-dim general one)
    -> (y, y_alt, n_ambiguous)."""
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    assert k.ndim == 1 and w.shape == k.shape and 1 <= k.shape[0] <= MAX_HEAD_DIM
    D = k.shape[0]
    y = np.empty(D, np.uint16)
    ya = np.empty(D, np.uint16)
    if D == HEAD_DIM:
        n = lib().dspark_oracle_gemma_knorm(_ptr(k), _ptr(w), ctypes.c_float(eps), _ptr(y), _ptr(ya))
    else:
        n = lib().dspark_oracle_gemma_knorm_n(_ptr(k), _ptr(w), D, ctypes.c_float(eps), _ptr(y), _ptr(ya))
    return y, ya, n


def rope_pair(x1: int, x2: int, c: int, s: int):
    o1 = ctypes.c_uint16()
    o2 = ctypes.c_uint16()
    lib().dspark_oracle_rope_pair(int(x1), int(x2), int(c), int(s), ctypes.byref(o1), ctypes.byref(o2))
    return o1.value, o2.value


def dest_row(slot: int, h: int, num_kv_heads: int, block_size: int, num_blocks: int) -> int:
    return int(lib().dspark_oracle_dest_row(int(slot), int(h), int(num_kv_heads), int(block_size),
                                            int(num_blocks)))


# ---------------------------------------------------------------- whole call

class Problem:
    """Host copies of one write call's inputs, kept alive for the C side.

    Arrays: all_kv ``[T, L, 2, H, D]`` / knorm_w ``[L, D]`` / cos_sin as
    uint16 bf16 bits, positions and slot_mapping int64, k_scale / v_scale
    float32 ``[L]``.  The head dim D is all_kv's last extent (128 on the
    pages); cache rows hold 2D elements."""

    def __init__(self, all_kv, knorm_w, positions, slot_mapping, cos_sin, k_scale, v_scale,
                 *, num_blocks: int, block_size: int, rotary_dim: int, kv_dtype: int, eps: float,
                 layer_slots=None):
        self.all_kv = np.ascontiguousarray(all_kv, dtype=np.uint16)
        T, L, two, H, D = self.all_kv.shape
        assert two == 2 and 1 <= D <= MAX_HEAD_DIM
        self.D, self.row = D, 2 * D
        self.knorm_w = np.ascontiguousarray(knorm_w, dtype=np.uint16).reshape(L, D)
        self.positions = np.ascontiguousarray(positions, dtype=np.int64).reshape(T)
        self.slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64).reshape(T)
        self.cos_sin = np.ascontiguousarray(cos_sin, dtype=np.uint16)
        assert self.cos_sin.ndim == 2 and self.cos_sin.shape[1] == rotary_dim
        self.k_scale = np.ascontiguousarray(k_scale, dtype=np.float32).reshape(L)
        self.v_scale = np.ascontiguousarray(v_scale, dtype=np.float32).reshape(L)
        self.T, self.L, self.H = T, L, H
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.rotary_dim, self.kv_dtype, self.eps = int(rotary_dim), int(kv_dtype), float(eps)
        # [L, T] one slot mapping per layer, or None (slot_mapping shared)
        self.layer_slots = None if layer_slots is None else \
            np.ascontiguousarray(layer_slots, dtype=np.int64).reshape(L, T)
        self.c = OracleInputs(
            _ptr(self.all_kv), _ptr(self.knorm_w), _ptr(self.positions), _ptr(self.slot_mapping),
            _ptr(self.cos_sin), _ptr(self.k_scale), _ptr(self.v_scale),
            T, self.cos_sin.shape[0], self.num_blocks, L, H, self.block_size, self.rotary_dim,
            self.kv_dtype, ctypes.c_float(self.eps).value,
            _ptr(self.layer_slots) if self.layer_slots is not None else None, D,
        )

    @property
    def elem_dtype(self):
        return np.uint8 if self.kv_dtype == KV_FP8_E4M3 else np.uint16

    def check(self):
        _check(lib().dspark_oracle_check_inputs(ctypes.byref(self.c)))

    def new_caches(self, fill_byte: int = 0xFF):
        shape = (self.num_blocks, self.H, self.block_size, self.row)
        out = []
        for _ in range(self.L):
            c = np.empty(shape, dtype=self.elem_dtype)
            c.view(np.uint8).fill(fill_byte)
            out.append(c)
        return out

    def write(self, caches, t_begin: int = 0, t_end: int | None = None, alt_cap: int | None = None):
        """Run the write into host ``caches`` (one array per layer).  Returns
        the admissible alternates as arrays (layer, element index, value)."""
        t_end = self.T if t_end is None else t_end
        for c in caches:
            assert c.flags["C_CONTIGUOUS"] and c.dtype == self.elem_dtype
        # about one tie per 2^9 norm outputs, each giving up to three more
        # candidates for itself and its rotation partner: D/16 per row is ample
        cap = alt_cap if alt_cap is not None else max(4096, (t_end - t_begin) * self.L * self.H * self.D // 16)
        ptrs = (ctypes.c_void_p * self.L)(*[_ptr(c) for c in caches])
        al = np.empty(cap, np.int32)
        ae = np.empty(cap, np.int64)
        av = np.empty(cap, np.uint16)
        n = ctypes.c_int64()
        rc = lib().dspark_oracle_write(ctypes.byref(self.c), ptrs, t_begin, t_end, _ptr(al), _ptr(ae),
                                       _ptr(av), cap, ctypes.byref(n))
        _check(rc)
        k = n.value
        return al[:k].copy(), ae[:k].copy(), av[:k].copy()

    def write_threads(self, caches, nthreads: int, t_begin: int = 0, t_end: int | None = None):
        """The same write split over ``nthreads`` host threads by token
        ranges (timing on every core); the alternates are not returned."""
        t_end = self.T if t_end is None else t_end
        for c in caches:
            assert c.flags["C_CONTIGUOUS"] and c.dtype == self.elem_dtype
        ptrs = (ctypes.c_void_p * self.L)(*[_ptr(c) for c in caches])
        _check(lib().dspark_oracle_write_threads(ctypes.byref(self.c), ptrs, t_begin, t_end, int(nthreads)))

    def rows(self, row_ids):
        """Stored 2D-element rows for flat row ids ``(t*L + l)*H + h``, with
        alternates as (index into row_ids, dim, value)."""
        ids = np.ascontiguousarray(row_ids, dtype=np.int64).reshape(-1)
        n = ids.shape[0]
        out = np.empty((n, self.row), dtype=self.elem_dtype)
        cap = max(1024, n * 8)
        ar = np.empty(cap, np.int64)
        ad = np.empty(cap, np.int32)
        av = np.empty(cap, np.uint16)
        cnt = ctypes.c_int64()
        rc = lib().dspark_oracle_rows(ctypes.byref(self.c), _ptr(ids), n, _ptr(out), _ptr(ar), _ptr(ad),
                                      _ptr(av), cap, ctypes.byref(cnt))
        _check(rc)
        k = cnt.value
        return out, (ar[:k].copy(), ad[:k].copy(), av[:k].copy())

    def dest_rows(self, row_ids):
        """Cache row (within its layer) that each flat row id is stored to,
        -1 for padding."""
        ids = np.asarray(row_ids, dtype=np.int64).reshape(-1)
        t = ids // (self.L * self.H)
        l = (ids // self.H) % self.L
        h = ids % self.H
        slot = self.slot_mapping[t] if self.layer_slots is None else self.layer_slots[l, t]
        return np.array([dest_row(int(s), int(hi), self.H, self.block_size, self.num_blocks)
                         for s, hi in zip(slot, h)], dtype=np.int64)


def problem_from_inputs(inp, layer_slots=None) -> Problem:
    """A Problem from a ``workloads.Inputs`` (CPU torch tensors); layer_slots
    ([L, T] int64) gives every layer its own slot mapping."""
    import torch  # local: the oracle's arithmetic does not use torch

    def bits(x):
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    wl = inp.workload
    return Problem(
        bits(inp.all_kv), bits(inp.knorm_w), inp.positions.cpu().numpy(), inp.slot_mapping.cpu().numpy(),
        bits(inp.cos_sin), inp.k_scale.cpu().numpy(), inp.v_scale.cpu().numpy(),
        num_blocks=wl.num_blocks, block_size=wl.block_size, rotary_dim=wl.rotary_dim,
        kv_dtype=KV_FP8_E4M3 if wl.kv_dtype == "fp8_e4m3" else KV_BF16, eps=inp.eps,
        layer_slots=None if layer_slots is None else np.asarray(layer_slots),
    )


# ---------------------------------------------------------------- draft-token QK insert

class QkOracleInputs(ctypes.Structure):
    _fields_ = [
        ("qkv", ctypes.c_void_p), ("q_norm_w", ctypes.c_void_p), ("k_norm_w", ctypes.c_void_p),
        ("positions", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p),
        ("num_tokens", ctypes.c_int64), ("max_pos", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("eps", ctypes.c_float),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float), ("q_scale", ctypes.c_float),
    ]


ALT_QKV, ALT_QFP8, ALT_CACHE = 0, 1, 2


class QkProblem:
    """Host copies of one draft-token QK-norm / RoPE / KV-insert call, kept
    alive for the C side (``qk_insert_oracle.c`` has the definition).

    Arrays: qkv ``[T, (Hq + 2 Hkv) * 128]``, the two norm weights ``[128]`` and
    cos_sin as uint16 bf16 bits; positions and slot_mapping int64."""

    def __init__(self, qkv, q_norm_w, k_norm_w, positions, slot_mapping, cos_sin, *, num_heads: int,
                 num_kv_heads: int, num_blocks: int, block_size: int, rotary_dim: int, kv_dtype: int,
                 eps: float, k_scale: float = 1.0, v_scale: float = 1.0, q_scale: float = 1.0):
        self.Hq, self.Hkv = int(num_heads), int(num_kv_heads)
        self.width = (self.Hq + 2 * self.Hkv) * HEAD_DIM
        self.qkv = np.ascontiguousarray(qkv, dtype=np.uint16).reshape(-1, self.width)
        self.T = self.qkv.shape[0]
        self.q_norm_w = np.ascontiguousarray(q_norm_w, dtype=np.uint16).reshape(HEAD_DIM)
        self.k_norm_w = np.ascontiguousarray(k_norm_w, dtype=np.uint16).reshape(HEAD_DIM)
        self.positions = np.ascontiguousarray(positions, dtype=np.int64).reshape(self.T)
        self.slot_mapping = None if slot_mapping is None else \
            np.ascontiguousarray(slot_mapping, dtype=np.int64).reshape(self.T)
        self.cos_sin = np.ascontiguousarray(cos_sin, dtype=np.uint16)
        assert self.cos_sin.ndim == 2 and self.cos_sin.shape[1] == rotary_dim
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.rotary_dim, self.kv_dtype, self.eps = int(rotary_dim), int(kv_dtype), float(eps)
        self.k_scale, self.v_scale, self.q_scale = float(k_scale), float(v_scale), float(q_scale)
        self.c = QkOracleInputs(
            _ptr(self.qkv), _ptr(self.q_norm_w), _ptr(self.k_norm_w), _ptr(self.positions),
            _ptr(self.slot_mapping) if self.slot_mapping is not None else None, _ptr(self.cos_sin),
            self.T, self.cos_sin.shape[0], self.num_blocks, self.Hq, self.Hkv, self.block_size,
            self.rotary_dim, self.kv_dtype, ctypes.c_float(self.eps).value,
            ctypes.c_float(self.k_scale).value, ctypes.c_float(self.v_scale).value,
            ctypes.c_float(self.q_scale).value,
        )

    @property
    def elem_dtype(self):
        return np.uint8 if self.kv_dtype == KV_FP8_E4M3 else np.uint16

    def new_cache(self, fill_byte: int = 0xFF):
        c = np.empty((self.num_blocks, self.Hkv, self.block_size, ROW), dtype=self.elem_dtype)
        c.view(np.uint8).fill(fill_byte)
        return c

    def run(self, cache=None, q_fp8: bool = False, t_begin: int = 0, t_end: int | None = None,
            qkv_out=None):
        """Run the call.  Returns (qkv_out, q_fp8_out or None, alternates),
        alternates as arrays (output ALT_*, element index, value); ``cache``
        (host, the cache dtype) is written in place when given."""
        t_end = self.T if t_end is None else t_end
        if qkv_out is None:
            qkv_out = self.qkv.copy()
        assert qkv_out.flags["C_CONTIGUOUS"] and qkv_out.shape == self.qkv.shape
        qf = np.full((self.T, self.Hq * HEAD_DIM), 0xFF, np.uint8) if q_fp8 else None
        if cache is not None:
            assert cache.flags["C_CONTIGUOUS"] and cache.dtype == self.elem_dtype
        elems = max(1, (t_end - t_begin) * (self.Hq + 2 * self.Hkv) * HEAD_DIM)
        cap = max(4096, elems // 16)
        aw = np.empty(cap, np.int32)
        ae = np.empty(cap, np.int64)
        av = np.empty(cap, np.uint16)
        n = ctypes.c_int64()
        rc = lib().dspark_oracle_qk_insert(
            ctypes.byref(self.c), t_begin, t_end, _ptr(qkv_out), _ptr(qf) if qf is not None else None,
            _ptr(cache) if cache is not None else None, _ptr(aw), _ptr(ae), _ptr(av), cap, ctypes.byref(n))
        _check(rc)
        k = n.value
        return qkv_out, qf, (aw[:k].copy(), ae[:k].copy(), av[:k].copy())


def qk_problem_from_inputs(inp, with_slots: bool = True) -> QkProblem:
    """A QkProblem from a ``workloads.QkInputs`` (CPU torch tensors)."""
    import torch  # local: the oracle's arithmetic does not use torch

    def bits(x):
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    wl = inp.workload
    return QkProblem(
        bits(inp.qkv), bits(inp.q_norm_w), bits(inp.k_norm_w), inp.positions.cpu().numpy(),
        inp.slot_mapping.cpu().numpy() if with_slots else None, bits(inp.cos_sin),
        num_heads=wl.num_heads, num_kv_heads=wl.num_kv_heads, num_blocks=wl.num_blocks,
        block_size=wl.block_size, rotary_dim=wl.rotary_dim,
        kv_dtype=KV_FP8_E4M3 if wl.kv_dtype == "fp8_e4m3" else KV_BF16, eps=inp.eps,
        k_scale=inp.k_scale, v_scale=inp.v_scale, q_scale=inp.q_scale,
    )
