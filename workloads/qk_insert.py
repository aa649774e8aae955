"""Seeded synthetic inputs for the DSpark draft-token fused QK-norm / RoPE /
KV insert (``dspark_qknorm_rope_kv_insert`` on the DSpark draft model page).

Like ``synth``, this module only draws random numbers, builds the RoPE
cos|sin table and lays out slot mappings the way a paged-KV block allocator
would; it holds none of the op's arithmetic.  Both the oracle-side tests and
the CUDA path consume the same tensors.

Layouts (the op's arguments on that page):

* ``qkv``        bf16 ``[T, (Hq + 2 Hkv) * 128]``: per token the Hq query
  heads, then the Hkv key heads, then the Hkv value heads
* ``q_norm_w``, ``k_norm_w``  bf16 ``[128]`` (Gemma weights, applied as ``1 + w``)
* ``positions``  int64 ``[T]``; ``slot_mapping`` int64 ``[T]`` (``-1`` = padding)
* ``cos_sin``    bf16 ``[max_pos, rotary_dim]`` (cos | sin)
* ``kv_cache``   ``[num_blocks, Hkv, block_size, 256]`` bf16, or uint8 holding
  fp8 e4m3 codes, prefilled with the byte 0xFF
* ``k_scale``, ``v_scale`` (fp8 cache) and ``q_scale`` (fp8 query output): fp32

A draft step carries 7 query rows per request (the drafter's block of query
rows on the ROCm drafter dispatch page): every request contributes 7
consecutive positions at a random offset, stored through its own block table.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

from .synth import HEAD_DIM, ROW_ELEMS, PREFILL_BYTE, BASE_SEED, KV_BF16, KV_FP8, rope_cos_sin_cache

QUERY_ROWS_PER_REQUEST = 7


@dataclass(frozen=True)
class QkWorkload:
    """Shape and value recipe of one insert call."""

    name: str
    requests: int
    num_heads: int
    num_kv_heads: int
    rotary_dim: int
    block_size: int
    num_blocks: int
    max_pos: int
    rope_theta: float
    kv_dtype: str = KV_BF16
    q_fp8: bool = False
    x_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    w_std: float = 0.1
    eps: float = 1e-6
    scale_lo: float = 0.05
    scale_hi: float = 0.5
    pad_count: int = 0
    seed: int = BASE_SEED + 100

    @property
    def num_tokens(self) -> int:
        return self.requests * QUERY_ROWS_PER_REQUEST

    @property
    def width(self) -> int:
        return (self.num_heads + 2 * self.num_kv_heads) * HEAD_DIM

    @property
    def elem_size(self) -> int:
        return 2 if self.kv_dtype == KV_BF16 else 1

    @property
    def capacity(self) -> int:
        return self.num_blocks * self.block_size

    def with_(self, **kw) -> "QkWorkload":
        return replace(self, **kw)


QK_WORKLOADS: list[QkWorkload] = [
    QkWorkload(name="qk_tiny", requests=1, num_heads=4, num_kv_heads=1, rotary_dim=64, block_size=16,
               num_blocks=4, max_pos=64, rope_theta=1e4, q_fp8=True, pad_count=1, seed=BASE_SEED + 100),
    QkWorkload(name="qk_draft", requests=64, num_heads=64, num_kv_heads=8, rotary_dim=64, block_size=16,
               num_blocks=4096, max_pos=32768, rope_theta=1e6, pad_count=9, seed=BASE_SEED + 101),
    QkWorkload(name="qk_draft_fp8", requests=64, num_heads=64, num_kv_heads=8, rotary_dim=64, block_size=16,
               num_blocks=4096, max_pos=32768, rope_theta=1e6, kv_dtype=KV_FP8, q_fp8=True, x_std=2.0,
               outlier_frac=0.01, outlier_mult=10.0, pad_count=9, seed=BASE_SEED + 102),
]

QK_WORKLOADS_BY_NAME = {w.name: w for w in QK_WORKLOADS}


@dataclass
class QkInputs:
    """CPU tensors of one insert call (see the module docstring for layouts)."""

    workload: QkWorkload
    qkv: torch.Tensor
    q_norm_w: torch.Tensor
    k_norm_w: torch.Tensor
    positions: torch.Tensor
    slot_mapping: torch.Tensor
    cos_sin: torch.Tensor
    k_scale: float
    v_scale: float
    q_scale: float
    eps: float
    extra: dict = field(default_factory=dict)

    @property
    def num_valid_tokens(self) -> int:
        return int((self.slot_mapping >= 0).sum())

    def to(self, device) -> "QkInputs":
        mv = lambda x: x.to(device)  # noqa: E731
        return QkInputs(self.workload, mv(self.qkv), mv(self.q_norm_w), mv(self.k_norm_w),
                        mv(self.positions), mv(self.slot_mapping), mv(self.cos_sin), self.k_scale,
                        self.v_scale, self.q_scale, self.eps, dict(self.extra))


def _positions_and_slots(wl: QkWorkload, g: torch.Generator):
    """7 consecutive positions per request at a random offset; each request's
    logical blocks map to distinct shuffled physical blocks."""
    R, n, bs = wl.requests, QUERY_ROWS_PER_REQUEST, wl.block_size
    offs = torch.randint(0, wl.max_pos - n + 1, (R,), generator=g, dtype=torch.int64)
    pool = torch.randperm(wl.num_blocks, generator=g).to(torch.int64)
    nxt = 0
    pos_l, slot_l = [], []
    for r in range(R):
        p = offs[r] + torch.arange(n, dtype=torch.int64)
        lb = p // bs
        first = int(lb[0])
        nlb = int(lb[-1]) - first + 1
        if nxt + nlb > wl.num_blocks:
            raise ValueError("not enough physical blocks")
        phys = pool[nxt: nxt + nlb]
        nxt += nlb
        pos_l.append(p)
        slot_l.append(phys[lb - first] * bs + p % bs)
    pos = torch.cat(pos_l).contiguous()
    slots = torch.cat(slot_l).contiguous()
    if wl.pad_count:
        pad = torch.randperm(wl.num_tokens, generator=g)[: wl.pad_count]
        slots[pad] = -1
    return pos, slots


def generate_qk(wl: QkWorkload, seed: int | None = None) -> QkInputs:
    """Draw the inputs of ``wl`` (fp32 samples rounded to bf16, RNE)."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    x = torch.randn((wl.num_tokens, wl.width), generator=g, dtype=torch.float32)
    if wl.x_std != 1.0:
        x.mul_(wl.x_std)
    if wl.outlier_frac > 0:
        hit = torch.rand(x.shape, generator=g) < wl.outlier_frac
        x = torch.where(hit, x * wl.outlier_mult, x)
    qkv = x.to(torch.bfloat16).contiguous()
    q_norm_w = (torch.randn(HEAD_DIM, generator=g) * wl.w_std).to(torch.bfloat16).contiguous()
    k_norm_w = (torch.randn(HEAD_DIM, generator=g) * wl.w_std).to(torch.bfloat16).contiguous()
    pos, slots = _positions_and_slots(wl, g)
    cos_sin = rope_cos_sin_cache(wl.max_pos, wl.rotary_dim, wl.rope_theta)
    sc = torch.empty(3, dtype=torch.float32).uniform_(wl.scale_lo, wl.scale_hi, generator=g).tolist()
    k_scale, v_scale = (sc[0], sc[1]) if wl.kv_dtype == KV_FP8 else (1.0, 1.0)
    q_scale = sc[2] if wl.q_fp8 else 1.0
    return QkInputs(wl, qkv, q_norm_w, k_norm_w, pos, slots, cos_sin, float(k_scale), float(v_scale),
                    float(q_scale), float(wl.eps))


def make_qk_cache(wl: QkWorkload, device="cpu", fill: int | None = PREFILL_BYTE) -> torch.Tensor:
    dtype = torch.bfloat16 if wl.kv_dtype == KV_BF16 else torch.uint8
    c = torch.empty((wl.num_blocks, wl.num_kv_heads, wl.block_size, ROW_ELEMS), dtype=dtype, device=device)
    if fill is not None:
        c.view(torch.uint8).fill_(fill)
    return c


def qk_compulsory_bytes(wl: QkWorkload, num_valid_tokens: int, num_tokens: int | None = None) -> int:
    """Bytes one call (or its first ``num_tokens`` tokens) must move at least:
    qkv read once; query and key heads written back; the K|V cache rows of
    valid tokens; the fp8 query output; per token its position, slot and
    cos|sin row; the two norm weights."""
    T = wl.num_tokens if num_tokens is None else num_tokens
    Hq, Hkv = wl.num_heads, wl.num_kv_heads
    read = T * wl.width * 2
    back = T * (Hq + Hkv) * HEAD_DIM * 2
    cache = num_valid_tokens * Hkv * ROW_ELEMS * wl.elem_size
    qf8 = T * Hq * HEAD_DIM if wl.q_fp8 else 0
    per_tok = T * (8 + 8 + 2 * wl.rotary_dim)
    return read + back + cache + qf8 + per_tok + 2 * HEAD_DIM * 2


def describe_qk(wl: QkWorkload) -> dict:
    return {
        "workload": wl.name, "num_tokens": wl.num_tokens, "requests": wl.requests,
        "num_heads": wl.num_heads, "nkv": wl.num_kv_heads, "head_dim": HEAD_DIM,
        "rotary_dim": wl.rotary_dim, "block_size": wl.block_size, "num_blocks": wl.num_blocks,
        "kv_cache_dtype": wl.kv_dtype, "q_fp8_out": wl.q_fp8, "max_pos": wl.max_pos,
    }
