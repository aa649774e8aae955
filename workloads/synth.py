"""Seeded synthetic inputs for the DSpark fused context-KV write.

This module produces the input tensors of one write call (``all_kv``, the
per-layer Gemma K-norm weights, positions, the shared slot mapping, the bf16
cos|sin cache and the per-layer fp32 k/v scales) for the five workloads the
hot path is measured on, plus arbitrary custom shapes for the edge-case tests.
It holds none of the write's own arithmetic: it only draws random numbers,
builds the RoPE cos|sin table (an input the rotary embedding module of the
model owns) and lays out slot mappings the way a paged-KV block allocator
would.  Both the oracle-side tests and the CUDA path consume the same tensors.

Layouts follow the vLLM DSpark context-KV writer page (module docstring and
``DSparkContextKVWriter.__call__``):

* ``all_kv``       bf16 ``[num_ctx, L, 2, nkv, 128]`` (K heads, then V heads)
* ``knorm_w``      bf16 ``[L, 128]`` (Gemma weights, applied as ``1 + w``)
* ``positions``    int64 ``[num_ctx]``
* ``slot_mapping`` int64 ``[num_ctx]``; ``-1`` marks padding
* ``cos_sin``      bf16 ``[max_pos, rotary_dim]``: cos in the first half, sin
  in the second
* ``k_scale``, ``v_scale``  fp32 ``[L]``
* per-layer caches ``[num_blocks, nkv, block_size, 256]`` (bf16, or uint8
  holding fp8 e4m3 codes), prefilled with the byte 0xFF
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

HEAD_DIM = 128
ROW_ELEMS = 2 * HEAD_DIM
PREFILL_BYTE = 0xFF
BASE_SEED = 20260

KV_BF16 = "bf16"
KV_FP8 = "fp8_e4m3"


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one write call."""

    name: str
    num_ctx: int
    num_layers: int
    num_kv_heads: int
    rotary_dim: int
    block_size: int
    num_blocks: int
    max_pos: int
    rope_theta: float
    kv_dtype: str = KV_BF16
    kv_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    w_std: float = 0.1
    eps: float = 1e-6
    scale_lo: float = 0.05
    scale_hi: float = 0.5
    # slot layout: "unique" (distinct random slots, random positions),
    # "perm" (first num_ctx of a permutation, positions 0..num_ctx-1),
    # "blocktable" (requests with positions 0..tpr-1 through per-request
    # block tables), "offset" (requests at random offsets, each logical
    # block on its own shuffled physical block)
    slots: str = "unique"
    pad_count: int = 0
    requests: int = 0
    tokens_per_request: int = 0
    blocks_per_request: int = 0
    seed: int = BASE_SEED
    # D of K and V: the pages' 128, or another head dim (64, 256) of the
    # general write; cache rows hold 2D elements
    head_dim: int = HEAD_DIM

    @property
    def row_elems(self) -> int:
        return 2 * self.head_dim

    @property
    def capacity(self) -> int:
        return self.num_blocks * self.block_size

    @property
    def elem_size(self) -> int:
        return 2 if self.kv_dtype == KV_BF16 else 1

    @property
    def layer_cache_bytes(self) -> int:
        return self.num_blocks * self.num_kv_heads * self.block_size * self.row_elems * self.elem_size

    @property
    def num_rows(self) -> int:
        return self.num_ctx * self.num_layers * self.num_kv_heads

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: tiny, draft step, fp8 draft step, prefill batch, long context.
WORKLOADS: list[Workload] = [
    Workload(
        name="tiny", num_ctx=16, num_layers=1, num_kv_heads=1, rotary_dim=64,
        block_size=16, num_blocks=4, max_pos=64, rope_theta=1e4,
        slots="perm", pad_count=2, seed=BASE_SEED + 0,
    ),
    Workload(
        name="draft_step", num_ctx=512, num_layers=5, num_kv_heads=8, rotary_dim=64,
        block_size=16, num_blocks=4096, max_pos=32768, rope_theta=1e6,
        slots="unique", pad_count=26, seed=BASE_SEED + 1,
    ),
    Workload(
        name="draft_step_fp8", num_ctx=512, num_layers=5, num_kv_heads=8, rotary_dim=64,
        block_size=16, num_blocks=4096, max_pos=32768, rope_theta=1e6,
        kv_dtype=KV_FP8, kv_std=2.0, outlier_frac=0.01, outlier_mult=10.0,
        slots="unique", pad_count=26, seed=BASE_SEED + 2,
    ),
    Workload(
        name="prefill_fp8", num_ctx=8192, num_layers=5, num_kv_heads=8, rotary_dim=32,
        block_size=64, num_blocks=2048, max_pos=32768, rope_theta=1e6,
        kv_dtype=KV_FP8, slots="blocktable", pad_count=164,
        requests=32, tokens_per_request=256, blocks_per_request=4, seed=BASE_SEED + 3,
    ),
    Workload(
        name="long_context", num_ctx=65536, num_layers=5, num_kv_heads=4, rotary_dim=16,
        block_size=128, num_blocks=8192, max_pos=131072, rope_theta=1e6,
        slots="offset", pad_count=0, requests=256, tokens_per_request=256, seed=BASE_SEED + 4,
    ),
]

WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS}

# Prefill-sized writes in layouts the pages' kernel refuses (head dims 64 and
# 256, rotary dims other than 16 / 32 / 64, block sizes that are not powers
# of two), for the general write: same value recipe, blocktable slots.
GENERAL_WORKLOADS: list[Workload] = [
    Workload(
        name="gen_head64", num_ctx=8192, num_layers=5, num_kv_heads=8, rotary_dim=64, head_dim=64,
        block_size=16, num_blocks=4096, max_pos=32768, rope_theta=1e6, slots="blocktable", pad_count=164,
        requests=32, tokens_per_request=256, blocks_per_request=16, seed=BASE_SEED + 10,
    ),
    Workload(
        name="gen_head256_fp8", num_ctx=8192, num_layers=5, num_kv_heads=4, rotary_dim=64, head_dim=256,
        block_size=32, num_blocks=2048, max_pos=32768, rope_theta=1e6, kv_dtype=KV_FP8, slots="blocktable",
        pad_count=164, requests=32, tokens_per_request=256, blocks_per_request=8, seed=BASE_SEED + 11,
    ),
    Workload(
        name="gen_block48_fp8", num_ctx=8192, num_layers=5, num_kv_heads=8, rotary_dim=32,
        block_size=48, num_blocks=2048, max_pos=32768, rope_theta=1e6, kv_dtype=KV_FP8, slots="blocktable",
        pad_count=164, requests=32, tokens_per_request=256, blocks_per_request=6, seed=BASE_SEED + 12,
    ),
    Workload(
        name="gen_rot24", num_ctx=8192, num_layers=5, num_kv_heads=8, rotary_dim=24,
        block_size=16, num_blocks=4096, max_pos=32768, rope_theta=1e6, slots="blocktable", pad_count=164,
        requests=32, tokens_per_request=256, blocks_per_request=16, seed=BASE_SEED + 13,
    ),
    Workload(
        name="gen_rot128", num_ctx=8192, num_layers=5, num_kv_heads=8, rotary_dim=128,
        block_size=64, num_blocks=2048, max_pos=32768, rope_theta=1e6, slots="blocktable", pad_count=164,
        requests=32, tokens_per_request=256, blocks_per_request=4, seed=BASE_SEED + 14,
    ),
]

GENERAL_WORKLOADS_BY_NAME = {w.name: w for w in GENERAL_WORKLOADS}


def pages_layout(wl: Workload) -> bool:
    """Whether the pages' kernel takes this layout (writer page,
    rotary_dims_supported and DSparkContextKVWriter._validate: head_dim 128,
    rotary_dim 16 / 32 / 64, a power-of-two block size)."""
    bs = wl.block_size
    return wl.head_dim == HEAD_DIM and wl.rotary_dim in (16, 32, 64) and bs > 0 and bs & (bs - 1) == 0


@dataclass
class Inputs:
    """CPU tensors of one write call (see the module docstring for layouts)."""

    workload: Workload
    all_kv: torch.Tensor
    knorm_w: torch.Tensor
    positions: torch.Tensor
    slot_mapping: torch.Tensor
    cos_sin: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    eps: float
    extra: dict = field(default_factory=dict)

    @property
    def num_valid_tokens(self) -> int:
        return int((self.slot_mapping >= 0).sum())

    def to(self, device) -> "Inputs":
        mv = lambda x: x.to(device)  # noqa: E731
        return Inputs(self.workload, mv(self.all_kv), mv(self.knorm_w), mv(self.positions),
                      mv(self.slot_mapping), mv(self.cos_sin), mv(self.k_scale),
                      mv(self.v_scale), self.eps, dict(self.extra))


def rope_cos_sin_cache(max_pos: int, rotary_dim: int, theta: float) -> torch.Tensor:
    """bf16 ``[max_pos, rotary_dim]`` table: cos(p*f_i) then sin(p*f_i), with
    ``f_i = theta**(-2i/rotary_dim)`` for ``i < rotary_dim/2`` (the NeoX
    rotary embedding's cos|sin cache, evaluated in fp64 and rounded to bf16)."""
    half = rotary_dim // 2
    i = torch.arange(half, dtype=torch.float64)
    inv_freq = theta ** (-2.0 * i / rotary_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return torch.cat([ang.cos(), ang.sin()], dim=1).float().to(torch.bfloat16).contiguous()


def _positions_and_slots(wl: Workload, g: torch.Generator):
    T = wl.num_ctx
    if wl.slots == "perm":
        pos = torch.arange(T, dtype=torch.int64)
        slots = torch.randperm(wl.capacity, generator=g)[:T].to(torch.int64)
    elif wl.slots == "unique":
        if T > wl.capacity:
            raise ValueError("more tokens than cache slots")
        pos = torch.randint(0, wl.max_pos, (T,), generator=g, dtype=torch.int64)
        slots = torch.randperm(wl.capacity, generator=g)[:T].to(torch.int64)
    elif wl.slots == "blocktable":
        R, tpr, bpr, bs = wl.requests, wl.tokens_per_request, wl.blocks_per_request, wl.block_size
        assert R * tpr == T and bpr * bs >= tpr and R * bpr <= wl.num_blocks
        tables = torch.randperm(wl.num_blocks, generator=g)[: R * bpr].view(R, bpr).to(torch.int64)
        p = torch.arange(tpr, dtype=torch.int64)
        pos = p.repeat(R)
        slots = (tables[:, p // bs] * bs + (p % bs)[None, :]).reshape(-1)
    elif wl.slots == "offset":
        R, tpr, bs = wl.requests, wl.tokens_per_request, wl.block_size
        assert R * tpr == T
        offs = torch.randint(0, wl.max_pos - tpr + 1, (R,), generator=g, dtype=torch.int64)
        phys_pool = torch.randperm(wl.num_blocks, generator=g).to(torch.int64)
        nxt = 0
        pos_l, slot_l = [], []
        for r in range(R):
            p = offs[r] + torch.arange(tpr, dtype=torch.int64)
            lb = p // bs
            first = int(lb[0])
            nlb = int(lb[-1]) - first + 1
            phys = phys_pool[nxt: nxt + nlb]
            nxt += nlb
            if nxt > wl.num_blocks:
                raise ValueError("not enough physical blocks")
            pos_l.append(p)
            slot_l.append(phys[lb - first] * bs + p % bs)
        pos = torch.cat(pos_l)
        slots = torch.cat(slot_l)
    else:
        raise ValueError(f"unknown slot layout {wl.slots!r}")
    if wl.pad_count:
        pad = torch.randperm(T, generator=g)[: wl.pad_count]
        slots = slots.clone()
        slots[pad] = -1
    return pos.contiguous(), slots.contiguous()


def generate(wl: Workload, seed: int | None = None, with_all_kv: bool = True) -> Inputs:
    """Draw the inputs of ``wl`` from a seeded torch CPU generator (fp32
    samples rounded to bf16 with round-to-nearest-even).  ``with_all_kv=False``
    skips the K/V draw (``all_kv`` is then an empty tensor): the caller
    computes it, e.g. from a projection."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    T, L, H = wl.num_ctx, wl.num_layers, wl.num_kv_heads
    if with_all_kv:
        kv = torch.randn((T, L, 2, H, wl.head_dim), generator=g, dtype=torch.float32)
        if wl.kv_std != 1.0:
            kv.mul_(wl.kv_std)
        if wl.outlier_frac > 0:
            hit = torch.rand(kv.shape, generator=g) < wl.outlier_frac
            kv = torch.where(hit, kv * wl.outlier_mult, kv)
        all_kv = kv.to(torch.bfloat16).contiguous()
        del kv
    else:
        all_kv = torch.empty((0,), dtype=torch.bfloat16)
    knorm_w = (torch.randn((L, wl.head_dim), generator=g) * wl.w_std).to(torch.bfloat16).contiguous()
    pos, slots = _positions_and_slots(wl, g)
    cos_sin = rope_cos_sin_cache(wl.max_pos, wl.rotary_dim, wl.rope_theta)
    if wl.kv_dtype == KV_FP8:
        k_scale = torch.empty(L, dtype=torch.float32).uniform_(wl.scale_lo, wl.scale_hi, generator=g)
        v_scale = torch.empty(L, dtype=torch.float32).uniform_(wl.scale_lo, wl.scale_hi, generator=g)
    else:
        k_scale = torch.ones(L, dtype=torch.float32)
        v_scale = torch.ones(L, dtype=torch.float32)
    return Inputs(wl, all_kv, knorm_w, pos, slots, cos_sin, k_scale, v_scale, float(wl.eps))


def make_caches(wl: Workload, device="cpu", fill: int | None = PREFILL_BYTE) -> list[torch.Tensor]:
    """One separately allocated ``[num_blocks, nkv, block_size, 2 * head_dim]``
    cache per layer, every byte set to ``fill`` (left uninitialised when
    ``fill`` is None)."""
    dtype = torch.bfloat16 if wl.kv_dtype == KV_BF16 else torch.uint8
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.row_elems)
    caches = []
    for _ in range(wl.num_layers):
        c = torch.empty(shape, dtype=dtype, device=device)
        if fill is not None:
            c.view(torch.uint8).fill_(fill)
        caches.append(c)
    return caches


def take_tokens(inp: Inputs, count: int) -> Inputs:
    """The first ``count`` tokens of ``inp`` (a bounded sample of the same call)."""
    wl = inp.workload.with_(num_ctx=count)
    return Inputs(wl, inp.all_kv[:count].contiguous(), inp.knorm_w, inp.positions[:count].contiguous(),
                  inp.slot_mapping[:count].contiguous(), inp.cos_sin, inp.k_scale, inp.v_scale, inp.eps)


def compulsory_bytes(wl: Workload, num_valid_tokens: int) -> int:
    """Bytes the write must move at least: per token its slot (and, when
    valid, its position and cos|sin row); per valid row the K|V read (512
    bytes at head dim 128) and the cache write (512 bytes bf16, 256 fp8);
    plus the K-norm weights and the 2*L scales."""
    L, H, r = wl.num_layers, wl.num_kv_heads, wl.rotary_dim
    valid_rows = num_valid_tokens * L * H
    out_row = wl.row_elems * wl.elem_size
    per_tok = 8 * wl.num_ctx + num_valid_tokens * (8 + 2 * r)
    return valid_rows * (wl.row_elems * 2 + out_row) + per_tok + L * wl.head_dim * 2 + 2 * L * 4


def describe(wl: Workload) -> dict:
    return {
        "workload": wl.name, "num_ctx": wl.num_ctx, "layers": wl.num_layers,
        "nkv": wl.num_kv_heads, "head_dim": wl.head_dim, "rotary_dim": wl.rotary_dim,
        "block_size": wl.block_size, "num_blocks": wl.num_blocks, "kv_cache_dtype": wl.kv_dtype,
        "max_pos": wl.max_pos,
    }


def layer_slot_mappings(inp: Inputs, groups: int = 2, seed: int = 0) -> torch.Tensor:
    """int64 ``[L, T]``: one slot mapping per layer for a draft whose layers
    span ``groups`` KV-cache groups (DSpark draft model page,
    ``_shared_slot_mapping``: such drafts have no shared mapping).  Layer l
    belongs to group ``l * groups // L``; group 0 keeps the workload's own
    mapping, every other group gets distinct random slots of the same cache
    size, and a few tokens padded in one group are valid in another."""
    wl = inp.workload
    T, L = wl.num_ctx, wl.num_layers
    g = torch.Generator().manual_seed(wl.seed * 7 + 11 + seed)
    maps = [inp.slot_mapping.clone()]
    for _ in range(1, groups):
        m = torch.randperm(wl.capacity, generator=g)[:T].to(torch.int64)
        flip = torch.rand(T, generator=g) < 0.05
        valid = (inp.slot_mapping >= 0) ^ flip
        maps.append(torch.where(valid, m, torch.full_like(m, -1)))
    out = torch.empty((L, T), dtype=torch.int64)
    for l in range(L):
        out[l] = maps[min(groups - 1, l * groups // L)]
    return out.contiguous()
