"""Seeded synthetic inputs for the fused context-KV projection and write.

The DSpark draft model page computes the context K/V of every draft layer
with one projection of the (normed) context states,
``all_kv = _project_context_kv_token_major(context_states, ...)``, whose
output the fused writer consumes (``all_kv [num_ctx, L, 2, nkv, 128]``).  A
projection workload is a context-KV write workload (positions, slots,
caches, norm weights, scales: ``synth``) plus the projection's inputs:

* ``x``     bf16 ``[num_ctx, hidden]``: the context states
* ``w_kv``  bf16 ``[L * 2 * nkv * 128, hidden]``: the stacked K and V
  projection rows of every layer, row ``((l * 2 + kv) * nkv + h) * 128 + d``
  producing ``all_kv[t, l, kv, h, d]``

Value recipes: ``gauss`` -- x ~ N(0, 1) (unit-RMS rows, as after the hidden
norm), w ~ N(0, 1/hidden) so that all_kv ~ N(0, 1); ``int`` -- x and w small
integers times powers of two (x in {-8..8}/8, w in {-8..8}/32), so that every
product and every partial sum of the projection is exact in fp32 whatever
the summation order: the projection's bf16 output is then unique, and the
fused write can be compared with the oracle under the write's own tolerance.
The hidden size is not on the pages; 4096 is a synthetic choice.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch

from .synth import HEAD_DIM, WORKLOADS_BY_NAME, Inputs, Workload, generate


@dataclass(frozen=True)
class ProjWorkload:
    name: str
    base: Workload
    hidden: int = 4096
    recipe: str = "gauss"   # "gauss" | "int"

    @property
    def n_out(self) -> int:
        return self.base.num_layers * 2 * self.base.num_kv_heads * HEAD_DIM

    def with_(self, **kw) -> "ProjWorkload":
        return replace(self, **kw)


PROJ_WORKLOADS: list[ProjWorkload] = [
    ProjWorkload("proj_tiny", WORKLOADS_BY_NAME["tiny"], hidden=256, recipe="int"),
    ProjWorkload("proj_draft_step", WORKLOADS_BY_NAME["draft_step"]),
    ProjWorkload("proj_draft_step_fp8", WORKLOADS_BY_NAME["draft_step_fp8"]),
    ProjWorkload("proj_prefill_fp8", WORKLOADS_BY_NAME["prefill_fp8"]),
    ProjWorkload("proj_long_context", WORKLOADS_BY_NAME["long_context"]),
]
PROJ_WORKLOADS_BY_NAME = {w.name: w for w in PROJ_WORKLOADS}


@dataclass
class ProjInputs:
    workload: ProjWorkload
    x: torch.Tensor       # bf16 [T, hidden]
    w_kv: torch.Tensor    # bf16 [N, hidden]
    ctx: Inputs           # the write's inputs (ctx.all_kv empty: it is the projection's output)

    def to(self, device) -> "ProjInputs":
        return ProjInputs(self.workload, self.x.to(device), self.w_kv.to(device), self.ctx.to(device))


def generate_proj(wl: ProjWorkload, seed: int | None = None) -> ProjInputs:
    base_seed = wl.base.seed + 500 if seed is None else seed
    ctx = generate(wl.base, seed=base_seed, with_all_kv=False)
    g = torch.Generator().manual_seed(base_seed + 1)
    T, H, N = wl.base.num_ctx, wl.hidden, wl.n_out
    if wl.recipe == "int":
        x = torch.randint(-8, 9, (T, H), generator=g).float() / 8.0
        w = torch.randint(-8, 9, (N, H), generator=g).float() / 32.0
    elif wl.recipe == "gauss":
        x = torch.randn((T, H), generator=g)
        w = torch.randn((N, H), generator=g) * (1.0 / H) ** 0.5
    else:
        raise ValueError(f"unknown recipe {wl.recipe!r}")
    return ProjInputs(wl, x.to(torch.bfloat16).contiguous(), w.to(torch.bfloat16).contiguous(), ctx)


def proj_flops(wl: ProjWorkload) -> int:
    return 2 * wl.base.num_ctx * wl.n_out * wl.hidden


def with_all_kv(inp: ProjInputs, all_kv_bits) -> Inputs:
    """The write's Inputs with all_kv set (e.g. to the oracle's projection)."""
    b = inp.workload.base
    kv = torch.from_numpy(all_kv_bits.view("int16")).view(torch.bfloat16).reshape(
        b.num_ctx, b.num_layers, 2, b.num_kv_heads, HEAD_DIM)
    c = inp.ctx
    return Inputs(b, kv, c.knorm_w, c.positions, c.slot_mapping, c.cos_sin, c.k_scale, c.v_scale, c.eps)
