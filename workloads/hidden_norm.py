"""Seeded synthetic inputs for the hidden-state Gemma RMSNorm of the context
states (DSpark draft model page: ``hidden_norm = _gemma_rms_norm(hidden_size,
eps)``, ``_normalize_context_states``).

* ``x``  bf16 ``[rows, hidden]``: context states, N(0, 2) with 0.1% of the
  elements scaled by 20 (hidden states carry outlier features)
* ``w``  bf16 ``[hidden]``: the Gemma weight, N(0, 0.1), applied as ``1 + w``

The hidden size is not on the pages; 4096 is a synthetic choice.  The row
counts follow the context-KV write workloads (draft step, prefill, long
context).  Holds none of the norm's arithmetic.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch

from .synth import BASE_SEED


@dataclass(frozen=True)
class NormWorkload:
    name: str
    rows: int
    hidden: int = 4096
    x_std: float = 2.0
    outlier_frac: float = 0.001
    outlier_mult: float = 20.0
    w_std: float = 0.1
    eps: float = 1e-6
    seed: int = BASE_SEED + 200

    def with_(self, **kw) -> "NormWorkload":
        return replace(self, **kw)


NORM_WORKLOADS: list[NormWorkload] = [
    NormWorkload("hn_tiny", rows=5, hidden=264, seed=BASE_SEED + 200),
    NormWorkload("hn_draft_step", rows=512, seed=BASE_SEED + 201),
    NormWorkload("hn_prefill", rows=8192, seed=BASE_SEED + 202),
    NormWorkload("hn_long_context", rows=65536, seed=BASE_SEED + 203),
]
NORM_WORKLOADS_BY_NAME = {w.name: w for w in NORM_WORKLOADS}


def generate_norm(wl: NormWorkload, seed: int | None = None):
    """(x, w, eps) on the CPU."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    x = torch.randn((wl.rows, wl.hidden), generator=g) * wl.x_std
    if wl.outlier_frac > 0:
        hit = torch.rand(x.shape, generator=g) < wl.outlier_frac
        x = torch.where(hit, x * wl.outlier_mult, x)
    w = torch.randn(wl.hidden, generator=g) * wl.w_std
    return x.to(torch.bfloat16).contiguous(), w.to(torch.bfloat16).contiguous(), float(wl.eps)


def norm_bytes(wl: NormWorkload) -> int:
    """Compulsory bytes: every row read and written once, the weight once."""
    return 2 * wl.rows * wl.hidden * 2 + wl.hidden * 2
