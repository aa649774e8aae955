"""Shared helpers of the parity tests: drive the CUDA path through the C ABI
on seeded inputs, and compare its caches with the oracle's.

Tolerance (the stated bar for this write):
  * placement and padding: bit-exact -- every row the oracle leaves at the
    0xFF prefill stays 0xFF on the GPU, byte for byte;
  * V in a bf16 cache: bit-exact (it is a copy);
  * K in a bf16 cache: within 1 bf16 ulp of the oracle's value or of one of
    its admissible alternates (the other bf16 neighbour of a norm output that
    lies within 2^-18 of a rounding midpoint, propagated through RoPE);
  * fp8 K and V: within 1 e4m3 code (same alternates for K).
Distances are taken on the sign-magnitude code as an ordered integer, so +0
and -0 are equal and neighbouring codes are 1 apart.
"""

from __future__ import annotations

import numpy as np
import torch

import workloads as wk

BF16_K_ULPS = 1
FP8_CODES = 1


def ordered(a: np.ndarray, fp8: bool) -> np.ndarray:
    a = a.astype(np.int64)
    sign = 0x80 if fp8 else 0x8000
    mag = a & (sign - 1)
    return np.where(a & sign, -mag, mag)


def _alt_ok(g_val, fp8, alts):
    return any(abs(int(ordered(np.array([a]), fp8)[0]) - int(ordered(np.array([g_val]), fp8)[0]))
               <= (FP8_CODES if fp8 else BF16_K_ULPS) for a in alts)


def compare_rows(gpu: np.ndarray, ora: np.ndarray, alt_index: dict, fp8: bool) -> list:
    """gpu, ora: [n, 2D] stored elements (K in [0, D), V in [D, 2D); D = 128
    on the pages); alt_index: {(row, dim): [values]}.  Returns a list of
    (row, dim, gpu, oracle) mismatches (empty = parity)."""
    assert gpu.shape == ora.shape and gpu.dtype == ora.dtype
    D = gpu.shape[1] // 2
    bad = []
    d = np.abs(ordered(gpu, fp8) - ordered(ora, fp8))
    if fp8:
        viol = d > FP8_CODES
    else:
        viol = np.zeros_like(d, dtype=bool)
        viol[:, :D] = d[:, :D] > BF16_K_ULPS
        viol[:, D:] = d[:, D:] != 0
    for r, c in np.argwhere(viol):
        if c < D and _alt_ok(gpu[r, c], fp8, alt_index.get((int(r), int(c)), ())):
            continue
        bad.append((int(r), int(c), int(gpu[r, c]), int(ora[r, c])))
    return bad


def alt_index_rows(alts) -> dict:
    ar, ad, av = alts
    idx: dict = {}
    for r, dm, v in zip(ar.tolist(), ad.tolist(), av.tolist()):
        idx.setdefault((r, dm), []).append(v)
    return idx


def compare_caches(gpu_caches, ora_caches, alts, fp8: bool):
    """Whole-cache comparison: unwritten rows byte-exact, written rows within
    the tolerance.  Returns a list of problems (empty = parity)."""
    al, ae, av = alts
    problems = []
    for l, (g, o) in enumerate(zip(gpu_caches, ora_caches)):
        row = o.shape[-1]
        g = g.reshape(-1, row)
        o = o.reshape(-1, row)
        fill = 0xFF if fp8 else 0xFFFF
        unwritten = (o == fill).all(axis=1)
        if not np.array_equal(g[unwritten], o[unwritten]):
            rows = np.nonzero(unwritten & ~(g == o).all(axis=1))[0]
            problems.append(f"layer {l}: {len(rows)} unaddressed rows changed, e.g. row {rows[:5].tolist()}")
        wr = np.nonzero(~unwritten)[0]
        sel = al == l
        idx = {}
        pos_of = {int(r): i for i, r in enumerate(wr)}
        for e, v in zip(ae[sel].tolist(), av[sel].tolist()):
            r, c = divmod(e, row)
            if r in pos_of:
                idx.setdefault((pos_of[r], c), []).append(v)
        bad = compare_rows(g[wr], o[wr], idx, fp8)
        if bad:
            problems.append(f"layer {l}: {len(bad)} elements out of tolerance, e.g. "
                            f"{[(int(wr[r]), c, hex(x), hex(y)) for r, c, x, y in bad[:5]]}")
    return problems


# ---------------------------------------------------------------- GPU driving

def device_inputs(inp: wk.Inputs, device="cuda"):
    d = inp.to(device)
    L = inp.workload.num_layers
    # one fp32 scalar tensor per layer, like the attention layers' _k_scale / _v_scale
    d.extra["k_scales"] = [d.k_scale[l:l + 1].clone() for l in range(L)]
    d.extra["v_scales"] = [d.v_scale[l:l + 1].clone() for l in range(L)]
    return d


def gpu_write(inp: wk.Inputs, caches=None, error_flags=None, stream=None, general=None):
    """Run the write on the GPU through the C ABI (ContextKVWriter; its
    general mode when asked or when the layout is not the pages') and return
    the device caches."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = inp.workload
    d = device_inputs(inp)
    if caches is None:
        caches = wk.make_caches(wl, device="cuda")
    if general is None:
        general = not wk.pages_layout(wl)
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"],
                           "fp8" if wl.kv_dtype == wk.KV_FP8 else "auto", general=general)
    w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping,
      stream=stream, error_flags=error_flags)
    torch.cuda.synchronize()
    return caches, w, d


def to_numpy_caches(caches, fp8: bool):
    out = []
    for c in caches:
        h = c.cpu()
        out.append(h.view(torch.uint8).numpy() if fp8 else h.view(torch.int16).numpy().view(np.uint16))
    return out


def oracle_full(inp: wk.Inputs):
    import oracle

    p = oracle.problem_from_inputs(inp)
    caches = p.new_caches()
    alts = p.write(caches)
    return p, caches, alts
