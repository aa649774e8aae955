"""GPU parity of the tensor-core context-KV projection and of the projection
with the write fused into its epilogue (DSpark draft model page,
precompute_and_store_context_kv: all_kv = the projection of the context
states, then the fused writer), through the C ABI.

* Exact-integer inputs (x in {-8..8}/8, w in {-8..8}/32): every fp32 partial
  sum is exact whatever the order of the tensor cores' accumulation, so the
  bf16 projection is unique -- the projection must equal the oracle's bit
  for bit, and the fused write must match the oracle's write of the oracle's
  projection within the write's own tolerance (tests/parity.py).
* Every case runs on both tile shapes (128 and 256 tokens per tile).
* Gaussian inputs: each projected element within |sum of fp32 rounding
  errors| <= hidden * 2^-24 * sum_k |x_k w_k| (any summation order) plus one
  bf16 rounding of the exact dot product; then the oracle writes that
  projection and the fused launch must match it at the write's tolerance.
"""

import numpy as np
import pytest
import torch

import workloads as wk
from parity import compare_caches, device_inputs, to_numpy_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["short", "tall"])
def tile(request, monkeypatch):
    """Every case on both tile shapes: 128-token tiles with the two
    accumulators alternating, and 256-token tiles filling both at once (the
    default picks one by the call's size)."""
    monkeypatch.setenv("DSPARK_PROJ_TILE", request.param)
    return request.param


def bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def proj_workload(name, recipe="int", **base_over):
    wl = wk.PROJ_WORKLOADS_BY_NAME[name].with_(recipe=recipe)
    if base_over:
        wl = wl.with_(base=wl.base.with_(**base_over))
    return wl


def gpu_project(inp: wk.ProjInputs):
    import speculative_decoding_draft_ctx_gb300 as dk

    b = inp.workload.base
    x, w = inp.x.cuda(), inp.w_kv.cuda()
    out = dk.project_context_kv(x, w, b.num_layers, b.num_kv_heads)
    torch.cuda.synchronize()
    return out


def gpu_project_write(inp: wk.ProjInputs, flags=None):
    import speculative_decoding_draft_ctx_gb300 as dk

    b = inp.workload.base
    d = device_inputs(inp.ctx)
    caches = wk.make_caches(b, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"],
                           "fp8" if b.kv_dtype == wk.KV_FP8 else "auto")
    w.project_and_write(inp.x.cuda(), inp.w_kv.cuda(), d.knorm_w, d.eps, d.positions, d.cos_sin, b.rotary_dim,
                        d.slot_mapping, error_flags=flags)
    torch.cuda.synchronize()
    return caches


PROJ_SHAPES = [
    # (base workload, overrides, hidden)
    ("proj_tiny", {}, 256),
    ("proj_draft_step", {}, 4096),
    ("proj_draft_step", {"num_ctx": 200, "pad_count": 9}, 136),       # a ragged row tile and a ragged k-block
    ("proj_draft_step", {"num_ctx": 129, "num_layers": 2, "num_kv_heads": 3, "pad_count": 4}, 72),
    ("proj_prefill_fp8", {}, 512),
]


@pytest.mark.parametrize("name,over,hidden", PROJ_SHAPES)
def test_projection_bit_exact_on_exact_inputs(oracle_lib, name, over, hidden):
    wl = proj_workload(name, **over).with_(hidden=hidden)
    inp = wk.generate_proj(wl)
    got = bits(gpu_project(inp)).reshape(wl.base.num_ctx, -1)
    ref = oracle_lib.project_context_kv(bits(inp.x), bits(inp.w_kv))
    bad = np.argwhere(got != ref)
    assert len(bad) == 0, (len(bad), bad[:5].tolist())


def test_projection_gaussian_within_the_fp32_bound(oracle_lib):
    wl = proj_workload("proj_draft_step", recipe="gauss", num_ctx=256, pad_count=5)
    inp = wk.generate_proj(wl)
    got, exact = _projection_within_fp32_bound(oracle_lib, inp, gpu_project(inp))
    # and most elements are the correctly rounded bf16 of the exact dot product
    ref = oracle_lib.bf16_values(oracle_lib.bf16_rne_array(exact))
    assert (got == ref).mean() > 0.995


FUSED = [
    ("proj_tiny", {}, 256),
    ("proj_draft_step", {}, 4096),
    ("proj_draft_step_fp8", {}, 4096),
    ("proj_draft_step", {"num_ctx": 200, "pad_count": 9, "rotary_dim": 16}, 136),
    ("proj_draft_step_fp8", {"num_ctx": 333, "num_layers": 3, "num_kv_heads": 5, "rotary_dim": 32,
                             "block_size": 4, "num_blocks": 2048, "pad_count": 20}, 264),
]


@pytest.mark.parametrize("name,over,hidden", FUSED)
def test_fused_write_matches_the_oracle_on_exact_inputs(oracle_lib, name, over, hidden):
    wl = proj_workload(name, **over).with_(hidden=hidden)
    inp = wk.generate_proj(wl)
    b = wl.base
    fp8 = b.kv_dtype == wk.KV_FP8
    caches = gpu_project_write(inp)
    all_kv = oracle_lib.project_context_kv(bits(inp.x), bits(inp.w_kv))
    ctx = wk.with_all_kv(inp, all_kv)
    p = oracle_lib.problem_from_inputs(ctx)
    ora = p.new_caches()
    alts = p.write(ora)
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


def test_fused_write_full_prefill_sampled(oracle_lib):
    """Prefill fp8 at full size (8192 tokens, hidden 4096): every written row
    of 512 sampled tokens against the oracle, and nothing else written."""
    wl = proj_workload("proj_prefill_fp8")
    inp = wk.generate_proj(wl)
    b = wl.base
    caches = gpu_project_write(inp)
    g = to_numpy_caches(caches, True)
    rng = np.random.default_rng(7)
    toks = np.sort(rng.choice(b.num_ctx, 512, replace=False))
    all_kv = oracle_lib.project_context_kv(bits(inp.x[toks]), bits(inp.w_kv))
    sub = wk.Inputs(b.with_(num_ctx=len(toks)),
                    torch.from_numpy(all_kv.view(np.int16)).view(torch.bfloat16).reshape(
                        len(toks), b.num_layers, 2, b.num_kv_heads, 128),
                    inp.ctx.knorm_w, inp.ctx.positions[toks].contiguous(), inp.ctx.slot_mapping[toks].contiguous(),
                    inp.ctx.cos_sin, inp.ctx.k_scale, inp.ctx.v_scale, inp.ctx.eps)
    p = oracle_lib.problem_from_inputs(sub)
    ids = np.arange(len(toks) * b.num_layers * b.num_kv_heads, dtype=np.int64)
    rows, (ar, ad, av) = p.rows(ids)
    dest = p.dest_rows(ids)
    keep = dest >= 0
    from parity import compare_rows

    for l in range(b.num_layers):
        sel = keep & ((ids // b.num_kv_heads) % b.num_layers == l)
        idx = {}
        pos_of = {int(i): k for k, i in enumerate(np.nonzero(sel)[0])}
        for r, dm, v in zip(ar.tolist(), ad.tolist(), av.tolist()):
            if r in pos_of:
                idx.setdefault((pos_of[r], dm), []).append(v)
        gl = g[l].reshape(-1, 256)[dest[sel]]
        bad = compare_rows(gl, rows[sel], idx, True)
        assert not bad, (l, len(bad), bad[:5])
    # exactly the valid tokens' rows were written
    valid = int((inp.ctx.slot_mapping >= 0).sum())
    for l in range(b.num_layers):
        written = (~(g[l].reshape(-1, 256) == 0xFF).all(axis=1)).sum()
        assert written == valid * b.num_kv_heads


def _projection_within_fp32_bound(oracle_lib, inp, all_kv):
    """Every element of the GPU projection within |sum of fp32 rounding
    errors| <= hidden * 2^-24 * sum_k |x_k w_k| (any summation order) plus
    one bf16 rounding of the exact dot product."""
    wl = inp.workload
    got = oracle_lib.bf16_values(bits(all_kv).reshape(wl.base.num_ctx, -1))
    x = oracle_lib.bf16_values(bits(inp.x))
    w = oracle_lib.bf16_values(bits(inp.w_kv))
    exact = x @ w.T
    bound = wl.hidden * 2.0**-24 / (1 - wl.hidden * 2.0**-24) * (np.abs(x) @ np.abs(w).T)
    # one bf16 rounding: half a bf16 ulp of the value (2^-8 relative), doubled for slack at binade edges
    ulp = np.abs(exact) * 2.0**-7 + 2.0**-133
    err = np.abs(got - exact)
    assert (err <= bound + ulp).all(), float((err - bound - ulp).max())
    return got, exact


@pytest.mark.parametrize("name,over", [
    ("proj_draft_step", {}),
    ("proj_draft_step_fp8", {}),
    ("proj_draft_step_fp8", {"num_ctx": 333, "num_layers": 3, "num_kv_heads": 5, "rotary_dim": 32,
                             "block_size": 4, "num_blocks": 2048, "pad_count": 20}),
])
def test_fused_write_gaussian_matches_the_oracle(oracle_lib, name, over):
    """Gaussian inputs: the projection of a Gaussian recipe has no unique
    bf16 value (the fp32 sum depends on the accumulation order), so the
    library's standalone projection -- the same tiles and the same tensor-core
    accumulation order as the fused launch -- is first held to the fp32
    accumulation bound above, then the oracle writes *that* all_kv, and the
    fused launch's caches must match the oracle's at the write's own
    tolerance (tests/parity.py: placement and padding exact, bf16 V exact,
    K within 1 ulp of an admissible value, fp8 within 1 code)."""
    wl = proj_workload(name, recipe="gauss", **over)
    inp = wk.generate_proj(wl)
    b = wl.base
    fp8 = b.kv_dtype == wk.KV_FP8
    all_kv = gpu_project(inp)
    _projection_within_fp32_bound(oracle_lib, inp, all_kv)
    p = oracle_lib.problem_from_inputs(wk.with_all_kv(inp, bits(all_kv).reshape(-1)))
    ora = p.new_caches()
    alts = p.write(ora)
    fused = to_numpy_caches(gpu_project_write(inp), fp8)
    problems = compare_caches(fused, ora, alts, fp8)
    assert not problems, problems


def test_fused_write_flags_out_of_range_rows(oracle_lib):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = proj_workload("proj_draft_step", num_ctx=130, pad_count=0)
    inp = wk.generate_proj(wl)
    inp.ctx.slot_mapping[3] = wl.base.capacity
    inp.ctx.positions[129] = wl.base.max_pos
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = gpu_project_write(inp, flags=flags)
    assert int(flags.item()) == dk.FLAG_SLOT_RANGE | dk.FLAG_POS_RANGE
    g = to_numpy_caches(caches, False)
    for c in g:
        written = (~(c.reshape(-1, 256) == 0xFFFF).all(axis=1)).sum()
        assert written == (130 - 2) * wl.base.num_kv_heads
