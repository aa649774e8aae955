"""GPU parity of the general write (head dims 64 / 128 / 256, any even rotary
dim up to the head dim, any block size) against the oracle, through the C
ABI -- the layouts the vLLM DSpark context-KV writer page's _validate and
rotary_dims_supported refuse, computed as its module docstring defines.

Tolerance as for the pages' layouts (tests/parity.py): placement, padding and
bf16 V bit-exact; K within 1 bf16 ulp of an admissible oracle value; fp8
within 1 e4m3 code.
"""

import numpy as np
import pytest
import torch

import workloads as wk
from parity import compare_caches, compare_rows, device_inputs, gpu_write, oracle_full, to_numpy_caches

pytestmark = pytest.mark.gpu


def layout(D, r, bs, fp8=False, T=300, L=3, H=5, nb=None, slots="unique", pad=11, seed=5):
    nb = nb or max(16, (2 * T) // bs + 4)
    return wk.Workload(name=f"d{D}_r{r}_bs{bs}_{'fp8' if fp8 else 'bf16'}_h{H}", num_ctx=T, num_layers=L,
                       num_kv_heads=H, rotary_dim=r, head_dim=D, block_size=bs, num_blocks=nb, max_pos=8192,
                       rope_theta=1e6, kv_dtype=wk.KV_FP8 if fp8 else wk.KV_BF16,
                       kv_std=2.0 if fp8 else 1.0, outlier_frac=0.01 if fp8 else 0.0,
                       outlier_mult=10.0 if fp8 else 1.0, slots=slots, pad_count=pad, seed=seed)


LAYOUTS = [
    layout(64, 64, 16), layout(64, 18, 3, fp8=True), layout(64, 6, 1, H=9), layout(64, 40, 24, H=1),
    layout(128, 24, 16), layout(128, 128, 48, fp8=True), layout(128, 2, 7), layout(128, 96, 12, fp8=True),
    layout(128, 64, 100, H=4),
    layout(256, 64, 32, fp8=True), layout(256, 256, 48), layout(256, 50, 100), layout(256, 2, 5, fp8=True, H=7),
    # rotary dims 16 / 32 / 64 at head dims 64 and 256: the pipelined kernel's
    # xor-shuffle RoPE; 16 heads x 8 layers of head dim 64 fill a 32 KB stage
    # with 128 rows (four row groups per consumer warp), 8 heads of head dim
    # 256 give one group per warp
    layout(64, 16, 8, fp8=True), layout(64, 32, 5), layout(64, 64, 16, H=16, L=8, T=120, fp8=True),
    layout(256, 16, 16), layout(256, 32, 12, fp8=True), layout(256, 32, 16, H=8, L=4, T=100),
]


@pytest.mark.parametrize("kernel", ["pipelined", "general"])
@pytest.mark.parametrize("wl", LAYOUTS, ids=lambda w: w.name)
def test_general_write_matches_the_oracle(oracle_lib, monkeypatch, wl, kernel):
    """Each layout through the pipelined kernel (the default) and through the
    general kernel (pinned)."""
    if kernel == "general":
        monkeypatch.setenv("DSPARK_CTX_KV_KERNEL", "general")
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    _, ora, alts = oracle_full(inp)
    fp8 = wl.kv_dtype == wk.KV_FP8
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_general_kernel_on_the_pages_layouts(oracle_lib, monkeypatch, idx):
    """The general kernel pinned for the pages' own layouts (head_dim 128,
    rotary_dim 16 / 32 / 64, power-of-two blocks) meets the same bar."""
    wl = wk.WORKLOADS[idx]
    if idx >= 3:
        wl = wl.with_(num_ctx=512, requests=2, pad_count=9)
    elif idx > 0:
        wl = wl.with_(num_ctx=200, pad_count=9)
    monkeypatch.setenv("DSPARK_CTX_KV_KERNEL", "general")
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp, general=True)
    _, ora, alts = oracle_full(inp)
    fp8 = wl.kv_dtype == wk.KV_FP8
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


@pytest.mark.parametrize("wl", [layout(256, 64, 16, H=40, T=60, L=2), layout(64, 18, 3, H=130, T=20, L=2)],
                         ids=lambda w: w.name)
def test_rows_too_wide_for_a_stage_fall_back(oracle_lib, wl):
    """nkv * 4 * head_dim above the pipelined kernel's 32 KB stage: the
    general kernel serves the call, to the same bar."""
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    _, ora, alts = oracle_full(inp)
    fp8 = wl.kv_dtype == wk.KV_FP8
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


def test_large_slots_with_a_divided_block_size(oracle_lib):
    """Block size 3 over 600,000 blocks: slots up to 1.8 million go through
    the multiply-high division; every row lands where the oracle puts it."""
    wl = layout(64, 32, 3, fp8=True, T=4096, L=1, H=1, nb=600_000, pad=40)
    inp = wk.generate(wl)
    assert int(inp.slot_mapping.max()) > 1_000_000
    caches, _, _ = gpu_write(inp)
    _, ora, alts = oracle_full(inp)
    problems = compare_caches(to_numpy_caches(caches, True), ora, alts, True)
    assert not problems, problems


@pytest.mark.parametrize("wl", [layout(256, 64, 24, fp8=True, L=4, H=3), layout(64, 18, 5, L=4, H=9)],
                         ids=lambda w: w.name)
def test_general_write_with_per_layer_slot_mappings(oracle_lib, wl):
    import speculative_decoding_draft_ctx_gb300 as dk

    inp = wk.generate(wl)
    ls = wk.layer_slot_mappings(inp, groups=2)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    fp8 = wl.kv_dtype == wk.KV_FP8
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8" if fp8 else "auto",
                           general=True)
    dls = ls.cuda()
    w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, [dls[l] for l in range(wl.num_layers)])
    torch.cuda.synchronize()
    p = oracle_lib.problem_from_inputs(inp, layer_slots=ls.numpy())
    ora = p.new_caches()
    alts = p.write(ora)
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


def test_general_write_flags_and_skips_out_of_range_rows(oracle_lib):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = layout(256, 40, 12, T=64, pad=4)
    inp = wk.generate(wl)
    valid = (inp.slot_mapping >= 0).nonzero().flatten().tolist()
    bad_slot, bad_pos = valid[0], valid[1]
    inp.slot_mapping[bad_slot] = wl.capacity + 5
    inp.positions[bad_pos] = wl.max_pos
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches, _, _ = gpu_write(inp, error_flags=flags)
    assert int(flags.item()) == dk.FLAG_SLOT_RANGE | dk.FLAG_POS_RANGE
    # the oracle on the same inputs with those two tokens padded
    ref = wk.Inputs(wl, inp.all_kv, inp.knorm_w, inp.positions.clone(), inp.slot_mapping.clone(), inp.cos_sin,
                    inp.k_scale, inp.v_scale, inp.eps)
    ref.slot_mapping[[bad_slot, bad_pos]] = -1
    ref.positions[bad_pos] = 0
    _, ora, alts = oracle_full(ref)
    problems = compare_caches(to_numpy_caches(caches, False), ora, alts, False)
    assert not problems, problems


def test_general_write_without_tokens_is_a_no_op():
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = layout(64, 18, 3, T=0, pad=0)
    caches = wk.make_caches(wl, device="cuda")
    ks = [torch.ones(1, device="cuda") for _ in range(wl.num_layers)]
    w = dk.ContextKVWriter(caches, ks, ks, "auto", general=True)
    empty = torch.empty((0, wl.num_layers, 2, wl.num_kv_heads, 64), dtype=torch.bfloat16, device="cuda")
    w(empty, torch.zeros((wl.num_layers, 64), dtype=torch.bfloat16, device="cuda"), 1e-6,
      torch.empty(0, dtype=torch.int64, device="cuda"),
      torch.zeros((16, 18), dtype=torch.bfloat16, device="cuda"), 18, torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    for c in caches:
        assert bool((c.view(torch.uint8) == 0xFF).all())


@pytest.mark.parametrize("name", [w.name for w in wk.GENERAL_WORKLOADS])
def test_full_size_general_workloads_sampled(oracle_lib, name):
    """Each general workload at full size, in the launch configuration the
    benchmark times: every written row of 256 sampled tokens against the
    oracle, and exactly the valid tokens' rows written."""
    wl = wk.GENERAL_WORKLOADS_BY_NAME[name]
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    fp8 = wl.kv_dtype == wk.KV_FP8
    g = to_numpy_caches(caches, fp8)
    D, L, H = wl.head_dim, wl.num_layers, wl.num_kv_heads
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(wl.num_ctx, 256, replace=False))
    p = oracle_lib.problem_from_inputs(inp)
    ids = (toks[:, None] * L * H + np.arange(L * H)[None, :]).reshape(-1)
    rows, (ar, ad, av) = p.rows(ids)
    dest = p.dest_rows(ids)
    keep = dest >= 0
    for l in range(L):
        sel = keep & ((ids // H) % L == l)
        pos_of = {int(i): k for k, i in enumerate(np.nonzero(sel)[0])}
        idx = {}
        for r, dm, v in zip(ar.tolist(), ad.tolist(), av.tolist()):
            if r in pos_of:
                idx.setdefault((pos_of[r], dm), []).append(v)
        got = g[l].reshape(-1, 2 * D)[dest[sel]]
        bad = compare_rows(got, rows[sel], idx, fp8)
        assert not bad, (l, len(bad), bad[:5])
    fill = 0xFF if fp8 else 0xFFFF
    for l in range(L):
        written = (~(g[l].reshape(-1, 2 * D) == fill).all(axis=1)).sum()
        assert written == inp.num_valid_tokens * H
