"""The synthetic inputs follow their stated recipe (shapes, seeds, padding
counts, slot structure, value ranges), so that every parity case and bench
line is run on the workloads it claims: the draft steps' distinct random
slots, the prefill's per-request block tables, the long context's shuffled
physical blocks, exact padding counts, and fp8 scales in their range.  CPU
only; the oracle is not involved."""

import numpy as np
import pytest
import torch

import workloads as wk

BY = wk.WORKLOADS_BY_NAME


def _valid(inp):
    s = inp.slot_mapping
    return s[s >= 0]


@pytest.mark.parametrize("name", ["tiny", "draft_step", "draft_step_fp8", "prefill_fp8"])
def test_shapes_dtypes_and_exact_padding(name):
    wl = BY[name]
    inp = wk.generate(wl)
    T, L, H = wl.num_ctx, wl.num_layers, wl.num_kv_heads
    assert inp.all_kv.shape == (T, L, 2, H, 128) and inp.all_kv.dtype == torch.bfloat16
    assert inp.knorm_w.shape == (L, 128) and inp.knorm_w.dtype == torch.bfloat16
    assert inp.positions.dtype == inp.slot_mapping.dtype == torch.int64
    assert inp.cos_sin.shape == (wl.max_pos, wl.rotary_dim) and inp.cos_sin.dtype == torch.bfloat16
    assert int((inp.slot_mapping < 0).sum()) == wl.pad_count
    v = _valid(inp)
    assert len(torch.unique(v)) == len(v)  # valid slots are distinct
    assert int(v.min()) >= 0 and int(v.max()) < wl.capacity
    assert int(inp.positions.min()) >= 0 and int(inp.positions.max()) < wl.max_pos


def test_seeds_make_each_workload_reproducible_and_distinct():
    a, b = wk.generate(BY["draft_step"]), wk.generate(BY["draft_step"])
    assert torch.equal(a.all_kv, b.all_kv) and torch.equal(a.slot_mapping, b.slot_mapping)
    c = wk.generate(BY["draft_step"], seed=BY["draft_step"].seed + 1)
    assert not torch.equal(a.all_kv, c.all_kv)
    seeds = [w.seed for w in wk.WORKLOADS]
    assert len(set(seeds)) == len(seeds)


def test_prefill_block_tables():
    wl = BY["prefill_fp8"]
    inp = wk.generate(wl, with_all_kv=False)
    R, tpr, bs = wl.requests, wl.tokens_per_request, wl.block_size
    pos = inp.positions.view(R, tpr)
    assert torch.equal(pos, torch.arange(tpr).expand(R, tpr))  # every request at positions 0..255
    s = inp.slot_mapping.view(R, tpr)
    valid = s >= 0
    assert torch.equal((s % bs)[valid], (pos % bs)[valid])  # offset in the block = position mod block size
    # one physical block per (request, logical block), distinct over all of them
    req = torch.arange(R).view(R, 1).expand(R, tpr)
    seen = {}
    for r, lb, blk in zip(req[valid].tolist(), (pos // bs)[valid].tolist(), (s // bs)[valid].tolist()):
        assert seen.setdefault((r, lb), blk) == blk
    assert len(set(seen.values())) == len(seen)
    assert max(lb for _, lb in seen) < wl.blocks_per_request


def test_long_context_offsets_and_shuffled_blocks():
    wl = BY["long_context"]
    inp = wk.generate(wl, with_all_kv=False)
    R, tpr, bs = wl.requests, wl.tokens_per_request, wl.block_size
    assert int((inp.slot_mapping < 0).sum()) == 0
    pos = inp.positions.view(R, tpr)
    assert (pos[:, 1:] - pos[:, :-1] == 1).all()  # consecutive positions within a request
    assert int(pos.min()) >= 0 and int(pos.max()) < wl.max_pos
    s = inp.slot_mapping.view(R, tpr)
    assert torch.equal(s % bs, pos % bs)
    # each (request, logical block) sits on one physical block of its own
    req = np.repeat(np.arange(R), tpr)
    keys = req * (wl.max_pos // bs + 1) + (inp.positions // bs).numpy()
    phys = (inp.slot_mapping // bs).numpy()
    uk, first = np.unique(keys, return_index=True)
    assert (phys == phys[first][np.searchsorted(uk, keys)]).all()  # one block per key
    assert len(np.unique(phys[first])) == len(uk)  # no block shared by two keys


def test_fp8_values_outliers_and_scales():
    wl = BY["draft_step_fp8"]
    inp = wk.generate(wl)
    ks, vs = inp.k_scale, inp.v_scale
    assert ((ks >= wl.scale_lo) & (ks <= wl.scale_hi)).all() and ((vs >= wl.scale_lo) & (vs <= wl.scale_hi)).all()
    x = inp.all_kv.float()
    # N(0, 2) with 1% of the elements x10: the tail beyond 8 sigma of the
    # base (|x| > 16) is the outliers' alone, about 1% x P(|N(0, 20)| > 16)
    frac = float((x.abs() > 16).float().mean())
    assert 0.003 < frac < 0.006
    assert abs(float(x.std()) - (4 * 0.99 + 400 * 0.01) ** 0.5) < 0.1
    bf = BY["draft_step"]
    assert (wk.generate(bf).k_scale == 1).all()  # bf16 caches: unit scales (ignored)


def test_cos_sin_rows_are_cos_then_sin_at_the_position_angle():
    wl = BY["draft_step"]
    cs = wk.rope_cos_sin_cache(wl.max_pos, wl.rotary_dim, wl.rope_theta).double()
    h = wl.rotary_dim // 2
    for p in (0, 1, 777, wl.max_pos - 1):
        ang = p * wl.rope_theta ** (-2.0 * torch.arange(h, dtype=torch.float64) / wl.rotary_dim)
        assert torch.allclose(cs[p, :h], torch.cos(ang), atol=2 ** -8)
        assert torch.allclose(cs[p, h:], torch.sin(ang), atol=2 ** -8)


@pytest.mark.parametrize("name", ["qk_tiny", "qk_draft", "qk_draft_fp8"])
def test_qk_insert_requests_of_seven_consecutive_rows(name):
    wl = wk.QK_WORKLOADS_BY_NAME[name]
    inp = wk.generate_qk(wl)
    R, n, bs = wl.requests, 7, wl.block_size
    assert wl.num_tokens == R * n
    assert inp.qkv.shape == (R * n, (wl.num_heads + 2 * wl.num_kv_heads) * 128)
    assert inp.qkv.dtype == torch.bfloat16
    pos = inp.positions.view(R, n)
    assert (pos[:, 1:] - pos[:, :-1] == 1).all() and int(pos.min()) >= 0 and int(pos.max()) < wl.max_pos
    s = inp.slot_mapping.view(R, n)
    assert int((s < 0).sum()) == wl.pad_count
    valid = s >= 0
    assert torch.equal((s % bs)[valid], (pos % bs)[valid])
    req = torch.arange(R).view(R, 1).expand(R, n)
    seen = {}
    for r, lb, blk in zip(req[valid].tolist(), (pos // bs)[valid].tolist(), (s // bs)[valid].tolist()):
        assert seen.setdefault((r, lb), blk) == blk
    assert len(set(seen.values())) == len(seen) and max(seen.values()) < wl.num_blocks


@pytest.mark.parametrize("wl", wk.GENERAL_WORKLOADS, ids=lambda w: w.name)
def test_general_layouts_are_outside_the_pages_kernel(wl):
    # each general workload breaks one of the pages' layout rules (head dim
    # 128, rotary dim 16 / 32 / 64, a power-of-two block size) and keeps the
    # prefill recipe: 32 requests x positions 0..255 through block tables
    assert not wk.pages_layout(wl)
    pages_rules = (wl.head_dim == 128, wl.rotary_dim in (16, 32, 64),
                   wl.block_size & (wl.block_size - 1) == 0)
    assert not all(pages_rules)
    inp = wk.generate(wl, with_all_kv=False)
    assert int((inp.slot_mapping < 0).sum()) == wl.pad_count
    R, tpr, bs = wl.requests, wl.tokens_per_request, wl.block_size
    pos = inp.positions.view(R, tpr)
    assert torch.equal(pos, torch.arange(tpr).expand(R, tpr))
    s = inp.slot_mapping.view(R, tpr)
    valid = s >= 0
    assert torch.equal((s % bs)[valid], (pos % bs)[valid])
    assert len(torch.unique(s[valid])) == int(valid.sum()) and int(s.max()) < wl.capacity
    assert inp.cos_sin.shape == (wl.max_pos, wl.rotary_dim)
