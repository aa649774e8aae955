"""GPU parity: the sm_103a write against the CPU oracle on the same seeded
inputs, element by element, through the C ABI.

Small workloads compare whole caches (every byte of every layer); the two
full-size workloads (prefill batch, long context) run in the same launch
configuration the benchmark times and compare every written row with the
oracle's, plus whole-cache properties: exactly the addressed rows changed.
The long-context write is also checked by a placement round trip with
tagged V rows.
Tolerance: see tests/parity.py.
"""

import numpy as np
import pytest
import torch

import workloads as wk
from parity import (alt_index_rows, compare_caches, compare_rows, device_inputs, gpu_write,
                    oracle_full, to_numpy_caches)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["default", "tma", "warp", "generic"])
def kernel(request, monkeypatch):
    """Run the test on the kernel the library picks (warp-private pipelines
    for small calls, else the pipelined bulk-copy kernel where the shape
    allows), on the pipelined kernel, on the warp-private pipelines (where
    they apply; elsewhere the default) and on the generic kernel."""
    if request.param == "default":
        monkeypatch.delenv("DSPARK_CTX_KV_KERNEL", raising=False)
    else:
        monkeypatch.setenv("DSPARK_CTX_KV_KERNEL", request.param)
    return request.param


def _parity(inp):
    wl = inp.workload
    fp8 = wl.kv_dtype == wk.KV_FP8
    caches, _, _ = gpu_write(inp)
    g = to_numpy_caches(caches, fp8)
    _, o, alts = oracle_full(inp)
    problems = compare_caches(g, o, alts, fp8)
    assert not problems, problems


@pytest.mark.parametrize("idx", [0, 1, 2], ids=["tiny", "draft_step", "draft_step_fp8"])
def test_parity_small_workloads(oracle_lib, kernel, idx):
    _parity(wk.generate(wk.WORKLOADS[idx]))


RAGGED = [
    # (T, L, H, r, bs, nb, kv, pad)
    (1, 1, 1, 16, 1, 4, wk.KV_BF16, 0),
    (7, 2, 3, 32, 2, 8, wk.KV_FP8, 2),
    (37, 3, 5, 64, 4, 16, wk.KV_BF16, 5),
    (37, 3, 6, 16, 8, 8, wk.KV_FP8, 3),
    (100, 7, 9, 32, 256, 1, wk.KV_BF16, 11),
    (333, 1, 2, 64, 32, 16, wk.KV_FP8, 0),
    (1000, 2, 4, 16, 16, 80, wk.KV_BF16, 100),
    (257, 4, 8, 64, 64, 8, wk.KV_FP8, 1),
    (50, 3, 64, 32, 16, 8, wk.KV_FP8, 5),     # one layer per stage: three pieces per token
    (20, 2, 40, 64, 4, 16, wk.KV_BF16, 2),   # 20 KB per layer: one layer per stage
    (30, 33, 2, 16, 16, 4, wk.KV_BF16, 0),   # more layers than the pipelined kernel stages
    (9, 1, 65, 16, 8, 2, wk.KV_FP8, 1),      # a layer larger than a stage
]


@pytest.mark.parametrize("T,L,H,r,bs,nb,kv,pad", RAGGED)
def test_parity_ragged_shapes(oracle_lib, kernel, T, L, H, r, bs, nb, kv, pad):
    wl = wk.Workload(name="ragged", num_ctx=T, num_layers=L, num_kv_heads=H, rotary_dim=r,
                     block_size=bs, num_blocks=nb, max_pos=3000, rope_theta=1e4, kv_dtype=kv,
                     pad_count=pad, kv_std=2.0 if kv == wk.KV_FP8 else 1.0,
                     outlier_frac=0.01 if kv == wk.KV_FP8 else 0.0, outlier_mult=10.0, seed=T * 31 + H)
    _parity(wk.generate(wl))


def test_parity_prefill_full_size(oracle_lib, kernel):
    """Prefill batch (8192 tokens, fp8, r=32, bs=64): every written row."""
    wl = wk.WORKLOADS[3]
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    _check_rows(inp, caches, row_ids=None)


def test_parity_long_context_full_size(oracle_lib, kernel):
    """Long context (65536 tokens, bf16, r=16, bs=128) at full size: every
    written row -- all 1,310,720 (token, layer, head) rows -- against the
    oracle, and exactly the addressed rows changed."""
    wl = wk.WORKLOADS[4]
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    _check_rows(inp, caches, row_ids=None)


def test_placement_long_context_tagged(oracle_lib, kernel):
    """Placement round trip at full size (long context): V of every row
    carries exact small-integer tags of its own (token, layer, head) -- token
    low byte, token high byte, layer, head, each an integer below 256 and so
    exact in bf16 -- and every written row of every layer's cache must
    decode back to a token whose slot (oracle placement rule) and head give
    exactly that row, in that layer; every layer holds exactly the valid
    tokens' rows (writer page: slots < 0 are padding and are not written)."""
    import oracle

    wl = wk.WORKLOADS[4]
    inp = wk.generate(wl)
    T, L, H = wl.num_ctx, wl.num_layers, wl.num_kv_heads
    t = torch.arange(T)
    v = inp.all_kv[:, :, 1]  # [T, L, H, 128] view
    v[..., 0] = (t & 255).to(torch.bfloat16)[:, None, None]
    v[..., 1] = (t >> 8).to(torch.bfloat16)[:, None, None]
    v[..., 2] = torch.arange(L, dtype=torch.bfloat16)[None, :, None]
    v[..., 3] = torch.arange(H, dtype=torch.bfloat16)[None, None, :]
    caches, _, _ = gpu_write(inp)
    slots = inp.slot_mapping.numpy()
    nvalid = int((slots >= 0).sum())
    for layer, c in enumerate(caches):
        rows = c.view(-1, 256)
        written = (rows.view(torch.int16) != -1).any(dim=1).nonzero().flatten()
        assert written.numel() == nvalid * H, (layer, written.numel(), nvalid * H)
        tags = rows[written][:, 128:132].float().cpu().numpy().astype(np.int64)
        tt = tags[:, 0] + 256 * tags[:, 1]
        assert (tags[:, 2] == layer).all()
        assert ((tt >= 0) & (tt < T)).all()
        assert (slots[tt] >= 0).all()
        dest = np.array([oracle.dest_row(int(s), int(h), H, wl.block_size, wl.num_blocks)
                         for s, h in zip(slots[tt], tags[:, 3])], np.int64)
        assert np.array_equal(dest, written.cpu().numpy())


def _check_rows(inp, caches, row_ids):
    import oracle

    wl = inp.workload
    fp8 = wl.kv_dtype == wk.KV_FP8
    p = oracle.problem_from_inputs(inp)
    L, H = wl.num_layers, wl.num_kv_heads
    slots = inp.slot_mapping
    if row_ids is None:
        valid_t = (slots >= 0).nonzero().flatten()
        row_ids = (valid_t[:, None] * (L * H) + torch.arange(L * H)[None, :]).flatten().numpy()
    row_ids = np.asarray(row_ids, np.int64)
    t = row_ids // (L * H)
    keep = slots.numpy()[t] >= 0
    row_ids = row_ids[keep]
    t = t[keep]
    l = (row_ids // H) % L
    h = row_ids % H
    ora, alts = p.rows(row_ids)
    # destination rows from the oracle's placement rule
    s = slots.numpy()[t]
    dest = np.array([oracle.dest_row(int(si), int(hi), H, wl.block_size, wl.num_blocks)
                     for si, hi in zip(s, h)], np.int64)
    assert (dest >= 0).all()
    gpu = np.empty_like(ora)
    for layer in range(L):
        m = l == layer
        if not m.any():
            continue
        rows = caches[layer].view(-1, 256)[torch.from_numpy(dest[m]).cuda()].cpu()
        gpu[m] = rows.view(torch.uint8).numpy() if fp8 else rows.view(torch.int16).numpy().view(np.uint16)
    # compared in chunks of rows, so that full-size workloads stay within a
    # few GB of host memory
    ar, ad, av = alts
    bad = []
    chunk = 1 << 17
    for c0 in range(0, len(row_ids), chunk):
        m = (ar >= c0) & (ar < c0 + chunk)
        bad += compare_rows(gpu[c0:c0 + chunk], ora[c0:c0 + chunk], alt_index_rows((ar[m] - c0, ad[m], av[m])), fp8)
    assert not bad, bad[:10]
    # whole caches: exactly the addressed rows differ from the 0xFF prefill
    nvalid = int((slots >= 0).sum())
    changed = 0
    for c in caches:
        b = c.view(torch.uint8).view(-1, 256 * c.element_size())
        changed += int((b != 0xFF).any(dim=1).sum())
    assert changed == nvalid * H * L


def test_fp8_v_codes_are_bit_exact(oracle_lib, kernel):
    """Beyond the 1-code tolerance: every fp8 V code equals the oracle's,
    i.e. the kernels' x / scale is the correctly rounded fp32 quotient and
    the pack rounds to nearest even with saturation, like the oracle."""
    wl = wk.WORKLOADS[2]
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    g = to_numpy_caches(caches, True)
    _, o, _ = oracle_full(inp)
    for l in range(wl.num_layers):
        gl, ol = g[l].reshape(-1, 256), o[l].reshape(-1, 256)
        wr = ~(ol == 0xFF).all(axis=1)
        assert np.array_equal(gl[wr, 128:], ol[wr, 128:])


def test_zero_tokens_launches_nothing_and_writes_nothing(oracle_lib):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[1].with_(num_ctx=0, pad_count=0)
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    for c in caches:
        assert bool((c.view(torch.uint8) == 0xFF).all())
    # the raw entry point with num_ctx 0 and null buffers is fine too
    dk.dspark_ctx_kv_write(0, 0, 0, 0, 0, 0, 1, 0, 1, 0, 0, 0, 1, 1, 16, 16, 1e-6, 0)


def test_all_padding_writes_nothing(oracle_lib):
    wl = wk.WORKLOADS[1].with_(num_ctx=64, pad_count=64)
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    for c in caches:
        assert bool((c.view(torch.uint8) == 0xFF).all())


def test_out_of_range_rows_are_skipped_and_flagged(oracle_lib, kernel):
    """Rows with a slot beyond the cache or a position beyond the cos|sin
    table are not written and set their bit in the error word; a padded
    token's position is never looked at; every other row is still exact."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[1].with_(num_ctx=200, pad_count=20)
    inp = wk.generate(wl)
    valid = (inp.slot_mapping >= 0).nonzero().flatten()
    pad = (inp.slot_mapping < 0).nonzero().flatten()
    bad_slot_t, bad_pos_t = int(valid[3]), int(valid[10])
    inp.slot_mapping[bad_slot_t] = wl.capacity + 5
    inp.positions[bad_pos_t] = wl.max_pos
    inp.positions[pad] = -(10**12)  # never read
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches, _, _ = gpu_write(inp, error_flags=flags)
    assert int(flags.item()) == dk.FLAG_SLOT_RANGE | dk.FLAG_POS_RANGE
    # the oracle's view of the same call without the two bad tokens
    ref = wk.generate(wl)
    ref.positions.copy_(inp.positions)
    ref.positions[pad] = 0
    ref.slot_mapping.copy_(inp.slot_mapping)
    ref.slot_mapping[[bad_slot_t, bad_pos_t]] = -1
    _, o, alts = oracle_full(ref)
    problems = compare_caches(to_numpy_caches(caches, False), o, alts, False)
    assert not problems, problems

    flags.zero_()
    ok_inp = wk.generate(wl)
    gpu_write(ok_inp, error_flags=flags)
    assert int(flags.item()) == 0


def test_layer_caches_in_one_buffer_with_negative_offsets(oracle_lib, kernel):
    """Layers carved from one allocation in reverse order: layer l > 0 lies
    before layer 0, so its element offset is negative."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[2].with_(num_ctx=300, pad_count=9)
    inp = wk.generate(wl)
    per = wl.num_blocks * wl.num_kv_heads * wl.block_size * 256
    gap = 16 * 3  # a 16-element aligned gap between layers
    buf = torch.full(((per + gap) * wl.num_layers,), 0xFF, dtype=torch.uint8, device="cuda")
    caches = []
    for l in range(wl.num_layers):
        start = (wl.num_layers - 1 - l) * (per + gap)
        caches.append(buf[start:start + per].view(wl.num_blocks, wl.num_kv_heads, wl.block_size, 256))
    gpu_write(inp, caches=caches)
    _, o, alts = oracle_full(inp)
    assert not compare_caches(to_numpy_caches(caches, True), o, alts, True)
    # the gaps were not touched
    for l in range(wl.num_layers):
        start = (wl.num_layers - 1 - l) * (per + gap) + per
        assert bool((buf[start:start + gap] == 0xFF).all())
    assert dk.STATUS_CODE["DSPARK_OK"] == 0


def test_zero_and_constant_rows(oracle_lib, kernel):
    """Degenerate K rows: all zero (normed to zero), constant (normed to
    1 + w), one-hot; and a token at position 0 (RoPE is the identity)."""
    wl = wk.WORKLOADS[1].with_(num_ctx=32, pad_count=0, num_layers=2)
    inp = wk.generate(wl)
    inp.all_kv[0, :, 0] = 0.0
    inp.all_kv[1, :, 0] = 0.75
    inp.all_kv[2, :, 0] = 0.0
    inp.all_kv[2, :, 0, :, 5] = -3.0
    inp.positions[3] = 0
    _parity(inp)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_cuda_graph_capture_and_replay(oracle_lib):
    """The write captured in a CUDA graph replays against new input values in
    the same buffers; the tables are not rebuilt on the same key, and a moved
    cache during capture is refused with DSPARK_ERR_CAPTURING."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[2].with_(num_ctx=256, pad_count=12)
    inp = wk.generate(wl)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)  # warm-up builds tables
    torch.cuda.synchronize()
    assert w.tables.builds == 1
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    assert w.tables.builds == 1
    # new values in the same buffers, caches reset, scales changed in place
    inp2 = wk.generate(wl, seed=999)
    for name in ("all_kv", "knorm_w", "positions", "slot_mapping"):
        getattr(d, name).copy_(getattr(inp2, name).cuda())
    for l in range(wl.num_layers):
        d.extra["k_scales"][l].fill_(float(inp2.k_scale[l]))
        d.extra["v_scales"][l].fill_(float(inp2.v_scale[l]))
    for c in caches:
        c.fill_(0xFF)
    g.replay()
    torch.cuda.synchronize()
    _, o, alts = oracle_full(inp2)
    assert not compare_caches(to_numpy_caches(caches, True), o, alts, True)
    # a cache that moves while capturing: refused, old tables kept
    moved = [c.clone() for c in caches]
    w2 = dk.ContextKVWriter(moved, d.extra["k_scales"], d.extra["v_scales"], "fp8")
    w2._tables = w.tables
    g2 = torch.cuda.CUDAGraph()
    with pytest.raises(dk.DSparkError) as ei:
        with torch.cuda.graph(g2, stream=s):
            w2(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    assert ei.value.name == "DSPARK_ERR_CAPTURING"
    w2._tables = None
    torch.cuda.synchronize()


def test_writer_validation_on_device_tensors(oracle_lib):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[1]
    ks = [torch.ones(1, device="cuda") for _ in range(2)]
    good = [torch.empty(8, 2, 16, 256, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    assert dk.ContextKVWriter.supported(good, ks, ks, "auto")
    bad_bs = [torch.empty(8, 2, 12, 256, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(dk.DSparkError, match="BLOCK_SIZE"):
        dk.ContextKVWriter(bad_bs, ks, ks, "auto")
    u8 = [torch.empty(8, 2, 16, 256, dtype=torch.uint8, device="cuda") for _ in range(2)]
    with pytest.raises(dk.DSparkError, match="DTYPE"):
        dk.ContextKVWriter(u8, ks, ks, "auto")
    assert dk.ContextKVWriter.supported(u8, ks, ks, "fp8")
    base = torch.empty(2 * 8 * 2 * 16 * 256 + 8, dtype=torch.bfloat16, device="cuda")
    n = 8 * 2 * 16 * 256
    mis = [base[:n].view(8, 2, 16, 256), base[8:8 + n].view(8, 2, 16, 256)]
    with pytest.raises(dk.DSparkError, match="ALIGNMENT"):
        dk.ContextKVWriter(mis, ks, ks, "auto")
    cpu_scales = [torch.ones(1) for _ in range(2)]
    assert not dk.ContextKVWriter.supported(good, cpu_scales, cpu_scales, "auto")
    nc = [torch.empty(8, 16, 2, 256, dtype=torch.bfloat16, device="cuda").transpose(1, 2) for _ in range(2)]
    assert not dk.ContextKVWriter.supported(nc, ks, ks, "auto")
    del wl


@pytest.mark.parametrize("which", ["tma", "warp"])
def test_expired_wait_reports_timeout_and_leaves_the_context_usable(oracle_lib, monkeypatch, which):
    """The timeout path of the pipelined and the warp-private kernels,
    exercised without a fault: with the test hook DSPARK_TEST_HOLD_NS set,
    each CTA's producer (each warp) first waits 2 ms on a device word that
    nothing sets; the wait runs out, it stops before issuing any copy (the
    pipelined kernel's consumers see the abort and leave), nothing is
    written, and DSPARK_FLAG_TIMEOUT reaches the caller's error word -- or
    the writer's own word when the caller passes none.  The next launch,
    hook off, matches the oracle: the context is still usable."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.WORKLOADS[2].with_(num_ctx=256, pad_count=12)
    inp = wk.generate(wl)
    monkeypatch.setenv("DSPARK_CTX_KV_KERNEL", which)
    monkeypatch.setenv("DSPARK_TEST_HOLD_NS", "2000000")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches, w, d = gpu_write(inp, error_flags=flags)
    assert int(flags.item()) == dk.FLAG_TIMEOUT
    for c in caches:
        assert bool((c.view(torch.uint8) == 0xFF).all())
    w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    assert w.error_flags() == dk.FLAG_TIMEOUT
    assert w.error_flags() == 0  # read and cleared
    monkeypatch.delenv("DSPARK_TEST_HOLD_NS")
    flags.zero_()
    caches, _, _ = gpu_write(inp, error_flags=flags)
    assert int(flags.item()) == 0
    _, o, alts = oracle_full(inp)
    assert not compare_caches(to_numpy_caches(caches, True), o, alts, True)
