"""GPU parity of the write with a dynamic tail (dspark_ctx_kv_write_sched):
calls large enough for the pipelined kernel to hand its last units out from a
caller-owned work counter, compared with the oracle on whole caches under the
write's tolerance (tests/parity.py), and the counter left at zero for the
next call."""

import dataclasses

import pytest
import torch

import workloads as wk
from parity import compare_caches, device_inputs, to_numpy_caches

pytestmark = pytest.mark.gpu

PREFILL = wk.WORKLOADS[3]  # 8192 tokens, 5 layers, 8 KV heads, r = 32, fp8
# the dynamic tail engages from 64 units per CTA (about 19.5k tokens here):
# 20480 tokens in 80 requests, 3 layers and 4 KV heads (a cheap oracle)
BIG = dataclasses.replace(PREFILL, name="thin_20k_fp8", num_ctx=20480, requests=80, num_layers=3,
                          num_kv_heads=4)
BIG_BF16 = dataclasses.replace(BIG, name="thin_20k_bf16", kv_dtype=wk.KV_BF16)


@pytest.fixture(autouse=True)
def default_kernel(monkeypatch):
    monkeypatch.delenv("DSPARK_CTX_KV_KERNEL", raising=False)


def write_sched(inp, counter, layer_slots=None):
    """One call of the scheduled entry on fresh caches; returns the caches and
    the call's error word."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = inp.workload
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    fp8 = wl.kv_dtype == wk.KV_FP8
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8" if fp8 else "auto")
    w.ensure_tables()
    t = w.tables
    slots = None
    if layer_slots is not None:
        slots = [layer_slots[l].cuda() for l in range(wl.num_layers)]
        t.update_slots(slots)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    dk.dspark_ctx_kv_write_sched(
        d.all_kv, d.knorm_w, d.positions, d.slot_mapping if slots is None else None,
        t.layer_slots if slots is not None else None, wl.num_ctx, d.cos_sin, d.cos_sin.shape[0], caches[0],
        wl.num_blocks, t.cache_offsets, t.k_scales, t.v_scales, wl.num_layers, wl.num_kv_heads, wl.block_size,
        wl.rotary_dim, d.eps, "fp8" if fp8 else "auto", flags, counter)
    torch.cuda.synchronize()
    return caches, int(flags.item())


def check_parity(oracle_lib, inp, caches, layer_slots=None):
    fp8 = inp.workload.kv_dtype == wk.KV_FP8
    p = oracle_lib.problem_from_inputs(inp, layer_slots=None if layer_slots is None else layer_slots.numpy())
    ora = p.new_caches()
    alts = p.write(ora)
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


@pytest.mark.parametrize("wl", [BIG, BIG_BF16], ids=["fp8", "bf16"])
def test_two_calls_in_a_row_share_one_counter(oracle_lib, wl):
    counter = torch.zeros(2, dtype=torch.int64, device="cuda")
    for seed in (wl.seed, wl.seed + 1):
        inp = wk.generate(wl, seed=seed)
        caches, _ = write_sched(inp, counter)
        assert counter.tolist() == [0, 0]  # every call leaves it at zero
        check_parity(oracle_lib, inp, caches)


def test_per_layer_mappings_with_a_counter(oracle_lib):
    counter = torch.zeros(2, dtype=torch.int64, device="cuda")
    inp = wk.generate(BIG)
    ls = wk.layer_slot_mappings(inp, groups=3)
    caches, _ = write_sched(inp, counter, ls)
    assert counter.tolist() == [0, 0]
    check_parity(oracle_lib, inp, caches, ls)


def test_out_of_range_rows_are_skipped_and_flagged_with_a_counter(oracle_lib):
    # a slot past the caches and a position past the cos|sin table, both in
    # the last units (those handed out from the counter): not written, their
    # bits raised, every other row exact
    import speculative_decoding_draft_ctx_gb300 as dk

    inp = wk.generate(BIG)
    valid = (inp.slot_mapping >= 0).nonzero().flatten()
    bad_slot_t, bad_pos_t = int(valid[-3]), int(valid[-10])
    inp.slot_mapping[bad_slot_t] = BIG.capacity + 5
    inp.positions[bad_pos_t] = BIG.max_pos
    counter = torch.zeros(2, dtype=torch.int64, device="cuda")
    caches, flags = write_sched(inp, counter)
    assert flags == dk.FLAG_SLOT_RANGE | dk.FLAG_POS_RANGE
    assert counter.tolist() == [0, 0]
    ref = wk.generate(BIG)
    ref.slot_mapping[[bad_slot_t, bad_pos_t]] = -1
    check_parity(oracle_lib, ref, caches)


def test_a_dirty_counter_is_flagged_and_left_zero(oracle_lib):
    # a counter far from zero hands out no unit (nothing is read past the
    # tail), raises its flag, and is zero again after the call; the next call
    # on it is exact
    import speculative_decoding_draft_ctx_gb300 as dk

    inp = wk.generate(BIG)
    counter = torch.tensor([1 << 40, 0], dtype=torch.int64, device="cuda")
    _, flags = write_sched(inp, counter)
    assert flags == dk.FLAG_COUNTER
    assert counter.tolist() == [0, 0]
    caches, flags = write_sched(inp, counter)
    assert flags == 0
    check_parity(oracle_lib, inp, caches)


def test_null_counter_is_the_fixed_split(oracle_lib):
    inp = wk.generate(PREFILL)
    caches, _ = write_sched(inp, None)
    check_parity(oracle_lib, inp, caches)


def test_graph_replays_reuse_the_counter(oracle_lib):
    # captured once, replayed twice on the capture stream's counter (made by
    # an eager call there first): the second replay starts from the zero the
    # first one left
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = BIG
    inp = wk.generate(wl)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # the tables, and the capture stream's counter
        w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    torch.cuda.synchronize()
    assert side.cuda_stream in w._work
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for c in caches:
            c.fill_(wk.PREFILL_BYTE)
        g.replay()
        torch.cuda.synchronize()
        check_parity(oracle_lib, inp, caches)
    assert all(int(v) == 0 for c in w._work.values() for v in c.tolist())


def test_capture_on_a_new_stream_takes_the_fixed_split(oracle_lib):
    # no counter is made under capture: the captured write takes the fixed
    # split and is exact, and no counter exists for that stream afterwards
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = BIG
    inp = wk.generate(wl)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8")
    w.ensure_tables()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    assert side.cuda_stream not in w._work
    g.replay()
    torch.cuda.synchronize()
    check_parity(oracle_lib, inp, caches)
