"""GPU parity of the write with one slot mapping per layer (DSpark draft
model page, _shared_slot_mapping: drafts whose layers span several KV-cache
groups) against the oracle, through the C ABI, on both kernels: whole caches
under the write's tolerance (tests/parity.py)."""

import numpy as np
import pytest
import torch

import workloads as wk
from parity import compare_caches, device_inputs, to_numpy_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["pipelined", "generic"])
def kernel(request, monkeypatch):
    if request.param == "generic":
        monkeypatch.setenv("DSPARK_CTX_KV_KERNEL", "generic")
    else:
        monkeypatch.delenv("DSPARK_CTX_KV_KERNEL", raising=False)
    return request.param


def run(inp, layer_slots, stream=None):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = inp.workload
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"],
                           "fp8" if wl.kv_dtype == wk.KV_FP8 else "auto")
    slots = [layer_slots[l].cuda() for l in range(wl.num_layers)]
    w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, slots, stream=stream)
    torch.cuda.synchronize()
    return caches, w


def parity(oracle_lib, inp, layer_slots):
    wl = inp.workload
    fp8 = wl.kv_dtype == wk.KV_FP8
    caches, _ = run(inp, layer_slots)
    p = oracle_lib.problem_from_inputs(inp, layer_slots=layer_slots.numpy())
    ora = p.new_caches()
    alts = p.write(ora)
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems


@pytest.mark.parametrize("idx,groups", [(1, 2), (2, 3), (1, 5)], ids=["draft2", "draft_fp8_3", "draft5"])
def test_layer_slots_draft_workloads(oracle_lib, kernel, idx, groups):
    inp = wk.generate(wk.WORKLOADS[idx])
    parity(oracle_lib, inp, wk.layer_slot_mappings(inp, groups=groups))


RAGGED = [
    # (T, L, H, r, bs, nb, kv, pad, groups)
    (7, 2, 3, 32, 2, 16, wk.KV_FP8, 2, 2),
    (37, 3, 5, 64, 4, 16, wk.KV_BF16, 5, 3),
    (100, 7, 9, 32, 256, 1, wk.KV_BF16, 11, 7),
    (257, 4, 8, 64, 64, 8, wk.KV_FP8, 1, 2),
    (50, 3, 64, 32, 16, 8, wk.KV_FP8, 5, 3),
]


@pytest.mark.parametrize("T,L,H,r,bs,nb,kv,pad,groups", RAGGED)
def test_layer_slots_ragged(oracle_lib, kernel, T, L, H, r, bs, nb, kv, pad, groups):
    wl = wk.Workload(name="ragged", num_ctx=T, num_layers=L, num_kv_heads=H, rotary_dim=r, block_size=bs,
                     num_blocks=nb, max_pos=3000, rope_theta=1e4, kv_dtype=kv, pad_count=pad,
                     kv_std=2.0 if kv == wk.KV_FP8 else 1.0, seed=T * 17 + H)
    inp = wk.generate(wl)
    parity(oracle_lib, inp, wk.layer_slot_mappings(inp, groups=groups))


def test_layer_slots_prefill_full_size(oracle_lib, kernel):
    inp = wk.generate(wk.WORKLOADS[3])
    parity(oracle_lib, inp, wk.layer_slot_mappings(inp, groups=2))


def test_one_tensor_repeated_is_the_shared_write(oracle_lib):
    inp = wk.generate(wk.WORKLOADS[1])
    L = inp.workload.num_layers
    from parity import gpu_write

    shared, _, _ = gpu_write(inp)
    import speculative_decoding_draft_ctx_gb300 as dk

    d = device_inputs(inp)
    caches = wk.make_caches(inp.workload, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "auto")
    w(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, inp.workload.rotary_dim, [d.slot_mapping] * L)
    torch.cuda.synchronize()
    for a, b in zip(shared, caches):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))  # the 0xFF prefill is NaN in bf16


def test_layer_slots_in_a_cuda_graph(oracle_lib):
    """Tables built before capture; the captured call replays on new values
    copied into the same buffers."""
    import speculative_decoding_draft_ctx_gb300 as dk

    inp = wk.generate(wk.WORKLOADS[2])
    wl = inp.workload
    ls = wk.layer_slot_mappings(inp, groups=2)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8")
    slots = [ls[l].cuda() for l in range(wl.num_layers)]
    kv = d.all_kv.clone()
    w(kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, slots)  # builds the tables
    builds = w.tables.builds
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w(kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, slots)
    torch.cuda.synchronize()
    assert w.tables.builds == builds
    other = wk.generate(wl, seed=wl.seed + 5)
    kv.copy_(other.all_kv.cuda())
    for c in caches:
        c.fill_(0xFF)
    g.replay()
    torch.cuda.synchronize()
    ref_inp = wk.Inputs(wl, other.all_kv, inp.knorm_w, inp.positions, inp.slot_mapping, inp.cos_sin, inp.k_scale,
                        inp.v_scale, inp.eps)
    p = oracle_lib.problem_from_inputs(ref_inp, layer_slots=ls.numpy())
    ora = p.new_caches()
    alts = p.write(ora)
    problems = compare_caches(to_numpy_caches(caches, True), ora, alts, True)
    assert not problems, problems
