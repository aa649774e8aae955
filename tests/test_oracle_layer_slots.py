"""Pins of the oracle's per-layer slot mappings (DSpark draft model page,
_shared_slot_mapping: drafts whose layers span several KV-cache groups have
no shared mapping; the context-KV writer page writes each layer's K|V rows
at that layer's slots).  The shared-mapping write is pinned on its own
(test_oracle_pins.py); here a per-layer write must equal, layer by layer,
the shared write run with that layer's mapping."""

import numpy as np
import pytest

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def small(idx):
    wl = wk.WORKLOADS[idx]
    return wl if idx == 0 else wl.with_(num_ctx=96, pad_count=7)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_same_mapping_everywhere_is_the_shared_write(oracle_lib, idx):
    inp = wk.generate(small(idx))
    L = inp.workload.num_layers
    ref = oracle_lib.problem_from_inputs(inp)
    rc = ref.new_caches()
    ref.write(rc)
    p = oracle_lib.problem_from_inputs(inp, layer_slots=np.tile(inp.slot_mapping.numpy(), (L, 1)))
    pc = p.new_caches()
    p.write(pc)
    for a, b in zip(rc, pc):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("idx,groups", [(1, 2), (2, 3), (1, 5)])
def test_each_layer_equals_the_shared_write_with_its_mapping(oracle_lib, idx, groups):
    inp = wk.generate(small(idx))
    ls = wk.layer_slot_mappings(inp, groups=groups)
    L = inp.workload.num_layers
    p = oracle_lib.problem_from_inputs(inp, layer_slots=ls.numpy())
    pc = p.new_caches()
    p.write(pc)
    assert len({tuple(ls[l].tolist()) for l in range(L)}) == groups
    for l in range(L):
        inp_l = wk.Inputs(inp.workload, inp.all_kv, inp.knorm_w, inp.positions, ls[l].clone(), inp.cos_sin,
                          inp.k_scale, inp.v_scale, inp.eps)
        ref = oracle_lib.problem_from_inputs(inp_l)
        rc = ref.new_caches()
        ref.write(rc)
        assert np.array_equal(pc[l], rc[l]), l


def test_duplicates_are_per_layer(oracle_lib):
    inp = wk.generate(small(1))
    ls = wk.layer_slot_mappings(inp, groups=2).numpy().copy()
    L = inp.workload.num_layers
    # the same slot in two different layers' caches is fine
    v0 = np.nonzero(ls[0] >= 0)[0][0]
    ls[L - 1, np.nonzero(ls[L - 1] >= 0)[0][0]] = ls[0, v0]
    p = oracle_lib.problem_from_inputs(inp, layer_slots=ls)
    p.write(p.new_caches())
    # twice in one layer is refused
    ls2 = ls.copy()
    valid = np.nonzero(ls2[L - 1] >= 0)[0]
    ls2[L - 1, valid[1]] = ls2[L - 1, valid[0]]
    p = oracle_lib.problem_from_inputs(inp, layer_slots=ls2)
    with pytest.raises(oracle_lib.OracleError, match="duplicate"):
        p.write(p.new_caches())


@pytest.mark.parametrize("nthreads", [1, 3, 7])
def test_threaded_oracle_write_equals_the_single_threaded_one(oracle_lib, nthreads):
    """The timing helper that splits the write over host threads by token
    ranges writes the same caches byte for byte."""
    inp = wk.generate(wk.WORKLOADS[2].with_(num_ctx=101, pad_count=5))
    p = oracle_lib.problem_from_inputs(inp)
    a = p.new_caches()
    p.write(a)
    b = p.new_caches()
    p.write_threads(b, nthreads)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
