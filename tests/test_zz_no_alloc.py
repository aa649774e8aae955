"""The no-allocation write (dspark_ctx_kv_write_noalloc: tables from host
memory into the library's fixed device array) against the existing entry
point (dspark_ctx_kv_write_sched with the tables object's device tables and
a caller-owned counter): two calls in a row, issued back to back on one
stream, each byte-identical to the existing entry's caches and error word.
Collected last so that it also runs after every other GPU test."""

import dataclasses

import pytest
import torch

import workloads as wk
from parity import device_inputs

pytestmark = pytest.mark.gpu

PREFILL = wk.WORKLOADS[3]
# past the dynamic tail's threshold (64 units per CTA): 20480 tokens
BIG = dataclasses.replace(PREFILL, name="thin_20k_fp8", num_ctx=20480, requests=80, num_layers=3, num_kv_heads=4)
BIG_BF16 = dataclasses.replace(BIG, name="thin_20k_bf16", kv_dtype=wk.KV_BF16)
DRAFT = wk.WORKLOADS[1]  # 512 tokens: the warp-private kernel


@pytest.fixture(autouse=True)
def default_kernel(monkeypatch):
    monkeypatch.delenv("DSPARK_CTX_KV_KERNEL", raising=False)


class Call:
    """One call's device inputs, its caches and error word, and (per-layer
    mappings) its slot tensors."""

    def __init__(self, wl, seed, groups):
        inp = wk.generate(wl, seed=seed)
        self.wl = wl
        self.d = device_inputs(inp)
        self.fp8 = wl.kv_dtype == wk.KV_FP8
        self.slots = None
        if groups:
            ls = wk.layer_slot_mappings(inp, groups=groups)
            self.slots = [ls[l].cuda() for l in range(wl.num_layers)]

    def fresh(self):
        return wk.make_caches(self.wl, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")

    def args(self):
        wl, d = self.wl, self.d
        return dict(num_ctx=wl.num_ctx, cos_sin=d.cos_sin, max_pos=d.cos_sin.shape[0], num_blocks=wl.num_blocks,
                    L=wl.num_layers, nkv=wl.num_kv_heads, block_size=wl.block_size, rotary_dim=wl.rotary_dim,
                    eps=d.eps, kv_dtype="fp8" if self.fp8 else "auto")

    def existing(self):
        """dspark_ctx_kv_write_sched through the tables object."""
        import speculative_decoding_draft_ctx_gb300 as dk

        caches, flags = self.fresh()
        d = self.d
        w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "fp8" if self.fp8 else "auto")
        w.ensure_tables()
        t = w.tables
        if self.slots is not None:
            t.update_slots(self.slots)
        counter = torch.zeros(2, dtype=torch.int64, device="cuda")
        dk.dspark_ctx_kv_write_sched(
            d.all_kv, d.knorm_w, d.positions, d.slot_mapping if self.slots is None else None,
            t.layer_slots if self.slots is not None else None, layer0_cache=caches[0],
            cache_offsets=t.cache_offsets, k_scales=t.k_scales, v_scales=t.v_scales, error_flags=flags,
            work_counter=counter, **self.args())
        torch.cuda.synchronize()
        return caches, flags

    def no_alloc(self, caches, flags):
        """dspark_ctx_kv_write_noalloc into ``caches``, enqueued (no
        synchronisation)."""
        import speculative_decoding_draft_ctx_gb300 as dk

        d = self.d
        offs = [(c.data_ptr() - caches[0].data_ptr()) // c.element_size() for c in caches]
        dk.dspark_ctx_kv_write_noalloc(
            d.all_kv, d.knorm_w, d.positions, d.slot_mapping if self.slots is None else None, self.slots,
            layer0_cache=caches[0], cache_offsets=offs,
            k_scales=d.extra["k_scales"] if self.fp8 else None, v_scales=d.extra["v_scales"] if self.fp8 else None,
            error_flags=flags, **self.args())
        return caches, flags


def same(a, b):
    ca, fa = a
    cb, fb = b
    assert int(fa.item()) == int(fb.item())
    for l, (x, y) in enumerate(zip(ca, cb)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), f"layer {l} differs"


@pytest.mark.parametrize("wl,groups", [(BIG, 0), (BIG_BF16, 0), (BIG, 3), (DRAFT, 0)],
                         ids=["dynamic_tail_fp8", "dynamic_tail_bf16", "per_layer_fp8", "draft_step"])
def test_two_calls_in_a_row_match_the_existing_entry(wl, groups):
    first, second = Call(wl, wl.seed, groups), Call(wl, wl.seed + 1, groups)
    want = [first.existing(), second.existing()]
    bufs = [first.fresh(), second.fresh()]
    torch.cuda.synchronize()
    # back to back on the current stream: the second call's table copy waits
    # for the first launch, which still reads the array
    got = [first.no_alloc(*bufs[0]), second.no_alloc(*bufs[1])]
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        same(g, w)
