"""Maximum sizes of the context-KV write (vLLM DSpark context-KV writer page,
module docstring), through the C ABI, against the oracle.

* all_kv above 2^31 elements (524,288 tokens of the long-context shape,
  5.4 GB): every kernel offset is 64-bit; rows of sampled tokens, the first
  and the last, against the oracle, and exactly the valid rows written;
* the widest layout the pipelined kernel stages (32 layers, 64 KV heads:
  one layer's K|V rows of a token fill its 32 KB stage) and the first ones
  past it (65 heads, 33 layers), which the generic kernel serves: whole
  caches against the oracle.
"""

import numpy as np
import pytest
import torch

import workloads as wk
from parity import compare_caches, compare_rows, gpu_write, oracle_full, to_numpy_caches

pytestmark = pytest.mark.gpu


def test_all_kv_above_two_to_the_31_elements(oracle_lib):
    import speculative_decoding_draft_ctx_gb300 as dk
    from parity import device_inputs

    T = 1 << 19
    wl = wk.WORKLOADS_BY_NAME["long_context"].with_(
        name="long_context_x8", num_ctx=T, slots="unique", pad_count=T // 50, num_blocks=T // 128,
        requests=0, tokens_per_request=0)
    L, H, D = wl.num_layers, wl.num_kv_heads, wl.head_dim
    assert T * L * 2 * H * D > 2**31
    inp = wk.generate(wl, with_all_kv=False)
    # K/V drawn on the device from a seeded generator (the same N(0, 1)
    # recipe); only the sampled tokens' rows are copied back for the oracle
    g = torch.Generator(device="cuda").manual_seed(wl.seed)
    all_kv = torch.randn((T, L, 2, H, D), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    d = device_inputs(inp)
    caches = wk.make_caches(wl, device="cuda")
    w = dk.ContextKVWriter(caches, d.extra["k_scales"], d.extra["v_scales"], "auto")
    w(all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping)
    torch.cuda.synchronize()

    rng = np.random.default_rng(11)
    toks = np.unique(np.concatenate([rng.choice(T, 256, replace=False), [0, T - 1]]))
    sub = wk.Inputs(wl.with_(num_ctx=len(toks)), all_kv[torch.from_numpy(toks).cuda()].cpu(), inp.knorm_w,
                    inp.positions[toks].contiguous(), inp.slot_mapping[toks].contiguous(), inp.cos_sin,
                    inp.k_scale, inp.v_scale, inp.eps)
    p = oracle_lib.problem_from_inputs(sub)
    ids = np.arange(len(toks) * L * H, dtype=np.int64)
    rows, (ar, ad, av) = p.rows(ids)
    dest = p.dest_rows(ids)
    keep = dest >= 0
    assert keep.sum() > 0
    for l in range(L):
        sel = keep & ((ids // H) % L == l)
        pos_of = {int(i): k for k, i in enumerate(np.nonzero(sel)[0])}
        idx = {}
        for r, dm, v in zip(ar.tolist(), ad.tolist(), av.tolist()):
            if r in pos_of:
                idx.setdefault((pos_of[r], dm), []).append(v)
        got = caches[l].view(-1, 2 * D)[torch.from_numpy(dest[sel]).cuda()].cpu()
        got = got.view(torch.int16).numpy().view(np.uint16)
        bad = compare_rows(got, rows[sel], idx, False)
        assert not bad, (l, len(bad), bad[:5])
    valid = int((inp.slot_mapping >= 0).sum())
    for c in caches:
        b = c.view(torch.uint8).view(-1, 4 * D)
        assert int((b != 0xFF).any(dim=1).sum()) == valid * H


@pytest.mark.parametrize("L,H,fp8", [(32, 64, False), (32, 64, True), (2, 65, True), (33, 2, False)],
                         ids=["32x64", "32x64_fp8", "65_heads", "33_layers"])
def test_widest_pipelined_layout_and_past_it(oracle_lib, L, H, fp8):
    wl = wk.Workload(name=f"wide_{L}x{H}", num_ctx=24, num_layers=L, num_kv_heads=H, rotary_dim=32,
                     block_size=8, num_blocks=8, max_pos=4096, rope_theta=1e6,
                     kv_dtype=wk.KV_FP8 if fp8 else wk.KV_BF16, slots="unique", pad_count=3, seed=31)
    inp = wk.generate(wl)
    caches, _, _ = gpu_write(inp)
    _, ora, alts = oracle_full(inp)
    problems = compare_caches(to_numpy_caches(caches, fp8), ora, alts, fp8)
    assert not problems, problems
