"""GPU parity of the draft-token fused QK-norm / RoPE / KV insert (DSpark
draft model page, dspark_qknorm_rope_kv_insert) against the CPU oracle on
the same seeded inputs, element by element, through the C ABI.

Every output is compared whole: the in-place qkv (query and key heads within
1 bf16 ulp of the oracle or of an admissible alternate, value heads
bit-exact), the fp8 query output (within 1 e4m3 code) and the whole cache
(unaddressed bytes keep the 0xFF prefill; bf16 V bit-exact, K within 1 ulp;
fp8 within 1 code).
"""

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.gpu

BF16_ULPS = 1
FP8_CODES = 1


def ordered(a: np.ndarray, sign: int) -> np.ndarray:
    a = a.astype(np.int64)
    mag = a & (sign - 1)
    return np.where(a & sign, -mag, mag)


def u16(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def mismatches(gpu: np.ndarray, ora: np.ndarray, tol: int, sign: int, alts: dict, exact=None) -> list:
    """Flat elements where gpu is more than ``tol`` codes from the oracle and
    from every admissible alternate; ``exact`` marks elements that must match
    bit for bit."""
    g, o = gpu.reshape(-1), ora.reshape(-1)
    d = np.abs(ordered(g, sign) - ordered(o, sign))
    bad = d > tol
    if exact is not None:
        ex = exact.reshape(-1)
        bad = np.where(ex, g != o, bad)
    out = []
    for e in np.nonzero(bad)[0]:
        if exact is not None and exact.reshape(-1)[e]:
            out.append((int(e), int(g[e]), int(o[e])))
            continue
        cand = alts.get(int(e), ())
        if any(abs(int(ordered(np.array([a]), sign)[0]) - int(ordered(g[e:e + 1], sign)[0])) <= tol for a in cand):
            continue
        out.append((int(e), int(g[e]), int(o[e])))
    return out


def alt_maps(alts, oracle_lib):
    aw, ae, av = alts
    maps = {oracle_lib.ALT_QKV: {}, oracle_lib.ALT_QFP8: {}, oracle_lib.ALT_CACHE: {}}
    for w, e, v in zip(aw.tolist(), ae.tolist(), av.tolist()):
        maps[w].setdefault(e, []).append(v)
    return maps


def run_gpu(inp: wk.QkInputs, insert=True, q_fp8=None, error_flags=None, cache=None):
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = inp.workload
    d = inp.to("cuda")
    q_fp8 = wl.q_fp8 if q_fp8 is None else q_fp8
    qf = torch.full((wl.num_tokens, wl.num_heads * 128), 0xFF, dtype=torch.uint8, device="cuda") if q_fp8 else None
    if cache is None and insert:
        cache = wk.make_qk_cache(wl, device="cuda")
    ks = torch.tensor([inp.k_scale], dtype=torch.float32, device="cuda")
    vs = torch.tensor([inp.v_scale], dtype=torch.float32, device="cuda")
    dk.qknorm_rope_kv_insert(d.qkv, d.q_norm_w, d.k_norm_w, d.cos_sin, d.positions, wl.num_heads,
                             wl.num_kv_heads, wl.rotary_dim, inp.eps,
                             slot_mapping=d.slot_mapping if insert else None, kv_cache=cache if insert else None,
                             k_scale=ks, v_scale=vs, q_fp8_out=qf, q_fp8_scale=inp.q_scale,
                             error_flags=error_flags)
    torch.cuda.synchronize()
    return d.qkv, qf, cache


def check_parity(oracle_lib, inp: wk.QkInputs, insert=True):
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    fp8 = wl.kv_dtype == wk.KV_FP8
    qkv, qf, cache = run_gpu(inp, insert=insert)
    p = oracle_lib.qk_problem_from_inputs(inp)
    oc = p.new_cache() if insert else None
    o_qkv, o_qf, alts = p.run(cache=oc, q_fp8=wl.q_fp8)
    maps = alt_maps(alts, oracle_lib)
    # in-place qkv: value heads exact, query and key heads within 1 ulp
    exact = np.zeros((T, Hq + 2 * Hkv, 128), bool)
    exact[:, Hq + Hkv:] = True
    bad = mismatches(u16(qkv), o_qkv, BF16_ULPS, 0x8000, maps[oracle_lib.ALT_QKV], exact)
    assert not bad, ("qkv", len(bad), bad[:5])
    if wl.q_fp8:
        bad = mismatches(qf.cpu().numpy(), o_qf, FP8_CODES, 0x80, maps[oracle_lib.ALT_QFP8])
        assert not bad, ("q_fp8", len(bad), bad[:5])
    if insert:
        g = cache.cpu()
        g = g.numpy() if fp8 else u16(g)
        fill = 0xFF if fp8 else 0xFFFF
        gr, orr = g.reshape(-1, 256), oc.reshape(-1, 256)
        unwritten = (orr == fill).all(axis=1)
        assert np.array_equal(gr[unwritten], orr[unwritten]), "unaddressed cache rows changed"
        assert (~unwritten).sum() == inp.num_valid_tokens * Hkv
        ex = np.zeros_like(gr, bool)
        if not fp8:
            ex[:, 128:] = True  # a bf16 V row is a copy
        bad = mismatches(gr, orr, FP8_CODES if fp8 else BF16_ULPS, 0x80 if fp8 else 0x8000,
                         maps[oracle_lib.ALT_CACHE], ex)
        assert not bad, ("cache", len(bad), bad[:5])


@pytest.mark.parametrize("name", ["qk_tiny", "qk_draft", "qk_draft_fp8"])
def test_qk_insert_parity_workloads(oracle_lib, name):
    check_parity(oracle_lib, wk.generate_qk(wk.QK_WORKLOADS_BY_NAME[name]))


RAGGED = [
    # (requests, Hq, Hkv, r, bs, nb, kv, q_fp8, pad)
    (1, 1, 1, 16, 1, 8, wk.KV_BF16, False, 0),      # W = 3: odd head count, half a warp idle
    (2, 3, 1, 32, 2, 16, wk.KV_FP8, True, 3),
    (5, 5, 2, 64, 4, 16, wk.KV_BF16, True, 1),
    (9, 6, 3, 16, 8, 24, wk.KV_FP8, False, 9),
    (13, 32, 4, 32, 256, 32, wk.KV_BF16, True, 2),
    (37, 16, 16, 64, 16, 80, wk.KV_FP8, True, 30),
    (3, 40, 1, 64, 64, 8, wk.KV_FP8, True, 21),      # every token padded: nothing inserted
]


@pytest.mark.parametrize("R,Hq,Hkv,r,bs,nb,kv,qf,pad", RAGGED)
def test_qk_insert_parity_ragged(oracle_lib, R, Hq, Hkv, r, bs, nb, kv, qf, pad):
    wl = wk.QkWorkload(name="ragged", requests=R, num_heads=Hq, num_kv_heads=Hkv, rotary_dim=r, block_size=bs,
                       num_blocks=nb, max_pos=2000, rope_theta=1e4, kv_dtype=kv, q_fp8=qf,
                       x_std=2.0 if kv == wk.KV_FP8 else 1.0, outlier_frac=0.01 if kv == wk.KV_FP8 else 0.0,
                       outlier_mult=10.0, pad_count=pad, seed=R * 131 + Hq)
    check_parity(oracle_lib, wk.generate_qk(wl))


def test_qk_without_insert(oracle_lib):
    check_parity(oracle_lib, wk.generate_qk(wk.QK_WORKLOADS_BY_NAME["qk_draft_fp8"]), insert=False)


def test_qk_out_of_range_rows_are_reported(oracle_lib):
    wl = wk.QK_WORKLOADS_BY_NAME["qk_draft"].with_(requests=3, pad_count=0)
    inp = wk.generate_qk(wl)
    src = inp.qkv.clone()
    bad_pos, bad_slot = 2, 5
    inp.positions[bad_pos] = wl.max_pos       # outside the cos|sin table: token untouched
    inp.slot_mapping[bad_slot] = wl.capacity  # beyond the cache: rotated, not inserted
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv, _, cache = run_gpu(inp, error_flags=flags)
    import speculative_decoding_draft_ctx_gb300 as dk

    assert int(flags.item()) == dk.FLAG_POS_RANGE | dk.FLAG_SLOT_RANGE
    g = qkv.cpu()
    assert torch.equal(g[bad_pos], src[bad_pos])
    assert not torch.equal(g[bad_slot], src[bad_slot])
    rows = u16(cache.cpu()).reshape(-1, 256)
    written = (~(rows == 0xFFFF).all(axis=1)).sum()
    assert written == (wl.num_tokens - 2) * wl.num_kv_heads
    # every other token matches the oracle (run on the unmodified inputs)
    o_qkv, _, alts = oracle_lib.qk_problem_from_inputs(wk.generate_qk(wl)).run()
    gg = u16(g).copy()
    gg[[bad_pos, bad_slot]] = o_qkv[[bad_pos, bad_slot]]
    exact = np.zeros((wl.num_tokens, wl.num_heads + 2 * wl.num_kv_heads, 128), bool)
    exact[:, wl.num_heads + wl.num_kv_heads:] = True
    bad = mismatches(gg, o_qkv, BF16_ULPS, 0x8000, alt_maps(alts, oracle_lib)[oracle_lib.ALT_QKV], exact)
    assert not bad, bad[:5]


def test_qk_insert_in_a_cuda_graph(oracle_lib):
    """Captured once, replayed on new inputs copied into the same buffers."""
    import speculative_decoding_draft_ctx_gb300 as dk

    wl = wk.QK_WORKLOADS_BY_NAME["qk_draft_fp8"]
    a, b = wk.generate_qk(wl), wk.generate_qk(wl, seed=wl.seed + 7)
    d = a.to("cuda")
    cache = wk.make_qk_cache(wl, device="cuda")
    qf = torch.zeros((wl.num_tokens, wl.num_heads * 128), dtype=torch.uint8, device="cuda")
    ks = torch.tensor([a.k_scale], dtype=torch.float32, device="cuda")
    vs = torch.tensor([a.v_scale], dtype=torch.float32, device="cuda")
    qkv = torch.empty_like(d.qkv)

    def call():
        dk.qknorm_rope_kv_insert(qkv, d.q_norm_w, d.k_norm_w, d.cos_sin, d.positions, wl.num_heads,
                                 wl.num_kv_heads, wl.rotary_dim, a.eps, slot_mapping=d.slot_mapping,
                                 kv_cache=cache, k_scale=ks, v_scale=vs, q_fp8_out=qf, q_fp8_scale=a.q_scale)

    qkv.copy_(d.qkv)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.synchronize()
    # replay on b's qkv (same positions and slots: b differs in values only)
    qkv.copy_(b.qkv.cuda())
    cache.view(torch.uint8).fill_(0xFF)
    g.replay()
    torch.cuda.synchronize()
    ref_qkv, ref_qf, ref_cache = run_gpu(wk.QkInputs(wl, b.qkv, a.q_norm_w, a.k_norm_w, a.positions,
                                                     a.slot_mapping, a.cos_sin, a.k_scale, a.v_scale,
                                                     a.q_scale, a.eps))
    assert torch.equal(qkv, ref_qkv)
    assert torch.equal(qf, ref_qf)
    assert torch.equal(cache, ref_cache)
