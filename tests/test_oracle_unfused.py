"""The oracle against an independent composition of the unfused pipeline.

The vLLM DSpark context-KV writer page (module docstring) says the fused write
replaces: a permute copy of the projection output, per-layer K-norm launches
followed by a stack, ``positions.repeat``, ``rotary_embedding`` and per-layer
``reshape_and_cache_flash`` calls.  This test builds that pipeline from plain
torch CPU ops (fp32 arithmetic, bf16 between stages, exactly as the unfused
path materialises it) and checks that the oracle's caches agree: placement,
padding and the bf16 V copy byte for byte, K within one bf16 ulp of an
admissible oracle value, fp8 codes within one code.  The same holds in the
layouts only the general write takes (head dims 64 and 256, rotary dims
other than 16 / 32 / 64, block sizes that are not powers of two).
"""

import numpy as np
import pytest
import torch

import workloads as wk


def unfused_write(inp: wk.Inputs):
    wl = inp.workload
    T, L, H, r, D = wl.num_ctx, wl.num_layers, wl.num_kv_heads, wl.rotary_dim, wl.head_dim
    half = r // 2
    # permute copy: [T, L, 2, H, D] -> per layer [T, H, D]
    all_k = inp.all_kv[:, :, 0].permute(1, 0, 2, 3).contiguous()
    all_v = inp.all_kv[:, :, 1].permute(1, 0, 2, 3).contiguous()
    # per-layer Gemma K-norm in fp32, materialised to bf16, then stacked
    normed = []
    for l in range(L):
        k = all_k[l].float()
        inv = torch.rsqrt(k.pow(2).mean(-1, keepdim=True) + inp.eps)
        normed.append((k * inv * (1.0 + inp.knorm_w[l].float())).to(torch.bfloat16))
    all_k = torch.stack(normed)
    # positions.repeat + NeoX rotary on the first r dims
    pos = inp.positions.repeat(L).view(L, T)
    cs = inp.cos_sin[pos.clamp(0, wl.max_pos - 1)].float()  # [L, T, r]
    cos, sin = cs[..., :half].unsqueeze(2), cs[..., half:].unsqueeze(2)
    x = all_k.float()
    x1, x2 = x[..., :half], x[..., half:r]
    rot = torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1).to(torch.bfloat16)
    all_k = torch.cat([rot, all_k[..., r:]], dim=-1)
    # per-layer reshape_and_cache_flash: [num_blocks, H, bs, 2D], K | V
    caches = wk.make_caches(wl)
    slots = inp.slot_mapping
    valid = (slots >= 0).nonzero().flatten()
    blk, off = slots[valid] // wl.block_size, slots[valid] % wl.block_size
    for l in range(L):
        kk, vv = all_k[l][valid], all_v[l][valid]
        if wl.kv_dtype == wk.KV_FP8:
            kk = (kk.float() / inp.k_scale[l]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            vv = (vv.float() / inp.v_scale[l]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        for h in range(H):
            caches[l][blk, h, off, :D] = kk[:, h]
            caches[l][blk, h, off, D:] = vv[:, h]
    return caches


def ordered(a: np.ndarray, fp8: bool) -> np.ndarray:
    a = a.astype(np.int64)
    sign = 0x80 if fp8 else 0x8000
    mag = a & (sign - 1)
    return np.where(a & sign, -mag, mag)


def small(wl: wk.Workload) -> wk.Workload:
    """96 tokens of a workload, or (blocktable slots) 2 requests of 48."""
    if wl.slots == "blocktable":
        return wl.with_(num_ctx=96, requests=2, tokens_per_request=48, pad_count=7)
    return wl.with_(num_ctx=96, pad_count=7)


CASES = [wk.WORKLOADS[0], small(wk.WORKLOADS[1]), small(wk.WORKLOADS[2])] + \
    [small(w) for w in wk.GENERAL_WORKLOADS] + \
    [small(wk.GENERAL_WORKLOADS[0]).with_(rotary_dim=18, block_size=3, num_blocks=64, blocks_per_request=16,
                                         name="head64_rot18_bs3"),
     small(wk.GENERAL_WORKLOADS[1]).with_(rotary_dim=256, block_size=5, num_blocks=64, blocks_per_request=10,
                                         name="head256_rot256_bs5")]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_oracle_equals_unfused_pipeline(oracle_lib, wl):
    D = wl.head_dim
    inp = wk.generate(wl)
    ref = unfused_write(inp)
    p = oracle_lib.problem_from_inputs(inp)
    caches = p.new_caches()
    al, ae, av = p.write(caches)
    fp8 = wl.kv_dtype == wk.KV_FP8
    for l in range(wl.num_layers):
        o = caches[l].reshape(-1, 2 * D)
        u = ref[l].view(torch.uint8 if fp8 else torch.int16).numpy().reshape(-1, 2 * D)
        u = u.view(np.uint8 if fp8 else np.uint16)
        # rows each side wrote (everything else is prefill on both sides)
        fill = 0xFF if fp8 else 0xFFFF
        ow = ~(o == fill).all(axis=1)
        uw = ~(u == fill).all(axis=1)
        assert np.array_equal(ow, uw)
        assert ow.sum() == inp.num_valid_tokens * wl.num_kv_heads
        if fp8:
            assert (np.abs(ordered(o[ow], True) - ordered(u[uw], True)) <= 1).all()
        else:
            assert np.array_equal(o[ow, D:], u[uw, D:])  # V bit-exact
            d = np.abs(ordered(o[ow, :D], False) - ordered(u[uw, :D], False))
            bad = np.argwhere(d > 1)
            rows_w = np.nonzero(ow)[0]
            for br, bc in bad:
                el = rows_w[br] * 2 * D + bc
                alts = av[(al == l) & (ae == el)]
                assert any(abs(int(ordered(np.array([a]), False)[0]) - int(ordered(u[rows_w[br], bc:bc + 1], False)[0])) <= 1
                           for a in alts), (l, br, bc)
