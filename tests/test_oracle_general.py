"""Pins of the oracle in the layouts only the general write takes: head dims
64 and 256, any even rotary dim up to the head dim, block sizes that are not
powers of two (vLLM DSpark context-KV writer page: the write of the module
docstring, in the layouts DSparkContextKVWriter._validate and
rotary_dims_supported send to the unfused path).

* position 0 (cos = 1, sin = 0 exactly): K' equals the hidden-state norm of
  the K row at width D (a separately pinned function) bit for bit, and V is
  copied at offset D of a 2D-element row -- catches a wrong n in the mean, a
  wrong weight row or a wrong K/V split;
* any position: the rotated dims agree with an exact 2 x 2 rotation of the
  normed row at angle pos * theta^(-2i/r) (fp64 trigonometry, not the bf16
  table) within the table's and the output's bf16 rounding, and dims >= r
  equal the normed row -- catches a wrong partner (d +- r/2 with r/2 odd or
  not a multiple of 8) or a wrong frequency index;
* placement: V rows tagged with exact small integers decode back to their
  (token, layer, head) at block slot // bs, offset slot % bs for block sizes
  1, 3, 48 and 100, and nothing else is written.
"""

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def layout(D, r, bs, T=24, L=2, H=3, fp8=False, nb=None):
    nb = nb or max(8, (T * 2) // bs + 2)
    return wk.Workload(name=f"d{D}_r{r}_bs{bs}", num_ctx=T, num_layers=L, num_kv_heads=H, rotary_dim=r,
                       head_dim=D, block_size=bs, num_blocks=nb, max_pos=4096, rope_theta=1e4,
                       kv_dtype=wk.KV_FP8 if fp8 else wk.KV_BF16, slots="unique", pad_count=3, seed=77)


LAYOUTS = [(64, 64, 16), (64, 18, 3), (64, 6, 1), (256, 64, 32), (256, 256, 48), (256, 50, 100),
           (128, 24, 16), (128, 128, 48), (128, 2, 7)]


@pytest.mark.parametrize("D,r,bs", LAYOUTS)
def test_position_zero_is_the_norm_at_width_d(oracle_lib, D, r, bs):
    wl = layout(D, r, bs)
    inp = wk.generate(wl)
    inp.positions.zero_()
    p = oracle_lib.problem_from_inputs(inp)
    ids = np.arange(wl.num_ctx * wl.num_layers * wl.num_kv_heads)
    rows, _ = p.rows(ids)
    assert rows.shape == (len(ids), 2 * D)
    kv = bits(inp.all_kv).reshape(wl.num_ctx, wl.num_layers, 2, wl.num_kv_heads, D)
    w = bits(inp.knorm_w).reshape(wl.num_layers, D)
    for i in ids:
        t, l, h = i // (wl.num_layers * wl.num_kv_heads), (i // wl.num_kv_heads) % wl.num_layers, i % wl.num_kv_heads
        y, _ = oracle_lib.gemma_norm_rows(kv[t, l, 0, h][None], w[l], inp.eps)
        assert np.array_equal(rows[i, :D], y[0]), (t, l, h)
        assert np.array_equal(rows[i, D:], kv[t, l, 1, h])


@pytest.mark.parametrize("D,r,bs", LAYOUTS)
def test_rotation_against_exact_trigonometry(oracle_lib, D, r, bs):
    wl = layout(D, r, bs)
    inp = wk.generate(wl)
    p = oracle_lib.problem_from_inputs(inp)
    ids = np.arange(wl.num_ctx * wl.num_layers * wl.num_kv_heads)
    rows, _ = p.rows(ids)
    kv = bits(inp.all_kv).reshape(wl.num_ctx, wl.num_layers, 2, wl.num_kv_heads, D)
    w = bits(inp.knorm_w).reshape(wl.num_layers, D)
    half = r // 2
    freq = np.array([wl.rope_theta ** (-2.0 * i / r) for i in range(half)])
    for i in ids:
        t, l, h = i // (wl.num_layers * wl.num_kv_heads), (i // wl.num_kv_heads) % wl.num_layers, i % wl.num_kv_heads
        y, _ = oracle_lib.gemma_norm_rows(kv[t, l, 0, h][None], w[l], inp.eps)
        yv = oracle_lib.bf16_values(y[0])
        got = oracle_lib.bf16_values(rows[i, :D])
        assert np.array_equal(rows[i, r:D], y[0, r:])  # pass-through dims
        ang = float(inp.positions[t]) * freq
        c, s = np.cos(ang), np.sin(ang)
        lo, hi = yv[:half], yv[half:r]
        exact = np.concatenate([lo * c - hi * s, hi * c + lo * s])
        bound = 2.0**-7 * np.concatenate([np.abs(lo) + np.abs(hi)] * 2) + 2.0**-133
        assert (np.abs(got[:r] - exact) <= bound).all(), (t, l, h, float(np.abs(got[:r] - exact).max()))


@pytest.mark.parametrize("D,bs", [(64, 1), (64, 3), (256, 48), (128, 100), (256, 7)])
def test_tagged_rows_decode_to_their_slot(oracle_lib, D, bs):
    wl = layout(D, 16, bs, T=40, L=3, H=2)
    inp = wk.generate(wl)
    T, L, H = wl.num_ctx, wl.num_layers, wl.num_kv_heads
    v = inp.all_kv[:, :, 1]
    tags = torch.zeros_like(v, dtype=torch.float32)
    tags[..., 0] = torch.arange(T, dtype=torch.float32)[:, None, None] + 1
    tags[..., 1] = torch.arange(L, dtype=torch.float32)[None, :, None] + 1
    tags[..., 2] = torch.arange(H, dtype=torch.float32)[None, None, :] + 1
    inp.all_kv[:, :, 1] = tags.to(torch.bfloat16)  # small integers: exact in bf16
    p = oracle_lib.problem_from_inputs(inp)
    caches = p.new_caches()
    p.write(caches)
    slots = inp.slot_mapping.numpy()
    for l in range(L):
        c = oracle_lib.bf16_values(caches[l])  # [nb, H, bs, 2D]
        written = ~(caches[l] == 0xFFFF).all(axis=3)
        assert written.sum() == int((slots >= 0).sum()) * H
        for b, h, o in zip(*np.nonzero(written)):
            t = int(c[b, h, o, D]) - 1
            assert int(c[b, h, o, D + 1]) - 1 == l and int(c[b, h, o, D + 2]) - 1 == h
            assert slots[t] == b * bs + o, (l, t, b, h, o)
            assert (c[b, h, o, D + 3:] == 0).all()


def test_general_layout_rules_of_the_oracle(oracle_lib):
    """The oracle accepts every even rotary dim up to the head dim and refuses
    an odd one or one beyond the head dim."""
    p = oracle_lib.problem_from_inputs(wk.generate(layout(64, 2, 16)))
    for r, ok in ((2, True), (64, True), (66, False), (7, False), (0, False)):
        p.c.rotary_dim = r  # the check reads only the sizes, not the table
        if ok:
            p.check()
        else:
            with pytest.raises(oracle_lib.OracleError):
                p.check()
