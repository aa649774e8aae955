"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one step of the oracle to something other than the oracle
itself: a closed form, an invariant, brute force over a finite code space, or
a special case where a library routine computes the same thing.  Each is
chosen so that a plausible mistake (a dropped term, a wrong sign, a wrong
index or denominator, a transposed operand) fails it.

Sources: vLLM DSpark context-KV writer page (module docstring: layout,
Gemma RMSNorm, partial NeoX RoPE, fp8 of x/scale, slots < 0 not written;
``rotary_dims_supported``), DSpark draft model page
(``precompute_and_store_context_kv``, ``_gemma_rms_norm``).
"""

import math
import struct

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bf16_of_f32(x: float) -> int:
    """torch's fp32 -> bf16 conversion (round to nearest even)."""
    t = torch.tensor([x], dtype=torch.float32).to(torch.bfloat16)
    return int(t.view(torch.int16).item()) & 0xFFFF


def bf16_bits_of(values) -> np.ndarray:
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def ordered(bits: np.ndarray, sign_bit: int) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & (sign_bit - 1)
    return np.where(b & sign_bit, -mag, mag)


# ------------------------------------------------------------------ bf16

def test_bf16_decode_matches_torch_on_every_code(oracle_lib):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle_lib.bf16_decode(int(c)) for c in codes[::7]])
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], r[~nan])


def test_bf16_rne_matches_torch_on_fp32_values(oracle_lib):
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(3000).astype(np.float32))
    vals += list((rng.standard_normal(500) * 1e-38).astype(np.float32))  # subnormal range
    vals += list((rng.standard_normal(500) * 1e30).astype(np.float32))
    # exact midpoints between neighbouring bf16 values: ties go to the even code
    for b in rng.integers(0, 0x7F00, 1000):
        lo = struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]
        mid_bits = (int(b) << 16) | 0x8000
        vals.append(np.float32(struct.unpack("<f", struct.pack("<I", mid_bits))[0]))
        vals.append(np.float32(-lo))
    for v in vals:
        assert oracle_lib.bf16_rne(float(v)) == bf16_of_f32(float(v)), v


def test_bf16_rne_rounds_once_from_fp64(oracle_lib):
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: just above it must round
    # up, just below it down, exactly on it to the even code (1.0).
    assert oracle_lib.bf16_rne(1 + 2**-8 + 2**-30) == 0x3F81
    assert oracle_lib.bf16_rne(1 + 2**-8 - 2**-30) == 0x3F80
    assert oracle_lib.bf16_rne(1 + 2**-8) == 0x3F80
    assert oracle_lib.bf16_rne(1 + 3 * 2**-8) == 0x3F82  # tie between 0x3F81 and 0x3F82 -> even
    assert oracle_lib.bf16_rne(-0.0) == 0x8000
    assert oracle_lib.bf16_rne(1e39) == 0x7F80


# ------------------------------------------------------------------ e4m3

def e4m3_value_from_definition(c: int) -> float:
    s = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * m * 2.0**-9
    return s * (8 + m) * 2.0 ** (e - 10)


def test_e4m3_decode_every_code(oracle_lib):
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle_lib.e4m3_decode(c)
        want = e4m3_value_from_definition(c)
        if math.isnan(want):
            assert math.isnan(got) and math.isnan(ref[c])
        else:
            assert got == want == ref[c], c
    assert oracle_lib.e4m3_decode(0x7E) == 448.0
    assert oracle_lib.e4m3_decode(0x01) == 2.0**-9


def test_e4m3_encode_round_trips_every_finite_code(oracle_lib):
    for c in range(256):
        v = e4m3_value_from_definition(c)
        if math.isnan(v):
            continue
        assert oracle_lib.e4m3_rne_sat(v) == c, hex(c)


def test_e4m3_midpoints_round_to_even(oracle_lib):
    pos = [c for c in range(0x7F)]  # 0x00 .. 0x7E, increasing values
    for a, b in zip(pos[:-1], pos[1:]):
        va, vb = e4m3_value_from_definition(a), e4m3_value_from_definition(b)
        mid = (va + vb) / 2
        even = a if a % 2 == 0 else b
        assert oracle_lib.e4m3_rne_sat(mid) == even, (hex(a), hex(b))
        assert oracle_lib.e4m3_rne_sat(-mid) == even | 0x80
        # a hair off the midpoint goes to the nearer code
        assert oracle_lib.e4m3_rne_sat(np.nextafter(np.float32(mid), np.float32(0))) == a
        assert oracle_lib.e4m3_rne_sat(np.nextafter(np.float32(mid), np.float32(1e9))) == b


def test_e4m3_saturates_and_keeps_nan(oracle_lib):
    for v in [448.0, 448.1, 464.0, 479.9, 480.0, 1e6, 3e38, math.inf]:
        assert oracle_lib.e4m3_rne_sat(v) == 0x7E
        assert oracle_lib.e4m3_rne_sat(-v) == 0xFE
    assert oracle_lib.e4m3_rne_sat(math.nan) & 0x7F == 0x7F
    assert oracle_lib.e4m3_rne_sat(0.0) == 0x00
    assert oracle_lib.e4m3_rne_sat(-0.0) == 0x80
    assert oracle_lib.e4m3_rne_sat(2.0**-10) == 0x00  # tie between 0 and 2^-9 -> even
    assert oracle_lib.e4m3_rne_sat(3 * 2.0**-10) == 0x02
    assert oracle_lib.e4m3_rne_sat(2.0) == 0x40


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(3000),
                           rng.standard_normal(1000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3_rne_sat(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ Gemma K-norm

def test_knorm_unit_rms_when_w_is_zero(oracle_lib):
    rng = np.random.default_rng(3)
    for scale in [1.0, 3.0, 0.25]:
        k = bf16_bits_of(rng.standard_normal(128) * scale)
        y, ya, _ = oracle_lib.gemma_knorm(k, np.zeros(128, np.uint16), 1e-6)
        yv = np.array([oracle_lib.bf16_decode(int(b)) for b in y])
        rms = math.sqrt(float(np.mean(yv**2)))
        assert abs(rms - 1.0) < 2e-3  # bf16 rounding of each element, eps ~1e-6


def test_knorm_constant_row_closed_form(oracle_lib):
    # mean(k^2) = a^2, so y_d = a / sqrt(a^2 + eps) * (1 + w_d); each w_d distinct
    w_vals = np.linspace(-0.5, 0.5, 128)
    w = bf16_bits_of(w_vals)
    wv = np.array([oracle_lib.bf16_decode(int(b)) for b in w])
    for a, eps in [(1.0, 1e-6), (-2.0, 1e-6), (0.01, 1e-3), (1e-3, 1e-6)]:
        k = bf16_bits_of(np.full(128, a))
        av = oracle_lib.bf16_decode(int(k[0]))
        eps32 = float(np.float32(eps))
        y, ya, _ = oracle_lib.gemma_knorm(k, w, eps)
        for d in range(128):
            exact = av / math.sqrt(av * av + eps32) * (1.0 + wv[d])
            assert y[d] == oracle_lib.bf16_rne(exact) or ya[d] == oracle_lib.bf16_rne(exact)
            got = oracle_lib.bf16_decode(int(y[d]))
            assert abs(got - exact) <= abs(exact) * 2**-8


def test_knorm_one_hot_row_uses_head_dim_128(oracle_lib):
    # k = a e_j: mean(k^2) = a^2/128, so y_j = sqrt(128) (1 + w_j), others 0
    w_vals = np.linspace(-0.3, 0.3, 128)
    w = bf16_bits_of(w_vals)
    for j in [0, 5, 63, 64, 127]:
        k = np.zeros(128, np.uint16)
        k[j] = bf16_bits_of([2.0])[0]
        y, ya, _ = oracle_lib.gemma_knorm(k, w, 0.0)
        exact = math.sqrt(128.0) * (1.0 + oracle_lib.bf16_decode(int(w[j])))
        assert y[j] == oracle_lib.bf16_rne(exact)
        assert all(y[d] == 0 for d in range(128) if d != j)


def test_knorm_zero_row_is_zero(oracle_lib):
    y, ya, _ = oracle_lib.gemma_knorm(np.zeros(128, np.uint16), bf16_bits_of(np.ones(128)), 1e-6)
    assert not y.any() and not ya.any()


def test_knorm_is_scale_free_without_eps(oracle_lib):
    rng = np.random.default_rng(4)
    k = bf16_bits_of(rng.standard_normal(128))
    k4 = bf16_bits_of(4.0 * np.array([oracle_lib.bf16_decode(int(b)) for b in k]))
    w = bf16_bits_of(rng.standard_normal(128) * 0.1)
    y1, _, _ = oracle_lib.gemma_knorm(k, w, 0.0)
    y2, _, _ = oracle_lib.gemma_knorm(k4, w, 0.0)
    assert np.array_equal(y1, y2)
    # and eps enters inside the root: a tiny row is damped by sqrt(eps)
    tiny = bf16_bits_of(np.full(128, 1e-3))
    y3, _, _ = oracle_lib.gemma_knorm(tiny, np.zeros(128, np.uint16), 1e-6)
    av = oracle_lib.bf16_decode(int(tiny[0]))
    assert oracle_lib.bf16_decode(int(y3[0])) == pytest.approx(av / math.sqrt(av * av + float(np.float32(1e-6))),
                                                               rel=2**-8)


def test_knorm_tie_reports_both_neighbours(oracle_lib):
    # constant row with eps=0 gives y_d = 1 + w_d exactly; w_d chosen so that
    # 1 + w_d is a bf16 midpoint (1 + 2^-8): both neighbours are admissible.
    w = np.zeros(128, np.uint16)
    w[:] = bf16_bits_of([2.0**-8])[0]
    k = bf16_bits_of(np.full(128, 1.0))
    y, ya, n = oracle_lib.gemma_knorm(k, w, 0.0)
    assert n == 128
    assert set([int(y[0]), int(ya[0])]) == {0x3F80, 0x3F81}


# ------------------------------------------------------------------ RoPE

def test_rope_identity_at_zero_angle(oracle_lib):
    one, zero = bf16_bits_of([1.0])[0], 0
    rng = np.random.default_rng(5)
    for x1, x2 in bf16_bits_of(rng.standard_normal(200)).reshape(-1, 2):
        assert oracle_lib.rope_pair(x1, x2, one, zero) == (x1, x2)


def test_rope_rotates_counterclockwise(oracle_lib):
    # NeoX: (x1, x2) -> (x1 c - x2 s, x2 c + x1 s)
    for ang in [0.3, 1.0, 2.5, -0.7]:
        c, s = bf16_bits_of([math.cos(ang), math.sin(ang)])
        one = bf16_bits_of([1.0])[0]
        o1, o2 = oracle_lib.rope_pair(one, 0, c, s)
        assert (o1, o2) == (c, s)
        o1, o2 = oracle_lib.rope_pair(0, one, c, s)
        assert o1 == (int(s) ^ 0x8000) and o2 == c


def test_rope_preserves_pair_norm(oracle_lib):
    rng = np.random.default_rng(6)
    for _ in range(300):
        ang = rng.uniform(-math.pi, math.pi)
        c, s = bf16_bits_of([math.cos(ang), math.sin(ang)])
        x1, x2 = bf16_bits_of(rng.standard_normal(2) * 3)
        o1, o2 = oracle_lib.rope_pair(x1, x2, c, s)
        dec = oracle_lib.bf16_decode
        cs2 = dec(int(c)) ** 2 + dec(int(s)) ** 2
        n_in = math.hypot(dec(int(x1)), dec(int(x2)))
        n_out = math.hypot(dec(int(o1)), dec(int(o2)))
        assert abs(n_out - n_in * math.sqrt(cs2)) <= n_in * 2**-7 + 1e-30
        assert abs(cs2 - 1.0) < 2**-6


# ------------------------------------------------------------------ whole rows

def _problem(wl, **over):
    import oracle

    inp = wk.generate(wl)
    for k, v in over.items():
        setattr(inp, k, v)
    return inp, oracle.problem_from_inputs(inp)


def _dec_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("r", [16, 32, 64])
def test_row_matches_direct_rotation_at_position_angle(oracle_lib, r):
    # K'_i, K'_{i+r/2} = 2x2 rotation of (y_i, y_{i+r/2}) by pos * theta^(-2i/r)
    # (computed here from math.cos/sin, not from the bf16 table), dims >= r = y
    theta = 1e6
    wl = wk.Workload(name="rot", num_ctx=24, num_layers=2, num_kv_heads=3, rotary_dim=r, block_size=8,
                     num_blocks=8, max_pos=4096, rope_theta=theta, seed=11)
    inp, p = _problem(wl)
    ids = np.arange(wl.num_rows)
    rows, _ = p.rows(ids)
    half = r // 2
    for rid in ids:
        t, l, h = rid // (wl.num_layers * 3), (rid // 3) % wl.num_layers, rid % 3
        k = inp.all_kv[t, l, 0, h].view(torch.int16).numpy().view(np.uint16)
        y, _, _ = oracle_lib.gemma_knorm(k, inp.knorm_w[l].view(torch.int16).numpy().view(np.uint16), inp.eps)
        yv = _dec_bf16(y)
        kp = _dec_bf16(rows[rid, :128])
        assert np.array_equal(rows[rid, r:128], y[r:])
        pos = int(inp.positions[t])
        for i in range(half):
            a = pos * theta ** (-2.0 * i / r)
            c, s = math.cos(a), math.sin(a)
            e1 = yv[i] * c - yv[i + half] * s
            e2 = yv[i + half] * c + yv[i] * s
            bound = (abs(yv[i]) + abs(yv[i + half])) * 2**-8 * 1.5
            assert abs(kp[i] - e1) <= bound + abs(e1) * 2**-8
            assert abs(kp[i + half] - e2) <= bound + abs(e2) * 2**-8


def test_row_at_position_zero_is_norm_only(oracle_lib):
    wl = wk.WORKLOADS[0]  # tiny: positions 0..15, so token 0 sits at position 0
    inp, p = _problem(wl)
    rows, _ = p.rows([0])
    k = inp.all_kv[0, 0, 0, 0].view(torch.int16).numpy().view(np.uint16)
    y, _, _ = oracle_lib.gemma_knorm(k, inp.knorm_w[0].view(torch.int16).numpy().view(np.uint16), inp.eps)
    assert np.array_equal(rows[0, :128], y)
    v = inp.all_kv[0, 0, 1, 0].view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rows[0, 128:], v)


def test_fp8_row_is_quantised_bf16_row(oracle_lib):
    # fp8 K = e4m3(bf16 K' / k_scale[l]), fp8 V = e4m3(V / v_scale[l]); scales
    # differ per layer and between k and v, so a swapped index fails
    wl = wk.WORKLOADS[2].with_(num_ctx=40)
    inp, p8 = _problem(wl)
    import oracle
    p16 = oracle.problem_from_inputs(
        wk.Inputs(wl.with_(kv_dtype=wk.KV_BF16), inp.all_kv, inp.knorm_w, inp.positions, inp.slot_mapping,
                  inp.cos_sin, inp.k_scale, inp.v_scale, inp.eps))
    ids = np.arange(wl.num_rows)
    r8, _ = p8.rows(ids)
    r16, _ = p16.rows(ids)
    ks, vs = inp.k_scale.numpy(), inp.v_scale.numpy()
    assert len(set(ks.tolist()) | set(vs.tolist())) == 2 * wl.num_layers
    dec = _dec_bf16(r16).astype(np.float32)
    for rid in ids[:: 7]:
        l = (rid // wl.num_kv_heads) % wl.num_layers
        want_k = [oracle_lib.e4m3_rne_sat(float(np.float32(x) / np.float32(ks[l]))) for x in dec[rid, :128]]
        want_v = [oracle_lib.e4m3_rne_sat(float(np.float32(x) / np.float32(vs[l]))) for x in dec[rid, 128:]]
        assert list(r8[rid, :128]) == want_k
        assert list(r8[rid, 128:]) == want_v


def test_fp8_v_known_values(oracle_lib):
    # V = 1.0 with v_scale 0.5 -> 2.0 -> code 0x40; V = -3 with 0.5 -> -6 -> 0xCC
    wl = wk.WORKLOADS[2].with_(num_ctx=2, num_layers=1, num_kv_heads=1, pad_count=0)
    inp = wk.generate(wl)
    inp.all_kv[0, 0, 1, 0, :] = 1.0
    inp.all_kv[1, 0, 1, 0, :] = -3.0
    inp.v_scale[:] = 0.5
    import oracle
    rows, _ = oracle.problem_from_inputs(inp).rows([0, 1])
    assert (rows[0, 128:] == 0x40).all()
    assert (rows[1, 128:] == 0xCC).all()


# ------------------------------------------------------------------ the whole write

def _tagged_inputs(wl):
    """V rows carry exact bf16 integer tags (t // 128, t % 128, l, h, 7), all
    below 256 and so exact in bf16, so every stored row names its source."""
    inp = wk.generate(wl)
    T, L, H = wl.num_ctx, wl.num_layers, wl.num_kv_heads
    assert T < 128 * 256 and L < 256 and H < 256
    tag = torch.zeros(T, L, H, 128)
    t = torch.arange(T)
    tag[:, :, :, 0] = (t // 128)[:, None, None].float()
    tag[:, :, :, 1] = (t % 128)[:, None, None].float()
    tag[:, :, :, 2] = torch.arange(L)[None, :, None].float()
    tag[:, :, :, 3] = torch.arange(H)[None, None, :].float()
    tag[:, :, :, 4] = 7.0
    inp.all_kv[:, :, 1] = tag.to(torch.bfloat16)
    return inp


@pytest.mark.parametrize("wl", [wk.WORKLOADS[0], wk.WORKLOADS[1],
                                wk.Workload(name="odd", num_ctx=37, num_layers=3, num_kv_heads=3,
                                            rotary_dim=32, block_size=4, num_blocks=32, max_pos=500,
                                            rope_theta=1e4, pad_count=5, seed=12)],
                         ids=lambda w: w.name)
def test_every_written_slot_round_trips_and_padding_is_untouched(oracle_lib, wl):
    import oracle

    inp = _tagged_inputs(wl)
    p = oracle.problem_from_inputs(inp)
    caches = p.new_caches()
    p.write(caches)
    H, bs, L = wl.num_kv_heads, wl.block_size, wl.num_layers
    slots = inp.slot_mapping.numpy()
    written = 0
    for l in range(L):
        rows = caches[l].reshape(-1, 256)
        hit = ~(rows.view(np.uint8).reshape(rows.shape[0], -1) == 0xFF).all(axis=1)
        idx = np.nonzero(hit)[0]
        written += len(idx)
        b, rem = np.divmod(idx, H * bs)  # row index = (b * H + h) * bs + o
        h, o = np.divmod(rem, bs)
        tags = _dec_bf16(rows[idx, 128:133]).astype(np.int64)
        t = tags[:, 0] * 128 + tags[:, 1]
        assert (tags[:, 4] == 7).all()
        assert (tags[:, 2] == l).all() and (tags[:, 3] == h).all()
        assert np.array_equal(slots[t], b * bs + o)  # each slot decodes to (block, offset)
    assert written == int((slots >= 0).sum()) * L * H


def test_padding_tokens_are_not_even_read(oracle_lib):
    import oracle

    wl = wk.WORKLOADS[0]
    inp = wk.generate(wl)
    pad = (inp.slot_mapping < 0).nonzero().flatten()
    assert len(pad) == 2
    inp.positions[pad] = 10**9  # a read of their cos|sin row would be out of range
    p = oracle.problem_from_inputs(inp)
    c1 = p.new_caches()
    p.write(c1)
    inp2 = wk.generate(wl)
    c2 = oracle.problem_from_inputs(inp2).new_caches()
    oracle.problem_from_inputs(inp2).write(c2)
    assert np.array_equal(c1[0], c2[0])


def test_preconditions_are_refused(oracle_lib):
    import oracle

    wl = wk.WORKLOADS[0]
    base = wk.generate(wl)
    valid = (base.slot_mapping >= 0).nonzero().flatten()
    dup = wk.generate(wl)
    dup.slot_mapping[valid[1]] = dup.slot_mapping[valid[0]]
    with pytest.raises(oracle.OracleError, match="duplicate"):
        oracle.problem_from_inputs(dup).check()
    far = wk.generate(wl)
    far.slot_mapping[valid[0]] = wl.capacity
    with pytest.raises(oracle.OracleError, match="beyond the cache"):
        oracle.problem_from_inputs(far).check()
    badpos = wk.generate(wl)
    badpos.positions[valid[0]] = wl.max_pos
    with pytest.raises(oracle.OracleError, match="position"):
        oracle.problem_from_inputs(badpos).check()


def test_dest_row_layout(oracle_lib):
    # [num_blocks, nkv, block_size, 256]: block = slot // bs, offset = slot % bs
    assert oracle_lib.dest_row(0, 0, 8, 16, 10) == 0
    assert oracle_lib.dest_row(1, 0, 8, 16, 10) == 1
    assert oracle_lib.dest_row(16, 0, 8, 16, 10) == 8 * 16
    assert oracle_lib.dest_row(17, 3, 8, 16, 10) == (1 * 8 + 3) * 16 + 1
    assert oracle_lib.dest_row(-1, 0, 8, 16, 10) == -1
    assert oracle_lib.dest_row(160, 0, 8, 16, 10) == -2
