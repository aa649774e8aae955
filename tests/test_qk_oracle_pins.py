"""Pins of the draft-token QK-norm / RoPE / KV-insert oracle.

The DSpark draft model page gives the op only as a signature and one
sentence (``dspark_qknorm_rope_kv_insert``: the fused QK-norm/RoPE on qkv,
also storing the draft tokens' k/v).  Each test ties the oracle to something
other than itself:

* the key path and the insert against the context-KV oracle, which the
  context-KV writer page pins independently (same norm, RoPE, encoding and
  cache layout on a one-layer problem built from the qkv rows);
* the query path against the same oracle with the query weight;
* an unfused torch-CPU composition (fp32 norm materialised to bf16, fp32
  rotation, one bf16 rounding, the fp8 query output through torch's e4m3);
* invariants the page fixes: value heads untouched, padded tokens rotated but
  not inserted, the identity rotation at position 0, the insert optional.
"""

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def ordered(a: np.ndarray, sign: int) -> np.ndarray:
    a = a.astype(np.int64)
    mag = a & (sign - 1)
    return np.where(a & sign, -mag, mag)


def bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def small(name: str, **kw) -> wk.QkWorkload:
    base = wk.QK_WORKLOADS_BY_NAME[name]
    if name != "qk_tiny":
        base = base.with_(requests=5, num_heads=8, num_kv_heads=2, pad_count=3, num_blocks=256)
    return base.with_(**kw)


def context_problem(oracle_lib, inp: wk.QkInputs, head_block: str, head: int = 0):
    """A one-layer context-KV problem whose K rows are the qkv's key heads (or
    query head ``head`` for every KV slot) and whose V rows are its value heads."""
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    q = inp.qkv.view(T, Hq + 2 * Hkv, 128)
    if head_block == "k":
        k = q[:, Hq:Hq + Hkv]
        w = inp.k_norm_w
    else:
        k = q[:, head:head + 1].expand(T, Hkv, 128)
        w = inp.q_norm_w
    v = q[:, Hq + Hkv:]
    all_kv = torch.stack([k, v], dim=1).unsqueeze(1).contiguous()  # [T, 1, 2, Hkv, 128]
    fp8 = wl.kv_dtype == wk.KV_FP8 and head_block == "k"
    return oracle_lib.Problem(
        bits(all_kv), bits(w.view(1, 128)), inp.positions.numpy(), inp.slot_mapping.numpy(),
        bits(inp.cos_sin), np.array([inp.k_scale], np.float32), np.array([inp.v_scale], np.float32),
        num_blocks=wl.num_blocks, block_size=wl.block_size, rotary_dim=wl.rotary_dim,
        kv_dtype=oracle_lib.KV_FP8_E4M3 if fp8 else oracle_lib.KV_BF16, eps=inp.eps)


@pytest.mark.parametrize("name", ["qk_tiny", "qk_draft", "qk_draft_fp8"])
def test_insert_equals_context_oracle_on_one_layer(oracle_lib, name):
    """Cache rows of the insert == the context-KV write of the same K|V rows:
    placement, padding, norm, RoPE and encoding, byte for byte."""
    inp = wk.generate_qk(small(name))
    p = oracle_lib.qk_problem_from_inputs(inp)
    cache = p.new_cache()
    p.run(cache=cache)
    ctx = context_problem(oracle_lib, inp, "k")
    ref = ctx.new_caches()
    ctx.write(ref)
    assert np.array_equal(cache, ref[0])
    written = ~(cache.reshape(-1, 256) == (0xFF if p.kv_dtype else 0xFFFF)).all(axis=1)
    assert written.sum() == inp.num_valid_tokens * inp.workload.num_kv_heads


@pytest.mark.parametrize("name", ["qk_tiny", "qk_draft"])
def test_key_and_query_heads_equal_context_oracle_rows(oracle_lib, name):
    """In-place key heads and query heads == the context oracle's bf16 K' of
    the same row under the same weight (k_norm_w for keys, q_norm_w for queries)."""
    inp = wk.generate_qk(small(name))
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    p = oracle_lib.qk_problem_from_inputs(inp)
    out, _, _ = p.run()
    heads = out.reshape(T, Hq + 2 * Hkv, 128)
    ids = np.arange(T * Hkv, dtype=np.int64)  # every (t, h) row of the one-layer problem
    krows, _ = context_problem(oracle_lib, inp, "k").rows(ids)
    assert np.array_equal(heads[:, Hq:Hq + Hkv].reshape(-1, 128), krows[:, :128])
    for i in (0, Hq - 1):
        qrows, _ = context_problem(oracle_lib, inp, "q", head=i).rows(np.arange(T, dtype=np.int64) * Hkv)
        assert np.array_equal(heads[:, i], qrows[:, :128]), i


def test_value_heads_untouched_and_padding_rotated_not_inserted(oracle_lib):
    inp = wk.generate_qk(small("qk_draft"))
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    p = oracle_lib.qk_problem_from_inputs(inp)
    cache = p.new_cache()
    out, _, _ = p.run(cache=cache)
    src = bits(inp.qkv).reshape(T, Hq + 2 * Hkv, 128)
    heads = out.reshape(T, Hq + 2 * Hkv, 128)
    assert np.array_equal(heads[:, Hq + Hkv:], src[:, Hq + Hkv:])
    pad = (inp.slot_mapping < 0).numpy()
    assert pad.sum() == wl.pad_count
    # padded tokens are normed and rotated like every other token
    assert (heads[pad, :Hq + Hkv] != src[pad, :Hq + Hkv]).any(axis=-1).all()
    # and nothing else than the valid tokens' rows left the 0xFF prefill
    rows = cache.reshape(-1, 256)
    assert (~(rows == 0xFFFF).all(axis=1)).sum() == (~pad).sum() * Hkv


def test_without_insert_qkv_is_the_same(oracle_lib):
    inp = wk.generate_qk(small("qk_draft_fp8"))
    a, qa, _ = oracle_lib.qk_problem_from_inputs(inp).run(cache=None, q_fp8=True)
    p = oracle_lib.qk_problem_from_inputs(inp)
    b, qb, _ = p.run(cache=p.new_cache(), q_fp8=True)
    c, _, _ = oracle_lib.qk_problem_from_inputs(inp, with_slots=False).run(cache=p.new_cache())
    assert np.array_equal(a, b) and np.array_equal(a, c) and np.array_equal(qa, qb)


def test_position_zero_is_the_norm_alone(oracle_lib):
    inp = wk.generate_qk(small("qk_draft"))
    inp.positions.zero_()
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    out, _, _ = oracle_lib.qk_problem_from_inputs(inp).run()
    heads = out.reshape(T, Hq + 2 * Hkv, 128)
    src = bits(inp.qkv).reshape(T, Hq + 2 * Hkv, 128)
    for t in (0, T - 1):
        for hh in (0, Hq - 1, Hq, Hq + Hkv - 1):
            w = bits(inp.q_norm_w if hh < Hq else inp.k_norm_w)
            y, _, _ = oracle_lib.gemma_knorm(src[t, hh], w, inp.eps)
            assert np.array_equal(heads[t, hh], y), (t, hh)


def unfused(inp: wk.QkInputs):
    """Plain torch CPU composition: per head fp32 Gemma norm -> bf16, NeoX
    rotation in fp32 -> bf16, fp8 query as e4m3(x / scale) with saturation."""
    wl = inp.workload
    T, Hq, Hkv, r = wl.num_tokens, wl.num_heads, wl.num_kv_heads, wl.rotary_dim
    half = r // 2
    x = inp.qkv.view(T, Hq + 2 * Hkv, 128)
    qk = x[:, :Hq + Hkv].float()
    w = torch.cat([inp.q_norm_w.float().expand(Hq, 128), inp.k_norm_w.float().expand(Hkv, 128)])
    inv = torch.rsqrt(qk.pow(2).mean(-1, keepdim=True) + inp.eps)
    y = (qk * inv * (1.0 + w)).to(torch.bfloat16).float()
    cs = inp.cos_sin[inp.positions].float()
    cos, sin = cs[:, None, :half], cs[:, None, half:]
    y1, y2 = y[..., :half], y[..., half:r]
    rot = torch.cat([y1 * cos - y2 * sin, y2 * cos + y1 * sin], dim=-1)
    out = torch.cat([rot, y[..., r:]], dim=-1).to(torch.bfloat16)
    qf8 = (out[:, :Hq].float() / inp.q_scale).clamp(-448, 448).to(torch.float8_e4m3fn)
    return out, qf8.view(torch.uint8).reshape(T, Hq * 128)


@pytest.mark.parametrize("name", ["qk_tiny", "qk_draft", "qk_draft_fp8"])
def test_oracle_equals_unfused_composition(oracle_lib, name):
    inp = wk.generate_qk(small(name, q_fp8=True))
    wl = inp.workload
    T, Hq, Hkv = wl.num_tokens, wl.num_heads, wl.num_kv_heads
    out, qf, (aw, ae, av) = oracle_lib.qk_problem_from_inputs(inp).run(q_fp8=True)
    ref, ref_q = unfused(inp)
    o = out.reshape(T, Hq + 2 * Hkv, 128)[:, :Hq + Hkv].reshape(T, -1)
    u = bits(ref).reshape(T, -1)
    d = np.abs(ordered(o, 0x8000) - ordered(u, 0x8000))
    width = (Hq + 2 * Hkv) * 128
    for t, c in np.argwhere(d > 1):
        el = t * width + c  # same element index: query and key heads lead the row
        alts = av[(aw == oracle_lib.ALT_QKV) & (ae == el)]
        assert any(abs(int(ordered(np.array([a]), 0x8000)[0]) - int(ordered(u[t, c:c + 1], 0x8000)[0])) <= 1
                   for a in alts), (t, c)
    dq = np.abs(ordered(qf, 0x80) - ordered(ref_q.numpy(), 0x80))
    assert dq.max() <= 1


def test_refuses_broken_preconditions(oracle_lib):
    # each case starts from freshly drawn inputs (the problem shares their memory)
    fresh = lambda: oracle_lib.qk_problem_from_inputs(wk.generate_qk(small("qk_draft")))  # noqa: E731
    p = fresh()
    valid = np.nonzero(p.slot_mapping >= 0)[0]
    p.slot_mapping[valid[1]] = p.slot_mapping[valid[0]]
    with pytest.raises(oracle_lib.OracleError, match="duplicate"):
        p.run(cache=p.new_cache())
    p = fresh()
    pad = np.nonzero(p.slot_mapping < 0)[0]
    p.positions[pad[0]] = p.cos_sin.shape[0]  # padded tokens are rotated too
    with pytest.raises(oracle_lib.OracleError, match="position"):
        p.run()
    p = fresh()
    p.slot_mapping[valid[0]] = p.num_blocks * p.block_size
    with pytest.raises(oracle_lib.OracleError, match="slot beyond"):
        p.run(cache=p.new_cache())
    p = fresh()
    p.c.q_scale = 0.0
    with pytest.raises(oracle_lib.OracleError, match="scale"):
        p.run(q_fp8=True)
