"""The oracle reproduces its stored golden fixtures byte for byte.

The fixtures (tests/golden/*.json) hold their own inputs, so this guards the
oracle's arithmetic against unintended change independently of any random
generator.  They were written by tests/golden/make_golden.py, which calls
only the oracle."""

import json
import os

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _arr(hexstr, dtype, shape=None):
    a = np.frombuffer(bytes.fromhex(hexstr), dtype=dtype).copy()
    return a.reshape(shape) if shape is not None else a


@pytest.mark.parametrize("fname", ["tiny_bf16.json", "tiny_fp8.json", "general_d64_r18_bs3.json",
                                   "general_d256_r50_bs5_fp8.json"])
def test_oracle_reproduces_golden(oracle_lib, fname):
    with open(os.path.join(HERE, fname)) as f:
        fx = json.load(f)
    s = fx["shape"]
    T, L, H, r = s["num_ctx"], s["layers"], s["nkv"], s["rotary_dim"]
    D = s.get("head_dim", 128)
    i = fx["inputs"]
    p = oracle_lib.Problem(
        _arr(i["all_kv"], np.uint16, (T, L, 2, H, D)), _arr(i["knorm_w"], np.uint16, (L, D)),
        np.array(i["positions"], np.int64), np.array(i["slot_mapping"], np.int64),
        _arr(i["cos_sin"], np.uint16, (s["max_pos"], r)), np.array(i["k_scale"], np.float32),
        np.array(i["v_scale"], np.float32), num_blocks=s["num_blocks"], block_size=s["block_size"],
        rotary_dim=r, kv_dtype=s["kv_dtype"], eps=s["eps"])
    caches = p.new_caches()
    al, ae, av = p.write(caches)
    seen = [np.zeros(c.reshape(-1, 2 * D).shape[0], bool) for c in caches]
    for l, ri, want in fx["expected_rows"]:
        assert caches[l].reshape(-1, 2 * D)[ri].tobytes().hex() == want
        seen[l][ri] = True
    for c, m in zip(caches, seen):
        rest = c.reshape(-1, 2 * D)[~m]
        assert (rest.view(np.uint8) == 0xFF).all()
    assert len(fx["expected_rows"]) == int((p.slot_mapping >= 0).sum()) * L * H
    assert al.tolist() == fx["alternates"]["layer"]
    assert ae.tolist() == fx["alternates"]["elem"]
    assert av.tolist() == fx["alternates"]["value"]
