"""Writes the golden fixtures under tests/golden/ from the CPU oracle alone.

The pages print no worked example with numbers, so every stored expected
value here is the oracle's, produced by this script (which calls only
``oracle/``), and the inputs are stored beside it so the fixture does not
depend on the random generator of any torch version.  Regenerate with
``python tests/golden/make_golden.py`` after a change to the oracle's
arithmetic that a passage of the pages justifies.
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as wk  # noqa: E402


def hexs(a: np.ndarray) -> str:
    return a.tobytes().hex()


def make(name: str, wl: wk.Workload) -> dict:
    inp = wk.generate(wl)
    p = oracle.problem_from_inputs(inp)
    caches = p.new_caches()
    al, ae, av = p.write(caches)
    shape = {"num_ctx": p.T, "layers": p.L, "nkv": p.H, "rotary_dim": p.rotary_dim,
             "block_size": p.block_size, "num_blocks": p.num_blocks, "max_pos": int(p.cos_sin.shape[0]),
             "kv_dtype": p.kv_dtype, "eps": p.eps}
    if p.D != oracle.HEAD_DIM:
        shape["head_dim"] = p.D  # rows of 2 * head_dim elements
    return {
        "name": name,
        "source": "oracle/ctx_kv_oracle.c via tests/golden/make_golden.py; definition: vLLM DSpark "
                  "context-KV writer page, module docstring (layout, norm, partial NeoX RoPE, fp8 of "
                  "x/scale, slots < 0 not written)",
        "shape": shape,
        "inputs": {
            "all_kv": hexs(p.all_kv), "knorm_w": hexs(p.knorm_w), "positions": p.positions.tolist(),
            "slot_mapping": p.slot_mapping.tolist(), "cos_sin": hexs(p.cos_sin),
            "k_scale": p.k_scale.tolist(), "v_scale": p.v_scale.tolist(),
        },
        # written rows only, as (layer, row index in [num_blocks*nkv*block_size], 2 * head_dim
        # stored elements as hex); every other byte of every cache keeps the 0xFF prefill
        "expected_rows": [[l, int(ri), hexs(c.reshape(-1, p.row)[ri])]
                          for l, c in enumerate(caches)
                          for ri in np.nonzero(~(c.reshape(-1, p.row).view(np.uint8).reshape(
                              c.reshape(-1, p.row).shape[0], -1) == 0xFF).all(axis=1))[0]],
        "alternates": {"layer": al.tolist(), "elem": ae.tolist(), "value": av.tolist()},
    }


def main():
    tiny = wk.WORKLOADS[0]
    fixtures = {
        "tiny_bf16.json": make("tiny_bf16", tiny),
        "tiny_fp8.json": make("tiny_fp8", tiny.with_(kv_dtype=wk.KV_FP8, num_layers=2, num_kv_heads=1,
                                                     rotary_dim=16, kv_std=2.0, seed=tiny.seed + 100)),
    }
    # layouts outside the pages' kernel: head dims 64 and 256, rotary dims 18
    # and 50 (pairs across chunk boundaries), block sizes 3 and 5
    gen = wk.Workload(name="g", num_ctx=8, num_layers=2, num_kv_heads=2, rotary_dim=18, head_dim=64,
                      block_size=3, num_blocks=8, max_pos=64, rope_theta=1e4, slots="unique", pad_count=1,
                      seed=tiny.seed + 200)
    fixtures["general_d64_r18_bs3.json"] = make("general_d64_r18_bs3", gen)
    fixtures["general_d256_r50_bs5_fp8.json"] = make(
        "general_d256_r50_bs5_fp8", gen.with_(head_dim=256, rotary_dim=50, block_size=5, kv_dtype=wk.KV_FP8,
                                              kv_std=2.0, seed=tiny.seed + 201))
    for fname, fx in fixtures.items():
        with open(os.path.join(HERE, fname), "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
