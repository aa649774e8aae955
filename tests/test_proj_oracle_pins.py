"""Pins of the oracle's context-KV projection step (all_kv = the fused
projection output of the context states, DSpark draft model page,
precompute_and_store_context_kv / _project_context_kv_token_major; layout
[num_ctx, L, 2, nkv, 128] from the context-KV writer page).

* a hand-worked 1 x 2 by 2 x 2 case;
* on the exact-integer recipe, the oracle equals an int64 matmul scaled back
  and rounded to bf16 by torch's own conversion (every value there is exact
  in fp32, so that conversion is a single correct rounding);
* tagged weight rows land at the all_kv index the layout names:
  row ((l * 2 + kv) * nkv + h) * 128 + d -> all_kv[t, l, kv, h, d].
"""

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_hand_worked_case(oracle_lib):
    x = np.array([[0x3F80, 0x4000]], np.uint16)                     # [1, 2]
    w = np.array([[0x3F80, 0x3F80], [0x4040, 0xBF80]], np.uint16)  # [[1, 1], [3, -1]]
    assert oracle_lib.project_context_kv(x, w).tolist() == [[0x4040, 0x3F80]]  # [3, 1]


def test_integer_recipe_equals_int64_matmul(oracle_lib):
    wl = wk.PROJ_WORKLOADS_BY_NAME["proj_draft_step"].with_(recipe="int", hidden=512)
    wl = wl.with_(base=wl.base.with_(num_ctx=64, pad_count=3))
    inp = wk.generate_proj(wl)
    xi = (inp.x.float() * 8).round().to(torch.int64)
    wi = (inp.w_kv.float() * 32).round().to(torch.int64)
    assert torch.equal(xi.float() / 8, inp.x.float()) and torch.equal(wi.float() / 32, inp.w_kv.float())
    exact = (xi @ wi.T).double() / 256.0
    assert exact.abs().max() < 2**15  # multiples of 2^-8 below 2^15: exact in fp32
    ref = bits(exact.float().to(torch.bfloat16))
    got = oracle_lib.project_context_kv(bits(inp.x), bits(inp.w_kv))
    assert np.array_equal(got, ref)
    assert (got != ref).sum() == 0 and len(np.unique(got)) > 100


def test_layout_of_the_projection_rows(oracle_lib):
    """x = e_0, w[n, 0] = tag(n): all_kv[t, l, kv, h, d] must be the tag of
    row ((l * 2 + kv) * nkv + h) * 128 + d."""
    L, nkv, hidden = 2, 3, 16
    N = L * 2 * nkv * 128
    x = torch.zeros((2, hidden))
    x[:, 0] = 1.0
    w = torch.zeros((N, hidden))
    n = torch.arange(N)
    w[:, 0] = (n % 251).float()  # exact small integers
    kv = oracle_lib.project_context_kv(bits(x.to(torch.bfloat16)), bits(w.to(torch.bfloat16)))
    vals = oracle_lib.bf16_values(kv).reshape(2, L, 2, nkv, 128)
    for l in range(L):
        for k in range(2):
            for h in range(nkv):
                for d in (0, 77, 127):
                    assert vals[1, l, k, h, d] == (((l * 2 + k) * nkv + h) * 128 + d) % 251
