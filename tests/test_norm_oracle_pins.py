"""Pins of the oracle's hidden-state Gemma RMSNorm (DSpark draft model page:
hidden_norm = _gemma_rms_norm(hidden_size, eps) on the context states; the
norm y = x * rsqrt(mean(x^2) + eps) * (1 + w) with an fp32 1 + w weight).

* at width 128 it equals the context-KV oracle's K norm, pinned on its own;
* a constant row a gives a / sqrt(a^2 + eps) * (1 + w_d) per dim (catches a
  wrong weight index or a missing "1 +");
* a one-hot row gives sqrt(n) (1 + w_j) at j (catches the n of the mean);
* with w = 0 a row's RMS is 1 within bf16 rounding;
* random rows agree with a torch fp64 textbook formula rounded once to bf16,
  except where the exact value lies in the admissible tie window.
"""

import math

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.usefixtures("oracle_lib")


def bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_width_128_equals_the_k_norm(oracle_lib):
    x, w, eps = wk.generate_norm(wk.NormWorkload("t", rows=7, hidden=128))
    y, ya = oracle_lib.gemma_norm_rows(bits(x), bits(w), eps)
    for r in range(7):
        ky, kya, _ = oracle_lib.gemma_knorm(bits(x[r]), bits(w), eps)
        assert np.array_equal(y[r], ky) and np.array_equal(ya[r], kya)


def test_constant_row_closed_form(oracle_lib):
    n, a, eps = 1000, 0.75, 1e-6
    x = torch.full((1, n), a).to(torch.bfloat16)
    w = (torch.arange(n) % 7 * 0.125 - 0.375).to(torch.bfloat16)
    y, _ = oracle_lib.gemma_norm_rows(bits(x), bits(w), eps)
    a_ = float(x[0, 0])
    expect = [a_ / math.sqrt(a_ * a_ + eps) * (1.0 + float(w[d])) for d in range(n)]
    assert np.array_equal(y[0], bits(torch.tensor(expect, dtype=torch.float64).float().to(torch.bfloat16)))


def test_one_hot_row(oracle_lib):
    n, j = 4096, 1234
    x = torch.zeros((1, n))
    x[0, j] = 3.0
    w = (torch.randn(n, generator=torch.Generator().manual_seed(1)) * 0.1).to(torch.bfloat16)
    y, _ = oracle_lib.gemma_norm_rows(bits(x.to(torch.bfloat16)), bits(w), 0.0)
    vals = oracle_lib.bf16_values(y[0])
    assert (vals[np.arange(n) != j] == 0).all()
    ref = math.sqrt(n) * (1.0 + float(w[j]))
    assert abs(vals[j] - ref) <= abs(ref) * 2.0**-8


def test_unit_rms_at_zero_weight(oracle_lib):
    x, _, eps = wk.generate_norm(wk.NormWorkload("t", rows=16, hidden=4096))
    y, _ = oracle_lib.gemma_norm_rows(bits(x), np.zeros(4096, np.uint16), eps)
    rms = np.sqrt((oracle_lib.bf16_values(y) ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 2e-3)


def test_random_rows_against_the_textbook_formula(oracle_lib):
    x, w, eps = wk.generate_norm(wk.NORM_WORKLOADS_BY_NAME["hn_tiny"].with_(rows=64, hidden=4096))
    y, ya = oracle_lib.gemma_norm_rows(bits(x), bits(w), eps)
    xd = x.double()
    ref = xd / torch.sqrt(xd.pow(2).mean(-1, keepdim=True) + eps) * (1.0 + w.double())
    rb = oracle_lib.bf16_rne_array(ref.numpy())
    diff = y != rb
    assert np.array_equal(ya[diff], rb[diff])   # only tie-window elements may differ
    assert diff.mean() < 1e-3
