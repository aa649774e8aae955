"""GPU parity of the hidden-state Gemma RMSNorm (DSpark draft model page:
hidden_norm = _gemma_rms_norm(hidden_size, eps) on the context states)
against the oracle, element by element, through the C ABI: every output
within 1 bf16 ulp of the oracle's correctly rounded value (an fp32 sum of
squares in another order moves the norm by far less than an ulp; a value
near a rounding midpoint may round either way)."""

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.gpu


def bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ordered(a):
    a = a.astype(np.int64)
    return np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)


def check(oracle_lib, wl, in_place=False, rows_sample=None):
    import speculative_decoding_draft_ctx_gb300 as dk

    x, w, eps = wk.generate_norm(wl)
    xd, wd = x.cuda(), w.cuda()
    out = dk.gemma_rms_norm(xd, wd, eps, out=xd if in_place else None)
    torch.cuda.synchronize()
    g = bits(out)
    xb = bits(x)
    if rows_sample is not None:
        rows = np.sort(np.random.default_rng(3).choice(wl.rows, rows_sample, replace=False))
        g, xb = g[rows], xb[rows]
    y, ya = oracle_lib.gemma_norm_rows(xb, bits(w), eps)
    d = np.minimum(np.abs(ordered(g) - ordered(y)), np.abs(ordered(g) - ordered(ya)))
    assert d.max() <= 1, (int(d.max()), np.argwhere(d > 1)[:5].tolist())


@pytest.mark.parametrize("hidden", [8, 264, 1024, 2048, 4096, 6144, 8192])
def test_norm_widths(oracle_lib, hidden):
    check(oracle_lib, wk.NormWorkload("t", rows=37, hidden=hidden))


@pytest.mark.parametrize("name", ["hn_tiny", "hn_draft_step", "hn_prefill"])
def test_norm_workloads(oracle_lib, name):
    check(oracle_lib, wk.NORM_WORKLOADS_BY_NAME[name])


def test_norm_long_context_sampled(oracle_lib):
    check(oracle_lib, wk.NORM_WORKLOADS_BY_NAME["hn_long_context"], rows_sample=1024)


def test_norm_in_place(oracle_lib):
    check(oracle_lib, wk.NORM_WORKLOADS_BY_NAME["hn_draft_step"], in_place=True)


def test_norm_zero_rows_and_zero_row():
    import speculative_decoding_draft_ctx_gb300 as dk

    x = torch.zeros((0, 4096), dtype=torch.bfloat16, device="cuda")
    dk.gemma_rms_norm(x, torch.zeros(4096, dtype=torch.bfloat16, device="cuda"), 1e-6)
    z = torch.zeros((3, 4096), dtype=torch.bfloat16, device="cuda")
    out = dk.gemma_rms_norm(z, torch.ones(4096, dtype=torch.bfloat16, device="cuda"), 1e-6)
    assert torch.equal(out, z)
