"""fa_softmax_rows (online normaliser, one row per CTA) against the fp64 oracle.

Errors are reported in fp32 ulps of each row's largest probability, the unit the pages use
for the same check ("LLM Architecture Refresh [3]", section 3: 1.5-3 ulp on one GPU backend,
3-4 ulp on CPU). Bound used here: 8 ulps for rows of up to 8192 elements; beyond that the
fp32 normaliser sums chains of n/1024 terms per accumulator, whose rounding error grows
like their length, so the bound is 8 + n/4096 ulps. Rows sum to 1 within 1e-5 and
|LSE - LSE_ref| <= 2e-6 * max(1, |LSE_ref|).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_util import fa_mod

pytestmark = pytest.mark.gpu

ULP_BOUND = 8.0


def _x(rows, n, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(rows, n, generator=g, dtype=torch.float32) * scale


def _check(x_cpu, what=""):
    fa = fa_mod()
    p, lse = fa.softmax_rows(x_cpu.cuda())
    fa.check()
    x64 = x_cpu.double().numpy()
    ref = oracle.online_softmax(x64, x64.shape[-1])
    p = p.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    pmax = ref["p"].max(axis=-1, keepdims=True)
    ulp = np.exp2(np.floor(np.log2(pmax)) - 23)
    err_ulps = float(np.max(np.abs(p - ref["p"]) / ulp))
    bound = ULP_BOUND + (x64.shape[-1] / 4096 if x64.shape[-1] > 8192 else 0)
    assert err_ulps <= bound, f"{what}: {err_ulps:.2f} ulps > {bound}"
    assert np.max(np.abs(p.sum(-1) - 1.0)) <= 1e-5, what
    assert np.all(np.abs(lse - ref["lse"]) <= 2e-6 * np.maximum(1.0, np.abs(ref["lse"]))), what
    return err_ulps


def test_four_rows_of_2048_times_8(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "online_softmax_check.json")))
    x = _x(g["rows"], g["n"], seed=3, scale=g["logit_scale"])
    e = _check(x, "P3 check")
    assert e <= g["max_ulps_fp32_printed"] * 2


@pytest.mark.parametrize("n", [1, 2, 3, 5, 100, 1023, 1024, 2048, 8192, 8196, 10000, 65536])
@pytest.mark.parametrize("rows", [1, 33])
def test_shapes(n, rows):
    _check(_x(rows, n, seed=n + rows, scale=4.0), f"rows={rows} n={n}")


def test_masked_entries_get_zero():
    x = _x(16, 3000, seed=5)
    mask = torch.rand(16, 3000, generator=torch.Generator().manual_seed(6)) < 0.7
    mask[:, 17] = False  # at least one finite entry per row
    x[mask] = float("-inf")
    fa = fa_mod()
    p, _ = fa.softmax_rows(x.cuda())
    fa.check()
    assert torch.all(p.cpu()[mask] == 0)
    _check(x, "masked")


def test_large_magnitudes_do_not_overflow():
    # Without the max shift, exp overflows fp32 past 88.7 ("LLM Architecture Refresh [3]",
    # section 3, "And the running max -- what is it for?"); logits here reach +-4000.
    _check(_x(8, 4096, seed=7, scale=1000.0), "large")


def test_many_rows_sampled():
    fa = fa_mod()
    x = _x(65536, 2048, seed=8, scale=2.0).cuda()
    p, lse = fa.softmax_rows(x)
    fa.check()
    rows = np.random.default_rng(9).integers(0, 65536, size=64)
    x64 = x[torch.as_tensor(rows, device=x.device)].cpu().double().numpy()
    ref = oracle.online_softmax(x64, 2048)
    got = p[torch.as_tensor(rows, device=x.device)].cpu().double().numpy()
    ulp = np.exp2(np.floor(np.log2(ref["p"].max(-1, keepdims=True))) - 23)
    assert np.max(np.abs(got - ref["p"]) / ulp) <= ULP_BOUND
