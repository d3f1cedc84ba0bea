"""Helpers shared by the GPU parity tests (not collected as tests).

Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs), fixed by the
specification of this library and written here once:
  forward : max |O - O_ref| <= 1e-2 beyond the bf16 quantisation of O, and
            max |LSE - LSE_ref| <= 1e-3
            O is stored in bf16, so even the exactly rounded answer differs from the fp64
            oracle by up to half a bf16 ulp (0.0156 for |O| in [4, 8)). The 1e-2 bound is
            therefore applied to the distance between O_ref and the interval of reals that
            round to the stored bf16 value: |O - O_ref| - ulp_bf16(O)/2 <= 1e-2.
  backward: ||X - X_ref||_F / ||X_ref||_F <= 2e-2 for X in dQ, dK, dV, and element by element
            max |X - X_ref| / max |X_ref| <= 2e-2 as well, so that one wrong row or column
            (a few elements out of millions, invisible in the Frobenius ratio) still fails.
            Where the kernel's arithmetic stands: P and dS are rounded to bf16 before their
            products (relative error 2^-9 per term, summed with random signs) and the result is
            stored in bf16 (2^-9 of the element at most), so both ratios come out near 1e-3 to
            5e-3; 2e-2 leaves a margin of about four.
The reference is always the fp64 CPU oracle on the same bf16 inputs.
"""

import numpy as np
import torch

import oracle
from online_softmax_09_gb300.inputs import to_f64

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 2e-2
GRAD_MAX_TOL = 2e-2


def fa_mod():
    from online_softmax_09_gb300 import build, fa

    build.build()
    return fa


def gpu_forward(q, k, v, causal, scale=None, counters=None):
    fa = fa_mod()
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, causal, scale, counters=counters)
    fa.check()
    return o, lse


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits; floor at the smallest normal)."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


def assert_fwd_close(o, lse, O_ref, L_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    if not o.size:
        return 0.0, 0.0
    d = np.abs(o - O_ref)
    excess = float(np.max(d - half_ulp_bf16(np.maximum(np.abs(o), np.abs(O_ref)))))
    eo = float(np.max(d))
    el = float(np.max(np.abs(lse - L_ref)))
    assert excess <= O_TOL, f"{what}: max|dO| = {eo:.3e}, beyond bf16 output rounding {excess:.3e} > {O_TOL}"
    assert el <= LSE_TOL, f"{what}: max|dLSE| = {el:.3e} > {LSE_TOL}"
    return eo, el


def check_fwd_full(q, k, v, causal, scale):
    o, lse = gpu_forward(q, k, v, causal, scale)
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    return assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, "full")


def check_fwd_rows(q, k, v, o, lse, causal, scale, heads, rows):
    """Compare selected (b, hq) heads at selected query rows against the oracle."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    worst = (0.0, 0.0)
    for b, h in heads:
        qr = to_f64(q[b, h, rows])
        O_ref, L_ref = oracle.attention_rows(qr, to_f64(k[b, h // G]), to_f64(v[b, h // G]), rows, causal, scale)
        og = o[b, h, torch.as_tensor(rows, device=o.device)].float().cpu().numpy()
        lg = lse[b, h, torch.as_tensor(rows, device=lse.device)].cpu().numpy()
        e = assert_fwd_close(og, lg, O_ref, L_ref, f"head ({b},{h})")
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    return worst


def sample_rows(N, n_random, seed):
    """Row 0, the last row, rows around every 128-row tile edge near the ends, plus random rows."""
    g = np.random.default_rng(seed)
    fixed = {0, 1, N - 1, min(127, N - 1), min(128, N - 1), max(N - 128, 0), max(N - 129, 0)}
    return sorted(fixed | set(g.integers(0, N, size=n_random).tolist()))


def rel_fro(x, ref, floor=0.0):
    """||x - ref||_F / max(||ref||_F, floor). The floor matters only where the exact gradient
    vanishes (e.g. N = 1, where the single weight is 1 and dQ = dK = 0 exactly)."""
    x = np.asarray(x, dtype=np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), floor, 1e-300))


def max_rel(x, ref, floor=0.0):
    """max |x - ref| / max(max |ref|, floor): the largest element-wise error against the
    tensor's scale (the floor as in rel_fro)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    return float(np.max(np.abs(x - ref)) / max(float(np.max(np.abs(ref))), floor, 1e-300))


def assert_grad_close(name, x, ref, fro_floor=0.0, max_floor=0.0, what=""):
    """Both gradient bounds (relative Frobenius and element-wise max, each with its floor as in
    rel_fro); returns the two ratios."""
    x = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(x)), f"{what} {name}: non-finite values"
    fro, mx = rel_fro(x, ref, fro_floor), max_rel(x, ref, max_floor)
    msg = f"{what} {name}: relative Frobenius {fro:.3e}, element-wise max |d| / max |ref| {mx:.3e}"
    print(msg)
    assert fro <= GRAD_REL_TOL and mx <= GRAD_MAX_TOL, msg
    return fro, mx
