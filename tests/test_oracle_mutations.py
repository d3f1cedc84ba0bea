"""Planted mistakes in the oracle (CPU only): each must be caught by a pin.

Each test patches one step of the oracle with a plausible bug, re-runs the
independent check that should catch it, and asserts that the check fails.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as A


def _brute_force_disagrees(causal):
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((6, 3)) for _ in range(3))
    O, lse = A.attention_forward_head(q, k, v, causal, 0.5)
    Ob, lb = A.brute_force_attention(q.tolist(), k.tolist(), v.tolist(), causal, 0.5)
    return np.max(np.abs(O - np.array(Ob))) > 1e-9 or np.max(np.abs(lse - np.array(lb))) > 1e-9


def test_off_by_one_causal_mask_is_caught(monkeypatch):
    orig = A._causal_mask
    monkeypatch.setattr(A, "_causal_mask", lambda nq, nk, qs=0, ks=0: orig(nq, nk, qs, ks - 1))
    assert _brute_force_disagrees(True)


def test_transposed_value_operand_is_caught(monkeypatch):
    orig = A.attention_forward_head

    def bad(q, k, v, causal, scale):
        return orig(q, k, np.asarray(v).T.copy() if np.asarray(v).shape[0] == np.asarray(v).shape[1] else v[::-1], causal, scale)

    monkeypatch.setattr(A, "attention_forward_head", bad)
    assert _brute_force_disagrees(False)


def test_dropped_correction_in_tiled_loop_is_caught(monkeypatch):
    # Dropping the rescale of acc (acc = acc + p V instead of acc*c + p V).
    rng = np.random.default_rng(2)
    q = rng.standard_normal((128, 8)) * 8
    k = rng.standard_normal((128, 8))
    k[100] = 20 * q.mean(0)
    v = rng.standard_normal((128, 8))
    O, _ = A.attention_forward_head(q, k, v, False, 0.35)
    real_exp = np.exp

    calls = {"n": 0}

    def exp_no_correction(x):
        # The tiled loop's correction factor is the only exp of an (rows,1) array.
        calls["n"] += 1
        x = np.asarray(x)
        if x.ndim == 2 and x.shape[1] == 1:
            return np.where(np.isneginf(x), 0.0, np.ones_like(x))
        return real_exp(x)

    monkeypatch.setattr(A.np, "exp", exp_no_correction)
    Ot, _, _ = A.tiled_attention(q, k, v, False, 0.35, 32, 32)
    monkeypatch.setattr(A.np, "exp", real_exp)
    assert calls["n"] > 0
    assert np.max(np.abs(Ot - O)) > 1e-3


def test_backward_without_delta_fails_finite_differences(monkeypatch):
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((1, 1, 4, 3)) for _ in range(4))
    orig_sum = np.sum

    def zero_delta(a, axis=None, keepdims=False, **kw):
        r = orig_sum(a, axis=axis, keepdims=keepdims, **kw)
        return r * 0.0 if (axis == 1 and keepdims) else r

    monkeypatch.setattr(A.np, "sum", zero_delta)
    dq, _, _ = oracle.attention_backward(q, k, v, do, False, 0.5)
    monkeypatch.setattr(A.np, "sum", orig_sum)
    h = 1e-6
    num = np.zeros_like(q)
    for i in range(4):
        for j in range(3):
            qp, qm = q.copy(), q.copy()
            qp[0, 0, i, j] += h
            qm[0, 0, i, j] -= h
            lp = float(orig_sum(oracle.attention_forward(qp, k, v, False, 0.5)[0] * do))
            lm = float(orig_sum(oracle.attention_forward(qm, k, v, False, 0.5)[0] * do))
            num[0, 0, i, j] = (lp - lm) / (2 * h)
    assert np.linalg.norm(dq - num) / np.linalg.norm(num) > 1e-3


@pytest.mark.parametrize("block", [128])
def test_wrong_skip_rule_is_caught(block, monkeypatch):
    # Skipping the diagonal tile too (j >= i) breaks the printed counts.
    def bad_counts(n, bq, bk, causal, batch=1, heads=1, dim=64, elem=4):
        computed = skipped = 0
        for i in range(0, n, bq):
            rows = min(bq, n - i)
            for j in range(0, n, bk):
                if causal and j >= i:
                    skipped += 1
                    continue
                computed += 1
        return {"computed": computed, "skipped": skipped, "matmul_flops": 0, "hbm_bytes": 0}

    monkeypatch.setattr(A, "tile_schedule_counts", bad_counts)
    assert A.causal_tile_counts(2048, block) != (136, 120)
