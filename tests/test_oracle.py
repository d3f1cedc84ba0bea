"""Pins for the fp64 oracle: checks against what the pages print and what the
mathematics fixes, never against the oracle's own formulas retyped."""

import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import attention as A


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# Online softmax: printed worked example, library softmax, invariants.
# ---------------------------------------------------------------------------


def test_rebase_walkthrough_matches_printed_values(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "rebase_walkthrough.json")))
    r = oracle.online_softmax(np.array(g["logits"]), g["block_size"])
    assert len(r["trace"]) == len(g["blocks"])
    for got, want in zip(r["trace"], g["blocks"]):
        assert abs(got["m"] - want["m"]) < 5e-5
        assert abs(got["l"] - want["l"]) < 5e-5
        if "correction" in want:
            assert abs(got["correction"] - want["correction"]) < 5e-5
    # The streamed sum equals the one-shot sum exp(x - max).
    assert abs(r["l"] - g["one_shot_sum"]) < 5e-5
    # Rebased history of block 1 = l_old * correction (printed 0.6532).
    assert abs(r["trace"][0]["l"] * r["trace"][1]["correction"] - g["blocks"][1]["rebased_history"]) < 5e-5


@pytest.mark.parametrize("block", [64, 128, 512, 2048])
def test_online_softmax_matches_library_softmax(block, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "online_softmax_check.json")))
    x = _rng(3).standard_normal((g["rows"], g["n"])) * g["logit_scale"]
    r = oracle.online_softmax(x, block)
    ref = scipy.special.softmax(x, axis=-1)
    assert np.max(np.abs(r["p"] - ref)) < 1e-15
    np.testing.assert_allclose(r["p"].sum(-1), g["rows_sum_to"], atol=1e-13)
    np.testing.assert_allclose(r["lse"], scipy.special.logsumexp(x, axis=-1), rtol=0, atol=1e-12)


def test_online_softmax_block_size_changes_nothing():
    x = _rng(4).standard_normal((3, 1000)) * 8
    outs = [oracle.online_softmax(x, b)["p"] for b in (1, 7, 64, 1000)]
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 1e-14  # a few fp64 ulp at p ~ 1


def test_rescale_counter_on_rows_with_known_answers():
    inc = np.arange(256, dtype=np.float64)  # every block raises the max
    dec = inc[::-1].copy()  # only the first block sets it
    assert oracle.online_softmax(inc, 64)["rescales"] == 4
    assert oracle.online_softmax(dec, 64)["rescales"] == 1
    # iid logits: expected number of record-setting blocks among b blocks is the
    # harmonic number H_b (first block included). 32 blocks -> H_32 ~ 4.06.
    x = _rng(5).standard_normal((20000, 32 * 8))
    mean = oracle.online_softmax(x, 8)["rescales"].mean()
    h32 = sum(1.0 / i for i in range(1, 33))
    assert abs(mean - h32) < 0.05


# ---------------------------------------------------------------------------
# Standard attention: special cases, brute force, library routines.
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_match_library_softmax(causal):
    rng = _rng(6)
    q, k = rng.standard_normal((40, 16)), rng.standard_normal((40, 16))
    P = oracle.attention_probs(q, k, causal, 0.25)
    np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-14)
    S = 0.25 * np.einsum("id,jd->ij", q, k)
    if causal:
        S[np.triu_indices(40, 1)] = -np.inf
        assert np.all(P[np.triu_indices(40, 1)] == 0.0)
    assert np.max(np.abs(P - scipy.special.softmax(S, axis=1))) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(causal):
    rng = _rng(7)
    N, d = 33, 8
    q = rng.standard_normal((N, d))
    k = np.tile(rng.standard_normal((1, d)), (N, 1))
    v = rng.standard_normal((N, d))
    O, lse = oracle.attention_forward_head(q, k, v, causal, 0.3)
    for i in range(N):
        vis = v[: i + 1] if causal else v
        np.testing.assert_allclose(O[i], vis.mean(0), atol=1e-13)
        s = 0.3 * float(q[i] @ k[0])
        assert abs(lse[i] - (s + math.log(len(vis)))) < 1e-12


def test_single_key_gives_v_and_lse_equals_score():
    rng = _rng(8)
    q, k, v = rng.standard_normal((1, 5)), rng.standard_normal((1, 5)), rng.standard_normal((1, 5))
    for causal in (False, True):
        O, lse = oracle.attention_forward_head(q, k, v, causal, 0.7)
        np.testing.assert_allclose(O, v, atol=1e-15)
        assert abs(lse[0] - 0.7 * float(q[0] @ k[0])) < 1e-15


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_loops_match(N, causal):
    rng = _rng(100 + N)
    B, Hq, Hkv, d = 1, 4, 2, 3
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    O, lse = oracle.attention_forward(q, k, v, causal, 0.6)
    for h in range(Hq):
        hk = h // (Hq // Hkv)
        Ob, lb = oracle.brute_force_attention(q[0, h].tolist(), k[0, hk].tolist(), v[0, hk].tolist(), causal, 0.6)
        np.testing.assert_allclose(O[0, h], np.array(Ob), atol=1e-12)
        np.testing.assert_allclose(lse[0, h], np.array(lb), atol=1e-12)


def test_rows_variant_matches_full():
    rng = _rng(9)
    q, k, v = (rng.standard_normal((64, 8)) for _ in range(3))
    O, lse = oracle.attention_forward_head(q, k, v, True, 0.4)
    rows = np.array([0, 1, 17, 63])
    Or, lr = oracle.attention_rows(q[rows], k, v, rows, True, 0.4)
    np.testing.assert_allclose(Or, O[rows], atol=1e-13)
    np.testing.assert_allclose(lr, lse[rows], atol=1e-13)


# ---------------------------------------------------------------------------
# The tiled loop equals the definition (the pages' exactness claim, in fp64).
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("bq,bk", [(64, 64), (128, 128), (256, 512), (48, 80)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_equals_standard(bq, bk, causal):
    rng = _rng(11)
    N, d = 600, 16  # ragged against every tile shape
    q, k, v = (rng.standard_normal((N, d)) * 2 for _ in range(3))
    O, lse = oracle.attention_forward_head(q, k, v, causal, 1 / 4)
    Ot, lt, cnt = oracle.tiled_attention(q, k, v, causal, 1 / 4, bq, bk)
    assert np.max(np.abs(Ot - O)) < 1e-12
    assert np.max(np.abs(lt - lse)) < 1e-12
    ref = oracle.tile_schedule_counts(N, bq, bk, causal, dim=d)
    assert cnt["tiles_computed"] == ref["computed"]
    assert cnt["tiles_skipped"] == ref["skipped"]
    assert cnt["matmul_flops"] == ref["matmul_flops"]


def test_tiled_handles_large_rescales():
    # A late key far above the rest forces a deep correction; the result must
    # still equal the definition.
    rng = _rng(12)
    N, d = 256, 8
    q = rng.standard_normal((N, d)) * 8
    k = rng.standard_normal((N, d))
    k[200] = 20 * q.mean(0)
    v = rng.standard_normal((N, d))
    O, lse = oracle.attention_forward_head(q, k, v, False, 1 / math.sqrt(d))
    Ot, lt, cnt = oracle.tiled_attention(q, k, v, False, 1 / math.sqrt(d), 64, 64)
    assert cnt["rescales"] > 0
    assert np.max(np.abs(Ot - O)) < 1e-12 and np.max(np.abs(lt - lse)) < 1e-12


# ---------------------------------------------------------------------------
# Counts: tiles, FLOPs, bytes (printed tables and closed forms).
# ---------------------------------------------------------------------------


def test_causal_tile_counts_printed(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "causal_tiles.json")))
    for row in g["rows"]:
        c, s = oracle.causal_tile_counts(g["n"], row["block"])
        assert (c, s) == (row["computed"], row["skipped"])
        assert round(100 * s / (c + s)) == row["fraction_skipped_pct"]


@pytest.mark.parametrize("Bblocks", [1, 2, 3, 7, 16, 32, 1024])
def test_skip_fraction_closed_form(Bblocks):
    c, s = oracle.causal_tile_counts(Bblocks * 128, 128)
    assert c == Bblocks * (Bblocks + 1) // 2
    assert s * 2 * Bblocks == (Bblocks - 1) * (c + s)  # s/(c+s) == (B-1)/(2B)


def test_flop_and_traffic_tables_printed(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flops_bytes.json")))
    H, d, e, blk = g["heads"], g["dim"], g["elem_bytes"], g["block"]
    MiB = 1024 ** 2
    for row in g["noncausal"]:
        nv = oracle.naive_counts(row["n"], heads=H, dim=d, elem=e)
        tl = oracle.tile_schedule_counts(row["n"], blk, blk, False, heads=H, dim=d, elem=e)
        assert nv["matmul_flops"] == tl["matmul_flops"]  # equal to the digit
        assert round(nv["matmul_flops"] / 1e9, 1) == row["naive_gflop"]
        assert round(tl["matmul_flops"] / 1e9, 1) == row["tiled_gflop"]
        assert nv["score_bytes"] == row["score_mib"] * MiB
    for row in g["causal"]:
        nv = oracle.naive_counts(row["n"], heads=H, dim=d, elem=e)
        tl = oracle.tile_schedule_counts(row["n"], blk, blk, True, heads=H, dim=d, elem=e)
        assert round(tl["matmul_flops"] / 1e9, 1) == row["tiled_gflop"]
        assert round(tl["matmul_flops"] / nv["matmul_flops"], 2) == row["ratio"]
        Bb = row["n"] // blk
        assert tl["matmul_flops"] * 2 * Bb == nv["matmul_flops"] * (Bb + 1)  # (B+1)/(2B)
    for row in g["all_tensor_traffic_mib"]:
        nv = oracle.naive_counts(row["n"], heads=H, dim=d, elem=e)
        tl = oracle.tile_schedule_counts(row["n"], blk, blk, False, heads=H, dim=d, elem=e)
        assert nv["hbm_bytes"] == row["naive"] * MiB
        assert tl["hbm_bytes"] == row["tiled"] * MiB
        assert row["n"] // blk == row["kv_rereads"]


def test_algorithmic_flops_closed_forms():
    # Non-causal: the naive count 4 N^2 d per head; causal counts visible pairs.
    assert oracle.algorithmic_flops(1, 8, 4096, 64, False) == oracle.naive_counts(4096, heads=8, dim=64)["matmul_flops"]
    N, d = 100, 16
    visible = sum(i + 1 for i in range(N))
    assert oracle.algorithmic_flops(2, 3, N, d, True) == 2 * 3 * 4 * d * visible
    # With one-row tiles the tiled loop computes exactly the visible pairs... plus
    # the masked diagonal entries of its 1x1 tiles, which are all visible.
    t = oracle.tile_schedule_counts(N, 1, 1, True, dim=d)
    assert t["matmul_flops"] == oracle.algorithmic_flops(1, 1, N, d, True)


# ---------------------------------------------------------------------------
# Backward: central finite differences of the forward, GQA group sums.
# ---------------------------------------------------------------------------


def _loss(q, k, v, do, causal, scale):
    O, _ = oracle.attention_forward(q, k, v, causal, scale)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (2, 1)])
def test_backward_matches_finite_differences(causal, Hq, Hkv):
    rng = _rng(21)
    B, N, d = 1, 5, 4
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, Hq, N, d))
    scale = 0.45
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            num[idx] = (lp - lm) / (2 * h)
        rel = np.linalg.norm(g - num) / np.linalg.norm(num)
        assert rel < 1e-7, (name, rel)


def test_backward_gqa_equals_duplicated_heads():
    rng = _rng(22)
    B, Hq, Hkv, N, d = 2, 4, 2, 9, 3
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, Hq, N, d))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, 0.5)
    kx, vx = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq2, dk2, dv2 = oracle.attention_backward(q, kx, vx, do, True, 0.5)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, 2, N, d).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, 2, N, d).sum(2), atol=1e-13)
    O, _ = oracle.attention_forward(q, kx, vx, True, 0.5)
    O2, _ = oracle.attention_forward(q, k, v, True, 0.5)
    np.testing.assert_allclose(O, O2, atol=1e-14)


def test_backward_head_subset():
    rng = _rng(23)
    q = rng.standard_normal((1, 4, 6, 2))
    k = rng.standard_normal((1, 2, 6, 2))
    v = rng.standard_normal((1, 2, 6, 2))
    do = rng.standard_normal((1, 4, 6, 2))
    full = oracle.attention_backward(q, k, v, do, False, 1.0)
    part = oracle.attention_backward(q, k, v, do, False, 1.0, heads=[(0, 1)])
    np.testing.assert_allclose(part[0][0, 2:], full[0][0, 2:])
    np.testing.assert_allclose(part[1][0, 1], full[1][0, 1])
    assert np.all(np.isnan(part[1][0, 0]))


def test_half_ulp_bf16_matches_torch_rounding():
    # The forward tolerance allows the bf16 output quantisation; check the helper's half-ulp
    # bound against torch's own round-to-nearest bf16 conversion.
    import torch
    from gpu_util import half_ulp_bf16

    x = np.concatenate([np.random.default_rng(30).standard_normal(20000) * s for s in (0.01, 1, 4, 100)])
    r = torch.tensor(x).to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(r - x) <= half_ulp_bf16(np.maximum(np.abs(x), np.abs(r))) * (1 + 1e-12))
    assert np.max(np.abs(r - x) / half_ulp_bf16(np.abs(x))) > 0.9  # the bound is tight


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_matches_full_backward(causal):
    rng = _rng(24)
    N, d = 70, 6
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, causal, 0.4)
    qr, kr = np.array([0, 5, 33, 69]), np.array([0, 1, 40, 69])
    rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, qr, kr, causal, 0.4, chunk=16)
    np.testing.assert_allclose(rq, dq[qr], atol=1e-12)
    np.testing.assert_allclose(rk, dk[kr], atol=1e-12)
    np.testing.assert_allclose(rv, dv[kr], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_query_blocks_sum_to_full_backward(causal):
    rng = _rng(25)
    N, d = 50, 5
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    O, lse = oracle.attention_forward_head(q, k, v, causal, 0.3)
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, causal, 0.3)
    sk, sv = np.zeros_like(dk), np.zeros_like(dv)
    for blk in (np.arange(0, 17), np.arange(17, 40), np.arange(40, 50)):
        Ob, lb, qb, kb, vb = oracle.attention_query_block(q, k, v, do, blk, causal, 0.3)
        np.testing.assert_allclose(Ob, O[blk], atol=1e-13)
        np.testing.assert_allclose(lb, lse[blk], atol=1e-13)
        np.testing.assert_allclose(qb, dq[blk], atol=1e-12)
        sk += kb
        sv += vb
    np.testing.assert_allclose(sk, dk, atol=1e-12)
    np.testing.assert_allclose(sv, dv, atol=1e-12)


# ---------------------------------------------------------------------------
# Sliding window ([P3] section 5) and split-then-merge ([P3] section 3).
# ---------------------------------------------------------------------------


def test_window_at_least_n_equals_causal():
    rng = _rng(31)
    q, k, v = (rng.standard_normal((40, 6)) for _ in range(3))
    for w in (40, 41, 1000):
        O, L = oracle.attention_forward_head(q, k, v, False, 0.5, window=w)
        Oc, Lc = oracle.attention_forward_head(q, k, v, True, 0.5)
        np.testing.assert_allclose(O, Oc, atol=1e-14)
        np.testing.assert_allclose(L, Lc, atol=1e-14)


def test_window_of_one_sees_only_itself():
    rng = _rng(32)
    q, k, v = (rng.standard_normal((17, 5)) for _ in range(3))
    O, L = oracle.attention_forward_head(q, k, v, False, 0.5, window=1)
    np.testing.assert_allclose(O, v, atol=1e-14)
    np.testing.assert_allclose(L, 0.5 * np.sum(q * k, axis=1), atol=1e-14)


@pytest.mark.parametrize("w", [1, 2, 3, 5])
def test_window_brute_force(w):
    rng = _rng(33 + w)
    q, k, v = (rng.standard_normal((7, 3)) for _ in range(3))
    O, L = oracle.attention_forward_head(q, k, v, False, 0.6, window=w)
    Ob, Lb = oracle.brute_force_attention(q.tolist(), k.tolist(), v.tolist(), False, 0.6, window=w)
    np.testing.assert_allclose(O, np.array(Ob), atol=1e-12)
    np.testing.assert_allclose(L, np.array(Lb), atol=1e-12)
    rows = np.array([0, 3, 6])
    Or, Lr = oracle.attention_rows(q[rows], k, v, rows, False, 0.6, window=w)
    np.testing.assert_allclose(Or, O[rows], atol=1e-13)
    np.testing.assert_allclose(Lr, L[rows], atol=1e-13)


def test_window_backward_finite_differences():
    rng = _rng(34)
    B, Hq, Hkv, N, d, w = 1, 2, 1, 6, 3, 3
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, Hq, N, d))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, 0.5, window=w)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = float(np.sum(oracle.attention_forward(args["q"], args["k"], args["v"], True, 0.5, window=w)[0] * do))
            args[name] = xm
            lm = float(np.sum(oracle.attention_forward(args["q"], args["k"], args["v"], True, 0.5, window=w)[0] * do))
            num[idx] = (lp - lm) / (2 * h)
        assert np.linalg.norm(g - num) / np.linalg.norm(num) < 1e-7, name


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 50])
@pytest.mark.parametrize("causal", [False, True])
def test_split_then_merge_equals_full(splits, causal):
    rng = _rng(35)
    q, k, v = (rng.standard_normal((50, 4)) * 2 for _ in range(3))
    O, L = oracle.attention_forward_head(q, k, v, causal, 0.4)
    Os, Ls = oracle.attention_split_forward_head(q, k, v, causal, 0.4, splits)
    np.testing.assert_allclose(Os, O, atol=1e-12)
    np.testing.assert_allclose(Ls, L, atol=1e-12)


def test_backward_rows_with_window_matches_full():
    rng = _rng(36)
    N, d, w = 60, 4, 9
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, True, 0.4, window=w)
    qr, kr = np.array([0, 8, 9, 59]), np.array([0, 30, 50, 59])
    rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, qr, kr, True, 0.4, chunk=16, window=w)
    np.testing.assert_allclose(rq, dq[qr], atol=1e-12)
    np.testing.assert_allclose(rk, dk[kr], atol=1e-12)
    np.testing.assert_allclose(rv, dv[kr], atol=1e-12)
