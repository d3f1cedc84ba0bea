"""Forward parity: libfa.so (through the C ABI) against the fp64 CPU oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_fwd_close, check_fwd_full, check_fwd_rows, fa_mod, gpu_forward, half_ulp_bf16,
                      sample_rows)
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu


def test_small_single_head_noncausal_d64():
    # B=1, H=1, N=256, d=64, non-causal, N(0,1) from seed 0.
    q, k, v, _ = make_qkv(1, 1, 1, 256, 64, seed=0)
    check_fwd_full(q, k, v, False, 1 / 8)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("adversarial", [False, True])
def test_b2_h8_n1024_d64(causal, adversarial):
    q, k, v, _ = make_qkv(2, 8, 8, 1024, 64, seed=1, adversarial=adversarial)
    check_fwd_full(q, k, v, causal, 1 / 8)


@pytest.mark.parametrize("N", [1, 7, 64, 128, 129, 300, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (6, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_and_gqa_shapes(N, d, heads, causal):
    Hq, Hkv = heads
    q, k, v, _ = make_qkv(2, Hq, Hkv, N, d, seed=1000 + N + d + Hq)
    check_fwd_full(q, k, v, causal, 1 / math.sqrt(d))


def test_explicit_scale_and_default_scale():
    q, k, v, _ = make_qkv(1, 2, 2, 200, 128, seed=5)
    check_fwd_full(q, k, v, True, 0.05)
    o1, l1 = gpu_forward(q, k, v, True, None)
    o2, l2 = gpu_forward(q, k, v, True, 1 / math.sqrt(128))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_is_deterministic():
    q, k, v, _ = make_qkv(2, 4, 2, 700, 128, seed=6)
    o1, l1 = gpu_forward(q, k, v, True)
    o2, l2 = gpu_forward(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_side_stream():
    fa = fa_mod()
    q, k, v, _ = make_qkv(1, 2, 1, 384, 64, seed=7)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.forward(qd, kd, vd, True)
    fa.check(stream=s)
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), True, 1 / 8)
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref)


def test_llama8b_shape_b4_h32_kv8_n4096_d128_causal():
    # GQA 4:1, N(0,1)*0.5 from seed 2. Four heads in full, 24 sampled rows on every head.
    q, k, v, _ = make_qkv(4, 32, 8, 4096, 128, seed=2, value_scale=0.5)
    o, lse = gpu_forward(q, k, v, True)
    scale = 1 / math.sqrt(128)
    for b, h in [(0, 0), (1, 13), (2, 22), (3, 31)]:
        O_ref, L_ref = oracle.attention_forward_head(to_f64(q[b, h]), to_f64(k[b, h // 4]), to_f64(v[b, h // 4]),
                                                     True, scale)
        assert_fwd_close(o[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), O_ref, L_ref, f"({b},{h})")
    heads = [(b, h) for b in range(4) for h in range(32)]
    check_fwd_rows(q, k, v, o, lse, True, scale, heads, sample_rows(4096, 16, seed=2))


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("d", [64, 128])
def test_sequence_sweep_16k_tokens(N, d):
    # B*N = 16384 tokens, H=16, N(0,1) from seed 3, causal and non-causal.
    B = 16384 // N
    q, k, v, _ = make_qkv(B, 16, 16, N, d, seed=3)
    scale = 1 / math.sqrt(d)
    heads = [(0, 0), (B - 1, 15), (B // 2, 7)]
    rows = sample_rows(N, 48, seed=N + d)
    for causal in (False, True):
        o, lse = gpu_forward(q, k, v, causal)
        check_fwd_rows(q, k, v, o, lse, causal, scale, heads, rows)


def test_long_context_n131072_memory_and_tile_counts():
    # B=1, Hq=32, Hkv=8, N=131072, d=128, causal, N(0,1)*0.5 from seed 4.
    fa = fa_mod()
    B, Hq, Hkv, N, d = 1, 32, 8, 131072, 128
    q, k, v, _ = make_qkv(B, Hq, Hkv, N, d, seed=4, value_scale=0.5)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    counters = torch.zeros(3, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    fa.forward(qd, kd, vd, True, out=o, lse=lse, counters=counters)
    fa.check()
    assert torch.cuda.max_memory_allocated() - base == 0  # no N^2 (or any) scratch buffer
    assert torch.cuda.mem_get_info()[0] >= free_before - (64 << 20)
    T = N // 128
    computed, skipped, _ = counters.cpu().tolist()
    assert computed == B * Hq * T * (T + 1) // 2
    assert skipped == B * Hq * T * (T - 1) // 2
    assert skipped * 2 * T == (T - 1) * (computed + skipped)  # (T-1)/(2T) = 1023/2048
    rows = sample_rows(N, 40, seed=4) + [N // 2, N // 2 + 127]
    check_fwd_rows(q, k, v, o, lse, True, 1 / math.sqrt(d), [(0, 0), (0, 9), (0, 18), (0, 31)], rows)


def test_tile_counters_noncausal_and_rescales():
    q, k, v, _ = make_qkv(2, 8, 8, 1024, 64, seed=1, adversarial=True)
    counters = torch.zeros(3, dtype=torch.int64, device="cuda")
    gpu_forward(q, k, v, False, counters=counters)
    computed, skipped, rescaled = counters.cpu().tolist()
    assert computed == 2 * 8 * 8 * 8 and skipped == 0
    assert rescaled > 0  # the planted key forces late rescales


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_stale_reference_max_staircase(causal, d):
    # Scores that climb by about 3 (base 2) from one key tile to the next, with one top key per
    # tile standing 8 to 12 above the tile's other keys: the kernel's reference max lags the true
    # max by up to 2^8 between rescales, and each row is dominated by a key whose weight against
    # that stale reference is not a bf16 number. Without the rounding correction of the
    # normaliser this input shows errors of about 1e-2 in O.
    # Built from seeded draws: q = sqrt(d) e_1 + noise, k_1 = r / log2(e) with r uniform in
    # [3t - 12, 3t - 8] on key tile t and r = 3t + U(-1/2, 1/2) on its last key, V ~ N(0, 1).
    B, H, N = 1, 4, 1024
    q, k, v, _ = make_qkv(B, H, H, N, d, seed=77, value_scale=0.05)
    g = torch.Generator().manual_seed(78)
    q[..., 0] = math.sqrt(d)
    r = torch.rand(B, H, N, generator=g) * 4.0 + 3.0 * (torch.arange(N) // 128).float() - 12.0
    r[..., 127::128] = 3.0 * torch.arange(N // 128).float() + torch.rand(B, H, N // 128, generator=g) - 0.5
    k[..., 0] = (r / math.log2(math.e)).to(torch.bfloat16)
    v = make_qkv(B, H, H, N, d, seed=79)[2]
    scale = 1 / math.sqrt(d)
    o, lse = gpu_forward(q, k, v, causal, scale)
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    o = o.float().cpu().numpy()
    assert_fwd_close(o, lse.cpu().numpy(), O_ref, L_ref, f"d={d} causal={causal}")
    excess = float(np.max(np.abs(o - O_ref) - half_ulp_bf16(np.maximum(np.abs(o), np.abs(O_ref)))))
    # Regression guard for the normaliser's rounding correction: measured at <= 2.7e-3 with it
    # and 5.8e-3 to 8.8e-3 without it on these four cases (both within the 1e-2 parity bound).
    assert excess <= 4e-3, f"excess {excess:.3e}: the dominant weights' bf16 rounding is not compensated"
