"""Backward parity: libfa.so fa_bwd (through the C ABI) against the fp64 CPU oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_grad_close, fa_mod, rel_fro, sample_rows
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(q, k, v, do, causal, scale=None):
    fa = fa_mod()
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal, scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dod, lse, causal, scale)
    fa.check()
    return o, lse, dq, dk, dv


def check_full(q, k, v, do, causal, scale):
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, do, causal, scale)
    ref = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), causal, scale)
    # dV never vanishes; it sets the gradient scale where the exact dQ and dK do (N = 1).
    fro_floor = 1e-3 * np.linalg.norm(ref[2])
    max_floor = 1e-3 * float(np.max(np.abs(ref[2])))
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        fro, _ = assert_grad_close(name, g.float().cpu().numpy(), r, fro_floor, max_floor, what="full")
        errs.append(fro)
    return errs


def test_b1_h1_n256_d64():
    q, k, v, do = make_qkv(1, 1, 1, 256, 64, seed=0, with_do=True)
    check_full(q, k, v, do, False, 1 / 8)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("adversarial", [False, True])
def test_b2_h8_n1024_d64(causal, adversarial):
    q, k, v, do = make_qkv(2, 8, 8, 1024, 64, seed=1, with_do=True, adversarial=adversarial)
    check_full(q, k, v, do, causal, 1 / 8)


@pytest.mark.parametrize("N", [1, 7, 128, 200, 300])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (6, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_and_gqa_shapes(N, d, heads, causal):
    Hq, Hkv = heads
    q, k, v, do = make_qkv(2, Hq, Hkv, N, d, seed=2000 + N + d + Hq, with_do=True)
    check_full(q, k, v, do, causal, 1 / math.sqrt(d))


def test_llama8b_shape_b4_h32_kv8_n4096_d128_causal():
    # GQA 4:1, N(0,1)*0.5 from seed 2; the full backward of kv groups (0,0) and (0,7), in the
    # first of the kernel's two launch bands of 16 (batch, kv head) pairs, and (3,7), the last
    # group of the second band.
    q, k, v, do = make_qkv(4, 32, 8, 4096, 128, seed=2, value_scale=0.5, with_do=True)
    scale = 1 / math.sqrt(128)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, do, True)
    for b, groups in ((0, [(0, 0), (0, 7)]), (3, [(0, 7)])):
        bs = slice(b, b + 1)
        ref = oracle.attention_backward(to_f64(q[bs]), to_f64(k[bs]), to_f64(v[bs]), to_f64(do[bs]), True, scale,
                                        heads=groups)
        for _, hk in groups:
            hq = slice(4 * hk, 4 * hk + 4)
            what = f"(b={b}, kv head {hk})"
            assert_grad_close("dq", dq[b, hq].float().cpu().numpy(), ref[0][0, hq], what=what)
            assert_grad_close("dk", dk[b, hk].float().cpu().numpy(), ref[1][0, hk], what=what)
            assert_grad_close("dv", dv[b, hk].float().cpu().numpy(), ref[2][0, hk], what=what)


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("d", [64, 128])
def test_sequence_sweep_16k_tokens(N, d):
    # B*N = 16384, H=16, N(0,1) from seed 3; one head checked per case (full for N <= 2048,
    # otherwise on sampled query rows for dQ and sampled key rows for dK, dV).
    B = 16384 // N
    q, k, v, do = make_qkv(B, 16, 16, N, d, seed=3, with_do=True)
    scale = 1 / math.sqrt(d)
    b, h = B - 1, 5
    rows = sample_rows(N, 48, seed=N + d)
    for causal in (False, True):
        _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, do, causal)
        args = (to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]), to_f64(do[b, h]))
        if N <= 2048:
            rq, rk, rv = oracle.attention_backward_head(*args, causal, scale)
            gq, gk, gv = dq[b, h], dk[b, h], dv[b, h]
        else:
            rq, rk, rv = oracle.attention_backward_rows(*args, rows, rows, causal, scale)
            idx = torch.as_tensor(rows, device=dq.device)
            gq, gk, gv = dq[b, h, idx], dk[b, h, idx], dv[b, h, idx]
        for name, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv)):
            assert_grad_close(name, g.float().cpu().numpy(), r, what=f"causal={causal}")


def test_dk_dv_deterministic_and_workspace_reuse():
    fa = fa_mod()
    q, k, v, do = make_qkv(2, 4, 2, 640, 128, seed=9, with_do=True)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, True)
    ws = torch.full((fa.workspace_bytes(2, 4, 2, 640, 128),), 0x7f, dtype=torch.uint8, device="cuda")
    g1 = fa.backward(qd, kd, vd, o, dod, lse, True, workspace=ws)
    g1 = [t.clone() for t in g1]
    g2 = fa.backward(qd, kd, vd, o, dod, lse, True, workspace=ws)  # stale workspace contents
    fa.check()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])  # dK, dV: no atomics
    assert rel_fro(g2[0].float().cpu().numpy(), g1[0].float().cpu().numpy()) < 1e-2


@pytest.mark.parametrize("shape", [(8, 4, 4, 1024, 128), (4, 8, 2, 3000, 64)])
def test_compute_stage_runs_again_without_a_new_prepare(shape):
    # The compute kernel hands out work items from a workspace counter and leaves it at zero,
    # so a second compute after one prepare redoes every item: dK and dV come out the same bit
    # for bit, and the dQ accumulator holds every contribution twice. Shapes with more work
    # items than SMs, so CTAs take several items each.
    fa = fa_mod()
    B, Hq, Hkv, N, d = shape
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=10 + N, with_do=True))
    o, lse = fa.forward(q, k, v, True)
    ref = [t.clone() for t in fa.backward(q, k, v, o, do, lse, True)]
    ws = torch.empty(fa.workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.backward_stages(q, k, v, o, do, lse, dq, dk, dv, ws, True, only=(0, 1))
    fa.backward_stages(q, k, v, o, do, lse, dq, dk, dv, ws, True, only=(1, 2))
    fa.check()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert rel_fro(dq.float().cpu().numpy(), 2 * ref[0].float().cpu().numpy()) < 1e-2


def test_backward_workspace_has_no_n_squared_term():
    fa = fa_mod()
    sizes = [fa.workspace_bytes(1, 32, 8, n, 128) for n in (4096, 8192, 16384)]
    assert sizes[2] - sizes[1] == 2 * (sizes[1] - sizes[0])
    # fp32 dQ accumulator + two fp32 row statistics + one 256-byte work counter, nothing else.
    assert sizes[0] == 32 * 4096 * (128 + 2) * 4 + 256


def _random_configs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        hkv = int(rng.choice([1, 2, 3, 4]))
        g = int(rng.choice([1, 2]))
        out.append((int(rng.integers(1, 17)), hkv * g, hkv, int(rng.integers(1, 800)), int(rng.choice([64, 128])),
                    bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", _random_configs(8, seed=2267))
def test_random_shapes_forward_and_backward(B, Hq, Hkv, N, d, causal):
    # Seeded random batch, GQA ratio, ragged N, head dim and mask (this seed gives three shapes
    # with more backward work items than SMs): the forward and the persistent backward in full
    # against the oracle.
    q, k, v, do = make_qkv(B, Hq, Hkv, N, d, seed=7000 + N, with_do=True)
    scale = 1 / math.sqrt(d)
    o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, do, causal)
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    from gpu_util import assert_fwd_close
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, "random shape")
    ref = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), causal, scale)
    fro_floor = 1e-3 * np.linalg.norm(ref[2])
    max_floor = 1e-3 * float(np.max(np.abs(ref[2])))
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_close(name, g.float().cpu().numpy(), r, fro_floor, max_floor, what="random shape")
