"""fa_fwd_bwd_host: forward + backward on host buffers with overlapped copies.

Checked against the device-resident path (same kernels on batch-element slices, so O, LSE, dK
and dV must be bit-identical; dQ is summed by bulk reductions in a timing-dependent order, so
it agrees to fp32 rounding), and once directly against the fp64 oracle with the tolerances of
gpu_util.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_fwd_close, assert_grad_close, fa_mod
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu


def _device_path(fa, q, k, v, do, causal):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dod, lse, causal)
    fa.check()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(3, 8, 2, 1000, 128, True), (2, 4, 4, 300, 64, False),
                                                (1, 2, 1, 129, 128, True), (4, 4, 1, 512, 64, True),
                                                # Chunks whose lse slices start off a 16-byte boundary.
                                                (2, 3, 1, 129, 64, True), (1, 4, 2, 129, 128, False),
                                                (3, 6, 3, 77, 128, True)])
def test_matches_device_path(B, Hq, Hkv, N, d, causal):
    fa = fa_mod()
    q, k, v, do = make_qkv(B, Hq, Hkv, N, d, seed=6000 + N + d, value_scale=0.5, with_do=True)
    q, k, v, do = (t.pin_memory() for t in (q, k, v, do))
    got = fa.fwd_bwd_host(q, k, v, do, causal)
    fa.check()
    ref = _device_path(fa, q, k, v, do, causal)
    for name, g, r in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]), (ref[0], ref[1], ref[3], ref[4])):
        assert torch.equal(g, r), name
    dq_err = float((got[2].float() - ref[2].float()).norm() / ref[2].float().norm())
    assert dq_err <= 1e-3, dq_err


def test_against_oracle():
    fa = fa_mod()
    B, Hq, Hkv, N, d = 2, 4, 2, 300, 64
    q, k, v, do = make_qkv(B, Hq, Hkv, N, d, seed=61, with_do=True)
    o, lse, dq, dk, dv = fa.fwd_bwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), do.pin_memory(), True)
    fa.check()
    scale = 1 / math.sqrt(d)
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), True, scale)
    assert_fwd_close(o.float().numpy(), lse.numpy(), O_ref, L_ref, "host step")
    ref = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), True, scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_close(name, g.float().numpy(), r, what="host step")


def test_pageable_buffers_and_back_to_back_calls_share_a_workspace():
    fa = fa_mod()
    B, Hq, Hkv, N, d = 2, 4, 2, 640, 128
    ins = [make_qkv(B, Hq, Hkv, N, d, seed=62 + i, value_scale=0.5, with_do=True) for i in range(2)]
    ws = torch.empty(fa.fwd_bwd_host_workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device="cuda")
    outs = [fa.fwd_bwd_host(*x, True, workspace=ws) for x in ins]  # pageable inputs, no sync between
    fa.check()
    for x, got in zip(ins, outs):
        ref = _device_path(fa, *x, True)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        assert torch.equal(got[3], ref[3]) and torch.equal(got[4], ref[4])


def test_workspace_errors():
    fa = fa_mod()
    q, k, v, do = make_qkv(1, 2, 2, 128, 64, seed=63, with_do=True)
    small = torch.empty(fa.fwd_bwd_host_workspace_bytes(1, 2, 2, 128, 64) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError):
        fa.fwd_bwd_host(q, k, v, do, True, workspace=small)
    with pytest.raises(ValueError):
        fa.fwd_bwd_host(q.cuda(), k, v, do, True)


def test_full_size_bench_workload_matches_device_path():
    # The shape and inputs the end-to-end benchmark times: B=4, Hq=32, Hkv=8, N=4096, d=128,
    # causal, N(0,1)*0.5 from seed 2 (two chunks of four kv heads per batch element).
    fa = fa_mod()
    B, Hq, Hkv, N, d = 4, 32, 8, 4096, 128
    q, k, v, do = (t.pin_memory() for t in make_qkv(B, Hq, Hkv, N, d, seed=2, value_scale=0.5, with_do=True))
    got = fa.fwd_bwd_host(q, k, v, do, True)
    fa.check()
    ref = _device_path(fa, q, k, v, do, True)
    for name, g, r in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]), (ref[0], ref[1], ref[3], ref[4])):
        assert torch.equal(g, r), name
    dq_err = float((got[2].float() - ref[2].float()).norm() / ref[2].float().norm())
    assert dq_err <= 1e-3, dq_err
