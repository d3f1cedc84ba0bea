"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (a plugin whose host runtime owns all device memory, a loop where cudaMalloc's
implicit synchronisation is not allowed) get the workspace from a fixed array inside the
library instead of passing one. These tests call the entry point through the C ABI and check
it against fa_bwd, the entry point that takes a caller-allocated workspace, on two calls in a
row with different shapes, so a second call cannot pass on stale scratch contents, and one
call directly against the fp64 oracle. The file is named so that pytest collects it last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import GRAD_REL_TOL, assert_grad_close, fa_mod, rel_fro
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu

_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


def _noalloc():
    fa = fa_mod()
    L = fa.lib()
    fn = L.fa_bwd_noalloc
    fn.argtypes = [_vp] * 9 + [_i, _i, _i, _i, _i, _i, _f, _vp]
    fn.restype = _i
    return fa, fn


def _compare_once(fa, fn, B, Hq, Hkv, N, d, causal, seed):
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=seed, with_do=True))
    o, lse = fa.forward(q, k, v, causal)
    ref = fa.backward(q, k, v, o, do, lse, causal)  # caller-allocated workspace
    got = [torch.full_like(t, float("nan")) for t in ref]
    stream = torch.cuda.current_stream().cuda_stream
    r = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
           got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), B, Hq, Hkv, N, d, int(causal), 0.0, stream)
    assert r == 0, fa.strerror(r)
    fa.check()
    for name, g, w in zip(("dq", "dk", "dv"), got, ref):
        g = g.float().cpu().numpy()
        w = w.float().cpu().numpy()
        assert np.all(np.isfinite(g)), name
        assert rel_fro(g, w) <= GRAD_REL_TOL, name


def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    fa, fn = _noalloc()
    _compare_once(fa, fn, 2, 4, 2, 640, 128, True, seed=41)
    _compare_once(fa, fn, 1, 6, 3, 300, 64, False, seed=42)


def test_noalloc_matches_the_oracle():
    # One call checked against the fp64 oracle itself, with the same bounds as every backward
    # parity test (relative Frobenius and element-wise), on a grouped, ragged causal shape.
    fa, fn = _noalloc()
    B, Hq, Hkv, N, d = 2, 4, 2, 333, 128
    qh, kh, vh, doh = make_qkv(B, Hq, Hkv, N, d, seed=44, with_do=True)
    q, k, v, do = (t.cuda() for t in (qh, kh, vh, doh))
    o, lse = fa.forward(q, k, v, True)
    got = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    stream = torch.cuda.current_stream().cuda_stream
    r = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
           got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), B, Hq, Hkv, N, d, 1, 0.0, stream)
    assert r == 0, fa.strerror(r)
    fa.check()
    ref = oracle.attention_backward(to_f64(qh), to_f64(kh), to_f64(vh), to_f64(doh), True, 1 / math.sqrt(d))
    for name, g, w in zip(("dq", "dk", "dv"), got, ref):
        assert_grad_close(name, g.float().cpu().numpy(), w, what="fa_bwd_noalloc")


def test_noalloc_rejects_problems_larger_than_its_scratch():
    fa, fn = _noalloc()
    # 64 MiB holds about 129,000 padded query rows at d = 128; 32 heads x 8192 rows is twice that.
    assert fa.workspace_bytes(1, 32, 8, 8192, 128) > 64 << 20
    dummy = 0x1000  # never dereferenced: the size check comes first and nothing is launched
    r = fn(*([dummy] * 9), 1, 32, 8, 8192, 128, 1, 0.0, None)
    assert r == -6, fa.strerror(r)


def test_python_binding_matches_fa_bwd():
    # fa.backward_noalloc marshals the same call: dK and dV (no reductions across CTAs) are
    # bit-identical to fa_bwd's, dQ agrees to its fp32 reduction order.
    fa, _ = _noalloc()
    q, k, v, do = (t.cuda() for t in make_qkv(2, 4, 2, 257, 128, seed=43, with_do=True))
    o, lse = fa.forward(q, k, v, True)
    ref = fa.backward(q, k, v, o, do, lse, True)
    got = fa.backward_noalloc(q, k, v, o, do, lse, True)
    fa.check()
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    assert rel_fro(got[0].float().cpu().numpy(), ref[0].float().cpu().numpy()) <= 1e-3
