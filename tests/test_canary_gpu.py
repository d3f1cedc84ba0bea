"""Guard bytes around every output and workspace buffer the kernels write.

Each buffer handed to the library is the middle of a larger allocation whose first and last
GUARD bytes hold a fixed pattern; after the call the pattern must be intact, so no kernel wrote
outside the buffer it was given (an out-of-bounds write the oracle comparisons cannot see when
it lands in memory no test reads). Shapes are ragged (N not a multiple of 128), grouped and
degenerate (N = 1), where the tile edges are.
"""

import pytest
import torch

from gpu_util import fa_mod
from online_softmax_09_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; a multiple of 256 keeps the inner buffer's alignment
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a guard-filled byte allocation."""

    def __init__(self, shape, dtype, device="cuda", pin=False):
        numel = 1
        for s in shape:
            numel *= s
        self.nbytes = numel * torch.empty((), dtype=dtype).element_size()
        if device == "cpu":
            self.buf = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, pin_memory=pin)
        else:
            self.buf = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def intact(self):
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _workspace(nbytes):
    return Guarded((max(int(nbytes), 16),), torch.uint8)


SHAPES = [(2, 4, 2, 129, 64, True), (1, 3, 1, 300, 128, False), (2, 2, 2, 1, 128, True), (1, 8, 2, 257, 128, True)]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SHAPES)
def test_forward_and_backward_stay_inside_their_buffers(B, Hq, Hkv, N, d, causal):
    fa = fa_mod()
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=9000 + N + d, value_scale=0.5, with_do=True))
    o = Guarded(q.shape, torch.bfloat16)
    lse = Guarded((B, Hq, N), torch.float32)
    fa.forward(q, k, v, causal, out=o.t, lse=lse.t)
    dq, dk, dv = (Guarded(t.shape, torch.bfloat16) for t in (q, k, k))
    ws = _workspace(fa.workspace_bytes(B, Hq, Hkv, N, d))
    fa.backward(q, k, v, o.t, do, lse.t, causal, dq=dq.t, dk=dk.t, dv=dv.t, workspace=ws.t)
    fa.check()
    for name, g in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv), ("workspace", ws)):
        assert g.intact(), name
    assert torch.isfinite(dq.t.float()).all() and torch.isfinite(o.t.float()).all()


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SHAPES[:2])
def test_staged_backward_stays_inside_its_buffers(B, Hq, Hkv, N, d, causal):
    fa = fa_mod()
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=9100 + N, value_scale=0.5, with_do=True))
    o, lse = fa.forward(q, k, v, causal)
    dq, dk, dv = (Guarded(t.shape, torch.bfloat16) for t in (q, k, k))
    ws = _workspace(fa.workspace_bytes(B, Hq, Hkv, N, d))
    fa.backward_stages(q, k, v, o, do, lse, dq.t, dk.t, dv.t, ws.t, causal)
    fa.check()
    assert all(g.intact() for g in (dq, dk, dv, ws))


@pytest.mark.parametrize("window", [1, 129])
def test_window_passes_stay_inside_their_buffers(window):
    fa = fa_mod()
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 64
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=9200 + window, value_scale=0.5, with_do=True))
    o = Guarded(q.shape, torch.bfloat16)
    lse = Guarded((B, Hq, N), torch.float32)
    fa.forward_window(q, k, v, window, out=o.t, lse=lse.t)
    dq, dk, dv = (Guarded(t.shape, torch.bfloat16) for t in (q, k, k))
    ws = _workspace(fa.workspace_bytes(B, Hq, Hkv, N, d))
    fa.backward_window(q, k, v, o.t, do, lse.t, window, dq=dq.t, dk=dk.t, dv=dv.t, workspace=ws.t)
    fa.check()
    assert all(g.intact() for g in (o, lse, dq, dk, dv, ws))


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_and_naive_stay_inside_their_buffers(causal):
    fa = fa_mod()
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_qkv(B, Hq, Hkv, N, d, seed=9300, value_scale=0.5))
    o = Guarded(q.shape, torch.bfloat16)
    lse = Guarded((B, Hq, N), torch.float32)
    ws = _workspace(fa.lib().fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, N, d, 3))
    fa.forward_splitkv(q, k, v, causal, 3, out=o.t, lse=lse.t, workspace=ws.t)
    fa.check()
    assert all(g.intact() for g in (o, lse, ws))
    o2 = Guarded(q.shape, torch.bfloat16)
    lse2 = Guarded((B, Hq, N), torch.float32)
    ws2 = _workspace(fa.lib().fa_naive_workspace_bytes(B, Hq, Hkv, N, d))
    fa.forward_naive(q, k, v, causal, out=o2.t, lse=lse2.t, workspace=ws2.t)
    fa.check()
    assert all(g.intact() for g in (o2, lse2, ws2))


@pytest.mark.parametrize("rows,n", [(37, 100), (37, 333), (5, 3000), (3, 20000), (2, 9001)])
def test_softmax_rows_stay_inside_their_buffers(rows, n):
    fa = fa_mod()
    g = torch.Generator().manual_seed(rows * n)
    x = (torch.randn(rows, n, generator=g) * 4).cuda()
    p = Guarded((rows, n), torch.float32)
    lse = Guarded((rows,), torch.float32)
    fa.softmax_rows(x, out=p.t, lse=lse.t)
    fa.check()
    assert p.intact() and lse.intact()


def test_host_step_stays_inside_its_buffers():
    fa = fa_mod()
    B, Hq, Hkv, N, d = 3, 6, 3, 129, 64
    q, k, v, do = (t.pin_memory() for t in make_qkv(B, Hq, Hkv, N, d, seed=9400, value_scale=0.5, with_do=True))
    outs = [Guarded(q.shape, torch.bfloat16, "cpu", pin=True), Guarded((B, Hq, N), torch.float32, "cpu", pin=True),
            Guarded(q.shape, torch.bfloat16, "cpu", pin=True), Guarded(k.shape, torch.bfloat16, "cpu", pin=True),
            Guarded(k.shape, torch.bfloat16, "cpu", pin=True)]
    ws = _workspace(fa.fwd_bwd_host_workspace_bytes(B, Hq, Hkv, N, d))
    fa.fwd_bwd_host(q, k, v, do, True, out=tuple(g.t for g in outs), workspace=ws.t)
    fa.check()
    assert all(g.intact() for g in outs) and ws.intact()
