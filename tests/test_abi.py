"""The C-ABI library builds, loads and exports every function include/fa.h declares.

No GPU needed: only argument checks that return before any CUDA call are exercised.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from online_softmax_09_gb300 import build, fa

    build.build()
    return fa.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*\*?\s*(fa_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_fwd_stats", "fa_check", "fa_strerror", "fa_version",
              "fa_bwd_prepare", "fa_bwd_compute", "fa_bwd_finalize"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    from online_softmax_09_gb300 import fa

    for s in range(0, -8, -1):
        assert fa.strerror(s) and fa.strerror(s) != "unknown status"
    assert fa.strerror(-99) == "unknown status"
    assert L.fa_version() >> 16 == 1


def _fwd(L, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, Hq=1, Hkv=1, N=128, d=128):
    return L.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, 0, 0.0, None)


def test_argument_errors_return_before_any_launch(L):
    assert _fwd(L, q=None) == -1  # null pointer
    assert _fwd(L, N=0) == -1
    assert _fwd(L, B=0) == -1
    assert _fwd(L, Hq=3, Hkv=2) == -1  # Hq % Hkv != 0
    assert _fwd(L, d=96) == -2  # unsupported head dim
    assert _fwd(L, d=256) == -2
    assert _fwd(L, k=0x1008) == -3  # misaligned
    assert _fwd(L, lse=0x1004) == -3
    assert L.fa_fwd_stats(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 1, 128, 128, 0, 0.0, None, None) == -1


def test_workspace_size_is_linear_in_n(L):
    ws = [L.fa_bwd_workspace_bytes(2, 8, 2, n, 128) for n in (1024, 2048, 4096)]
    assert ws[2] - ws[1] == 2 * (ws[1] - ws[0])  # affine in N: no N^2 term
    assert ws[0] >= 2 * 8 * 1024 * (128 + 2) * 4
    assert L.fa_bwd_workspace_bytes(1, 3, 2, 128, 128) == 0  # invalid sizes
    # Backward argument errors.
    args = [0x1000] * 9
    assert L.fa_bwd(*args, 0x1000, 0, 1, 1, 1, 128, 128, 0, 0.0, None) == -6  # workspace too small
    assert L.fa_bwd(*args, None, 1 << 30, 1, 1, 1, 128, 128, 0, 0.0, None) == -6
    assert L.fa_bwd(*args, 0x1001, 1 << 30, 1, 1, 1, 128, 128, 0, 0.0, None) == -3


def _host_step_bytes(L, B, Hq, Hkv, N, d):
    """The documented layout: each batch element in s chunks of Hkv/s kv heads (s the smallest
    divisor of Hkv with B*s >= 8, else Hkv); device copies of the nine tensors, each chunk's lse
    from a 256-byte boundary, and one chunk-sized backward workspace per compute stream
    (min(B*s, 4) streams)."""
    a = lambda x: (x + 255) // 256 * 256
    s = next((s for s in range(1, Hkv + 1) if Hkv % s == 0 and B * s >= 8), Hkv)
    nkv = Hkv // s
    nq = nkv * (Hq // Hkv)
    q, kv = B * Hq * N * d * 2, B * Hkv * N * d * 2
    return (4 * a(q) + 4 * a(kv) + B * s * a(nq * N * 4)
            + min(B * s, 4) * a(L.fa_bwd_workspace_bytes(1, nq, nkv, N, d)))


def test_host_step_workspace_and_argument_errors(L):
    B, Hq, Hkv, N, d = 2, 8, 2, 1000, 128
    for shape in [(B, Hq, Hkv, N, d), (4, 32, 8, 4096, 128), (1, 32, 8, 4096, 128), (16, 16, 16, 1024, 64),
                  (1, 1, 1, 128, 128), (3, 6, 3, 333, 64), (2, 3, 1, 129, 64), (5, 8, 4, 77, 128)]:
        assert L.fa_fwd_bwd_host_workspace_bytes(*shape) == _host_step_bytes(L, *shape), shape
    # The Llama-3.1-8B shape: each batch element in 2 chunks of four kv heads (16 query heads);
    # the nine tensors (all sizes multiples of 256 B) plus 4 chunk-sized workspaces.
    tensors = 4 * (4 * 32 * 4096 * 128 * 2) + 4 * (4 * 8 * 4096 * 128 * 2) + 4 * 32 * 4096 * 4
    assert L.fa_fwd_bwd_host_workspace_bytes(4, 32, 8, 4096, 128) == tensors + 4 * L.fa_bwd_workspace_bytes(
        1, 16, 4, 4096, 128)
    assert L.fa_fwd_bwd_host_workspace_bytes(B, 3, 2, N, d) == 0  # Hq % Hkv != 0
    assert L.fa_fwd_bwd_host_workspace_bytes(0, Hq, Hkv, N, d) == 0
    ptrs = [0x1000] * 9
    ws = L.fa_fwd_bwd_host_workspace_bytes(1, 1, 1, 128, 128)
    assert L.fa_fwd_bwd_host(*ptrs, 1, 1, 1, 128, 128, 0, 0.0, 0x1000, ws - 1, None) == -6  # too small
    assert L.fa_fwd_bwd_host(*ptrs, 1, 1, 1, 128, 128, 0, 0.0, None, ws, None) == -6
    assert L.fa_fwd_bwd_host(*ptrs, 1, 1, 1, 128, 128, 0, 0.0, 0x1080, ws, None) == -3  # not 256-aligned
    assert L.fa_fwd_bwd_host(None, *ptrs[1:], 1, 1, 1, 128, 128, 0, 0.0, 0x1000, ws, None) == -1
    assert L.fa_fwd_bwd_host(*ptrs, 1, 1, 1, 128, 96, 0, 0.0, 0x1000, ws, None) == -1  # d = 96: no layout


def test_splitkv_auto_choice(L):
    # Host-only cost model: no split when the GPU is full or the work items are already short,
    # a split when a few long causal items would otherwise run alone.
    assert L.fa_fwd_splitkv_auto(4, 32, 8, 4096, 128, 1, 152) == 1   # 2048 work items
    assert L.fa_fwd_splitkv_auto(1, 8, 8, 8192, 128, 1, 152) == 1    # enough work per SM already
    assert L.fa_fwd_splitkv_auto(1, 16, 16, 1024, 128, 1, 152) == 1  # items of at most 8 key tiles
    assert L.fa_fwd_splitkv_auto(1, 2, 2, 8192, 128, 1, 152) > 1     # 64 items, the longest 64 tiles
    assert L.fa_fwd_splitkv_auto(1, 4, 4, 4096, 128, 1, 152) > 1
    for shape in [(1, 1, 1, 1, 64, 0), (1, 2, 1, 300, 128, 1), (2, 4, 2, 131072, 64, 0)]:
        assert 1 <= L.fa_fwd_splitkv_auto(*shape, 152) <= 16
    assert L.fa_fwd_splitkv_auto(1, 2, 1, 300, 128, 1, 1) >= 1
    assert L.fa_fwd_splitkv_auto(1, 3, 2, 300, 128, 1, 152) < 0      # Hq % Hkv != 0
    assert L.fa_fwd_splitkv_auto(1, 2, 1, 300, 96, 1, 152) < 0       # d = 96
    assert L.fa_fwd_splitkv_auto(1, 2, 1, 300, 128, 1, 0) < 0        # no SMs


def test_noalloc_checks_arguments_before_any_cuda_call(L):
    # fa_bwd_noalloc takes its checks in the order of the other entry points: sizes and
    # pointers, then its fixed scratch's size limit, both before any CUDA call (so they hold on
    # a machine without a GPU), then the device, then the scratch lookup.
    fn = L.fa_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    ok = [0x1000] * 9
    assert fn(None, *ok[1:], 1, 1, 1, 128, 128, 1, 0.0, None) == -1      # null pointer
    assert fn(*ok[:8], 0x1008, 1, 1, 1, 128, 128, 1, 0.0, None) == -3    # misaligned dv
    assert fn(*ok, 1, 3, 2, 128, 128, 1, 0.0, None) == -1                # Hq % Hkv != 0
    assert fn(*ok, 1, 1, 1, 128, 96, 1, 0.0, None) == -2                 # unsupported d
    assert fn(*ok, 1, 32, 8, 8192, 128, 1, 0.0, None) == -6              # beyond the 64 MiB scratch
