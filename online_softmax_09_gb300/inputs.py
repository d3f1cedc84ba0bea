"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no attention arithmetic: it only draws random tensors.
Recipe: one CPU ``torch.Generator`` seeded with ``seed``; ``randn`` drawn in
the order Q, K, V, dO, each ``[B, H, N, d]`` float32, multiplied by
``value_scale``, then rounded to bfloat16. Both the CUDA path and the fp64
oracle consume exactly these bf16 values (the oracle upcasts them exactly).

The adversarial variant (many running-max rescales): after the draws, Q is
multiplied by 8; for every (b, kv-head) one key index ``j`` is drawn uniformly
from the same generator and that key is set to ``20 * qbar``, where ``qbar``
is the mean over positions (and over the group's query heads) of the scaled Q.
"""

from __future__ import annotations

import torch


def make_qkv(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int, value_scale: float = 1.0,
             with_do: bool = False, adversarial: bool = False):
    """Return ``(q, k, v, do)`` as contiguous CPU bfloat16 tensors (``do`` may be None)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32) * value_scale
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32) * value_scale
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32) * value_scale
    do = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32) if with_do else None
    if adversarial:
        q = q * 8.0
        G = Hq // Hkv
        qbar = q.mean(dim=2).reshape(B, Hkv, G, d).mean(dim=2)  # [B, Hkv, d]
        j = torch.randint(0, N, (B, Hkv), generator=g)
        for b in range(B):
            for h in range(Hkv):
                k[b, h, int(j[b, h])] = 20.0 * qbar[b, h]
    out = [t.to(torch.bfloat16).contiguous() for t in (q, k, v)]
    out.append(do.to(torch.bfloat16).contiguous() if do is not None else None)
    return tuple(out)


def to_f64(t):
    """Exact upcast of a bf16 tensor to a float64 numpy array (no arithmetic)."""
    return t.detach().to("cpu", torch.float64).numpy()
