"""Plain, slow, fp64 definitions of softmax attention and of the tiled method.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Conventions (the plainest reading where the pages leave a point open):

* Tensors are ``[B, H, N, d]`` float64 arrays (the pages slice queries as
  ``q[:, :, i:i+block]``, [P3] section 4). Queries and keys have the same
  length N ([P3] appendix: a single pass over one sequence, so the score
  matrix is square).
* Grouped-query attention: query head ``hq`` reads key/value head
  ``hq // G`` with ``G = Hq // Hkv`` (contiguous groups). The pages mention GQA
  only for Llama's head counts ([P3] section 6); this mapping is a reading.
* Causal: query ``i`` sees keys ``0..i`` inclusive; scores above the diagonal
  become minus infinity ([P3] section 5).
* The per-row statistic saved for the backward pass is the natural-log
  log-sum-exp ``LSE_i = m_i + ln(l_i)`` of the scaled scores. [P3] section 8
  mentions only statistics kept from the forward pass; LSE is the one scalar that lets P be
  recomputed as ``exp(S - LSE)``.
"""

from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Standard attention (the definition the method must reproduce exactly).
# --------------------------------------------------------------------------


def _kv_head(hq: int, Hq: int, Hkv: int) -> int:
    """Key/value head read by query head ``hq`` (contiguous GQA groups)."""
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // (Hq // Hkv)


def _causal_mask(n_q: int, n_k: int, q_start: int = 0, k_start: int = 0) -> np.ndarray:
    """Boolean mask, True where key position > query position (the future).

    [P3] section 5: causal attention forces the scores above the diagonal to
    minus infinity so the softmax gives them weight zero.
    """
    qi = np.arange(q_start, q_start + n_q)[:, None]
    kj = np.arange(k_start, k_start + n_k)[None, :]
    return kj > qi


def _masked(n_q: int, n_k: int, causal: bool, window=None, q_start: int = 0, k_start: int = 0):
    """True where a key is invisible to a query: in the future (causal), or, with a sliding
    window of w keys, older than the w most recent ones: key < query - w + 1 ([P3] section 5,
    sliding_window_attention's too_old mask, which is causal as well). None: nothing masked."""
    mask = None
    if causal or window is not None:
        mask = _causal_mask(n_q, n_k, q_start, k_start)
    if window is not None:
        qi = np.arange(q_start, q_start + n_q)[:, None]
        kj = np.arange(k_start, k_start + n_k)[None, :]
        mask = mask | (kj < qi - window + 1)
    return mask


def attention_probs(q: np.ndarray, k: np.ndarray, causal: bool, scale: float, window=None) -> np.ndarray:
    """Row-softmax weights P for ONE head: q [N,d], k [N,d] -> P [N,N].

    Numerically stable softmax with the row max subtracted ([P3] section 2,
    [P1] "The Running Statistics"): ``P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)``.
    """
    S = scale * (q @ k.T)
    mask = _masked(q.shape[0], k.shape[0], causal, window)
    if mask is not None:
        S = np.where(mask, -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    return P / P.sum(axis=1, keepdims=True)


def attention_forward_head(q, k, v, causal: bool, scale: float, window=None):
    """Standard attention for one head, fully materialised ([P3] section 1).

    ``S = scale * Q K^T``; masked if causal; ``m = rowmax(S)``;
    ``P = exp(S - m)``; ``l = rowsum(P)``; ``O = (P / l) V``; ``LSE = m + ln l``.
    Returns ``(O [N,d], LSE [N])``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S = scale * (q @ k.T)
    mask = _masked(q.shape[0], k.shape[0], causal, window)
    if mask is not None:
        S = np.where(mask, -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    O = (P / l) @ v
    lse = m[:, 0] + np.log(l[:, 0])
    return O, lse


def attention_forward(q, k, v, causal: bool, scale: float, window=None):
    """Standard attention over ``[B,Hq,N,d]`` / ``[B,Hkv,N,d]`` arrays.

    Head by head (to bound memory); returns ``(O [B,Hq,N,d], LSE [B,Hq,N])``.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    O = np.empty((B, Hq, N, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, Hq, N), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            hk = _kv_head(h, Hq, Hkv)
            O[b, h], lse[b, h] = attention_forward_head(q[b, h], k[b, hk], v[b, hk], causal, scale, window)
    return O, lse


def attention_rows(q_rows, k, v, rows, causal: bool, scale: float, window=None):
    """Standard attention for SELECTED query rows of one head.

    ``q_rows`` [R,d] holds the queries at absolute positions ``rows`` (for the
    causal mask); ``k``, ``v`` [N,d] hold every key of the head. Used where the
    full N x N matrix is too large for the CPU, e.g. N = 131072.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows)
    S = scale * (q_rows @ k.T)
    if causal or window is not None:
        S = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, S)
    if window is not None:
        S = np.where(np.arange(k.shape[0])[None, :] < rows[:, None] - window + 1, -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    return (P / l) @ v, m[:, 0] + np.log(l[:, 0])


# --------------------------------------------------------------------------
# Backward pass.
# --------------------------------------------------------------------------


def attention_backward_head(q, k, v, do, causal: bool, scale: float, window=None):
    """Gradients of standard attention for one head.

    [P3] section 8 (its paragraph on the backward pass) says only that the
    probabilities are recomputed from Q, K, V and statistics kept from the
    forward pass. The
    gradient itself is the textbook one for ``O = softmax(scale Q K^T) V``:
    ``dV = P^T dO``; ``dP = dO V^T``; ``delta = rowsum(dO * O)``;
    ``dS = P * (dP - delta)``; ``dQ = scale dS K``; ``dK = scale dS^T Q``.
    Returns ``(dQ, dK, dV)`` for this head.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    P = attention_probs(q, k, causal, scale, window)
    O = P @ v
    dV = P.T @ do
    dP = do @ v.T
    delta = np.sum(do * O, axis=1, keepdims=True)
    dS = P * (dP - delta)
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV


def attention_backward(q, k, v, do, causal: bool, scale: float, heads=None, window=None):
    """Gradients over ``[B,Hq,N,d]`` arrays; dK, dV summed over each GQA group.

    ``heads`` optionally restricts the computation to a list of ``(b, hkv)``
    groups (the other entries of the returned arrays are NaN), for configs
    whose full backward is too slow on the CPU.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    groups = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for b, hk in groups:
        dk[b, hk] = 0.0
        dv[b, hk] = 0.0
        for hq in range(hk * G, (hk + 1) * G):
            gq, gk, gv = attention_backward_head(q[b, hq], k[b, hk], v[b, hk], do[b, hq], causal, scale, window)
            dq[b, hq] = gq
            dk[b, hk] += gk
            dv[b, hk] += gv
    return dq, dk, dv


# --------------------------------------------------------------------------
# Brute force (explicit loops, no matrix products) for tiny inputs.
# --------------------------------------------------------------------------


def brute_force_attention(q, k, v, causal: bool, scale: float, window=None):
    """Softmax attention by explicit scalar loops (one head, small N only).

    Written straight from the softmax definition of [P1] ("Here's the
    challenge") without the max shift: ``w_ij = e^{s_ij} / sum_j e^{s_ij}``.
    Returns ``(O, LSE)`` as nested Python lists of floats.
    """
    N, d = len(q), len(q[0])
    dv = len(v[0])
    O, lse = [], []
    for i in range(N):
        keys = range(i + 1) if (causal or window is not None) else range(N)
        if window is not None:
            keys = range(max(0, i - window + 1), i + 1)
        s = {}
        for j in keys:
            acc = 0.0
            for t in range(d):
                acc += float(q[i][t]) * float(k[j][t])
            s[j] = scale * acc
        z = sum(math.exp(s[j]) for j in keys)
        row = []
        for c in range(dv):
            row.append(sum(math.exp(s[j]) / z * float(v[j][c]) for j in keys))
        O.append(row)
        lse.append(math.log(z))
    return O, lse


# --------------------------------------------------------------------------
# The online softmax and the tiled loop, step by step as the pages state them.
# --------------------------------------------------------------------------


def _rebase(m_old, m_new):
    """exp(m_old - m_new), taken as 0 where nothing has been seen yet (m_old = -inf)."""
    seen = ~np.isneginf(m_old)
    return np.where(seen, np.exp(np.where(seen, m_old - m_new, 0.0)), 0.0)


def online_softmax(x, block_size: int):
    """Single-pass online normaliser over the last axis ([P3] section 2, [P1]).

    The row is cut into blocks of ``block_size`` values. Each block has its own
    partial statistics, its maximum ``m_b`` and ``l_b = sum(exp(block - m_b))``;
    they are merged into the running ``(m, l)`` by rebasing both to the larger
    maximum ([P3] section 3, "Partial softmaxes compose"):
    ``m_new = max(m, m_b)``, ``correction = exp(m - m_new)``,
    ``l = l * correction + l_b * exp(m_b - m_new)`` -- the same running sum as
    ``l * correction + sum(exp(block - m_new))``. A second pass forms
    ``exp(x - m) / l``.

    Returns a dict: ``p`` (probabilities, same shape as x), ``m``, ``l``,
    ``lse`` (= m + ln l), ``trace`` (per block: m, correction, l for the
    first row) and ``rescales`` (per row: how many blocks moved the max,
    counting the first block).
    """
    x = np.asarray(x, dtype=np.float64)
    width = x.shape[-1]
    lead = x.shape[:-1]
    run_m = np.full(lead + (1,), -np.inf)
    run_l = np.zeros(lead + (1,))
    moved = np.zeros(lead, dtype=np.int64)
    trace = []
    first_row = (0,) * len(lead) + (0,)
    for part in np.split(x, np.arange(block_size, width, block_size), axis=-1):
        part_m = part.max(axis=-1, keepdims=True)
        part_l = np.exp(part - part_m).sum(axis=-1, keepdims=True)
        new_m = np.maximum(run_m, part_m)
        correction = _rebase(run_m, new_m)
        moved += (new_m > run_m)[..., 0]
        run_l = run_l * correction + part_l * np.exp(part_m - new_m)
        run_m = new_m
        trace.append({"m": float(run_m[first_row]), "correction": float(correction[first_row]),
                      "l": float(run_l[first_row])})
    p = np.exp(x - run_m) / run_l
    return {"p": p, "m": run_m[..., 0], "l": run_l[..., 0], "lse": run_m[..., 0] + np.log(run_l[..., 0]),
            "trace": trace, "rescales": moved}


def _tile_edges(length: int, block: int):
    """(start, stop) of the consecutive blocks of ``block`` rows covering ``length``."""
    starts = np.arange(0, length, block)
    return [(int(lo), int(min(lo + block, length))) for lo in starts]


def tiled_attention(q, k, v, causal: bool, scale: float, block_q: int, block_k: int):
    """The tiled two-level computation of [P3] section 4, in fp64, for one head.

    Query blocks of ``block_q`` rows each visit the key/value blocks of
    ``block_k`` rows. Every (query block, key block) tile yields a partial
    result relative to its own row maxima -- ``m_t = rowmax(s)``,
    ``p = exp(s - m_t)``, ``l_t = rowsum(p)``, ``o_t = p V`` -- which is merged
    into the query block's running ``(m, l, acc)`` by rebasing both sides to
    ``m_new = max(m, m_t)``: ``acc = acc exp(m - m_new) + o_t exp(m_t - m_new)``
    and likewise for ``l`` ([P3] section 3, "Partial softmaxes compose"; the
    pages fold the two factors into one correction of the running state). After
    the last tile ``O = acc / l``. With ``causal``, a tile whose first key lies
    after the block's last query is skipped ([P3] section 7) and diagonal tiles
    are masked element-wise ([P3] section 5).

    Returns ``(O, LSE, counters)``; counters follow [P3] section 8's tallies
    (two matmuls, i.e. ``4 rows cols d`` FLOPs, and the K and V tiles read, per
    computed tile) plus tile and rescale counts.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, d = q.shape
    O = np.empty((n_q, v.shape[1]))
    lse = np.empty(n_q)
    counters = {"tiles_computed": 0, "tiles_skipped": 0, "matmul_flops": 0,
                "kv_elements_read": 0, "rescales": 0}
    key_tiles = _tile_edges(k.shape[0], block_k)
    for q_lo, q_hi in _tile_edges(n_q, block_q):
        q_tile = q[q_lo:q_hi]
        m = np.full((q_hi - q_lo, 1), -np.inf)
        l = np.zeros((q_hi - q_lo, 1))
        acc = np.zeros((q_hi - q_lo, v.shape[1]))
        for k_lo, k_hi in key_tiles:
            if causal and k_lo >= q_hi:  # every key of the tile is after every query
                counters["tiles_skipped"] += 1
                continue
            k_tile, v_tile = k[k_lo:k_hi], v[k_lo:k_hi]
            counters["tiles_computed"] += 1
            counters["matmul_flops"] += 4 * q_tile.shape[0] * k_tile.shape[0] * d
            counters["kv_elements_read"] += k_tile.size + v_tile.size
            s = (q_tile @ k_tile.T) * scale
            if causal:
                s = np.where(_causal_mask(q_hi - q_lo, k_hi - k_lo, q_lo, k_lo), -np.inf, s)
            m_t = s.max(axis=1, keepdims=True)
            p = np.exp(s - np.where(np.isneginf(m_t), 0.0, m_t))
            m_new = np.maximum(m, m_t)
            keep = _rebase(m, m_new)
            take = _rebase(m_t, m_new)
            counters["rescales"] += int(np.sum((m_new > m) & ~np.isneginf(m)))
            l = l * keep + p.sum(axis=1, keepdims=True) * take
            acc = acc * keep + (p @ v_tile) * take
            m = m_new
        O[q_lo:q_hi] = acc / l
        lse[q_lo:q_hi] = m[:, 0] + np.log(l[:, 0])
    return O, lse, counters


# --------------------------------------------------------------------------
# Counts (no timing): tiles, FLOPs and HBM bytes as [P3] sections 7-8 tally them.
# --------------------------------------------------------------------------


def tile_schedule_counts(n: int, block_q: int, block_k: int, causal: bool,
                         batch: int = 1, heads: int = 1, dim: int = 64, elem: int = 4):
    """The tiled schedule's tallies, without arithmetic ([P3] sections 7-8).

    A tile is computed unless causal masking hides it whole (its first key
    after its last query). Per computed tile of ``rows`` queries and ``cols``
    keys the two matmuls cost ``4 rows cols dim`` FLOPs per (batch, head), and
    the K and V tiles are read from HBM (``2 cols dim`` elements); Q is read and
    O written once (``2 n dim`` elements) for the all-tensor traffic total.
    """
    visible = [(q_hi - q_lo, k_hi - k_lo)
               for q_lo, q_hi in _tile_edges(n, block_q)
               for k_lo, k_hi in _tile_edges(n, block_k)
               if not (causal and k_lo >= q_hi)]
    total_tiles = len(_tile_edges(n, block_q)) * len(_tile_edges(n, block_k))
    heads_total = batch * heads
    pair_count = sum(rows * cols for rows, cols in visible)
    key_rows = sum(cols for _, cols in visible)
    return {"computed": len(visible), "skipped": total_tiles - len(visible),
            "matmul_flops": 4 * heads_total * dim * pair_count,
            "hbm_bytes": heads_total * dim * elem * (2 * key_rows + 2 * n)}


def naive_counts(n: int, batch: int = 1, heads: int = 1, dim: int = 64, elem: int = 4):
    """Standard attention's counts ([P3] sections 1 and 8).

    FLOPs: the two matmuls over the whole matrix, ``2 (2 b h n n d)``.
    Score traffic: S written, read, P written, read: ``4 b h n^2 elem``.
    All-tensor traffic adds Q, K, V reads and the O write: ``4 b h n d elem``.
    """
    flops = 2 * (2 * batch * heads * n * n * dim)
    score = 4 * batch * heads * n * n * elem
    return {"matmul_flops": flops, "score_bytes": score,
            "hbm_bytes": score + 4 * batch * heads * n * dim * elem}


def causal_tile_counts(n: int, block: int):
    """(computed, skipped) square tiles for causal attention ([P3] section 7)."""
    c = tile_schedule_counts(n, block, block, True)
    return c["computed"], c["skipped"]


def algorithmic_flops(B: int, Hq: int, N: int, d: int, causal: bool) -> int:
    """Forward matmul FLOPs counted over VISIBLE (query, key) pairs only.

    Each visible pair costs one multiply-add in ``Q K^T`` and one in ``P V``
    per head-dimension element: ``4 d`` FLOPs ([P3] section 8's 2-per-MAC
    convention). Non-causal: ``4 N^2 d`` per head; causal:
    ``4 d N (N+1) / 2``.
    """
    pairs = N * (N + 1) // 2 if causal else N * N
    return 4 * d * pairs * B * Hq


def attention_backward_rows(q, k, v, do, q_rows, k_rows, causal: bool, scale: float, chunk: int = 1024,
                            window=None):
    """Backward of standard attention for ONE head, on selected rows only.

    Returns ``(dQ[q_rows], dK[k_rows], dV[k_rows])`` without forming the N x N matrices:
    the row statistics (LSE, delta) are computed over query chunks of ``chunk`` rows, then
    ``dQ_i = scale sum_j P_ij (dP_ij - delta_i) K_j`` for the selected queries and
    ``dV_j = sum_i P_ij dO_i``, ``dK_j = scale sum_i P_ij (dP_ij - delta_i) Q_i`` for the
    selected keys, with ``P_ij = exp(scale q_i.k_j - LSE_i)`` and ``dP_ij = dO_i . v_j``.
    Same definitions as :func:`attention_backward_head`, evaluated on a subset.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    N = q.shape[0]
    lse = np.empty(N)
    delta = np.empty(N)
    for s in range(0, N, chunk):
        rows = np.arange(s, min(N, s + chunk))
        O_c, lse[rows] = attention_rows(q[rows], k, v, rows, causal, scale, window)
        delta[rows] = np.sum(do[rows] * O_c, axis=1)
    q_rows = np.asarray(q_rows)
    k_rows = np.asarray(k_rows)
    # dQ for the selected queries.
    S = scale * (q[q_rows] @ k.T)
    if causal or window is not None:
        S = np.where(np.arange(N)[None, :] > q_rows[:, None], -np.inf, S)
    if window is not None:
        S = np.where(np.arange(N)[None, :] < q_rows[:, None] - window + 1, -np.inf, S)
    P = np.exp(S - lse[q_rows, None])
    dS = P * (do[q_rows] @ v.T - delta[q_rows, None])
    dQ = scale * (dS @ k)
    # dK, dV for the selected keys.
    dK = np.zeros((len(k_rows), q.shape[1]))
    dV = np.zeros((len(k_rows), v.shape[1]))
    for s in range(0, N, chunk):
        rows = np.arange(s, min(N, s + chunk))
        St = scale * (q[rows] @ k[k_rows].T)
        if causal or window is not None:
            St = np.where(k_rows[None, :] > rows[:, None], -np.inf, St)
        if window is not None:
            St = np.where(k_rows[None, :] < rows[:, None] - window + 1, -np.inf, St)
        Pt = np.exp(St - lse[rows, None])
        dSt = Pt * (do[rows] @ v[k_rows].T - delta[rows, None])
        dV += Pt.T @ do[rows]
        dK += scale * (dSt.T @ q[rows])
    return dQ, dK, dV


def attention_query_block(q, k, v, do, rows, causal: bool, scale: float):
    """Forward and backward share of ONE block of query rows of one head.

    Standard attention is row-separable in the queries: O, LSE and dQ of a query row
    depend only on that row, and dK, dV are sums over query rows of per-row terms
    (``dV = sum_i P_i^T dO_i``, ``dK = scale sum_i dS_i^T Q_i``). This returns, for the
    rows ``rows``: ``O_R``, ``LSE_R``, ``dQ_R`` and the rows' contributions ``dK_R``,
    ``dV_R`` (full N x d arrays), with the same definitions as
    :func:`attention_forward_head` and :func:`attention_backward_head`. Summing the
    contributions over a partition of the rows gives the full dK and dV.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    rows = np.asarray(rows)
    S = scale * (q[rows] @ k.T)
    if causal:
        S = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    P = P / l
    O = P @ v
    delta = np.sum(do[rows] * O, axis=1, keepdims=True)
    dS = P * (do[rows] @ v.T - delta)
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q[rows])
    dV = P.T @ do[rows]
    return O, m[:, 0] + np.log(l[:, 0]), dQ, dK, dV


def attention_split_forward_head(q, k, v, causal: bool, scale: float, splits: int):
    """Forward of one head computed as `splits` partial softmaxes over contiguous key ranges,
    then merged ([P3] section 3, "Partial softmaxes compose"): each range gives a partial
    output O_s (normalised over its own keys) and LSE_s (minus infinity when a row sees none
    of its keys); with m = max_s LSE_s and w_s = exp(LSE_s - m),
    O = sum_s w_s O_s / sum_s w_s and LSE = m + ln(sum_s w_s)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N = k.shape[0]
    bounds = np.linspace(0, N, splits + 1).astype(int)
    parts = []
    for s0, s1 in zip(bounds[:-1], bounds[1:]):
        S = scale * (q @ k[s0:s1].T)
        if causal:
            S = np.where(_causal_mask(q.shape[0], s1 - s0, 0, s0), -np.inf, S)
        m = S.max(axis=1, keepdims=True) if s1 > s0 else np.full((q.shape[0], 1), -np.inf)
        with np.errstate(invalid="ignore"):
            P = np.exp(S - np.where(np.isneginf(m), 0.0, m))
        l = P.sum(axis=1, keepdims=True)
        with np.errstate(invalid="ignore", divide="ignore"):
            O_s = np.where(l > 0, (P @ v[s0:s1]) / np.where(l > 0, l, 1.0), 0.0)
            lse_s = np.where(l[:, 0] > 0, m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
        parts.append((O_s, lse_s))
    m = np.max([ls for _, ls in parts], axis=0)
    w = [np.exp(ls - m) for _, ls in parts]
    wsum = np.sum(w, axis=0)
    O = sum(wi[:, None] * Oi for wi, (Oi, _) in zip(w, parts)) / wsum[:, None]
    return O, m + np.log(wsum)
