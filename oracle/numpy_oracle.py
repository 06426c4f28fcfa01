"""numpy FP64 restatement of the pages' attention algorithms -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
anything under ``oracle/``.  This module shares no code with the CUDA path.

It restates, in float64 and in the pages' own notation, the algorithms of
"flash_lab.py -- FlashAttention, flash-decoding and megakernel in numpy"
(CS349E lecture 11 shared module):

* section 1 (online softmax): ``softmax_3pass``, ``softmax_online``,
  ``partial_state``, ``merge_states``;
* section 2 (standard attention): ``causal_mask``, ``standard_attention``;
* section 2 (standard attention backward): ``standard_attention_bwd``;
* section 3 (FlashAttention): ``flash_fwd_tiled`` -- the FlashAttention-2 loop
  order (outer loop over query tiles, inner loop over key/value tiles, the
  running max m and sum l rescaled by exp(m_old - m_new), one division by l
  at the end, L = m + log l, and the causal "stop at the first fully masked
  tile" rule), and ``flash_bwd_tiled`` -- the FlashAttention-2 form of the
  backward (outer loop over key/value tiles, P recomputed as exp(S - L));
* section 4 (flash-decoding): ``split_kv_decode`` -- split the keys into
  segments, normalise each segment's output, keep its log-sum-exp, merge.

The C library in this directory (``fa_oracle.c``) is the fast form of the
same definition used for large parity checks; this module is the second,
independent statement used to pin it on small shapes and to model the tiled
algorithm's masking and skipping on the CPU.
"""
from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------
# section 1: online softmax
# --------------------------------------------------------------------------
def softmax_3pass(x):
    """Safe softmax along the last axis: max, then sum of exp(x - max), then divide."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def softmax_online(x, block=128):
    """One pass for (m, l) over blocks, rescaling l by exp(m - m_new); a second pass divides."""
    x = np.asarray(x, dtype=np.float64)
    m = np.full(x.shape[:-1] + (1,), -np.inf)
    l = np.zeros(x.shape[:-1] + (1,))
    for start in range(0, x.shape[-1], block):
        xb = x[..., start:start + block]
        m_new = np.maximum(m, xb.max(axis=-1, keepdims=True))
        l = l * np.exp(m - m_new) + np.exp(xb - m_new).sum(axis=-1, keepdims=True)
        m = m_new
    return np.exp(x - m) / l


def partial_state(x, v=None):
    """(m, l, o) of one segment: m = max, l = sum exp(x - m), o = sum exp(x - m) v."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1)
    p = np.exp(x - m[..., None])
    l = p.sum(axis=-1)
    o = None if v is None else p @ np.asarray(v, dtype=np.float64)
    return m, l, o


def merge_states(a, b):
    """Associative, commutative merge of two (m, l, o) states; an all -inf state has weight 0."""
    ma, la, oa = a
    mb, lb, ob = b
    m = np.maximum(ma, mb)
    with np.errstate(invalid="ignore"):
        wa = np.where(np.isneginf(ma), 0.0, np.exp(ma - m))
        wb = np.where(np.isneginf(mb), 0.0, np.exp(mb - m))
    l = la * wa + lb * wb
    o = None if oa is None else oa * wa[..., None] + ob * wb[..., None]
    return m, l, o


# --------------------------------------------------------------------------
# section 2: standard attention
# --------------------------------------------------------------------------
def causal_mask(nq, nk, q0=0, k0=0, offset=0):
    """Boolean [nq, nk]: True where allowed.  Query q0+r sits at offset+q0+r, key k0+c at k0+c."""
    qpos = offset + q0 + np.arange(nq)[:, None]
    kpos = k0 + np.arange(nk)[None, :]
    return kpos <= qpos


def standard_attention(Q, K, V, causal=False, scale=None):
    """S = Q K^T * scale, causal mask (offset Nk - N), 3-pass softmax, O = P V.

    Returns (O, LSE, P).  A row with no visible key gets O = 0, LSE = -inf and
    a zero P row (the reading the C oracle also takes).
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    N, d = Q.shape
    Nk = K.shape[0]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    S = (Q @ K.T) * scale
    if causal:
        S = np.where(causal_mask(N, Nk, offset=Nk - N), S, -np.inf)
    m = S.max(axis=1) if Nk > 0 else np.full(N, -np.inf)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])
    l = E.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    O = P @ V
    return O, lse, P


def standard_attention_bwd(Q, K, V, dO, causal=False, scale=None, return_terms=False):
    """Backward of standard attention with the full P materialised.

    dV = P^T dO; dP = dO V^T; D_i = sum_c dO_ic O_ic; dS = P o (dP - D);
    dQ = dS K scale; dK = dS^T Q scale.  Returns (dQ, dK, dV), followed by
    (P, dS) when ``return_terms``.
    """
    Q, K, V, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, dO))
    d = Q.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O, _, P = standard_attention(Q, K, V, causal, scale)
    D = np.sum(dO * O, axis=1)
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - D[:, None])
    if return_terms:
        return dS @ K * scale, dS.T @ Q * scale, dV, P, dS
    return dS @ K * scale, dS.T @ Q * scale, dV


# --------------------------------------------------------------------------
# section 3: FlashAttention, FlashAttention-2 loop order (tiled model)
# --------------------------------------------------------------------------
def flash_fwd_tiled(Q, K, V, Br, Bc, causal=False, scale=None):
    """Tiled forward in the FlashAttention-2 order.

    For each query tile (Br rows) keep m, l and the unnormalised accumulator
    on chip; for each key tile (Bc keys) form the masked score tile, update
    m_new = max(m, rowmax), alpha = exp(m - m_new), P = exp(S - m_new),
    l = alpha l + rowsum P, acc = alpha acc + P V; stop at the first tile
    whose first key lies after the tile's last query position (every later
    tile is masked too).  At the end O = acc / l and L = m + log l.

    Returns (O, L, visited) where ``visited`` lists the (query tile, key
    tile) pairs that were computed, for checking the skipping rule.
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    N, d = Q.shape
    Nk, dv = V.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    off = Nk - N
    O = np.zeros((N, dv))
    L = np.full(N, -np.inf)
    visited = []
    for i0 in range(0, N, Br):
        br = min(Br, N - i0)
        m = np.full(br, -np.inf)
        l = np.zeros(br)
        acc = np.zeros((br, dv))
        for j0 in range(0, Nk, Bc):
            if causal and off + i0 + br - 1 < j0:
                break
            bc = min(Bc, Nk - j0)
            visited.append((i0 // Br, j0 // Bc))
            S = (Q[i0:i0 + br] @ K[j0:j0 + bc].T) * scale
            if causal:
                S = np.where(causal_mask(br, bc, i0, j0, off), S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            m_use = np.where(np.isneginf(m_new), 0.0, m_new)
            alpha = np.where(np.isneginf(m), 0.0, np.exp(m - m_use))
            P = np.exp(S - m_use[:, None])
            l = alpha * l + P.sum(axis=1)
            acc = alpha[:, None] * acc + P @ V[j0:j0 + bc]
            m = m_new
        seen = l > 0
        with np.errstate(invalid="ignore", divide="ignore"):
            O[i0:i0 + br] = np.where(seen[:, None], acc / np.where(seen, l, 1.0)[:, None], 0.0)
            L[i0:i0 + br] = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)
    return O, L, visited


def flash_bwd_tiled(Q, K, V, O, dO, L, Br, Bc, causal=False, scale=None):
    """Tiled backward in the FlashAttention-2 order (recompute S and P from L).

    D_i = sum dO_i o O_i first.  The outer loop walks key/value tiles j (their
    dK_j, dV_j accumulate on chip), the inner loop walks query tiles i, skipping
    a tile whose last query position lies before the key tile's first key.
    Per (i, j): S = Q_i K_j^T scale (masked), P = exp(S - L_i),
    dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P o (dP - D_i),
    dQ_i += dS K_j scale, dK_j += dS^T Q_i scale.

    Returns (dQ, dK, dV, visited) with ``visited`` the (query tile, key tile)
    pairs computed.  A row with L = -inf (no visible key) gets P = 0.
    """
    Q, K, V, O, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, O, dO))
    L = np.asarray(L, dtype=np.float64)
    N, d = Q.shape
    Nk, dv = V.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    off = Nk - N
    D = (dO * O).sum(axis=1)
    dQ, dK, dV = np.zeros((N, d)), np.zeros((Nk, d)), np.zeros((Nk, dv))
    visited = []
    for j0 in range(0, Nk, Bc):
        bc = min(Bc, Nk - j0)
        dKj, dVj = np.zeros((bc, d)), np.zeros((bc, dv))
        for i0 in range(0, N, Br):
            br = min(Br, N - i0)
            if causal and off + i0 + br - 1 < j0:
                continue
            visited.append((i0 // Br, j0 // Bc))
            S = (Q[i0:i0 + br] @ K[j0:j0 + bc].T) * scale
            if causal:
                S = np.where(causal_mask(br, bc, i0, j0, off), S, -np.inf)
            Li = L[i0:i0 + br, None]
            with np.errstate(invalid="ignore"):
                P = np.where(np.isneginf(Li), 0.0, np.exp(S - np.where(np.isneginf(Li), 0.0, Li)))
            dVj += P.T @ dO[i0:i0 + br]
            dP = dO[i0:i0 + br] @ V[j0:j0 + bc].T
            dS = P * (dP - D[i0:i0 + br, None])
            dQ[i0:i0 + br] += dS @ K[j0:j0 + bc] * scale
            dKj += dS.T @ Q[i0:i0 + br] * scale
        dK[j0:j0 + bc] = dKj
        dV[j0:j0 + bc] = dVj
    return dQ, dK, dV, visited


# --------------------------------------------------------------------------
# section 4: flash-decoding (split KV, merge by log-sum-exp)
# --------------------------------------------------------------------------
def split_bounds(S, n_splits):
    """Segment boundaries for splitting S keys into n_splits parts (linspace, rounded)."""
    return np.linspace(0, S, n_splits + 1).round().astype(int)


def split_state(q, K, V, a, b, scale):
    """Normalised output o_s and log-sum-exp lse_s of queries q over keys [a, b)."""
    s = (q @ K[a:b].T) * scale
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p @ V[a:b]) / l, (m + np.log(l))[:, 0]


def merge_lse(parts):
    """lse = log sum_s exp(lse_s) (max-shifted); o = sum_s exp(lse_s - lse) o_s."""
    lses = np.stack([p[1] for p in parts])
    top = lses.max(axis=0)
    lse = top + np.log(np.exp(lses - top).sum(axis=0))
    o = sum(np.exp(ls - lse)[:, None] * o_s for o_s, ls in parts)
    return o, lse


def split_kv_decode(q, K, V, n_splits, scale=None, bounds=None):
    """Split the keys into segments, attend within each, merge.  Empty segments are skipped."""
    q, K, V = (np.asarray(t, dtype=np.float64) for t in (q, K, V))
    S, d = K.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    bounds = split_bounds(S, n_splits) if bounds is None else np.asarray(bounds)
    parts = [split_state(q, K, V, a, b, scale) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    o, lse = merge_lse(parts)
    return o, lse, parts
