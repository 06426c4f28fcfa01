"""numpy FP64 second statement of exact attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
anything under ``oracle/``.  This module shares no code with the CUDA path.

What it states, in float64, and where the pages define it
("flash_lab.py -- FlashAttention, flash-decoding and megakernel in numpy",
CS349E lecture 11 shared module):

* ``attention_definition`` / ``attention_bwd_definition``: exact attention and
  its gradients with the score matrix materialised (section 2, standard
  attention and its backward); the value every tiled form must reach.
* ``RowState``: the per-row streaming normaliser of section 1 -- a running
  maximum, a running sum of exponentials taken relative to it and an
  accumulator of exponential-weighted value rows.  Absorbing a block whose
  maximum exceeds the running one re-expresses the old sum and accumulator
  relative to the new maximum (they are multiplied by exp(old - new)).
* ``segment_state`` / ``combine``: a partial result kept in log-sum-exp form,
  (normalised output, log of the segment's normaliser), and the exact merge of
  two such states (section 1's merge, section 4's combine).  The merge is
  written here in that form: the merged log-normaliser is the log of the sum of
  the two normalisers, and each side's output is weighted by its share.
* ``tiled_forward`` / ``tiled_backward``: the FlashAttention-2 loop orders of
  section 3 as a walk over the (query tile, key tile) grid that visits exactly
  the tiles holding at least one visible (query, key) pair (``tile_visible``,
  derived below from the causal convention), built from ``RowState``.
* ``split_decode``: section 4's split-KV decoding with near-equal integer
  segment bounds; segments are combined with ``combine``.

The causal convention is that of "02_flash_forward.py -- FlashAttention forward"
demo 1: query i of N sits at position Nk - N + i, key j at position j, and a
key is visible when its position does not exceed the query's.

The C library in this directory (``fa_oracle.c``) is the fast statement of the
same definition used for large parity checks; this module pins it on small
shapes and models the tiled kernels' masking and tile skipping on the CPU.
"""
from __future__ import annotations

import math
from functools import reduce

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# positions and visibility
# --------------------------------------------------------------------------
def visibility(N, Nk, causal, q_lo=0, q_hi=None, k_lo=0, k_hi=None):
    """Boolean block [q_lo:q_hi, k_lo:k_hi] of the N x Nk visibility matrix.

    Without a mask every key is visible.  With one, query row i sits at
    position Nk - N + i and sees key j exactly when j <= Nk - N + i.
    """
    q_hi = N if q_hi is None else q_hi
    k_hi = Nk if k_hi is None else k_hi
    rows, cols = q_hi - q_lo, k_hi - k_lo
    if not causal:
        return np.ones((rows, cols), dtype=bool)
    last_key = (Nk - N) + np.arange(q_lo, q_hi)  # position of each query = its last visible key
    return np.arange(k_lo, k_hi)[None, :] <= last_key[:, None]


def tile_visible(N, Nk, causal, q_lo, q_hi, k_lo):
    """Whether the tile of queries [q_lo, q_hi) and keys starting at k_lo holds a visible pair.

    Visibility only grows with the query index (its position Nk - N + i grows)
    and only shrinks with the key index, so the most visible corner of a tile
    is (its last query, its first key): the tile holds a visible pair iff that
    corner is visible, i.e. k_lo <= Nk - N + (q_hi - 1).  Without a mask every
    tile does.
    """
    return (not causal) or k_lo <= (Nk - N) + (q_hi - 1)


# --------------------------------------------------------------------------
# softmax: the plain definition and the streaming normaliser
# --------------------------------------------------------------------------
def softmax_safe(x):
    """Softmax along the last axis in three passes: the maximum, the sum of
    exponentials relative to it, the division."""
    x = np.asarray(x, dtype=np.float64)
    top = np.max(x, axis=-1, keepdims=True)
    w = np.exp(x - top)
    return w / np.sum(w, axis=-1, keepdims=True)


class RowState:
    """Streaming normaliser of a block of rows.

    Holds, per row, the largest score absorbed so far (``top``; -inf while
    nothing visible has been seen), the sum of exp(score - top) over absorbed
    scores (``total``) and, when value rows are supplied, the sum of
    exp(score - top) * value (``acc``).  Masked scores are -inf and contribute
    exp(-inf) = 0.
    """

    def __init__(self, rows, width=0):
        self.top = np.full(rows, NEG_INF)
        self.total = np.zeros(rows)
        self.acc = np.zeros((rows, width))

    @staticmethod
    def _anchor(top):
        # A row with nothing visible has top = -inf; measuring its exponentials
        # from 0 instead keeps every exp argument free of (-inf) - (-inf).
        return np.where(np.isfinite(top), top, 0.0)

    def absorb(self, scores, values=None):
        """Fold a block of scores [rows, n] (and value rows [n, width]) into the state."""
        scores = np.asarray(scores, dtype=np.float64)
        block_top = scores.max(axis=1) if scores.shape[1] else np.full(scores.shape[0], NEG_INF)
        new_top = np.maximum(self.top, block_top)
        new_anchor = self._anchor(new_top)
        # the old sums were taken relative to the old maximum; re-express them relative to the
        # new one (a row that had seen nothing has empty sums: factor 0)
        shrink = np.exp(np.where(np.isfinite(self.top), self.top - new_anchor, NEG_INF))
        w = np.exp(scores - new_anchor[:, None])
        self.total = self.total * shrink + w.sum(axis=1)
        if values is not None:
            self.acc = self.acc * shrink[:, None] + w @ np.asarray(values, dtype=np.float64)
        self.top = new_top

    def log_normaliser(self):
        """log of sum over absorbed scores of exp(score); -inf for a row that saw nothing."""
        seen = self.total > 0
        return np.where(seen, self._anchor(self.top) + np.log(np.where(seen, self.total, 1.0)), NEG_INF)

    def output(self):
        """acc / total: the softmax-weighted mean of the absorbed value rows (0 where nothing was seen)."""
        seen = self.total > 0
        return np.where(seen[:, None], self.acc / np.where(seen, self.total, 1.0)[:, None], 0.0)


def softmax_streaming(x, block):
    """Softmax along the last axis of a 2-D array from one streaming pass over
    column blocks of width ``block`` (for the normaliser) and one final pass."""
    x = np.asarray(x, dtype=np.float64)
    st = RowState(x.shape[0])
    for c in range(0, x.shape[1], block):
        st.absorb(x[:, c:c + block])
    return np.exp(x - st.log_normaliser()[:, None])


# --------------------------------------------------------------------------
# partial states in log-sum-exp form, and their merge
# --------------------------------------------------------------------------
def segment_state(scores, values):
    """(o, lse) of one segment: o = softmax(scores) @ values over the segment, lse = log sum exp(scores).

    A row whose scores are all -inf has o = 0 and lse = -inf (it carries no weight)."""
    st = RowState(np.shape(scores)[0], np.shape(values)[1])
    st.absorb(scores, values)
    return st.output(), st.log_normaliser()


def combine(a, b):
    """Exact merge of two log-sum-exp-form states covering disjoint key sets.

    With Z = exp(lse) the normaliser of each side, the union has Z = Z_a + Z_b
    and its output is the Z-weighted mean of the two outputs.  In logs:
    lse = logaddexp(lse_a, lse_b) and the weight of side a is exp(lse_a - lse).
    A side with lse = -inf has weight 0; if both are empty the result is
    (0, -inf)."""
    (oa, la), (ob, lb) = a, b
    lse = np.logaddexp(la, lb)
    empty = np.isneginf(lse)
    ref = np.where(empty, 0.0, lse)
    wa = np.exp(la - ref)  # exp(-inf) = 0 for an empty side
    wb = np.exp(lb - ref)
    return wa[:, None] * oa + wb[:, None] * ob, lse


# --------------------------------------------------------------------------
# exact attention: the definitions
# --------------------------------------------------------------------------
def attention_definition(Q, K, V, causal=False, scale=None):
    """O = softmax(mask(Q K^T * scale)) V with the full score matrix; LSE = log of each row's normaliser.

    Returns (O, LSE, P).  A row with no visible key gets O = 0, LSE = -inf and a zero P row.
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    N, d = Q.shape
    Nk = K.shape[0]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    vis = visibility(N, Nk, causal)
    S = np.where(vis, scale * (Q @ K.T), NEG_INF)
    has_key = vis.any(axis=1)
    P = np.zeros_like(S)
    P[has_key] = softmax_safe(S[has_key])
    lse = np.full(N, NEG_INF)
    if has_key.any():
        rows = S[has_key]
        top = rows.max(axis=1)
        lse[has_key] = top + np.log(np.exp(rows - top[:, None]).sum(axis=1))
    return P @ V, lse, P


def attention_bwd_definition(Q, K, V, dO, causal=False, scale=None, return_terms=False):
    """Gradients of sum(O * dO) with the full P materialised.

    With O = P V and P = softmax of the scaled, masked scores:
    dV = P^T dO; dP = dO V^T; D_i = sum_c dO_ic O_ic; dS = P * (dP - D)
    (the softmax Jacobian applied row by row); the scores are scale * Q K^T, so
    dQ = scale dS K and dK = scale dS^T Q.  Returns (dQ, dK, dV), followed by
    (P, dS) when ``return_terms``.
    """
    Q, K, V, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, dO))
    scale = 1.0 / math.sqrt(Q.shape[1]) if scale is None else scale
    O, _, P = attention_definition(Q, K, V, causal, scale)
    dP = dO @ V.T
    D = np.einsum("ic,ic->i", dO, O)
    dS = P * (dP - D[:, None])
    grads = (scale * (dS @ K), scale * (dS.T @ Q), P.T @ dO)
    return grads + (P, dS) if return_terms else grads


# --------------------------------------------------------------------------
# the tiled loop orders (models of the kernels' walks)
# --------------------------------------------------------------------------
def _tiles(n, size):
    return [(lo, min(lo + size, n)) for lo in range(0, n, size)]


def tiled_forward(Q, K, V, Br, Bc, causal=False, scale=None):
    """Query tiles of Br rows each walk the key tiles of Bc keys that hold a visible pair,
    folding each masked score tile and its value rows into a ``RowState``; O and LSE come
    from the state once the walk ends.

    Returns (O, LSE, visited), ``visited`` the (query tile, key tile) indices computed.
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    N, d = Q.shape
    Nk, dv = V.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O, L, visited = np.zeros((N, dv)), np.full(N, NEG_INF), []
    for ti, (q_lo, q_hi) in enumerate(_tiles(N, Br)):
        st = RowState(q_hi - q_lo, dv)
        for tj, (k_lo, k_hi) in enumerate(_tiles(Nk, Bc)):
            if not tile_visible(N, Nk, causal, q_lo, q_hi, k_lo):
                continue
            visited.append((ti, tj))
            S = scale * (Q[q_lo:q_hi] @ K[k_lo:k_hi].T)
            st.absorb(np.where(visibility(N, Nk, causal, q_lo, q_hi, k_lo, k_hi), S, NEG_INF), V[k_lo:k_hi])
        O[q_lo:q_hi], L[q_lo:q_hi] = st.output(), st.log_normaliser()
    return O, L, visited


def tiled_backward(Q, K, V, O, dO, L, Br, Bc, causal=False, scale=None):
    """Key tiles own their dK and dV; each walks the query tiles that hold a visible pair with it,
    rebuilding that tile's probabilities from the forward's log-normaliser L
    (P = exp(S - L), 0 for a row with L = -inf), and adds its share of dQ.

    Returns (dQ, dK, dV, visited).
    """
    Q, K, V, O, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, O, dO))
    L = np.asarray(L, dtype=np.float64)
    N, d = Q.shape
    Nk, dv = V.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    D = np.einsum("ic,ic->i", dO, O)
    dQ, dK, dV, visited = np.zeros((N, d)), np.zeros((Nk, d)), np.zeros((Nk, dv)), []
    for tj, (k_lo, k_hi) in enumerate(_tiles(Nk, Bc)):
        Kj, Vj = K[k_lo:k_hi], V[k_lo:k_hi]
        for ti, (q_lo, q_hi) in enumerate(_tiles(N, Br)):
            if not tile_visible(N, Nk, causal, q_lo, q_hi, k_lo):
                continue
            visited.append((ti, tj))
            vis = visibility(N, Nk, causal, q_lo, q_hi, k_lo, k_hi)
            Li = L[q_lo:q_hi]
            finite = np.isfinite(Li)
            S = scale * (Q[q_lo:q_hi] @ Kj.T)
            P = np.exp(np.where(vis, S, NEG_INF) - np.where(finite, Li, 0.0)[:, None]) * finite[:, None]
            g = dO[q_lo:q_hi]
            dS = P * ((g @ Vj.T) - D[q_lo:q_hi, None])
            dV[k_lo:k_hi] += P.T @ g
            dK[k_lo:k_hi] += scale * (dS.T @ Q[q_lo:q_hi])
            dQ[q_lo:q_hi] += scale * (dS @ Kj)
    return dQ, dK, dV, visited


# --------------------------------------------------------------------------
# split-KV decoding
# --------------------------------------------------------------------------
def split_bounds(n_keys, n_splits):
    """n_splits + 1 near-equal integer cut points of [0, n_keys]: cut s is floor(s * n_keys / n_splits).
    With more splits than keys some segments are empty."""
    return [(s * n_keys) // n_splits for s in range(n_splits + 1)]


def split_decode(q, K, V, n_splits, scale=None, bounds=None):
    """Queries q [R, d] over keys K [n, d], values V [n, dv]: each non-empty segment of keys gives a
    log-sum-exp-form state, and the states are merged with ``combine``.

    Returns (o, lse, parts) with ``parts`` the per-segment (o_s, lse_s)."""
    q, K, V = (np.asarray(t, dtype=np.float64) for t in (q, K, V))
    scale = 1.0 / math.sqrt(q.shape[1]) if scale is None else scale
    cuts = split_bounds(K.shape[0], n_splits) if bounds is None else list(bounds)
    parts = [segment_state(scale * (q @ K[a:b].T), V[a:b]) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    o, lse = reduce(combine, parts)
    return o, lse, parts
