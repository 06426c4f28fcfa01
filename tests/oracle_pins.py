"""Checks that pin the CPU oracle to facts fixed outside itself.

Each check takes an ``attention(q, k, v, causal, scale) -> (O, LSE)`` callable
so that the same pins can be run against a deliberately broken build of the
oracle (see ``test_oracle_pins.test_planted_mistakes_are_caught``).

Pins used here, none of which re-runs the oracle's own formula:
  * brute force: a pure-Python evaluation of the softmax *definition*
    exp(s_j) / sum_k exp(s_k) (no max subtraction, math.fsum sums) on the
    small shapes of the pages' correctness demos;
  * hand-derived closed-form fixtures under ``tests/golden/``;
  * closed forms: Q = 0 averages the visible prefix with LSE = log(count);
    a causal first row returns V[0] exactly with LSE = scale * q0.k0;
  * a near one-hot construction K = c * Q[perm] that makes each query pick
    one value row (catches transposed operands and index slips).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Shapes (N, Nk, d) from the pages' correctness demos: 02_flash_forward.py demo 1 and
# the flash_lab.py self-test.  (77, 513, 32) exercises the causal offset Nk - N = 436.
BRUTE_SHAPES = ((77, 513, 32), (7, 33, 8), (50, 50, 8), (64, 64, 16), (1, 1000, 64))


def brute_attention(Q, K, V, causal, scale):
    """Softmax taken literally from its definition, in pure Python with exact-rounded sums."""
    Q, K, V = (np.asarray(t, dtype=np.float64).tolist() for t in (Q, K, V))
    N, Nk = len(Q), len(K)
    dv = len(V[0]) if Nk else 0
    O, L = [], []
    for i in range(N):
        qpos = Nk - N + i
        w = []
        for j in range(Nk):
            if causal and j > qpos:
                w.append(0.0)
            else:
                w.append(math.exp(scale * math.fsum(a * b for a, b in zip(Q[i], K[j]))))
        Z = math.fsum(w)
        if Z == 0.0:
            O.append([0.0] * dv)
            L.append(-math.inf)
            continue
        O.append([math.fsum(w[j] * V[j][c] for j in range(Nk)) / Z for c in range(dv)])
        L.append(math.log(Z))
    return np.array(O), np.array(L)


def brute_visible(N, Nk, causal):
    """Boolean [N, Nk] visibility, element by element: query i at position Nk - N + i sees key j
    when j is at or before that position ("02_flash_forward.py" demo 1)."""
    out = np.ones((N, Nk), dtype=bool)
    if causal:
        for i in range(N):
            for j in range(Nk):
                out[i, j] = j <= Nk - N + i
    return out


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)

    def arr(x):
        return np.array([[float(v) for v in row] if isinstance(row, list) else float(row) for row in x])

    out = {}
    for key, val in g.items():
        if isinstance(val, list):
            if val and isinstance(val[0], list) and val[0] and isinstance(val[0][0], list):
                out[key] = np.array([arr(v) for v in val])
            else:
                out[key] = arr(val)
        else:
            out[key] = val
    return out


ATTENTION_GOLDEN = ("two_key_weights.json", "causal_offset_means.json", "causal_square.json",
                    "no_visible_key.json")


def _close(a, b, tol):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    same_inf = (np.isinf(a) == np.isinf(b)) & (np.sign(a) == np.sign(b))
    if not np.all(same_inf[np.isinf(a) | np.isinf(b)]):
        return False
    fin = np.isfinite(a) & np.isfinite(b)
    return bool(np.all(np.abs(a[fin] - b[fin]) <= tol)) and not np.any(np.isnan(a) | np.isnan(b))


def check_golden(attention):
    """Failures (list of strings) of ``attention`` against the hand-derived fixtures."""
    bad = []
    for name in ATTENTION_GOLDEN:
        g = load_golden(name)
        O, L = attention(g["Q"], g["K"], g["V"], g["causal"], g["scale"])
        if not (_close(O, g["O"], g["tol"]) and _close(L, g["LSE"], g["tol"])):
            bad.append(f"golden {name}")
    return bad


def check_brute(attention, shapes=BRUTE_SHAPES, seed=0, tol=1e-12):
    bad = []
    rng = np.random.default_rng(seed)
    for (N, Nk, d) in shapes:
        Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, d))
        scale = 1.0 / math.sqrt(d)
        for causal in (False, True):
            O, L = attention(Q, K, V, causal, scale)
            Ob, Lb = brute_attention(Q, K, V, causal, scale)
            if not (_close(O, Ob, tol) and _close(L, Lb, tol)):
                bad.append(f"brute N={N} Nk={Nk} d={d} causal={causal}")
    return bad


def check_q_zero(attention, seed=3):
    """Q = 0: O is the mean of the visible V rows, LSE = log(count of visible keys)."""
    bad = []
    rng = np.random.default_rng(seed)
    for (N, Nk, d, dv) in ((5, 9, 4, 3), (9, 9, 8, 2), (1, 17, 4, 4)):
        Q = np.zeros((N, d))
        K, V = rng.standard_normal((Nk, d)), rng.standard_normal((Nk, dv))
        for causal in (False, True):
            O, L = attention(Q, K, V, causal, 0.3)
            for i in range(N):
                n = (Nk - N + i + 1) if causal else Nk
                if not (_close(O[i], V[:n].mean(axis=0), 1e-14) and _close(L[i], math.log(n), 1e-14)):
                    bad.append(f"q_zero N={N} Nk={Nk} causal={causal} row={i}")
                    break
    return bad


def check_causal_first_row(attention, seed=4):
    """Causal N = Nk: row 0 sees only key 0, so O[0] = V[0] exactly and LSE[0] = scale * q0.k0."""
    bad = []
    rng = np.random.default_rng(seed)
    N, d, dv, scale = 16, 8, 5, 0.35
    Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((N, d)), rng.standard_normal((N, dv))
    O, L = attention(Q, K, V, True, scale)
    if not np.array_equal(O[0], V[0]):
        bad.append("causal first row O != V[0]")
    if abs(L[0] - scale * float(np.dot(Q[0], K[0]))) > 1e-14:
        bad.append("causal first row LSE")
    return bad


def check_one_hot(attention, seed=5):
    """K = c * Q[perm] with unit-norm rows: each query attends (almost) only to the key built from itself."""
    bad = []
    rng = np.random.default_rng(seed)
    N, d, dv = 24, 64, 7
    Q = rng.standard_normal((N, d))
    Q /= np.linalg.norm(Q, axis=1, keepdims=True)
    perm = rng.permutation(N)
    K = 200.0 * Q[perm]
    V = rng.standard_normal((N, dv))
    O, L = attention(Q, K, V, False, 1.0)
    inv = np.argsort(perm)  # key j was built from query perm[j]; query i matches key inv[i]
    if not _close(O, V[inv], 1e-10):
        bad.append("one-hot O")
    if not _close(L, 200.0 * np.ones(N), 1e-8):
        bad.append("one-hot LSE")
    return bad


def run_all(attention):
    return (check_golden(attention) + check_brute(attention, shapes=((77, 513, 32), (7, 33, 8), (1, 1000, 64)))
            + check_q_zero(attention) + check_causal_first_row(attention) + check_one_hot(attention))


# --------------------------------------------------------------------------
# backward pins
# --------------------------------------------------------------------------
# Each check takes ``bwd(q, k, v, do, causal, scale) -> (dQ, dK, dV)``.  None of
# them re-runs the oracle's own formula:
#   * hand-derived fixtures under ``tests/golden/`` (bwd_*.json);
#   * central finite differences of f = sum(O o dO), with O from the pure-Python
#     brute-force forward above, for every input entry (the flash_lab.py
#     self-test checks one entry of dQ this way with eps 1e-6 and tolerance 1e-7);
#   * invariants that follow from softmax rows summing to 1 and from f being
#     bilinear in (Q, K) and linear in V;
#   * torch autograd through the plain float64 forward (an independent library).
BWD_GOLDEN = ("bwd_two_keys.json", "bwd_causal_uniform.json", "bwd_no_visible_key.json")


def check_bwd_golden(bwd):
    bad = []
    for name in BWD_GOLDEN:
        g = load_golden(name)
        dQ, dK, dV = bwd(g["Q"], g["K"], g["V"], g["dO"], g["causal"], g["scale"])
        if not (_close(dQ, g["dQ"], g["tol"]) and _close(dK, g["dK"], g["tol"]) and _close(dV, g["dV"], g["tol"])):
            bad.append(f"bwd golden {name}")
    return bad


def _objective(Q, K, V, dO, causal, scale):
    O, _ = brute_attention(Q, K, V, causal, scale)
    return math.fsum((O * dO).ravel().tolist())


def check_bwd_finite_differences(bwd, seed=21, eps=1e-6, tol=1e-7):
    """Every entry of dQ, dK, dV against a central difference of sum(O o dO)."""
    bad = []
    rng = np.random.default_rng(seed)
    for (N, Nk, d, dv, causal) in ((5, 7, 3, 2, False), (5, 7, 3, 2, True), (6, 4, 3, 2, True)):
        Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, dv))
        dO = rng.standard_normal((N, dv))
        scale = 0.7
        grads = bwd(Q, K, V, dO, causal, scale)
        for which, (X, G) in enumerate(zip((Q, K, V), grads)):
            num = np.zeros_like(X)
            for idx in np.ndindex(X.shape):
                args_p = [Q.copy(), K.copy(), V.copy()]
                args_m = [Q.copy(), K.copy(), V.copy()]
                args_p[which][idx] += eps
                args_m[which][idx] -= eps
                num[idx] = (_objective(*args_p, dO, causal, scale) - _objective(*args_m, dO, causal, scale)) / (2 * eps)
            if not _close(G, num, tol):
                bad.append(f"finite difference {'QKV'[which]} N={N} Nk={Nk} causal={causal}")
    return bad


def check_bwd_invariants(bwd, seed=22):
    """Rows of dS sum to 0 (so sum_j dK_j = 0); sum_j dV_j = sum_i dO_i; Euler identities
    sum dQ o Q = sum dK o K (scores bilinear in Q, K) and sum dV o V = sum O o dO (O linear in V);
    equal key rows give dQ = 0."""
    bad = []
    rng = np.random.default_rng(seed)
    for (N, Nk, d, dv, causal) in ((19, 41, 16, 6, False), (23, 23, 8, 8, True), (9, 30, 4, 5, True)):
        Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, dv))
        dO = rng.standard_normal((N, dv))
        scale = 0.4
        dQ, dK, dV = (np.asarray(x) for x in bwd(Q, K, V, dO, causal, scale))
        O, _ = brute_attention(Q, K, V, causal, scale)
        tag = f"N={N} Nk={Nk} causal={causal}"
        if not _close(dK.sum(axis=0), np.zeros(d), 1e-12):
            bad.append(f"sum dK {tag}")
        if not _close(dV.sum(axis=0), dO.sum(axis=0), 1e-12):
            bad.append(f"sum dV {tag}")
        if abs(float((dQ * Q).sum() - (dK * K).sum())) > 1e-11:
            bad.append(f"euler QK {tag}")
        if abs(float((dV * V).sum() - (O * dO).sum())) > 1e-11:
            bad.append(f"euler V {tag}")
        Kc = np.repeat(rng.standard_normal((1, d)), Nk, axis=0)
        dQc, _, _ = bwd(Q, Kc, V, dO, causal, scale)
        if not _close(dQc, np.zeros((N, d)), 1e-12):
            bad.append(f"equal keys dQ {tag}")
    return bad


def check_bwd_autograd(bwd, seed=23):
    """torch autograd (float64, CPU) through S = Q K^T scale, mask, softmax, O = P V."""
    import torch
    bad = []
    g = torch.Generator().manual_seed(seed)
    for (N, Nk, d, dv, causal) in ((33, 33, 16, 16, True), (20, 45, 8, 12, False), (1, 300, 32, 32, False)):
        Q, K, V = (torch.randn(s, generator=g, dtype=torch.float64, requires_grad=True)
                   for s in ((N, d), (Nk, d), (Nk, dv)))
        dO = torch.randn((N, dv), generator=g, dtype=torch.float64)
        scale = 1.0 / math.sqrt(d)
        S = Q @ K.T * scale
        if causal:
            S = S.masked_fill(torch.arange(Nk)[None, :] > (Nk - N + torch.arange(N))[:, None], float("-inf"))
        O = torch.softmax(S, dim=-1) @ V
        O.backward(dO)
        ref = [t.grad.numpy() for t in (Q, K, V)]
        got = bwd(Q.detach().numpy(), K.detach().numpy(), V.detach().numpy(), dO.numpy(), causal, scale)
        for name, a, b in zip("QKV", got, ref):
            if not _close(a, b, 1e-12):
                bad.append(f"autograd d{name} N={N} Nk={Nk} causal={causal}")
    return bad


def run_all_bwd(bwd):
    return (check_bwd_golden(bwd) + check_bwd_finite_differences(bwd) + check_bwd_invariants(bwd)
            + check_bwd_autograd(bwd))
