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
