"""The CPU oracle pinned to facts outside itself (runs without a GPU).

Tolerances 1e-15 / 1e-12 / 1e-13 are the ones the flash_lab.py self-test
(CS349E lecture 11 shared module) uses for the same comparisons in float64.
"""
from __future__ import annotations

import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
from oracle import numpy_oracle as no
from tests import oracle_pins as pins


def c_attention(Q, K, V, causal, scale):
    return oracle.attention(np.asarray(Q), np.asarray(K), np.asarray(V), causal=causal, scale=scale)


def np_attention(Q, K, V, causal, scale):
    O, L, _ = no.attention_definition(Q, K, V, causal, scale)
    return O, L


@pytest.mark.parametrize("impl", [c_attention, np_attention], ids=["c", "numpy"])
def test_golden_fixtures(impl):
    assert pins.check_golden(impl) == []


@pytest.mark.parametrize("impl", [c_attention, np_attention], ids=["c", "numpy"])
def test_brute_force_definition(impl):
    assert pins.check_brute(impl) == []


@pytest.mark.parametrize("impl", [c_attention, np_attention], ids=["c", "numpy"])
def test_closed_forms(impl):
    assert pins.check_q_zero(impl) == []
    assert pins.check_causal_first_row(impl) == []
    assert pins.check_one_hot(impl) == []


@pytest.mark.parametrize("N,Nk,d,dv", [(33, 33, 16, 16), (20, 45, 8, 12), (1, 300, 32, 32)])
def test_library_sdpa(N, Nk, d, dv):
    """torch's scaled_dot_product_attention (float64, CPU) as an independent library routine."""
    g = torch.Generator().manual_seed(7)
    Q, K, V = (torch.randn(s, generator=g, dtype=torch.float64) for s in ((N, d), (Nk, d), (Nk, dv)))
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        mask = None
        if causal:
            mask = torch.arange(Nk)[None, :] <= (Nk - N + torch.arange(N))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], V[None], attn_mask=mask,
                                                              scale=scale)[0]
        S = Q @ K.T * scale
        if causal:
            S = S.masked_fill(~mask, float("-inf"))
        lse_ref = torch.logsumexp(S, dim=-1)
        O, L = oracle.attention(Q, K, V, causal=causal, scale=scale)
        assert np.abs(O - ref.numpy()).max() < 1e-12
        assert np.abs(L - lse_ref.numpy()).max() < 1e-12


def test_invariants():
    rng = np.random.default_rng(11)
    N, Nk, d, dv = 19, 41, 16, 6
    Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, dv))
    s = 0.25
    O, L = oracle.attention(Q, K, V, causal=False, scale=s)
    # rows of P sum to 1
    _, _, P = no.attention_definition(Q, K, V, False, s)
    assert np.abs(P.sum(axis=1) - 1).max() < 1e-13
    # a constant added to every score leaves O alone and shifts LSE (extra coordinate trick)
    c = 3.5
    Q2 = np.concatenate([Q, np.ones((N, 1))], axis=1)
    K2 = np.concatenate([K, np.full((Nk, 1), c / s)], axis=1)
    O2, L2 = oracle.attention(Q2, K2, V, causal=False, scale=s)
    assert np.abs(O2 - O).max() < 1e-12 and np.abs(L2 - (L + c)).max() < 1e-12
    # affine in V: O(a V + 1 b^T) = a O(V) + b  (P rows sum to 1)
    a, b = -1.7, rng.standard_normal(dv)
    O3, L3 = oracle.attention(Q, K, a * V + b, causal=False, scale=s)
    assert np.abs(O3 - (a * O + b)).max() < 1e-12 and np.array_equal(L3, L)
    # permuting keys and values together changes nothing (non-causal)
    p = rng.permutation(Nk)
    O4, L4 = oracle.attention(Q, K[p], V[p], causal=False, scale=s)
    assert np.abs(O4 - O).max() < 1e-13 and np.abs(L4 - L).max() < 1e-13
    # the scale multiplies the scores: O(2Q, s/2) = O(Q, s)
    O5, L5 = oracle.attention(2 * Q, K, V, causal=False, scale=s / 2)
    assert np.abs(O5 - O).max() < 1e-13 and np.abs(L5 - L).max() < 1e-13


def test_large_values_stable():
    """Scores in the thousands neither overflow nor lose the winning row."""
    rng = np.random.default_rng(12)
    N, Nk, d, dv = 12, 40, 16, 5
    Q, K, V = (100 * rng.standard_normal(s) for s in ((N, d), (Nk, d), (Nk, dv)))
    for causal in (False, True):
        O, L = oracle.attention(Q, K, V, causal=causal, scale=0.25)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
        S = Q @ K.T * 0.25
        for i in range(N):
            vis = np.arange(Nk) <= (Nk - N + i) if causal else np.ones(Nk, bool)
            row = np.where(vis, S[i], -np.inf)
            top = np.sort(row)[::-1]
            assert V[vis].min(axis=0).min() - 1e-9 <= O[i].min() and O[i].max() <= V[vis].max() + 1e-9
            if top[0] - top[1] > 60:
                assert np.abs(O[i] - V[np.argmax(row)]).max() < 1e-12
                assert abs(L[i] - top[0]) <= 1e-15 * abs(top[0]) + 1e-12


def test_online_softmax_equals_3pass():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 300)) * 4
    assert np.abs(no.softmax_safe(x) - no.softmax_streaming(x, block=37)).max() < 1e-15
    # a block that raises the maximum by far more than exp's range must rescale, not overflow
    x[:, 200] += 900.0
    assert np.abs(no.softmax_safe(x) - no.softmax_streaming(x, block=37)).max() < 1e-15


def test_segment_state_is_the_library_definition():
    """(o, lse) of one segment against scipy's logsumexp and softmax (independent library routines)."""
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(4)
    x = rng.standard_normal((7, 90)) * 5
    x[3, :] = -np.inf  # a row with nothing visible
    x[5, 10:] = -np.inf
    v = rng.standard_normal((90, 3))
    o, lse = no.segment_state(x, v)
    live = np.arange(7) != 3
    assert np.abs(lse[live] - logsumexp(x[live], axis=1)).max() < 1e-13
    assert np.abs(o[live] - softmax(x[live], axis=1) @ v).max() < 1e-13
    assert np.isneginf(lse[3]) and np.all(o[3] == 0)


def test_merge_states_any_split_any_order():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 500)) * 3
    v = rng.standard_normal((500, 4))
    o_full, lse_full = no.segment_state(x, v)
    empty = (np.zeros((6, 4)), np.full(6, -np.inf))
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, 500), size=rng.integers(1, 12), replace=False))
        bounds = [0, *cuts.tolist(), 500]
        states = [no.segment_state(x[:, a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        # an empty (fully masked) segment must not change anything
        states.append(empty)
        order = rng.permutation(len(states))
        pool = [states[i] for i in order]
        while len(pool) > 1:  # random tree: merge a random adjacent pair
            k = int(rng.integers(0, len(pool) - 1))
            pool[k:k + 2] = [no.combine(pool[k], pool[k + 1])]
        o, lse = pool[0]
        assert np.abs(lse - lse_full).max() < 1e-13
        assert np.abs(o - o_full).max() < 1e-12
    o, lse = no.combine(empty, empty)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("n_splits", [1, 3, 16, 999])
def test_split_kv_decode_equals_oracle(n_splits):
    rng = np.random.default_rng(0)
    q = rng.standard_normal((4, 32))
    K, V = rng.standard_normal((1000, 32)), rng.standard_normal((1000, 32))
    o, lse, parts = no.split_decode(q, K, V, n_splits)
    O, L = oracle.attention(q, K, V, causal=False, scale=1 / math.sqrt(32))
    assert np.abs(o - O).max() < 1e-13 and np.abs(lse - L).max() < 1e-13
    # the C combine of the same split states, in a shuffled order, agrees too
    perm = rng.permutation(len(parts))
    op = np.stack([parts[i][0] for i in perm])
    lp = np.stack([parts[i][1] for i in perm])
    o2, l2 = oracle.merge_lse(op, lp)
    assert np.abs(o2 - O).max() < 1e-13 and np.abs(l2 - L).max() < 1e-13


def test_c_merge_golden_and_empty_rows():
    g = pins.load_golden("lse_merge.json")
    o, lse = oracle.merge_lse(g["o_parts"], g["lse_parts"])
    assert np.abs(o - g["o"]).max() < g["tol"] and np.abs(lse - g["lse"]).max() < g["tol"]
    o, lse = oracle.merge_lse(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("N,Nk,Br,Bc", [(300, 513, 128, 128), (513, 300, 128, 128), (77, 513, 16, 50),
                                        (50, 50, 16, 12), (7, 33, 16, 12), (256, 256, 64, 128)])
def test_tiled_model_matches_oracle_and_skips_exactly_masked_tiles(N, Nk, Br, Bc):
    rng = np.random.default_rng(N * 7 + Nk)
    d = 16
    Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, d))
    for causal in (False, True):
        O, L = oracle.attention(Q, K, V, causal=causal, scale=0.25)
        Ot, Lt, visited = no.tiled_forward(Q, K, V, Br, Bc, causal, scale=0.25)
        assert pins._close(Ot, O, 1e-12) and pins._close(Lt, L, 1e-12)
        # a tile is visited iff some element of it is visible (the skip rule drops only fully masked tiles)
        allowed = pins.brute_visible(N, Nk, causal)
        expect = {(i // Br, j // Bc) for i in range(0, N, Br) for j in range(0, Nk, Bc)
                  if allowed[i:i + Br, j:j + Bc].any()}
        assert set(visited) == expect


def test_decode_oracle_matches_per_head_attention():
    from fa_inputs import decode_inputs
    q, k, v, lens = decode_inputs(3, 2, 96, 16, 8, seed=5, lo=1, hi=96)
    O, L = oracle.decode(q, k, v, lens, scale=0.3)
    assert np.all(np.isfinite(O))  # NaN padding past each length is never read
    for b in range(3):
        n = int(lens[b])
        Oh, Lh = oracle.attention(q[b], k[b, :, :n], v[b, :, :n], causal=False, scale=0.3)
        assert np.array_equal(O[b], Oh) and np.array_equal(L[b], Lh)


def test_bf16_inputs_are_widened_exactly():
    from fa_inputs import attention_inputs
    q, k, v = attention_inputs(2, 2, 40, 70, 16, 16, seed=3, mult=2.0)
    O1, L1 = oracle.attention(q, k, v, causal=True)
    O2, L2 = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal=True)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_row_subset_matches_full():
    from fa_inputs import attention_inputs
    q, k, v = attention_inputs(1, 3, 200, 200, 32, 32, seed=9)
    O, L = oracle.attention(q, k, v, causal=True)
    Os, Ls = oracle.attention(q, k, v, causal=True, rows=(70, 133))
    assert np.array_equal(Os, O[:, :, 70:133]) and np.array_equal(Ls, L[:, :, 70:133])


# Mistakes a hand-written attention is likely to contain, planted in a copy of
# the oracle's C source.  Every one of them must make at least one pin fail.
MUTATIONS = {
    "mask_off_by_one": ("if (j > qpos) {\n            s[j] = -INFINITY;", "if (j >= qpos) {\n            s[j] = -INFINITY;"),
    "dropped_scale": ("s[j] = acc * scale;", "s[j] = acc;"),
    "wrong_sign_in_exp": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j] + m);"),
    "dropped_max_in_lse": ("*lse = m + log(l);", "*lse = log(l);"),
    "missing_normalisation": ("double p = s[j] / l;", "double p = s[j];"),
    "value_index_reversed": ("const double* v = V + j * dv;", "const double* v = V + (Nk - 1 - j) * dv;"),
    "top_left_causal": ("long qpos = jb->causal ? jb->Nk - jb->N + i : jb->Nk;",
                        "long qpos = jb->causal ? i : jb->Nk;"),
    "query_row_off_by_one": ("bh * jb->q_stride_bh + i * jb->d, jb->d, qb)",
                             "bh * jb->q_stride_bh + (i > 0 ? i - 1 : 0) * jb->d, jb->d, qb)"),
}


def test_planted_mistakes_are_caught(tmp_path):
    src = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")
    text = open(src).read()
    assert pins.run_all(c_attention) == []
    for name, (old, new) in MUTATIONS.items():
        assert text.count(old) == 1, name
        path = tmp_path / f"mut_{name}.c"
        path.write_text(text.replace(old, new))
        lib = oracle.open_library(oracle.compile_library(str(path), str(tmp_path / f"libmut_{name}.so")))

        def mutated(Q, K, V, causal, scale, _lib=lib):
            # the bf16 route reads Q through the per-row fetch, like production inputs
            return oracle.attention(np.asarray(Q), np.asarray(K), np.asarray(V), causal=causal, scale=scale,
                                    lib=_lib)

        def mutated_bf16(Q, K, V, causal, scale, _lib=lib):
            tq, tk, tv = (torch.tensor(np.asarray(x)).to(torch.bfloat16) for x in (Q, K, V))
            return oracle.attention(tq, tk, tv, causal=causal, scale=scale, lib=_lib)

        failures = pins.run_all(mutated)
        if not failures:
            # mistakes on the bf16 input route show up once inputs are bf16 (brute force on the same values)
            def bf16_pin(_m=mutated_bf16):
                rng = np.random.default_rng(0)
                Q, K, V = (torch.tensor(rng.standard_normal(s)).to(torch.bfloat16).double().numpy()
                           for s in ((20, 16), (30, 16), (30, 8)))
                Om, Lm = _m(Q, K, V, True, 0.25)
                Ob, Lb = pins.brute_attention(Q, K, V, True, 0.25)
                return [] if pins._close(Om, Ob, 1e-12) and pins._close(Lm, Lb, 1e-12) else ["bf16 brute"]
            failures = bf16_pin()
        assert failures, f"planted mistake {name} was not caught by any pin"
    shutil.rmtree(tmp_path, ignore_errors=True)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
def c_attention_bwd(Q, K, V, dO, causal, scale, lib=None):
    return oracle.attention_bwd(np.asarray(Q), np.asarray(K), np.asarray(V), np.asarray(dO), causal=causal,
                                scale=scale, lib=lib)


def np_attention_bwd(Q, K, V, dO, causal, scale):
    return no.attention_bwd_definition(Q, K, V, dO, causal, scale)


@pytest.mark.parametrize("impl", [c_attention_bwd, np_attention_bwd], ids=["c", "numpy"])
def test_bwd_pins(impl):
    assert pins.run_all_bwd(impl) == []


@pytest.mark.parametrize("N,Nk,Br,Bc", [(12, 12, 4, 5), (77, 513, 128, 128), (300, 200, 128, 128),
                                         (200, 300, 37, 64)])
def test_tiled_bwd_model_matches_oracle_and_skips_exactly_masked_tiles(N, Nk, Br, Bc):
    """The FlashAttention-2-order backward (recompute P from L) equals the definition; the
    (query tile, key tile) pairs it skips are exactly those with no visible pair."""
    rng = np.random.default_rng(31)
    d = dv = 8
    Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, dv))
    dO = rng.standard_normal((N, dv))
    for causal in (False, True):
        O, L = oracle.attention(Q, K, V, causal=causal, scale=0.3)
        dQ, dK, dV, visited = no.tiled_backward(Q, K, V, O, dO, L, Br, Bc, causal, 0.3)
        ref = oracle.attention_bwd(Q, K, V, dO, causal=causal, scale=0.3)
        for a, b in zip((dQ, dK, dV), ref):
            assert np.abs(a - b).max() < 1e-12
        mask = pins.brute_visible(N, Nk, causal)
        want = {(i, j) for i in range(-(-N // Br)) for j in range(-(-Nk // Bc))
                if mask[i * Br:(i + 1) * Br, j * Bc:(j + 1) * Bc].any()}
        assert set(visited) == want


def test_bwd_bf16_inputs_are_widened_exactly():
    rng = np.random.default_rng(32)
    t = [torch.tensor(rng.standard_normal(s)).to(torch.bfloat16) for s in ((2, 9, 16), (2, 14, 16), (2, 14, 8),
                                                                          (2, 9, 8))]
    got = oracle.attention_bwd(*t, causal=True, scale=0.25)
    want = oracle.attention_bwd(*(x.double() for x in t), causal=True, scale=0.25)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


BWD_MUTATIONS = {
    "dropped_D": ("double ds = p[j] * (dp - D);", "double ds = p[j] * dp;"),
    "D_sign": ("double ds = p[j] * (dp - D);", "double ds = p[j] * (dp + D);"),
    "dq_without_scale": ("dq[c] += scale * ds * K[j * d + c];", "dq[c] += ds * K[j * d + c];"),
    "dk_from_k": ("dK[j * d + c] += scale * ds * q[c];", "dK[j * d + c] += scale * ds * K[j * d + c];"),
    "dv_from_ds": ("dV[j * dv + c] += p[j] * g[c];", "dV[j * dv + c] += ds * g[c];"),
    "dp_from_k": ("dp += g[c] * V[j * dv + c];", "dp += g[c] * K[j * d + c % d];"),
    "mask_off_by_one": ("            if (j > qpos) {\n                p[j] = -INFINITY;",
                        "            if (j >= qpos) {\n                p[j] = -INFINITY;"),
    "top_left_causal": ("long qpos = causal ? Nk - N + i : Nk;", "long qpos = causal ? i : Nk;"),
    "unnormalised_p": ("for (long j = 0; j < Nk; ++j) p[j] /= l;", "(void)l;"),
}


def test_bwd_planted_mistakes_are_caught(tmp_path):
    src = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")
    text = open(src).read()
    for name, (old, new) in BWD_MUTATIONS.items():
        assert text.count(old) == 1, name
        path = tmp_path / f"mutbwd_{name}.c"
        path.write_text(text.replace(old, new))
        lib = oracle.open_library(oracle.compile_library(str(path), str(tmp_path / f"libmutbwd_{name}.so")))

        def mutated(Q, K, V, dO, causal, scale, _lib=lib):
            return c_attention_bwd(Q, K, V, dO, causal, scale, lib=_lib)

        assert pins.run_all_bwd(mutated), f"planted mistake {name} was not caught by any pin"
    shutil.rmtree(tmp_path, ignore_errors=True)
