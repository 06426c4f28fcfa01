"""fa_bwd (CUDA, through the C ABI) against the CPU FP64 oracle on the same bf16 inputs.

Tolerance (derived from the arithmetic; the gradients carry no tolerance of their own on
the pages).  The kernel feeds the tensor core bf16 operands: P (for dV = P^T dO) and
dS scale (for dQ and dK), each rounded to nearest with unit roundoff u = 2^-8; every
other step is fp32.  One rounding of each product's bf16 operand bounds the error of
element X[a, c] = sum_b A[a, b] B[b, c] by u * M[a, c] with M = |A| |B|.  The row term
D_i = sum_c dO_ic O_ic is formed from the forward's output O, whose own bf16 rounding of
P gives |dO_i| . |Delta O_i| <= u sum_c |dO_ic| (P |V|)_ic = u R_i, and dS_ij carries
P_ij times that.  With E = |dS| + P o R (R broadcast along rows):
    M_dV = P^T |dO|,   M_dK = scale E^T |Q|,   M_dQ = scale E |K|
(P and dS taken from the FP64 oracle).  A CPU emulation of all these roundings on the
shapes below reaches 0.4 u M; the gate is twice u (2^-7) M plus 1e-4, leaving room
for the fp32 effects (ex2.approx, accumulation order) and for a bf16 O, whose output
rounding doubles R.  bf16 gradients add the output rounding 2^-8 |X_ref|.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import attention_inputs, grad_output, sample_slices
from oracle import numpy_oracle as no
from tests.parity import to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
TAU = 2.0 ** -7
FLOOR = 1e-4
BF16_REL = 2.0 ** -8


def fa():
    import exact_tiled_attention_fa_gb300 as m
    return m


def gpu_grads(q, k, v, do, causal, scale, out_dtype=torch.float32):
    o, lse = fa().fwd(q, k, v, causal=causal, scale=scale, out_dtype=torch.float32)
    dq, dk, dv = fa().bwd(q, k, v, o, lse, do, causal=causal, scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    return dq, dk, dv


def magnitudes(q, k, v, do, causal, scale):
    """Per-head (M_dQ, M_dK, M_dV) from the numpy oracle's P and dS, for [..., rows, cols] inputs."""
    Q, K, V, G = (to_np(t).reshape((-1,) + tuple(t.shape[-2:])) for t in (q, k, v, do))
    out = [[], [], []]
    for h in range(Q.shape[0]):
        _, _, _, P, dS = no.attention_bwd_definition(Q[h], K[h], V[h], G[h], causal, scale, return_terms=True)
        R = (np.abs(G[h]) * (P @ np.abs(V[h]))).sum(axis=1)
        E = np.abs(dS) + P * R[:, None]
        out[0].append(scale * E @ np.abs(K[h]))
        out[1].append(scale * E.T @ np.abs(Q[h]))
        out[2].append(P.T @ np.abs(G[h]))
    return [np.stack(m) for m in out]


def check(got, ref, mags, bf16_out=False, what=""):
    for name, g, r, m in zip(("dQ", "dK", "dV"), got, ref, mags):
        a = to_np(g).reshape(m.shape)
        b = np.asarray(r).reshape(m.shape)
        assert not np.any(np.isnan(a)), f"{what} {name}: NaN"
        bound = TAU * m + FLOOR + (BF16_REL * np.abs(b) if bf16_out else 0.0)
        excess = a - b
        ratio = float((np.abs(excess) / bound).max()) if a.size else 0.0
        assert ratio <= 1.0, f"{what} {name}: error reaches {ratio:.2f} x the bound (max |err| {np.abs(excess).max():.3e})"


# (B, H, N, Nk, d, mult): several tiles with ragged tails, the pages' 77 x 513 demo with causal
# offset 436, N > Nk (causal rows with no visible key), exact tiles, a single query.
SMALL = [
    (1, 2, 300, 300, 64, 1.0),
    (2, 2, 77, 513, 32, 2.0),
    (1, 2, 513, 200, 128, 1.0),
    (2, 1, 256, 384, 128, 1.0),
    (1, 1, 1, 1000, 64, 1.0),
    (1, 3, 129, 129, 32, 1.0),
    (1, 1, 640, 640, 64, 2.0),
]


@pytest.mark.parametrize("B,H,N,Nk,d,mult", SMALL)
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes_full_oracle(B, H, N, Nk, d, mult, causal):
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=3, mult=mult, device=DEV)
    do = grad_output(B, H, N, d, seed=3, device=DEV)
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), causal=causal, scale=scale)
    mags = magnitudes(q.cpu(), k.cpu(), v.cpu(), do.cpu(), causal, scale)
    got = gpu_grads(q, k, v, do, causal, scale)
    check(got, ref, mags, what=f"fp32 {B,H,N,Nk,d} causal={causal}")
    got_b = gpu_grads(q, k, v, do, causal, scale, out_dtype=torch.bfloat16)
    check(got_b, ref, mags, bf16_out=True, what=f"bf16 {B,H,N,Nk,d} causal={causal}")


def test_bf16_forward_output_is_accepted():
    """D = sum dO o O computed from a bf16 O (the production format) stays within the bound."""
    B, H, N, d = 1, 2, 384, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=5, device=DEV)
    do = grad_output(B, H, N, d, seed=5, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa().fwd(q, k, v, causal=True, scale=scale, out_dtype=torch.bfloat16)
    got = fa().bwd(q, k, v, o, lse, do, causal=True, scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), causal=True, scale=scale)
    check(got, ref, magnitudes(q.cpu(), k.cpu(), v.cpu(), do.cpu(), True, scale), what="bf16 O")


def test_causal_first_row_has_zero_dq():
    """Causal N = Nk: query 0 sees key 0 only, so dS[0, :] = 0 and dQ[0] = 0 exactly."""
    q, k, v = attention_inputs(1, 2, 256, 256, 64, 64, seed=6, device=DEV)
    do = grad_output(1, 2, 256, 64, seed=6, device=DEV)
    dq, _, _ = gpu_grads(q, k, v, do, True, 0.125)
    assert torch.all(dq[:, :, 0, :] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_sampled_heads(causal):
    """GPT-2-medium shape B=64, H=16, N=Nk=1024, d=64 in the benchmark's launch; 6 seeded heads
    against the oracle."""
    B, H, N, d = 64, 16, 1024, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=0, device=DEV)
    do = grad_output(B, H, N, d, seed=0, device=DEV)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = gpu_grads(q, k, v, do, causal, scale, out_dtype=torch.bfloat16)
    heads = sample_slices(B * H, 6, seed=1)
    flat = [t.reshape(B * H, *t.shape[2:]) for t in (q, k, v, do, dq, dk, dv)]
    sel = [t[heads].cpu() for t in flat]
    ref = oracle.attention_bwd(sel[0], sel[1], sel[2], sel[3], causal=causal, scale=scale)
    mags = magnitudes(sel[0], sel[1], sel[2], sel[3], causal, scale)
    check(sel[4:], ref, mags, bf16_out=True, what=f"C2 causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_persistent_items_per_cta(d, causal, grad_dtype):
    """More (head, key tile) items than SMs, so each CTA walks several, short causal walks right
    after long ones; every third head against the oracle.  bf16 gradients with d = 64 leave
    through the staging tiles (reused item after item), the others row by row."""
    B, H, N = 2, 16, 1024
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=8, device=DEV)
    do = grad_output(B, H, N, d, seed=8, device=DEV)
    scale = 1.0 / math.sqrt(d)
    got = gpu_grads(q, k, v, do, causal, scale, out_dtype=grad_dtype)
    heads = range(0, B * H, 3)
    flat = [t.reshape(B * H, *t.shape[2:]) for t in (q, k, v, do) + tuple(got)]
    sel = [t[list(heads)].cpu() for t in flat]
    ref = oracle.attention_bwd(sel[0], sel[1], sel[2], sel[3], causal=causal, scale=scale)
    check(sel[4:], ref, magnitudes(sel[0], sel[1], sel[2], sel[3], causal, scale),
          bf16_out=(grad_dtype == torch.bfloat16), what=f"items d={d} causal={causal} {grad_dtype}")


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_no_writes_past_gradients(d, grad_dtype):
    """Ragged Nk (the last key tile has 44 keys): the memory right after dQ, dK and dV stays
    untouched, whether the tiles leave through bulk tensor stores or row by row."""
    B, H, N, Nk = 2, 2, 300, 300
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=11, device=DEV)
    do = grad_output(B, H, N, d, seed=11, device=DEV)
    o, lse = fa().fwd(q, k, v, causal=True, out_dtype=torch.float32)
    guard = 4096
    bufs = [torch.full((B * H * n * d + guard,), float("nan"), dtype=grad_dtype, device=DEV) for n in (N, Nk, Nk)]
    grads = tuple(b[: B * H * n * d].view(B, H, n, d) for b, n in zip(bufs, (N, Nk, Nk)))
    fa().bwd(q, k, v, o, lse, do, causal=True, grads=grads)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    for b, g, n in zip(bufs, grads, (N, Nk, Nk)):
        assert not torch.isnan(g).any()
        assert torch.isnan(b[B * H * n * d:]).all()


def test_rejects_small_workspace_and_bad_args():
    B, H, N, d = 1, 1, 128, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=0, device=DEV)
    do = grad_output(B, H, N, d, device=DEV)
    o, lse = fa().fwd(q, k, v)
    small = torch.empty(fa().bwd_workspace_size(B, H, N, d) - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa().FaError) as e:
        fa().bwd(q, k, v, o, lse, do, workspace=small)
    assert e.value.status == fa().FA_ERR_WORKSPACE
    q48 = torch.zeros((1, 1, 8, 48), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa().FaError) as e:
        fa().bwd(q48, q48, q48, q48.float(), torch.zeros((1, 1, 8), device=DEV), q48)
    assert e.value.status == fa().FA_ERR_UNSUPPORTED


def test_bounded_wait_reports_timeout_and_context_survives():
    """A 1 ns wait limit makes the backward's first barrier waits run out: the kernel records
    FA_ERR_TIMEOUT, drains its copies and MMAs and returns; the next call is correct."""
    B, H, N, d = 2, 8, 1024, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=9, device=DEV)
    do = grad_output(B, H, N, d, seed=9, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa().fwd(q, k, v, causal=True, scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    fa().set_wait_timeout_ns(1)
    try:
        fa().bwd(q, k, v, o, lse, do, causal=True, scale=scale, out_dtype=torch.float32)
        status = fa().get_device_error()
    finally:
        fa().set_wait_timeout_ns(0)
    assert status == fa().FA_ERR_TIMEOUT
    q2, k2, v2, do2 = (t[:, :2].contiguous() for t in (q, k, v, do))
    got = gpu_grads(q2, k2, v2, do2, True, scale)
    sel = [t.reshape(B * 2, N, d).cpu() for t in (q2, k2, v2, do2)]
    ref = oracle.attention_bwd(*sel, causal=True, scale=scale)
    check([g.reshape(B * 2, N, d) for g in got], ref, magnitudes(*sel, True, scale), what="after a timed-out launch")
