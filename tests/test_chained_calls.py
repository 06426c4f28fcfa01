"""Calls that consume the previous call's output on the same stream, with no synchronisation in
between, equal each call made on its own.

The kernels are launched as programmatic dependents: each may start its setup while the previous
kernel on the stream is still running, and waits for that kernel to complete before its first
global read or write.  Feeding every call the output of the call before it makes a missing or
misplaced wait visible: after the chain, each call is repeated alone on the inputs the chain gave
it and must give the same bits (the kernels are deterministic; dQ, whose fp32 atomic additions may
land in any order, within one bf16 rounding).
"""
from __future__ import annotations

import pytest
import torch

from fa_inputs import attention_inputs, decode_inputs, gqa_decode_inputs, grad_output

pytestmark = pytest.mark.gpu

DEV = "cuda"


def fa():
    import exact_tiled_attention_fa_gb300 as m
    return m


def done():
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_forward_chain(d):
    # Each forward's query is the previous forward's output; the mask alternates, so non-causal and
    # causal kernels follow one another.
    q, k, v = attention_inputs(2, 4, 384, 384, d, d, seed=11, device=DEV)
    xs, outs = [q], []
    for i in range(6):
        o, lse = fa().fwd(xs[-1], k, v, causal=i % 2 == 1)
        outs.append((o, lse))
        xs.append(o)
    done()
    for i, (o, lse) in enumerate(outs):
        o1, lse1 = fa().fwd(xs[i].clone(), k, v, causal=i % 2 == 1)
        done()
        assert torch.equal(o, o1) and torch.equal(lse, lse1), f"call {i}"


@pytest.mark.parametrize("causal", [False, True])
def test_forward_backward_chain(causal):
    # forward -> backward on its O and LSE -> forward with dQ as the query -> backward again
    B, H, N, d = 2, 3, 320, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=12, device=DEV)
    do = grad_output(B, H, N, d, seed=12, device=DEV)
    o1, l1 = fa().fwd(q, k, v, causal=causal)
    g1 = fa().bwd(q, k, v, o1, l1, do, causal=causal)
    o2, l2 = fa().fwd(g1[0], k, v, causal=causal)
    g2 = fa().bwd(g1[0], k, v, o2, l2, do, causal=causal)
    done()
    for (qq, o, lse, g) in ((q, o1, l1, g1), (g1[0].clone(), o2, l2, g2)):
        oa, la = fa().fwd(qq, k, v, causal=causal)
        done()
        assert torch.equal(o, oa) and torch.equal(lse, la)
        ga = fa().bwd(qq, k, v, oa, la, do, causal=causal)
        done()
        assert torch.equal(g[1], ga[1]) and torch.equal(g[2], ga[2])
        diff = (g[0].float() - ga[0].float()).abs()
        assert bool((diff <= ga[0].float().abs() * 2.0 ** -7 + 1e-6).all())


@pytest.mark.parametrize("fused", [False, True])
def test_decode_chain(fused):
    # each decode's query is the previous decode's output
    B, H, Nk_max, d = 4, 8, 4096, 128
    q, kc, vc, lens = decode_inputs(B, H, Nk_max, d, d, seed=13, lo=100, hi=4096, device=DEV)
    lens = lens.to(DEV)
    if fused:
        ws = fa().decode_fused_workspace(B, H, Nk_max, d, device=DEV)
        call = lambda q_, k_, v_, l_: fa().decode_splitkv_fused(q_, k_, v_, l_, ws)  # noqa: E731
    else:
        call = fa().decode_splitkv
    xs, outs = [q], []
    for _ in range(6):
        o, lse = call(xs[-1], kc, vc, lens)
        outs.append((o, lse))
        xs.append(o)
    done()
    for i, (o, lse) in enumerate(outs):
        o1, lse1 = call(xs[i].clone(), kc, vc, lens)
        done()
        assert torch.equal(o, o1) and torch.equal(lse, lse1), f"call {i}"


@pytest.mark.parametrize("Hkv", [8, 4, 2])  # 4, 8 and 16 query heads per key/value head
def test_gqa_decode_chain(Hkv):
    B, Hq, Nk_max, d = 2, 32, 4096, 128
    q, kc, vc, lens = gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, d, seed=14, lo=100, hi=4096, device=DEV)
    lens = lens.to(DEV)
    xs, outs = [q], []
    for _ in range(6):
        o, lse = fa().decode_splitkv_gqa(xs[-1], kc, vc, lens)
        outs.append((o, lse))
        xs.append(o)
    done()
    for i, (o, lse) in enumerate(outs):
        o1, lse1 = fa().decode_splitkv_gqa(xs[i].clone(), kc, vc, lens)
        done()
        assert torch.equal(o, o1) and torch.equal(lse, lse1), f"call {i}"


def test_splitkv_prefill_chain():
    B, H, N, Nk, d = 1, 4, 256, 4096, 128
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=15, device=DEV)
    xs, outs = [q], []
    for i in range(4):
        o, lse = fa().fwd_splitkv(xs[-1], k, v, causal=i % 2 == 0)
        outs.append((o, lse))
        xs.append(o)
    done()
    for i, (o, lse) in enumerate(outs):
        o1, lse1 = fa().fwd_splitkv(xs[i].clone(), k, v, causal=i % 2 == 0)
        done()
        assert torch.equal(o, o1) and torch.equal(lse, lse1), f"call {i}"
