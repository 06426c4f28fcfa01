"""Every entry point captured into a CUDA graph and replayed on new inputs equals the eager call.

The calls launch their kernels on the caller's stream and, once a device has been used, allocate
nothing, synchronise nothing and look up no device state: a decode or prefill step can be captured
once and replayed without the per-call launch cost (the short decodes are launch-bound).  After the
capture the inputs are overwritten in place; the replay must then reproduce an eager call on the new
inputs bit for bit (the kernels are deterministic), except dQ, whose fp32 atomic additions may land
in any order (within one bf16 rounding of the eager value).
"""
from __future__ import annotations

import pytest
import torch

from fa_inputs import attention_inputs, decode_inputs, gqa_decode_inputs, merge_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def fa():
    import exact_tiled_attention_fa_gb300 as m
    return m


def capture(fn):
    """Run fn once on a side stream (first-use set-up), then capture it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def refill(tensors, seed):
    """Overwrite the captured inputs in place with new N(0, 1) values."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    for t in tensors:
        t.copy_(torch.randn(t.shape, generator=gen, device=DEV, dtype=torch.float32).to(t.dtype))


def replay(g, outs, times=1):
    for _ in range(times):
        g.replay()
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    return [t.clone() for t in outs]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_graph(causal, d):
    q, k, v = attention_inputs(2, 3, 300, 333, d, d, seed=d, device=DEV)
    o = torch.empty((2, 3, 300, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((2, 3, 300), dtype=torch.float32, device=DEV)
    g = capture(lambda: fa().fwd(q, k, v, causal=causal, out=o, lse=lse))
    refill((q, k, v), seed=1)
    o_g, lse_g = replay(g, (o, lse))
    o_e, lse_e = fa().fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e)


def test_bwd_graph():
    B, H, N, d = 2, 2, 256, 64
    q, k, v = attention_inputs(B, H, N, N, d, d, seed=5, device=DEV)
    o, lse = fa().fwd(q, k, v, causal=True)
    do = torch.empty_like(o)
    refill((do,), seed=6)
    grads = tuple(torch.empty_like(t) for t in (q, k, v))
    ws = torch.empty(fa().bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=DEV)
    g = capture(lambda: fa().bwd(q, k, v, o, lse, do, causal=True, grads=grads, workspace=ws))
    refill((do,), seed=7)
    dq_g, dk_g, dv_g = replay(g, grads)
    dq_e, dk_e, dv_e = fa().bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dk_g, dk_e) and torch.equal(dv_g, dv_e)
    assert torch.allclose(dq_g.float(), dq_e.float(), rtol=2 ** -7, atol=1e-6)


def test_decode_graphs():
    B, H, Nk_max, d = 3, 4, 700, 128
    lens = torch.tensor([0, 5, 700], dtype=torch.int32)
    q, k, v, _ = decode_inputs(B, H, Nk_max, d, d, seed=3, device=DEV, seqlens=lens)
    ld = lens.to(DEV)
    n = fa().decode_default_splits(B, H, Nk_max, fa().num_sms())
    ws = torch.empty(fa().decode_workspace_size(B, H, d, n), dtype=torch.uint8, device=DEV)
    wsf = fa().decode_fused_workspace(B, H, Nk_max, d, n_splits=n, device=DEV)
    o2 = torch.empty((B, H, 1, d), dtype=torch.float32, device=DEV)
    l2 = torch.empty((B, H, 1), dtype=torch.float32, device=DEV)
    o1, l1 = torch.empty_like(o2), torch.empty_like(l2)

    def step():
        fa().decode_splitkv(q, k, v, ld, n_splits=n, out=o2, lse=l2, workspace=ws)
        fa().decode_splitkv_fused(q, k, v, ld, wsf, n_splits=n, out=o1, lse=l1)

    g = capture(step)
    refill((q, k, v), seed=4)
    outs = replay(g, (o2, l2, o1, l1), times=3)  # the fused combine's counters reset every replay
    e2 = fa().decode_splitkv(q, k, v, ld, n_splits=n, out_dtype=torch.float32)
    e1 = fa().decode_splitkv_fused(q, k, v, ld, wsf, n_splits=n, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for got, want in zip(outs, (*e2, *e1)):
        assert torch.equal(got, want)
    assert int(wsf[fa().decode_workspace_size(B, H, d, n):].count_nonzero()) == 0


@pytest.mark.parametrize("Hkv", [16, 8, 4, 1])  # groups of 2 (CUDA cores), 4, 8 and 32 (tensor core)
def test_gqa_decode_graph(Hkv):
    B, Hq, Nk_max, d = 2, 32, 1500, 128
    lens = torch.tensor([1500, 129], dtype=torch.int32)
    q, k, v, _ = gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, d, seed=Hkv, device=DEV, seqlens=lens)
    ld = lens.to(DEV)
    n = fa().decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, fa().num_sms())
    ws = torch.empty(fa().decode_workspace_size(B, Hq, d, n), dtype=torch.uint8, device=DEV)
    o = torch.empty((B, Hq, 1, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=DEV)
    g = capture(lambda: fa().decode_splitkv_gqa(q, k, v, ld, n_splits=n, out=o, lse=lse, workspace=ws))
    refill((q, k, v), seed=Hkv + 100)
    o_g, lse_g = replay(g, (o, lse))
    o_e, lse_e = fa().decode_splitkv_gqa(q, k, v, ld, n_splits=n)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e)


def test_fwd_splitkv_and_merge_graph():
    B, H, N, Nk, d = 1, 2, 200, 3000, 128
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=9, device=DEV)
    n = fa().fwd_splitkv_default_splits(B, H, N, Nk, fa().num_sms())
    ws = torch.empty(fa().fwd_splitkv_workspace_size(B, H, N, d, n), dtype=torch.uint8, device=DEV)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    op, lp = merge_inputs(5, 33, 128, seed=2, empty_frac=0.3, device=DEV)
    mo = torch.empty((33, 128), dtype=torch.float32, device=DEV)
    ml = torch.empty((33,), dtype=torch.float32, device=DEV)

    def step():
        fa().fwd_splitkv(q, k, v, causal=True, n_splits=n, out=o, lse=lse, workspace=ws)
        fa().merge_states(op, lp, out=mo, lse=ml)

    g = capture(step)
    refill((q, k, v, op), seed=10)
    outs = replay(g, (o, lse, mo, ml))
    want = (*fa().fwd_splitkv(q, k, v, causal=True, n_splits=n), *fa().merge_states(op, lp))
    torch.cuda.synchronize()
    for got, w in zip(outs, want):
        assert torch.equal(got, w)
