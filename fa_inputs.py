"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the attention arithmetic: it only draws random
numbers, rounds them to bf16 and lays them out.  Both the CUDA path and the
CPU oracle read the very same buffers it returns (the oracle after an exact
bf16 -> float64 up-cast), so the generator's device never affects parity.

Recipe (all configurations):
  * ``torch.randn`` in float32 from ``torch.Generator(device).manual_seed(seed)``,
    drawn in the order Q, K, V, then rounded to bf16 (round to nearest even);
  * an optional power-of-two multiplier applied *after* rounding (exact in bf16);
  * layout ``[B, H, rows, d]``, last dimension contiguous.
Decode caches additionally draw per-sequence lengths with
``torch.randint(lo, hi + 1)`` from a CPU generator (so the lengths do not
depend on the device) and fill every cache row past a sequence's length with
bf16 NaN, so that any read past the length poisons the result.
"""
from __future__ import annotations

import torch

BF16 = torch.bfloat16


def _gen(device, seed):
    return torch.Generator(device=device).manual_seed(int(seed))


def attention_inputs(B, H, N, Nk, d, dv, seed=0, mult=1.0, device="cpu"):
    """Q [B,H,N,d], K [B,H,Nk,d], V [B,H,Nk,dv] in bf16, iid N(0,1) (times ``mult``)."""
    g = _gen(device, seed)
    out = []
    for shape in ((B, H, N, d), (B, H, Nk, d), (B, H, Nk, dv)):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(BF16)
        if mult != 1.0:
            x = x * mult
        out.append(x.contiguous())
    return tuple(out)


def grad_output(B, H, N, dv, seed=0, device="cpu"):
    """Upstream gradient dO [B,H,N,dv] for the backward: bf16, iid N(0,1), its own generator stream."""
    g = _gen(device, int(seed) + 7919)
    return torch.randn((B, H, N, dv), generator=g, device=device, dtype=torch.float32).to(BF16).contiguous()


def decode_lengths(B, lo, hi, seed=0):
    """Per-sequence cached lengths drawn uniformly from the closed interval [lo, hi] (int32, CPU)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def decode_inputs(B, H, Nk_max, d, dv, seed=0, lo=1024, hi=None, device="cpu", seqlens=None):
    """Single-query decode inputs.

    Returns q [B,H,1,d], k_cache [B,H,Nk_max,d], v_cache [B,H,Nk_max,dv] (bf16,
    NaN past each sequence's length) and seqlens int32 [B] on the CPU.
    """
    hi = Nk_max if hi is None else hi
    if seqlens is None:
        seqlens = decode_lengths(B, lo, hi, seed)
    g = _gen(device, seed)
    q = torch.randn((B, H, 1, d), generator=g, device=device, dtype=torch.float32).to(BF16)
    k = torch.randn((B, H, Nk_max, d), generator=g, device=device, dtype=torch.float32).to(BF16)
    v = torch.randn((B, H, Nk_max, dv), generator=g, device=device, dtype=torch.float32).to(BF16)
    nan = float("nan")
    for b in range(B):
        n = int(seqlens[b])
        k[b, :, n:, :] = nan
        v[b, :, n:, :] = nan
    return q.contiguous(), k.contiguous(), v.contiguous(), seqlens


def gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, dv, seed=0, lo=1024, hi=None, device="cpu", seqlens=None):
    """Single-query decode inputs with grouped key/value heads: q [B,Hq,1,d], k_cache [B,Hkv,Nk_max,d],
    v_cache [B,Hkv,Nk_max,dv] (bf16, NaN past each sequence's length) and seqlens int32 [B] on the CPU.
    Drawn like ``decode_inputs`` (q, then K, then V from one generator)."""
    hi = Nk_max if hi is None else hi
    if seqlens is None:
        seqlens = decode_lengths(B, lo, hi, seed)
    g = _gen(device, seed)
    q = torch.randn((B, Hq, 1, d), generator=g, device=device, dtype=torch.float32).to(BF16)
    k = torch.randn((B, Hkv, Nk_max, d), generator=g, device=device, dtype=torch.float32).to(BF16)
    v = torch.randn((B, Hkv, Nk_max, dv), generator=g, device=device, dtype=torch.float32).to(BF16)
    nan = float("nan")
    for b in range(B):
        n = int(seqlens[b])
        k[b, :, n:, :] = nan
        v[b, :, n:, :] = nan
    return q.contiguous(), k.contiguous(), v.contiguous(), seqlens


def sample_slices(total, k, seed=1):
    """k distinct indices in [0, total) drawn with a seeded random permutation (sorted)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    idx = torch.randperm(int(total), generator=g)[: int(k)]
    return sorted(int(i) for i in idx)


def merge_inputs(n_parts, rows, dv, seed=0, empty_frac=0.0, device="cpu"):
    """Partial (o_s, lse_s) states for the merge entry point.

    o_parts float32 [n_parts, rows, dv] iid N(0,1); lse_parts float32
    [n_parts, rows] iid N(0, 4); a seeded fraction of the states are empty
    (lse = -inf, o = 0), the convention for a split with no visible key.
    """
    g = _gen(device, seed)
    o = torch.randn((n_parts, rows, dv), generator=g, device=device, dtype=torch.float32)
    lse = torch.randn((n_parts, rows), generator=g, device=device, dtype=torch.float32) * 2.0
    if empty_frac > 0:
        u = torch.rand((n_parts, rows), generator=g, device=device)
        empty = u < empty_frac
        lse = torch.where(empty, torch.full_like(lse, float("-inf")), lse)
        o = torch.where(empty[..., None], torch.zeros_like(o), o)
    return o.contiguous(), lse.contiguous()
