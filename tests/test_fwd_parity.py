"""fa_fwd (CUDA, through the C ABI) against the CPU FP64 oracle on the same bf16 inputs."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import attention_inputs, sample_slices
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def fa():
    import exact_tiled_attention_fa_gb300 as m
    return m


def run(q, k, v, causal, scale=None, out_dtype=torch.float32):
    o, lse = fa().fwd(q, k, v, causal=causal, scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    return o, lse


# (B, H, N, Nk, d, mult): the single-head 256 x 256 case, the pages' demo shapes (77 x 513 with
# causal offset 436, 300 x 300, a single query over 1000 keys), several tiles with ragged tails,
# N > Nk (causal rows with no visible key), and 160 heads of 333 rows at d = 128 (320 items for 152
# CTAs: without a mask the walk crosses from the full query pairs to the one-tile last pairs).
SMALL = [
    (4, 40, 333, 333, 128, 1.0),
    (1, 1, 256, 256, 64, 1.0),
    (8, 8, 77, 513, 32, 2.0),
    (2, 3, 300, 300, 64, 1.0),
    (1, 2, 1, 1000, 64, 1.0),
    (2, 2, 333, 700, 128, 1.0),
    (1, 2, 700, 333, 128, 1.0),
    (1, 1, 200, 100, 64, 1.0),
    (3, 1, 129, 129, 32, 2.0),
    (1, 1, 1, 1, 128, 1.0),
]


@pytest.mark.parametrize("B,H,N,Nk,d,mult", SMALL)
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes_full_oracle(B, H, N, Nk, d, mult, causal):
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, mult=mult, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, scale=scale)
    o, lse = run(q, k, v, causal, scale, torch.float32)
    assert_close(o, lse, o_ref, lse_ref, what=f"fp32 {B,H,N,Nk,d} causal={causal}")
    ob, lseb = run(q, k, v, causal, scale, torch.bfloat16)
    assert_close(ob, lseb, o_ref, lse_ref, bf16_out=True, what=f"bf16 {B,H,N,Nk,d} causal={causal}")


def test_causal_first_row_is_v0_exactly():
    q, k, v = attention_inputs(2, 3, 256, 256, 64, 64, seed=4, device=DEV)
    o, lse = run(q, k, v, True, 0.125, torch.float32)
    assert torch.equal(o[:, :, 0, :], v[:, :, 0, :].float())
    ref = (q[:, :, 0, :].double() * k[:, :, 0, :].double()).sum(-1) * 0.125
    assert float((lse[:, :, 0].double() - ref).abs().max()) <= 1e-5


def test_rows_without_visible_keys():
    q, k, v = attention_inputs(1, 2, 300, 100, 64, 64, seed=5, device=DEV)
    o, lse = run(q, k, v, True, 0.125, torch.float32)
    assert torch.all(o[:, :, :200] == 0) and torch.all(torch.isneginf(lse[:, :, :200]))


@pytest.mark.parametrize("d", [128, 64, 32])
def test_deterministic_and_no_writes_past_output(d):
    # d <= 64 writes O through a staging tile and bulk tensor stores, d = 128 row by row; at an
    # output 32-byte aligned or only 16-byte aligned, both must leave the memory around O untouched
    # (the last query tile is ragged) and give the same bits.
    B, H, N, Nk = 2, 2, 333, 257
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=6, device=DEV)
    guard = 4096
    n = B * H * N * d
    for causal in (False, True):
        for dt in (torch.float32, torch.bfloat16):
            o2, lse2 = fa().fwd(q, k, v, causal=causal, out_dtype=dt)
            for shift in (0, 16 // torch.empty((), dtype=dt).element_size()):  # 0 or 16 bytes past 32-byte alignment
                buf = torch.full((n + 2 * guard,), float("nan"), dtype=dt, device=DEV)
                lbuf = torch.full((B * H * N + guard,), float("nan"), dtype=torch.float32, device=DEV)
                o = buf[guard + shift: guard + shift + n].view(B, H, N, d)
                lse = lbuf[: B * H * N].view(B, H, N)
                fa().fwd(q, k, v, causal=causal, out=o, lse=lse)
                torch.cuda.synchronize()
                assert not torch.isnan(o).any() and not torch.isnan(lse).any()
                assert torch.isnan(buf[: guard + shift]).all() and torch.isnan(buf[guard + shift + n:]).all()
                assert torch.isnan(lbuf[B * H * N:]).all()
                assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_q_zero_averages_visible_values():
    B, H, N, Nk, d = 1, 2, 130, 390, 64
    _, k, v = attention_inputs(B, H, N, Nk, d, d, seed=7, device=DEV)
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=DEV)
    for causal in (False, True):
        o, lse = run(q, k, v, causal, 0.125, torch.float32)
        vv = to_np(v)
        for i in (0, 1, 77, 129):
            n = Nk - N + i + 1 if causal else Nk
            assert np.abs(to_np(o)[:, :, i] - vv[:, :, :n].mean(axis=2)).max() <= 1e-4
            assert np.abs(to_np(lse)[:, :, i] - math.log(n)).max() <= 1e-5


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("N,Nk,j", [(512, 512, 300), (512, 512, 200), (512, 512, 511), (512, 512, 5),
                                    (300, 512, 400)])
@pytest.mark.parametrize("bad", [float("nan"), float("inf")], ids=["nan", "inf"])
def test_causal_hidden_key_does_not_reach_earlier_rows(d, N, Nk, j, bad):
    """Under the causal mask a key reaches only the rows that see it: with every element of key j
    non-finite, the rows placed before position j must equal the oracle on the clean keys.  Key 300
    lies in the second 32-column chunk of diagonal tile 2 (a chunk hidden from the tile's first warp
    and cut by its second), key 200 in the third chunk of tile 1, key 511 in the last chunk of the
    last tile; with N < Nk the rows sit at positions Nk - N + i."""
    B, H = 1, 2
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=8, device=DEV)
    scale = 1.0 / math.sqrt(d)
    r1 = j - (Nk - N)  # rows 0 .. r1 - 1 do not see key j
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=scale, rows=(0, r1))
    kb = k.clone()
    kb[:, :, j, :] = bad
    o, lse = run(q, kb, v, True, scale, torch.float32)
    assert_close(o[:, :, :r1], lse[:, :, :r1], o_ref, lse_ref, what=f"d={d} N={N} Nk={Nk} key {j} = {bad}")


def _sampled_check(B, H, N, Nk, d, mult, causal, n_slices, rows=None, seed=0, out_dtype=torch.float32):
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=seed, mult=mult, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(q, k, v, causal, scale, out_dtype)
    for idx in sample_slices(B * H, n_slices, seed=1):
        b, h = divmod(idx, H)
        for (r0, r1) in rows or [(0, N)]:
            o_ref, lse_ref = oracle.attention(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), causal=causal,
                                              scale=scale, rows=(r0, r1))
            assert_close(o[b, h, r0:r1], lse[b, h, r0:r1], o_ref, lse_ref,
                         bf16_out=(out_dtype == torch.bfloat16), what=f"(b,h)=({b},{h}) rows {r0}:{r1}")


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_medium_shape_sampled(causal):
    """B=64, H=16, N=Nk=1024, d=64: 32 seeded (b, h) slices against the oracle."""
    _sampled_check(64, 16, 1024, 1024, 64, 1.0, causal, 32)


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_medium_shape_bf16_out_sampled(causal):
    _sampled_check(64, 16, 1024, 1024, 64, 1.0, causal, 4, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_4097_sampled(causal, out_dtype):
    """B=4, H=16, N=Nk=4097, d=128, inputs x2: 3 heads, first and last 384 rows (the ragged tail tile),
    with fp32 O and with the benchmark's bf16 O."""
    _sampled_check(4, 16, 4097, 4097, 128, 2.0, causal, 3, rows=[(0, 384), (3713, 4097)], out_dtype=out_dtype)


def test_ragged_77_513_full():
    """B=8, H=8, N=77, Nk=513, d=32, inputs x2, causal offset 436 (every head)."""
    q, k, v = attention_inputs(8, 8, 77, 513, 32, 32, seed=0, mult=2.0, device=DEV)
    scale = 1.0 / math.sqrt(32)
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, scale=scale)
        for dt in (torch.float32, torch.bfloat16):
            o, lse = run(q, k, v, causal, scale, dt)
            assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16), what=f"77x513 causal={causal} {dt}")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_long_causal_sampled(out_dtype):
    """B=2, H=32, N=Nk=16384, d=128, causal: 4 heads x first 2048 rows, and the last 128 rows of one head,
    with fp32 O and with the benchmark's bf16 O."""
    _sampled_check(2, 32, 16384, 16384, 128, 1.0, True, 4, rows=[(0, 2048)], out_dtype=out_dtype)
    _sampled_check(2, 32, 16384, 16384, 128, 1.0, True, 1, rows=[(16256, 16384)], out_dtype=out_dtype)


def test_bounded_wait_reports_timeout_and_context_survives():
    """A 1 ns wait limit makes the kernel's first barrier wait run out: the kernel records
    FA_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and returns; the
    context stays usable and the next call (default limit) is correct."""
    q, k, v = attention_inputs(2, 4, 1024, 1024, 64, 64, seed=8, device=DEV)
    fa().set_wait_timeout_ns(1)
    try:
        fa().fwd(q, k, v, causal=False, out_dtype=torch.float32)
        status = fa().get_device_error()
    finally:
        fa().set_wait_timeout_ns(0)
    assert status == fa().FA_ERR_TIMEOUT
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=0.125)
    o, lse = run(q, k, v, True, 0.125, torch.float32)
    assert_close(o, lse, o_ref, lse_ref, what="after a timed-out launch")


# Split-KV forward: few query tiles, keys cut into chunks of whole 128-key tiles and merged.
SPLIT = [
    (8, 8, 77, 513, 32, 2.0),     # the pages' ragged demo shape, causal offset 436
    (1, 2, 300, 1000, 64, 1.0),
    (2, 1, 700, 333, 128, 1.0),   # N > Nk: causal rows with no visible key
    (1, 1, 1, 2000, 64, 1.0),
    (1, 3, 256, 4097, 128, 2.0),
    (4, 16, 300, 2000, 64, 1.0),  # 128 heads x 2 query pairs: several split items per CTA
    (2, 3, 500, 260, 64, 1.0),    # N > Nk at d = 64: causal rows with no visible key, ragged key tail
]


@pytest.mark.parametrize("B,H,N,Nk,d,mult", SPLIT)
@pytest.mark.parametrize("n_splits", [1, 3, 0])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_splitkv_full_oracle(B, H, N, Nk, d, mult, n_splits, causal):
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=2, mult=mult, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, scale=scale)
    for dt in (torch.float32, torch.bfloat16):
        o, lse = fa().fwd_splitkv(q, k, v, causal=causal, scale=scale, n_splits=n_splits, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16),
                     what=f"splitkv {B,H,N,Nk,d} n={n_splits} causal={causal} {dt}")


@pytest.mark.parametrize("B,H,N,Nk,d", [(1, 2, 300, 1000, 64), (2, 1, 700, 333, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_splitkv_one_key_tile_per_split(B, H, N, Nk, d, causal):
    """n_splits = 999 (reduced to Nk, then to one 128-key tile per split): the most split items,
    each with a single key tile (the last one ragged)."""
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=3, device=DEV)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, scale=1.0 / math.sqrt(d))
    o, lse = fa().fwd_splitkv(q, k, v, causal=causal, n_splits=999, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    assert_close(o, lse, o_ref, lse_ref, what=f"splitkv one tile per split {B,H,N,Nk,d} causal={causal}")


def test_fwd_splitkv_long_context_sampled():
    """Few query tiles over a long context (B=1, H=8, N=512, Nk=32768, d=128, causal): the
    benchmark's split-KV prefill workload; two heads' last 256 rows against the oracle."""
    B, H, N, Nk, d = 1, 8, 512, 32768, 128
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, device=DEV)
    o, lse = fa().fwd_splitkv(q, k, v, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    for h in sample_slices(H, 2, seed=1):
        o_ref, l_ref = oracle.attention(q[0, h].cpu(), k[0, h].cpu(), v[0, h].cpu(), causal=True,
                                        scale=1 / math.sqrt(d), rows=(N - 256, N))
        assert_close(o[0, h, N - 256:], lse[0, h, N - 256:], o_ref, l_ref, what=f"long ctx h={h}")


def test_splitkv_bounded_wait_reports_timeout_and_context_survives():
    """The split-KV kernel under a 1 ns wait limit (prefill and packed-group decode) records
    FA_ERR_TIMEOUT and returns; the next calls are correct."""
    from fa_inputs import gqa_decode_inputs
    q, k, v = attention_inputs(1, 4, 256, 4096, 128, 128, seed=10, device=DEV)
    # 8 query heads per key/value head: d = 128 runs the transposed kernel, d = 64 the row kernel
    qd, kc, vc, lens = gqa_decode_inputs(2, 16, 2, 2048, 128, 128, seed=10, lo=100, hi=2048, device=DEV)
    q6, k6, v6, l6 = gqa_decode_inputs(2, 16, 2, 2048, 64, 64, seed=10, lo=100, hi=2048, device=DEV)
    fa().set_wait_timeout_ns(1)
    try:
        fa().fwd_splitkv(q, k, v, causal=True, n_splits=4, out_dtype=torch.float32)
        s1 = fa().get_device_error()
        fa().decode_splitkv_gqa(qd, kc, vc, lens.to(DEV), n_splits=4, out_dtype=torch.float32)
        s2 = fa().get_device_error()
        fa().decode_splitkv_gqa(q6, k6, v6, l6.to(DEV), n_splits=4, out_dtype=torch.float32)
        s3 = fa().get_device_error()
    finally:
        fa().set_wait_timeout_ns(0)
    assert s1 == fa().FA_ERR_TIMEOUT and s2 == fa().FA_ERR_TIMEOUT and s3 == fa().FA_ERR_TIMEOUT
    o, lse = fa().decode_splitkv_gqa(qd, kc, vc, lens.to(DEV), n_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    for b in range(2):
        n = int(lens[b])
        for h in range(16):
            o_ref, l_ref = oracle.attention(qd[b, h].cpu(), kc[b, h // 8, :n].cpu(), vc[b, h // 8, :n].cpu(),
                                            scale=1 / math.sqrt(128))
            assert_close(o[b, h], lse[b, h], o_ref, l_ref, what=f"gqa after a timed-out launch b={b} h={h}")
    o, lse = fa().fwd_splitkv(q, k, v, causal=True, n_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=1 / math.sqrt(128))
    assert_close(o, lse, o_ref, lse_ref, what="splitkv after a timed-out launch")
