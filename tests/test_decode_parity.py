"""fa_decode_splitkv and fa_merge_states (CUDA, through the C ABI) against the CPU FP64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import decode_inputs, gqa_decode_inputs, merge_inputs
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def fa():
    import exact_tiled_attention_fa_gb300 as m
    return m


def oracle_decode_compact(q, k, v, lens, scale):
    """Oracle on each sequence's own prefix (never copies the padding to the host)."""
    B, H = q.shape[0], q.shape[1]
    dv = v.shape[-1]
    O = np.zeros((B, H, 1, dv))
    L = np.zeros((B, H, 1))
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            L[b] = -np.inf
            continue
        o_b, l_b = oracle.attention(q[b].cpu(), k[b, :, :n].cpu(), v[b, :, :n].cpu(), causal=False, scale=scale)
        O[b], L[b] = o_b, l_b
    return O, L


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("n_splits", [1, 3, 16, 0, 999])
def test_small_decode(d, n_splits):
    B, H, Nk_max = 4, 3, 1000
    lens = torch.tensor([1, 64, 65, 1000], dtype=torch.int32)
    q, k, v, _ = decode_inputs(B, H, Nk_max, d, d, seed=d, device=DEV, seqlens=lens)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle_decode_compact(q, k, v, lens, scale)
    for dt in (torch.float32, torch.bfloat16):
        o, lse = fa().decode_splitkv(q, k, v, lens.to(DEV), scale=scale, n_splits=n_splits, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16), what=f"d={d} n={n_splits} {dt}")


def test_zero_length_and_clamped_lengths():
    B, H, Nk_max, d = 3, 2, 300, 64
    lens_in = torch.tensor([0, -5, 310], dtype=torch.int32)  # -5 and 310 are out of range
    q, k, v, _ = decode_inputs(B, H, Nk_max, d, d, seed=1, device=DEV, seqlens=torch.tensor([0, 0, 300]))
    o, lse = fa().decode_splitkv(q, k, v, lens_in.to(DEV), n_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == fa().FA_ERR_INVALID_ARG  # recorded, lengths clamped to [0, 300]
    assert fa().get_device_error() == 0  # reading cleared it
    assert torch.all(o[:2] == 0) and torch.all(torch.isneginf(lse[:2]))
    o_ref, lse_ref = oracle_decode_compact(q[2:], k[2:], v[2:], [300], 1 / 8)
    assert_close(o[2:], lse[2:], o_ref, lse_ref, what="clamped length")


def test_split_invariance_and_determinism():
    B, H, Nk_max, d = 2, 4, 4096, 128
    q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=3, lo=1, hi=Nk_max, device=DEV)
    outs = []
    for n in (1, 2, 7, 32, 64):
        o, lse = fa().decode_splitkv(q, k, v, lens.to(DEV), n_splits=n, out_dtype=torch.float32)
        o2, lse2 = fa().decode_splitkv(q, k, v, lens.to(DEV), n_splits=n, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert float((o - outs[0][0]).abs().max()) <= 2e-3
        assert float((lse - outs[0][1]).abs().max()) <= 2e-4


def test_full_decode_config():
    """B=16, H=32, d=128, lengths ~ U{1024..32768} (seed 0), caches padded to 32768 with NaN:
    every one of the 512 heads against the oracle."""
    B, H, Nk_max, d = 16, 32, 32768, 128
    q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=0, lo=1024, hi=32768, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle_decode_compact(q, k, v, lens, scale)
    for dt in (torch.float32, torch.bfloat16):  # fp32 O, and the benchmark's bf16 O
        o, lse = fa().decode_splitkv(q, k, v, lens.to(DEV), scale=scale, n_splits=0, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16), what=f"decode B16 H32 Nk<=32768 {dt}")


@pytest.mark.parametrize("n_parts,rows,dv,empty", [(1, 5, 128, 0.0), (16, 333, 128, 0.3), (999, 7, 64, 0.5),
                                                   (3, 64, 512, 0.0), (4, 10, 33, 1.0), (16, 50, 256, 0.2),
                                                   (77, 9, 32, 0.4)])
def test_merge_states_against_oracle(n_parts, rows, dv, empty):
    o_parts, lse_parts = merge_inputs(n_parts, rows, dv, seed=n_parts, empty_frac=empty, device=DEV)
    o_ref, lse_ref = oracle.merge_lse(o_parts.cpu(), lse_parts.cpu())
    o, lse = fa().merge_states(o_parts, lse_parts, out_dtype=torch.float32)
    torch.cuda.synchronize()
    a, b = to_np(lse), lse_ref
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = ~np.isneginf(b)
    if fin.any():
        assert np.abs(a[fin] - b[fin]).max() <= 1e-5 * max(1.0, np.abs(b[fin]).max())
    assert np.abs(to_np(o) - o_ref).max() <= 1e-5


@pytest.mark.parametrize("dv,offset", [(128, 0), (33, 0), (64, 1), (512, 0)])
def test_merge_states_never_reads_empty_parts(dv, offset):
    """Empty parts (lse = -inf) may hold anything: a split with no visible key writes nothing.
    With NaN there the merge must equal the oracle on the zero-filled states.  offset = 1 starts
    the parts 4 bytes past a 16-byte boundary (the scalar-load form of the merge)."""
    n_parts, rows = 37, 21
    o_parts, lse_parts = merge_inputs(n_parts, rows, dv, seed=dv + offset, empty_frac=0.6, device=DEV)
    o_ref, lse_ref = oracle.merge_lse(o_parts.cpu(), lse_parts.cpu())
    buf = torch.empty(n_parts * rows * dv + offset, dtype=torch.float32, device=DEV)
    o_bad = buf[offset:].view(n_parts, rows, dv)
    o_bad.copy_(torch.where(torch.isneginf(lse_parts)[..., None], torch.full_like(o_parts, float("nan")), o_parts))
    o, lse = fa().merge_states(o_bad, lse_parts, out_dtype=torch.float32)
    torch.cuda.synchronize()
    a, b = to_np(lse), lse_ref
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = ~np.isneginf(b)
    assert np.abs(a[fin] - b[fin]).max() <= 1e-5 * max(1.0, np.abs(b[fin]).max())
    assert np.isfinite(to_np(o)).all() and np.abs(to_np(o) - o_ref).max() <= 1e-5


def oracle_gqa_compact(q, k, v, lens, scale):
    """Oracle for grouped heads: query head h attends with key/value head h // R over its
    sequence's prefix; each group's cache rows are repeated for its R query heads (the pages'
    packing of a group's query heads against one K, V)."""
    B, Hq = q.shape[0], q.shape[1]
    R = Hq // k.shape[1]
    dv = v.shape[-1]
    O = np.zeros((B, Hq, 1, dv))
    L = np.zeros((B, Hq, 1))
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            L[b] = -np.inf
            continue
        kb = k[b, :, :n].cpu().repeat_interleave(R, dim=0)
        vb = v[b, :, :n].cpu().repeat_interleave(R, dim=0)
        O[b], L[b] = oracle.attention(q[b].cpu(), kb, vb, causal=False, scale=scale)
    return O, L


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 40])  # 24: a padded fourth warp set
@pytest.mark.parametrize("n_splits", [1, 5, 0])
def test_gqa_decode(d, R, n_splits):
    B, Hkv, Nk_max = 3, 2, 700
    lens = torch.tensor([1, 300, 700], dtype=torch.int32)
    q, k, v, _ = gqa_decode_inputs(B, Hkv * R, Hkv, Nk_max, d, d, seed=R + d, device=DEV, seqlens=lens)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle_gqa_compact(q, k, v, lens, scale)
    for dt in (torch.float32, torch.bfloat16):
        o, lse = fa().decode_splitkv_gqa(q, k, v, lens.to(DEV), scale=scale, n_splits=n_splits, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16), what=f"gqa d={d} R={R} n={n_splits}")


@pytest.mark.parametrize("R", [3, 8, 40], ids=["R3_transposed", "R8_transposed", "R40_row_tile"])
def test_gqa_zero_and_clamped_lengths(R):
    """Grouped decode on the tensor core (d = 128) with a zero-length sequence, lengths just past a
    128-key tile and an out-of-range length: the last is clamped to the cache and reported, a sequence
    with no keys gives O = 0 and LSE = -inf, the others match the oracle."""
    B, Hkv, Nk_max, d = 4, 2, 640, 128
    lens_ok = torch.tensor([0, 129, 257, 640], dtype=torch.int32)
    q, k, v, _ = gqa_decode_inputs(B, Hkv * R, Hkv, Nk_max, d, d, seed=R, device=DEV, seqlens=lens_ok)
    lens_in = torch.tensor([0, 129, 257, 700], dtype=torch.int32)  # 700 > Nk_max: clamped to 640
    o, lse = fa().decode_splitkv_gqa(q, k, v, lens_in.to(DEV), n_splits=3, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == fa().FA_ERR_INVALID_ARG
    assert fa().get_device_error() == 0
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    o_ref, lse_ref = oracle_gqa_compact(q[1:], k[1:], v[1:], lens_ok[1:], 1 / math.sqrt(d))
    assert_close(o[1:], lse[1:], o_ref, lse_ref, what=f"gqa lengths R={R}")


@pytest.mark.parametrize("Hkv", [8, 4, 1], ids=["R4_tensor_core", "R8_tensor_core", "R32_four_warp_sets"])
def test_gqa_full_size_sampled(Hkv):
    """The benchmark's GQA workloads (B=16, Hq=32 over Hkv=8 or 4, d=128, lengths U[1024, 32768]) in
    their launch configuration, and the same cache with 32 heads per group (four warp sets of the
    transposed kernel), with fp32 O and with the benchmark's bf16 O; 24 seeded query heads against
    the oracle."""
    B, Hq, Nk_max, d = 16, 32, 32768, 128
    q, k, v, lens = gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, d, seed=0, lo=1024, hi=Nk_max, device=DEV)
    R = Hq // Hkv
    refs = {}
    for idx in sample_slices_gqa(B * Hq, 24):
        b, h = divmod(idx, Hq)
        n = int(lens[b])
        refs[(b, h)] = oracle.attention(q[b, h].cpu(), k[b, h // R, :n].cpu(), v[b, h // R, :n].cpu(),
                                        scale=1 / math.sqrt(d))
    for dt in (torch.float32, torch.bfloat16):
        o, lse = fa().decode_splitkv_gqa(q, k, v, lens.to(DEV), out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        for (b, h), (o_ref, l_ref) in refs.items():
            assert_close(o[b, h], lse[b, h], o_ref, l_ref, bf16_out=(dt == torch.bfloat16),
                         what=f"gqa full R={R} b={b} h={h} {dt}")


def sample_slices_gqa(total, k):
    from fa_inputs import sample_slices
    return sample_slices(total, k, seed=1)


def test_gqa_rejects_bad_groups():
    q = torch.zeros((1, 6, 1, 64), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((1, 4, 128, 64), dtype=torch.bfloat16, device=DEV)
    lens = torch.full((1,), 128, dtype=torch.int32, device=DEV)
    with pytest.raises(fa().FaError) as e:  # 6 query heads over 4 key/value heads
        fa().decode_splitkv_gqa(q, k, k, lens)
    assert e.value.status == fa().FA_ERR_INVALID_ARG
    q3 = torch.zeros((1, 256, 1, 64), dtype=torch.bfloat16, device=DEV)
    k3 = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa().FaError) as e:  # a group of 256 heads does not fit a 128-row tile
        fa().decode_splitkv_gqa(q3, k3, k3, lens)
    assert e.value.status == fa().FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("n_splits", [1, 3, 16, 0])
def test_fused_combine(d, n_splits):
    """The combine done by each row's last split: oracle parity, counters left zero, and bit-equal
    to itself on a second call with the same workspace."""
    B, H, Nk_max = 5, 3, 1000
    lens = torch.tensor([0, 1, 64, 65, 1000], dtype=torch.int32)
    q, k, v, _ = decode_inputs(B, H, Nk_max, d, d, seed=d + 1, device=DEV, seqlens=lens)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle_decode_compact(q, k, v, lens, scale)
    ws = fa().decode_fused_workspace(B, H, Nk_max, d, n_splits=n_splits, device=DEV)
    parts = fa().decode_workspace_size(B, H, d, max(1, n_splits or fa().decode_default_splits(B, H, Nk_max, fa().num_sms())))
    first = None
    for dt in (torch.float32, torch.bfloat16, torch.float32):
        o, lse = fa().decode_splitkv_fused(q, k, v, lens.to(DEV), ws, scale=scale, n_splits=n_splits, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa().get_device_error() == 0
        assert int(ws[parts:].count_nonzero()) == 0, "arrival counters not reset"
        assert_close(o, lse, o_ref, lse_ref, bf16_out=(dt == torch.bfloat16), what=f"fused d={d} n={n_splits}")
        if dt == torch.float32:
            if first is None:
                first = (o.clone(), lse.clone())
            else:
                assert torch.equal(o, first[0]) and torch.equal(lse, first[1])


def test_fused_combine_full_size_matches_two_kernel_path():
    B, H, Nk_max, d = 16, 32, 32768, 128
    q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=0, lo=1024, hi=Nk_max, device=DEV)
    ld = lens.to(DEV)
    o2, l2 = fa().decode_splitkv(q, k, v, ld, out_dtype=torch.float32)
    ws = fa().decode_fused_workspace(B, H, Nk_max, d, device=DEV)
    o1, l1 = fa().decode_splitkv_fused(q, k, v, ld, ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa().get_device_error() == 0
    # same splits, same partials, the same merge arithmetic in a different kernel
    assert float((o1 - o2).abs().max()) <= 1e-6 and float((l1 - l2).abs().max()) <= 1e-6
