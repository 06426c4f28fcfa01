"""fa_decode_splitkv_noalloc: split-KV decode for callers that cannot allocate device memory.

Such callers (code whose device memory belongs to another allocator, or that runs under a
fixed memory budget) cannot hand fa_decode_splitkv a workspace of their own; this entry point
keeps the split partials in a scratch array owned by the library instead.  The tests call it
through the C ABI on consecutive calls that reuse the same scratch array and check that
  * its output is bit for bit that of fa_decode_splitkv (with a workspace) at the same split
    count: both run the same kernels on the same inputs, so any difference is a fault;
  * it matches the FP64 oracle within the parity tolerances, for fp32 and bf16 O and
    head sizes 32, 64 and 128;
  * problems whose partials do not fit are rejected with FA_ERR_WORKSPACE before anything is
    launched (outputs untouched), for an explicit split count and for the automatic one.
This file is collected last, so that a run stopping at its first failure has run every other
test before it.
"""
from __future__ import annotations

import ctypes
import math

import pytest
import torch

import oracle
from fa_inputs import decode_inputs
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def _entry():
    import exact_tiled_attention_fa_gb300 as fa
    lib = ctypes.CDLL(fa.LIB_PATH)  # the library the binding uses
    f = lib.fa_decode_splitkv_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp]
    f.restype = i
    return fa, f


def _call(fa, f, q, k, v, lens, n_splits, out_dtype=torch.float32):
    B, H, _, d = q.shape
    Nk_max = k.shape[2]
    o = torch.full((B, H, 1, d), float("nan"), dtype=out_dtype, device=q.device)
    lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device=q.device)
    st = f(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
           ctypes.c_void_p(lens.data_ptr()), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
           B, H, Nk_max, d, d, 1.0 / math.sqrt(d), n_splits, fa.FA_F32 if out_dtype == torch.float32 else fa.FA_BF16,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def _oracle(q, k, v, lens):
    """FP64 oracle on each sequence's valid cache prefix (the NaN padding is never read)."""
    B = q.shape[0]
    outs = [oracle.decode(q[b:b + 1].cpu(), k[b:b + 1, :, :int(lens[b])].cpu(), v[b:b + 1, :, :int(lens[b])].cpu(),
                          [int(lens[b])]) for b in range(B)]
    import numpy as np
    return np.concatenate([o for o, _ in outs]), np.concatenate([l for _, l in outs])


def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls():
    fa, f = _entry()
    cases = [  # (B, H, Nk_max, d, n_splits, seed, O dtype): a different problem on each call, then the first again
        (4, 8, 4096, 128, 0, 11, torch.float32),
        (2, 16, 2048, 64, 7, 12, torch.bfloat16),
        (3, 4, 1500, 32, 5, 13, torch.float32),
        (2, 6, 777, 32, 0, 14, torch.bfloat16),
        (4, 8, 4096, 128, 0, 11, torch.float32),
    ]
    first = None
    for B, H, Nk_max, d, n_splits, seed, dt in cases:
        q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=seed, lo=1, hi=Nk_max, device="cuda")
        lens_d = lens.to("cuda")
        st, o, lse = _call(fa, f, q, k, v, lens_d, n_splits, dt)
        torch.cuda.synchronize()
        assert st == fa.FA_OK, fa.status_string(st)
        assert fa.get_device_error() == fa.FA_OK
        n = n_splits or fa.decode_default_splits(B, H, Nk_max, fa.num_sms())
        o_ref, lse_ref = fa.decode_splitkv(q, k, v, lens_d, n_splits=n, out_dtype=dt)
        torch.cuda.synchronize()
        what = f"B={B} H={H} Nk_max={Nk_max} d={d} n_splits={n_splits} {dt}"
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), what  # same kernels, same inputs
        o_or, lse_or = _oracle(q, k, v, lens)
        assert_close(o, lse, o_or, lse_or, bf16_out=(dt == torch.bfloat16), what=what)
        if first is None:
            first = (o, lse)
        elif (B, H, Nk_max, d) == (4, 8, 4096, 128):
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1])


@pytest.mark.parametrize("B,H,Nk,n_splits", [(64, 64, 256, 64), (128, 160, 64, 0)],
                         ids=["explicit_splits", "automatic_splits"])
def test_noalloc_rejects_problems_larger_than_its_scratch(B, H, Nk, n_splits):
    """64*64 heads x 64 splits, or 128*160 heads with the automatic count (one split each): the
    fp32 partials, B*H*n*(128+1)*4 bytes, exceed the 8 MiB scratch."""
    fa, f = _entry()
    d = 128
    q = torch.zeros((B, H, 1, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((B,), Nk, dtype=torch.int32, device="cuda")
    n = n_splits or fa.decode_default_splits(B, H, Nk, fa.num_sms())
    assert fa.decode_workspace_size(B, H, d, n) > 8 << 20
    st, o, lse = _call(fa, f, q, k, k, lens, n_splits)
    torch.cuda.synchronize()
    assert st == fa.FA_ERR_WORKSPACE
    assert torch.isnan(o).all() and torch.isnan(lse).all()  # nothing was launched
    assert fa.get_device_error() == fa.FA_OK
