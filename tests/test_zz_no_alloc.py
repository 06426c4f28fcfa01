"""fa_decode_splitkv_noalloc: split-KV decode for callers that cannot allocate device memory.

Such callers (code whose device memory belongs to another allocator, or that runs under a
fixed memory budget) cannot hand fa_decode_splitkv a workspace of their own; this entry point
keeps the split partials in a scratch array owned by the library instead.  The test calls it
through the C ABI and checks that its results match fa_decode_splitkv (with a workspace) within
the parity tolerances, on consecutive calls that reuse the same scratch array.
"""
from __future__ import annotations

import ctypes
import math

import pytest
import torch

from fa_inputs import decode_inputs
from tests.parity import TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


def _entry():
    import exact_tiled_attention_fa_gb300 as fa
    lib = ctypes.CDLL(fa.LIB_PATH)  # the library the binding uses
    f = lib.fa_decode_splitkv_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp]
    f.restype = i
    return fa, f


def _call(f, q, k, v, lens, n_splits):
    B, H, _, d = q.shape
    Nk_max = k.shape[2]
    o = torch.full((B, H, 1, d), float("nan"), dtype=torch.float32, device=q.device)
    lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device=q.device)
    st = f(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
           ctypes.c_void_p(lens.data_ptr()), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
           B, H, Nk_max, d, d, 1.0 / math.sqrt(d), n_splits, 1,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    fa, f = _entry()
    cases = [  # (B, H, Nk_max, d, n_splits, seed): a different problem on each call, then the first again
        (4, 8, 4096, 128, 0, 11),
        (2, 16, 2048, 64, 7, 12),
        (4, 8, 4096, 128, 0, 11),
    ]
    first = None
    for B, H, Nk_max, d, n_splits, seed in cases:
        q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=seed, lo=1, hi=Nk_max, device="cuda")
        lens_d = lens.to("cuda")
        st, o, lse = _call(f, q, k, v, lens_d, n_splits)
        torch.cuda.synchronize()
        assert st == fa.FA_OK, fa.status_string(st)
        assert fa.get_device_error() == fa.FA_OK
        o_ref, lse_ref = fa.decode_splitkv(q, k, v, lens_d, n_splits=n_splits, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert not torch.isnan(o).any() and not torch.isnan(lse).any()
        assert float((o - o_ref).abs().max()) <= TOL_O
        assert float((lse - lse_ref).abs().max()) <= TOL_LSE
        if first is None:
            first = (o, lse)
        elif (B, H, Nk_max, d) == (4, 8, 4096, 128):
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1])


def test_noalloc_rejects_problems_larger_than_its_scratch():
    fa, f = _entry()
    B, H, d = 64, 64, 128
    q = torch.zeros((B, H, 1, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, 256, d), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((B,), 256, dtype=torch.int32, device="cuda")
    st, _, _ = _call(f, q, k, k, lens, 64)  # 64*64*64*(128+1)*4 bytes of partials > 8 MiB
    assert st == fa.FA_ERR_WORKSPACE
