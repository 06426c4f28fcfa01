"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments on the host before launching anything."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import exact_tiled_attention_fa_gb300 as fa
from exact_tiled_attention_fa_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

# A fake but 256-byte-aligned device address: argument checks reject the call before it is used.
P = ctypes.c_void_p(0x10000000)
NULL = ctypes.c_void_p(0)


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_decode_splitkv", "fa_merge_states", "fa_get_device_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def _fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=8, Nk=8, d=64, dv=64, causal=0, scale=0.125, odt=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, Nk, d, dv, causal, scale, odt, NULL)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, q=NULL) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, o=NULL) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, N=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, Nk=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, odt=7) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, q=ctypes.c_void_p(0x10000008)) == fa.FA_ERR_INVALID_ARG  # not 16-byte aligned
    assert _fwd(lib, lse=ctypes.c_void_p(0x10000002)) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=48, dv=48) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=64, dv=128) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256, dv=256) == fa.FA_ERR_UNSUPPORTED


def test_sizes_past_the_index_limits_are_rejected(lib):
    # The kernels index work items (and, in split mode, rows) with 32-bit integers; sizes whose
    # item or row count passes the stated limits return FA_ERR_INVALID_ARG before any launch.  Each
    # case has a control just under the limit that gets past the size check and is then rejected by
    # a later one (head size or workspace), so nothing is launched on the fake pointers.
    assert _fwd(lib, B=32768, H=32768, N=256, Nk=256) == fa.FA_ERR_INVALID_ARG  # 2^30 items
    assert _fwd(lib, B=32767, H=32767, N=256, Nk=256, d=48, dv=48) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, B=16384, H=32768, N=512, Nk=256) == fa.FA_ERR_INVALID_ARG
    bwd = lib.fa_bwd
    def call_bwd(B, H, ws_bytes):
        return bwd(P, P, P, P, P, P, P, P, P, P, ws_bytes, B, H, 128, 128, 64, 64, 0, 0.125, 0, 0, NULL)
    assert call_bwd(32768, 32768, 1 << 40) == fa.FA_ERR_INVALID_ARG  # 2^30 key-tile items
    assert call_bwd(32767, 32767, 0) == fa.FA_ERR_WORKSPACE
    skv = lib.fa_fwd_splitkv
    def call_skv(B, H, N, Nk, n, d=64):
        return skv(P, P, P, P, P, P, 1 << 60, B, H, N, Nk, d, d, 0, 0.125, n, 0, NULL)
    assert call_skv(65536, 32768, 1, 128, 1) == fa.FA_ERR_INVALID_ARG  # B*H*N = 2^31 rows
    assert call_skv(65535, 32768, 1, 128, 1, d=48) == fa.FA_ERR_UNSUPPORTED
    gqa = lib.fa_decode_splitkv_gqa
    def call_gqa(B, d=128):
        return gqa(P, P, P, P, P, P, P, 1 << 40, B, 8, 2, 1000, d, d, 0.1, 4, 0, NULL)
    assert call_gqa(65536) == fa.FA_ERR_INVALID_ARG
    assert call_gqa(65535, d=96) == fa.FA_ERR_UNSUPPORTED


def _dec(lib, ws_bytes=1 << 20, n_splits=4, q=P, ws=P, B=2, H=2, Nk=1000, d=128, dv=128, scale=0.1, odt=0):
    return lib.fa_decode_splitkv(q, P, P, P, P, P, ws, ws_bytes, B, H, Nk, d, dv, scale, n_splits, odt, NULL)


def test_decode_rejects_bad_arguments(lib):
    assert _dec(lib, q=NULL) == fa.FA_ERR_INVALID_ARG
    assert _dec(lib, ws=NULL) == fa.FA_ERR_INVALID_ARG
    assert _dec(lib, ws=ctypes.c_void_p(0x10000010)) == fa.FA_ERR_INVALID_ARG  # workspace not 256-aligned
    assert _dec(lib, n_splits=-1) == fa.FA_ERR_INVALID_ARG
    assert _dec(lib, Nk=0) == fa.FA_ERR_INVALID_ARG
    assert _dec(lib, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert _dec(lib, d=96, dv=96) == fa.FA_ERR_UNSUPPORTED
    need = lib.fa_decode_workspace_size(2, 2, 128, 4)
    assert _dec(lib, ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert _dec(lib, ws_bytes=0) == fa.FA_ERR_WORKSPACE


def test_gqa_decode_rejects_bad_arguments(lib):
    f = lib.fa_decode_splitkv_gqa
    def call(B=2, Hq=8, Hkv=2, Nk=1000, d=128, ws=P, ws_bytes=1 << 20, n=4):
        return f(P, P, P, P, P, P, ws, ws_bytes, B, Hq, Hkv, Nk, d, d, 0.1, n, 0, NULL)
    assert call(Hkv=0) == fa.FA_ERR_INVALID_ARG
    assert call(Hq=6, Hkv=4) == fa.FA_ERR_INVALID_ARG   # Hkv must divide Hq
    assert call(Hq=512, Hkv=2) == fa.FA_ERR_UNSUPPORTED  # group of 256 heads exceeds a 128-row tile
    need = lib.fa_decode_workspace_size(2, 8, 128, 4)
    assert call(ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


def test_fwd_splitkv_rejects_bad_arguments(lib):
    f = lib.fa_fwd_splitkv
    def call(q=P, ws=P, ws_bytes=1 << 24, B=1, H=2, N=100, Nk=1000, d=64, causal=0, n=4, scale=0.125):
        return f(q, P, P, P, P, ws, ws_bytes, B, H, N, Nk, d, d, causal, scale, n, 0, NULL)
    assert call(q=NULL) == fa.FA_ERR_INVALID_ARG
    assert call(ws=NULL) == fa.FA_ERR_INVALID_ARG
    assert call(n=-1) == fa.FA_ERR_INVALID_ARG
    assert call(causal=3) == fa.FA_ERR_INVALID_ARG
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED
    need = lib.fa_fwd_splitkv_workspace_size(1, 2, 100, 64, 4)
    assert need == (2 * 100 * 4 * 64 * 4 + 255) // 256 * 256 + (2 * 100 * 4 * 4 + 255) // 256 * 256
    assert call(ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    ds = lib.fa_fwd_splitkv_default_splits
    assert ds(1, 1, 1, 100000, 152) >= 2 and ds(64, 16, 1024, 1024, 152) == 1
    assert 1 <= ds(8, 8, 77, 513, 152) <= 5
    # one round: the most splits for which pairs of query tiles x splits fit one CTA per SM
    assert ds(1, 8, 512, 32768, 152) == 9 and ds(1, 4, 128, 131072, 152) == 38 and ds(2, 8, 384, 16384, 152) == 4
    for (B, H, N, Nk) in ((1, 8, 512, 32768), (1, 3, 200, 50000), (2, 5, 129, 9000), (1, 1, 64, 1000)):
        pairs, n = B * H * -(-N // 256), ds(B, H, N, Nk, 152)
        assert n == min(max(1, 152 // pairs), -(-Nk // 128))


def test_merge_rejects_bad_arguments(lib):
    m = lib.fa_merge_states
    assert m(NULL, P, 2, 3, 4, P, P, 0, NULL) == fa.FA_ERR_INVALID_ARG
    assert m(P, P, 0, 3, 4, P, P, 0, NULL) == fa.FA_ERR_INVALID_ARG
    assert m(P, P, 2, 0, 4, P, P, 0, NULL) == fa.FA_ERR_INVALID_ARG
    assert m(P, P, 2, 3, 513, P, P, 0, NULL) == fa.FA_ERR_INVALID_ARG
    assert m(P, P, 2, 3, 4, P, P, 5, NULL) == fa.FA_ERR_INVALID_ARG


def test_workspace_and_split_heuristic(lib):
    ws = lib.fa_decode_workspace_size
    assert ws(0, 1, 1, 1) == 0 and ws(1, 1, 1, 0) == 0
    # fp32 partial outputs then fp32 partial lse, each rounded up to 256 bytes
    assert ws(16, 32, 128, 10) == (16 * 32 * 10 * 128 * 4 + 255) // 256 * 256 + (16 * 32 * 10 * 4 + 255) // 256 * 256
    ds = lib.fa_decode_default_splits
    assert ds(0, 1, 1, 1) == 0
    for (B, H, Nk, sms) in ((16, 32, 32768, 148), (1, 1, 100000, 152), (64, 64, 256, 152), (1, 1, 1, 152)):
        n = ds(B, H, Nk, sms)
        assert 1 <= n <= max(1, -(-Nk // 256))
    # more SMs never means fewer splits
    assert ds(4, 8, 32768, 152) >= ds(4, 8, 32768, 76)


def test_gqa_split_heuristic(lib):
    g, ds = lib.fa_decode_gqa_default_splits, lib.fa_decode_default_splits
    assert g(0, 32, 8, 1024, 128, 152) == 0 and g(1, 6, 4, 1024, 128, 152) == 0
    assert g(1, 8, 8, 1024, 128, 0) == 0 and g(1, 8, 8, 1024, 0, 152) == 0
    # groups of 1 and 2 heads, and of 4 at d != 128 (CUDA cores), follow the B * Hq query heads
    for (B, Hq, Hkv, d) in ((16, 32, 32, 128), (16, 32, 16, 128), (16, 32, 8, 64), (3, 8, 2, 32)):
        assert g(B, Hq, Hkv, 32768, d, 152) == ds(B, Hq, 32768, 152)
    # other groups (tensor core): floor(1.7 * slots / (B * Hkv)) with two CTA slots per SM for 3-8
    # heads at d = 128 (the transposed kernel), one otherwise; at least 2 while the groups leave
    # SMs idle; no split longer than 64 key tiles (up to 4 heads) or 32 (more); clamped to
    # [1, ceil(Nk_max / 128)]
    assert g(16, 32, 4, 32768, 128, 152) == 8 and g(16, 32, 2, 32768, 128, 152) == 8
    assert g(16, 32, 1, 32768, 128, 152) == 16
    assert g(16, 32, 8, 32768, 128, 152) == 4  # 4 heads at d = 128: 608 / 128 slots per group
    assert g(16, 24, 8, 32768, 128, 152) == 4 and g(4, 32, 8, 32768, 128, 152) == 16
    assert g(64, 32, 8, 32768, 128, 152) == 4  # 256 tiles / 64 per split
    assert g(4, 32, 4, 32768, 128, 152) == 32 and g(4, 40, 8, 32768, 128, 152) == 16  # 8 and 5 heads
    assert g(4, 32, 4, 32768, 64, 152) == 16  # 8 heads at d = 64: row tiles, one slot per SM
    assert g(64, 32, 4, 4096, 128, 152) == 2 and g(1000, 32, 4, 4096, 128, 152) == 1
    assert g(64, 32, 4, 32768, 128, 152) == 8 and g(1000, 32, 4, 32768, 128, 152) == 8  # 32 tiles per split
    assert g(4, 32, 1, 256, 128, 152) == 2 and g(1, 128, 1, 100, 128, 152) == 1
    assert g(1, 24, 8, 1 << 20, 64, 152) == 128  # 3 heads at d = 64: 32 by the slots, 8192 tiles / 64


def test_status_strings(lib):
    for s in range(6):
        assert isinstance(fa.status_string(s), str) and fa.status_string(s)
    assert "timed out" in fa.status_string(fa.FA_ERR_TIMEOUT)
