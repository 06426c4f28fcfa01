"""Exact tiled attention on GB300 (sm_103a): Python binding of ``libfa.so``.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/fa.h``; torch supplies device
memory and the current stream.  There is no CPU fallback: if ``libfa.so`` is
missing or cannot be loaded, every entry point raises.

Entry points (same names as the C ABI, without the ``fa_`` prefix):
  fwd              exact attention forward (tiled, online softmax)
  fwd_splitkv      the forward with the keys split and merged (few query tiles)
  bwd              exact attention backward (dQ, dK, dV; P recomputed from LSE)
  decode_splitkv   split-KV single-query decode with log-sum-exp combine
  decode_splitkv_gqa  the same with grouped key/value heads (query heads of a group packed)
  decode_splitkv_fused  the same with the combine done by each row's last split (one launch)
  merge_states     log-sum-exp combine of partial states
  decode_default_splits, decode_gqa_default_splits, decode_workspace_size, get_device_error,
  set_wait_timeout_ns, status_string
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_WORKSPACE, FA_ERR_TIMEOUT = range(6)
FA_BF16, FA_F32 = 0, 1

_lib = None


class FaError(RuntimeError):
    """A libfa entry point returned a status other than FA_OK."""

    def __init__(self, status, where):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {int(status)})")


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libfa.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz, ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_decode_default_splits.argtypes = [i, i, i, i]
    lib.fa_decode_default_splits.restype = i
    lib.fa_decode_gqa_default_splits.argtypes = [i, i, i, i, i, i]
    lib.fa_decode_gqa_default_splits.restype = i
    lib.fa_decode_workspace_size.argtypes = [i, i, i, i]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, i, vp]
    lib.fa_decode_splitkv.restype = i
    lib.fa_fwd_splitkv_default_splits.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_default_splits.restype = i
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_workspace_size.restype = sz
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_decode_fused_workspace_size.argtypes = [i, i, i, i]
    lib.fa_decode_fused_workspace_size.restype = sz
    lib.fa_decode_splitkv_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, i, vp]
    lib.fa_decode_splitkv_fused.restype = i
    lib.fa_decode_splitkv_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_decode_splitkv_gqa.restype = i
    lib.fa_merge_states.argtypes = [vp, vp, i, i, i, vp, vp, i, vp]
    lib.fa_merge_states.restype = i
    lib.fa_get_device_error.argtypes = [vp]
    lib.fa_get_device_error.restype = i
    lib.fa_set_wait_timeout_ns.argtypes = [ull]
    lib.fa_set_wait_timeout_ns.restype = None
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def library():
    """The loaded ctypes handle (loads it on first use)."""
    return _load()


def status_string(status):
    return _load().fa_status_string(int(status)).decode()


def _check(status, where):
    if status != FA_OK:
        raise FaError(status, where)


# The current stream's raw handle; torch's own lookup (a plain int) when it has one, which avoids
# building a Stream object on every call.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device):
    idx = device.index if isinstance(device, torch.device) else int(device)
    if _raw_stream is not None:
        return _raw_stream(idx)
    return torch.cuda.current_stream(idx).cuda_stream


class _on_device:
    """Makes `index` the current CUDA device for the call (switching only when it is not)."""

    __slots__ = ("index", "ctx")

    def __init__(self, index):
        self.index = index
        self.ctx = None

    def __enter__(self):
        if torch.cuda.current_device() != self.index:
            self.ctx = torch.cuda.device(self.index)
            self.ctx.__enter__()

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)


def _odt(dtype):
    if dtype == torch.bfloat16:
        return FA_BF16
    if dtype == torch.float32:
        return FA_F32
    raise ValueError(f"output dtype must be bfloat16 or float32, not {dtype}")


def _need(t, name, dtype, device=None):
    """Checks a tensor argument; returns its CUDA device index.  `device` (a torch.device or an
    index) is the device the other arguments are on."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    di = t.get_device()
    if di < 0:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None:
        want = device.index if isinstance(device, torch.device) else device
        if di != want:
            raise ValueError(f"{name} is on cuda:{di}, expected cuda:{want}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return di


def _ptr(t):
    return t.data_ptr() if t is not None else None


def fwd(q, k, v, causal=False, scale=None, out_dtype=torch.bfloat16, out=None, lse=None, return_lse=True):
    """Exact attention forward.  q [B,H,N,d], k [B,H,Nk,d], v [B,H,Nk,dv], bf16, contiguous, on one GPU.

    Returns (O [B,H,N,dv] of ``out_dtype``, LSE fp32 [B,H,N] or None).
    """
    lib = _load()
    di = _need(q, "q", torch.bfloat16)  # device index; the other tensors must be on it
    _need(k, "k", torch.bfloat16, di)
    _need(v, "v", torch.bfloat16, di)
    if len(q.shape) != 4 or len(k.shape) != 4 or len(v.shape) != 4:
        raise ValueError("q, k, v must be [B, H, rows, head_dim]")
    B, H, N, d = q.shape
    Nk, dv = v.shape[2], v.shape[3]
    if k.shape != (B, H, Nk, d) or v.shape[:2] != (B, H):
        raise ValueError("shape mismatch between q, k, v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=out_dtype, device=q.device)
    _need(out, "out", out.dtype, di)
    if out.shape != (B, H, N, dv):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, di)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            B, H, N, Nk, d, dv, 1 if causal else 0, scale, _odt(out.dtype))
    if torch.cuda.current_device() == di:
        st = lib.fa_fwd(*args, _stream(di))
    else:
        with torch.cuda.device(di):
            st = lib.fa_fwd(*args, _stream(di))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return out, lse


def bwd_workspace_size(B, H, N, d):
    return int(_load().fa_bwd_workspace_size(B, H, N, d))


def bwd(q, k, v, o, lse, do, causal=False, scale=None, out_dtype=torch.bfloat16, grads=None, workspace=None):
    """Exact attention backward for the upstream gradient ``do`` of the forward output ``o``.

    q [B,H,N,d], k [B,H,Nk,d], v [B,H,Nk,dv], do [B,H,N,dv] bf16; o [B,H,N,dv] bf16 or fp32 and
    lse fp32 [B,H,N] as returned by ``fwd`` with the same ``causal`` and ``scale``.  ``grads`` is an
    optional (dq, dk, dv) triple to write into; ``workspace`` a uint8 CUDA tensor of at least
    ``bwd_workspace_size`` bytes (allocated here when omitted).  Returns (dq, dk, dv) of ``out_dtype``.
    """
    lib = _load()
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    _need(do, "do", torch.bfloat16, dev)
    _need(o, "o", o.dtype, dev)
    _need(lse, "lse", torch.float32, dev)
    B, H, N, d = q.shape
    Nk, dv = v.shape[2], v.shape[3]
    if (tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape[:2]) != (B, H) or tuple(o.shape) != (B, H, N, dv)
            or tuple(do.shape) != (B, H, N, dv) or tuple(lse.shape) != (B, H, N)):
        raise ValueError("shape mismatch between q, k, v, o, lse, do")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if grads is None:
        grads = (torch.empty((B, H, N, d), dtype=out_dtype, device=dev),
                 torch.empty((B, H, Nk, d), dtype=out_dtype, device=dev),
                 torch.empty((B, H, Nk, dv), dtype=out_dtype, device=dev))
    dq, dk, dv_ = grads
    for t, name in ((dq, "dq"), (dk, "dk"), (dv_, "dv")):
        _need(t, name, dq.dtype, dev)
    if tuple(dq.shape) != (B, H, N, d) or tuple(dk.shape) != (B, H, Nk, d) or tuple(dv_.shape) != (B, H, Nk, dv):
        raise ValueError("gradient buffers have the wrong shape")
    if workspace is None:
        workspace = torch.empty(bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    with _on_device(dev.index):
        st = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv_),
                        _ptr(workspace), workspace.numel(), B, H, N, Nk, d, dv, int(bool(causal)), scale,
                        _odt(o.dtype), _odt(dq.dtype), _stream(dev))
    _check(st, "fa_bwd")
    return dq, dk, dv_


def fwd_splitkv_default_splits(B, H, N, Nk, num_sms):
    return int(_load().fa_fwd_splitkv_default_splits(B, H, N, Nk, num_sms))


def fwd_splitkv_workspace_size(B, H, N, dv, n_splits):
    return int(_load().fa_fwd_splitkv_workspace_size(B, H, N, dv, n_splits))


def fwd_splitkv(q, k, v, causal=False, scale=None, n_splits=0, out_dtype=torch.bfloat16, out=None, lse=None,
                workspace=None, return_lse=True):
    """Forward with the keys split into chunks and merged; same inputs and result as ``fwd``."""
    lib = _load()
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    B, H, N, d = q.shape
    Nk, dv = v.shape[2], v.shape[3]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape[:2]) != (B, H):
        raise ValueError("shape mismatch between q, k, v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n = int(n_splits) if n_splits else fwd_splitkv_default_splits(B, H, N, Nk, num_sms(dev))
    if workspace is None:
        workspace = torch.empty(max(fwd_splitkv_workspace_size(B, H, N, dv, max(1, min(n, Nk))), 256),
                                dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    with _on_device(dev.index):
        st = lib.fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                B, H, N, Nk, d, dv, int(bool(causal)), scale, n, _odt(out.dtype), _stream(dev))
    _check(st, "fa_fwd_splitkv")
    return out, lse


def decode_default_splits(B, H, Nk_max, num_sms):
    return int(_load().fa_decode_default_splits(B, H, Nk_max, num_sms))


def decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, num_sms):
    return int(_load().fa_decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, num_sms))


def decode_workspace_size(B, H, dv, n_splits):
    return int(_load().fa_decode_workspace_size(B, H, dv, n_splits))


def num_sms(device=None):
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def decode_splitkv(q, k_cache, v_cache, seqlens, scale=None, n_splits=0, out_dtype=torch.bfloat16, out=None,
                   lse=None, workspace=None, return_lse=True):
    """Split-KV decode.  q [B,H,1,d], caches [B,H,Nk_max,d|dv] bf16, seqlens int32 [B] on the same GPU.

    ``workspace`` is a uint8 CUDA tensor of at least ``decode_workspace_size`` bytes (allocated here
    when omitted).  Returns (O [B,H,1,dv], LSE fp32 [B,H,1] or None).
    """
    lib = _load()
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query per (b, h)")
    Nk_max, dv = v_cache.shape[2], v_cache.shape[3]
    if tuple(k_cache.shape) != (B, H, Nk_max, d) or tuple(v_cache.shape[:2]) != (B, H) or seqlens.numel() != B:
        raise ValueError("shape mismatch between q, caches and seqlens")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n = int(n_splits) if n_splits else decode_default_splits(B, H, Nk_max, num_sms(dev))
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_size(B, H, dv, max(1, min(n, Nk_max))), 256),
                                dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if out is None:
        out = torch.empty((B, H, 1, dv), dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    with _on_device(dev.index):
        st = lib.fa_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out), _ptr(lse),
                                   _ptr(workspace), workspace.numel(), B, H, Nk_max, d, dv, scale, n,
                                   _odt(out.dtype), _stream(dev))
    _check(st, "fa_decode_splitkv")
    return out, lse


def decode_splitkv_gqa(q, k_cache, v_cache, seqlens, scale=None, n_splits=0, out_dtype=torch.bfloat16, out=None,
                       lse=None, workspace=None, return_lse=True):
    """Split-KV decode with grouped key/value heads: q [B,Hq,1,d], caches [B,Hkv,Nk_max,d|dv] bf16 with Hkv
    dividing Hq (query head h uses key/value head h // (Hq // Hkv)), seqlens int32 [B] on the same GPU.

    Returns (O [B,Hq,1,dv], LSE fp32 [B,Hq,1] or None).
    """
    lib = _load()
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    B, Hq, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query per (b, h)")
    Hkv, Nk_max, dv = k_cache.shape[1], v_cache.shape[2], v_cache.shape[3]
    if (tuple(k_cache.shape) != (B, Hkv, Nk_max, d) or tuple(v_cache.shape[:2]) != (B, Hkv)
            or seqlens.numel() != B):
        raise ValueError("shape mismatch between q, caches and seqlens")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    # (0 for groups the library rejects; the call below then reports why)
    n = int(n_splits) if n_splits else decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, num_sms(dev))
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_size(B, Hq, dv, max(1, min(n, Nk_max))), 256),
                                dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if out is None:
        out = torch.empty((B, Hq, 1, dv), dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    with _on_device(dev.index):
        st = lib.fa_decode_splitkv_gqa(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out), _ptr(lse),
                                       _ptr(workspace), workspace.numel(), B, Hq, Hkv, Nk_max, d, dv, scale,
                                       int(n_splits), _odt(out.dtype), _stream(dev))
    _check(st, "fa_decode_splitkv_gqa")
    return out, lse


def decode_fused_workspace_size(B, H, dv, n_splits):
    return int(_load().fa_decode_fused_workspace_size(B, H, dv, n_splits))


def decode_fused_workspace(B, H, Nk_max, dv, n_splits=0, device=None):
    """A workspace for ``decode_splitkv_fused`` with its counters zeroed (reuse it across calls)."""
    n = int(n_splits) if n_splits else decode_default_splits(B, H, Nk_max, num_sms(device))
    return torch.zeros(decode_fused_workspace_size(B, H, dv, max(1, min(n, Nk_max))), dtype=torch.uint8,
                       device=device or "cuda")


def decode_splitkv_fused(q, k_cache, v_cache, seqlens, workspace, scale=None, n_splits=0, out_dtype=torch.bfloat16,
                         out=None, lse=None, return_lse=True):
    """Split-KV decode with the combine fused into the split kernel.  ``workspace`` comes from
    ``decode_fused_workspace`` (its counters must be zero; each completed call leaves them zero)."""
    lib = _load()
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query per (b, h)")
    Nk_max, dv = v_cache.shape[2], v_cache.shape[3]
    if tuple(k_cache.shape) != (B, H, Nk_max, d) or tuple(v_cache.shape[:2]) != (B, H) or seqlens.numel() != B:
        raise ValueError("shape mismatch between q, caches and seqlens")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, 1, dv), dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    with _on_device(dev.index):
        st = lib.fa_decode_splitkv_fused(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out), _ptr(lse),
                                         _ptr(workspace), workspace.numel(), B, H, Nk_max, d, dv, scale,
                                         int(n_splits), _odt(out.dtype), _stream(dev))
    _check(st, "fa_decode_splitkv_fused")
    return out, lse


def merge_states(o_parts, lse_parts, out_dtype=torch.float32, out=None, lse=None):
    """Log-sum-exp combine: o_parts fp32 [P, rows, dv], lse_parts fp32 [P, rows] -> (o [rows, dv], lse [rows])."""
    lib = _load()
    _need(o_parts, "o_parts", torch.float32)
    dev = o_parts.device
    _need(lse_parts, "lse_parts", torch.float32, dev)
    P, rows, dv = o_parts.shape
    if tuple(lse_parts.shape) != (P, rows):
        raise ValueError("lse_parts must be [P, rows]")
    if out is None:
        out = torch.empty((rows, dv), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    with _on_device(dev.index):
        st = lib.fa_merge_states(_ptr(o_parts), _ptr(lse_parts), P, rows, dv, _ptr(out), _ptr(lse),
                                 _odt(out.dtype), _stream(dev))
    _check(st, "fa_merge_states")
    return out, lse


def get_device_error(device=None):
    """Synchronise the current stream and return (and clear) the device status word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on_device(dev.index):
        return int(_load().fa_get_device_error(_stream(dev)))


def set_wait_timeout_ns(ns):
    _load().fa_set_wait_timeout_ns(int(ns))
