"""CPU FP64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA path: the C
library ``fa_oracle.c`` (built here with gcc into ``liboracle.so``) is the
plain definition of standard attention and of its backward in float64, and
``numpy_oracle`` is a second, independent numpy statement of the same definitions.

Inputs are torch tensors or numpy arrays.  bf16 tensors are handed to the C
library as raw bit patterns and widened exactly there; everything else is
converted to float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import numpy_oracle  # noqa: F401  (re-exported for the tests)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def compile_library(src, out):
    """Compile an oracle C source into a shared library with gcc (portable flags only)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force=False):
    """Compile ``fa_oracle.c`` into ``liboracle.so`` (skipped when up to date)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_library(_SRC, _LIB)


def open_library(path):
    """ctypes handle on an oracle library at ``path`` with its signatures declared."""
    lib = ctypes.CDLL(path)
    vp, L, i, d, dp = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.oracle_attention.argtypes = [vp, vp, vp, i, L, L, L, L, L, i, d, L, L, dp, dp, i]
    lib.oracle_attention.restype = i
    lib.oracle_decode.argtypes = [vp, vp, vp, i, vp, L, L, L, L, L, d, dp, dp, i]
    lib.oracle_decode.restype = i
    lib.oracle_merge_lse.argtypes = [dp, dp, L, L, L, dp, dp]
    lib.oracle_merge_lse.restype = i
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i, L, L, L, L, L, i, d, dp, dp, dp, i]
    lib.oracle_attention_bwd.restype = i
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = open_library(_LIB)
    return _lib


def cores():
    """Threads the C oracle uses by default (all host cores)."""
    return os.cpu_count() or 1


def _as_input(t):
    """(buffer keeping memory alive, pointer, is_bf16) for a torch tensor or array."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").contiguous()
        if t.dtype == torch.bfloat16:
            arr = t.view(torch.int16).numpy().view(np.uint16)
            arr = np.ascontiguousarray(arr)
            return arr, arr.ctypes.data, 1
        arr = np.ascontiguousarray(t.to(torch.float64).numpy())
        return arr, arr.ctypes.data, 0
    arr = np.ascontiguousarray(np.asarray(t, dtype=np.float64))
    return arr, arr.ctypes.data, 0


def attention(q, k, v, causal=False, scale=None, rows=None, threads=None, lib=None):
    """Standard attention for inputs shaped [..., N, d] / [..., Nk, d] / [..., Nk, dv].

    Leading dimensions are flattened into independent heads.  ``rows`` =
    (row0, row1) restricts the computed query rows.  Returns float64 numpy
    arrays O [..., rows, dv] and LSE [..., rows].
    """
    qs, ks, vs = tuple(q.shape), tuple(k.shape), tuple(v.shape)
    lead = qs[:-2]
    N, d = qs[-2], qs[-1]
    Nk, dv = vs[-2], vs[-1]
    assert ks[-2] == Nk and ks[-1] == d and ks[:-2] == lead and vs[:-2] == lead
    BH = int(np.prod(lead)) if lead else 1
    row0, row1 = (0, N) if rows is None else rows
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    bq, pq, fq = _as_input(q)
    bk, pk, fk = _as_input(k)
    bv, pv, fv = _as_input(v)
    if not (fq == fk == fv):  # mixed input types: widen everything to float64
        bq, pq, _ = _as_input(np.asarray(_widen(q)))
        bk, pk, _ = _as_input(np.asarray(_widen(k)))
        bv, pv, _ = _as_input(np.asarray(_widen(v)))
        fq = 0
    nr = row1 - row0
    O = np.zeros((BH, nr, dv), dtype=np.float64)
    LSE = np.zeros((BH, nr), dtype=np.float64)
    rc = (lib or _load()).oracle_attention(pq, pk, pv, fq, BH, N, Nk, d, dv, int(bool(causal)), scale, row0,
                                  row1, O.ctypes.data, LSE.ctypes.data, threads or cores())
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed with code {rc}")
    return O.reshape(lead + (nr, dv)), LSE.reshape(lead + (nr,))


def attention_bwd(q, k, v, do, causal=False, scale=None, threads=None, lib=None):
    """Gradients (dQ, dK, dV) of standard attention for the upstream gradient ``do``.

    Shapes [..., N, d] / [..., Nk, d] / [..., Nk, dv] / [..., N, dv]; leading
    dimensions are independent heads.  Returns float64 numpy arrays.
    """
    qs, vs = tuple(q.shape), tuple(v.shape)
    lead = qs[:-2]
    N, d = qs[-2], qs[-1]
    Nk, dv = vs[-2], vs[-1]
    assert tuple(k.shape) == lead + (Nk, d) and tuple(do.shape) == lead + (N, dv)
    BH = int(np.prod(lead)) if lead else 1
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    ins = [_as_input(t) for t in (q, k, v, do)]
    if len({f for _, _, f in ins}) != 1:  # mixed input types: widen everything to float64
        ins = [_as_input(np.asarray(_widen(t))) for t in (q, k, v, do)]
    (bq, pq, fq), (bk, pk, _), (bv, pv, _), (bg, pg, _) = ins
    dQ = np.zeros((BH, N, d))
    dK = np.zeros((BH, Nk, d))
    dV = np.zeros((BH, Nk, dv))
    rc = (lib or _load()).oracle_attention_bwd(pq, pk, pv, pg, fq, BH, N, Nk, d, dv, int(bool(causal)), scale,
                                               dQ.ctypes.data, dK.ctypes.data, dV.ctypes.data,
                                               threads or cores())
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd failed with code {rc}")
    return dQ.reshape(lead + (N, d)), dK.reshape(lead + (Nk, d)), dV.reshape(lead + (Nk, dv))


def decode(q, k_cache, v_cache, seqlens, scale=None, threads=None, lib=None):
    """Single-query attention of q [B,H,1,d] over the first seqlens[b] cache rows.

    Returns O [B,H,1,dv] and LSE [B,H,1] as float64 numpy arrays.
    """
    B, H, one, d = tuple(q.shape)
    assert one == 1
    Nk_max, dv = tuple(v_cache.shape)[-2], tuple(v_cache.shape)[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    bq, pq, fq = _as_input(q)
    bk, pk, fk = _as_input(k_cache)
    bv, pv, fv = _as_input(v_cache)
    assert fq == fk == fv
    lens = np.ascontiguousarray(np.asarray([int(x) for x in seqlens], dtype=np.int32))
    O = np.zeros((B * H, dv), dtype=np.float64)
    LSE = np.zeros((B * H,), dtype=np.float64)
    rc = (lib or _load()).oracle_decode(pq, pk, pv, fq, lens.ctypes.data, B, H, Nk_max, d, dv, scale,
                               O.ctypes.data, LSE.ctypes.data, threads or cores())
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed with code {rc}")
    return O.reshape(B, H, 1, dv), LSE.reshape(B, H, 1)


def merge_lse(o_parts, lse_parts, lib=None):
    """Log-sum-exp combine of P partial states: o_parts [P, rows, dv], lse_parts [P, rows]."""
    op = np.ascontiguousarray(_widen(o_parts))
    lp = np.ascontiguousarray(_widen(lse_parts))
    P, rows, dv = op.shape
    o = np.zeros((rows, dv), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    rc = (lib or _load()).oracle_merge_lse(op.ctypes.data, lp.ctypes.data, P, rows, dv, o.ctypes.data,
                                  lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_merge_lse failed with code {rc}")
    return o, lse


def _widen(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)
