"""CPU oracle for the chunked gated delta rule with state/W fake QDQ.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import or call anything in this
package.  The CUDA library never links it, and it never imports the CUDA
library; the two share no code.

Contents
  qdq.c          bit-exact fp32 dynamic QDQ (E4M3 / INT8), plain C
  recurrent.c    O1: fp64 token-by-token recurrence with state QDQ, plain C + OpenMP
  chunked.py     O2: fp64 chunked (WY) form with state and W QDQ, torch CPU + autograd
  recurrent_torch.py  small-case fp64 recurrence in torch (autograd), for gradient pins
  decode.py      decode QAT step (state QDQ before every token), numpy fp64
  kda.py         KDA recurrence (decay per key channel) with state QDQ, numpy fp64
  two_precision.py  two-precision GDN profile: fp32 anchor + E4M3 read copy, numpy fp64

The C part is compiled with gcc into ``oracle/liboracle.so`` by ``build()``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "qdq.c"), os.path.join(_HERE, "recurrent.c")]
_lock = threading.Lock()
_lib = None

QDQ_NONE, QDQ_E4M3, QDQ_INT8 = 0, 1, 2
MODES = {"none": QDQ_NONE, "e4m3": QDQ_E4M3, "int8": QDQ_INT8}


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP, no contraction, no fast-math)."""
    newest = max(os.path.getmtime(s) for s in _SOURCES)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp] + _SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            L.oracle_qdq_groups.argtypes = [P, P, P, P, i64, i64, i64, i64, ctypes.c_int]
            L.oracle_qdq_groups.restype = ctypes.c_int
            L.oracle_e4m3_encode_array.argtypes = [P, P, i64]
            L.oracle_e4m3_decode_array.argtypes = [P, P, i64]
            L.oracle_int8_encode_array.argtypes = [P, P, i64]
            ci = ctypes.c_int
            L.oracle_gdn_recurrent.argtypes = [P, P, P, P, P, P, P, ci, ci, ci, ci, ci, ci, ci,
                                               ctypes.c_double, ci, ci, ci, P, P, P, P, P, ci]
            L.oracle_gdn_recurrent.restype = ctypes.c_int
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _mode(m) -> int:
    return MODES[m] if isinstance(m, str) else int(m)


# ----------------------------------------------------------------------------
# QDQ
# ----------------------------------------------------------------------------
def qdq_groups(x, group_cols: int, mode, with_codes: bool = False):
    """Grouped fake QDQ of a [batch, rows, cols] fp32 array (see qdq.c).

    One scale per (batch, block of ``group_cols`` columns) spanning all rows.
    Returns (y, scales[batch, cols/group_cols]) or (y, scales, codes u8).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    shp = x.shape
    if x.ndim == 1:
        x3 = x.reshape(1, 1, -1)
    elif x.ndim == 2:
        x3 = x.reshape(1, *shp)
    else:
        x3 = x.reshape(-1, shp[-2], shp[-1])
    b, r, c = x3.shape
    y = np.empty_like(x3)
    sc = np.zeros((b, c // group_cols), dtype=np.float32)
    cd = np.zeros(x3.shape, dtype=np.uint8) if with_codes else None
    rc = lib().oracle_qdq_groups(_ptr(x3), _ptr(y), _ptr(sc), _ptr(cd), b, r, c, group_cols,
                                 _mode(mode))
    if rc != 0:
        raise ValueError("oracle_qdq_groups: bad arguments")
    y = y.reshape(shp)
    if with_codes:
        return y, sc, cd.reshape(shp)
    return y, sc


def e4m3_encode(u):
    u = np.ascontiguousarray(u, dtype=np.float32)
    c = np.empty(u.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(u), _ptr(c), u.size)
    return c


def e4m3_decode(c):
    c = np.ascontiguousarray(c, dtype=np.uint8)
    y = np.empty(c.shape, dtype=np.float32)
    lib().oracle_e4m3_decode_array(_ptr(c), _ptr(y), c.size)
    return y


def int8_encode(u):
    u = np.ascontiguousarray(u, dtype=np.float32)
    c = np.empty(u.shape, dtype=np.int8)
    lib().oracle_int8_encode_array(_ptr(u), _ptr(c), u.size)
    return c


# ----------------------------------------------------------------------------
# O1: token recurrence
# ----------------------------------------------------------------------------
def dense_chunk_base(lengths, chunk: int = 64):
    """Chunk index of each sequence's first chunk when chunks are numbered
    densely, sequence after sequence."""
    base = np.zeros(len(lengths), dtype=np.int64)
    acc = 0
    for i, L in enumerate(lengths):
        base[i] = acc
        acc += -(-int(L) // chunk)
    return base, acc


def recurrent(q, k, v, beta, g, h0=None, cu_seqlens=None, scale=1.0, state_mode="none",
              block_v=64, chunk=64, record_states=False, n_threads=0):
    """O1.  q, k [B,T,Hk,Dk]; v [B,T,Hv,Dv]; beta, g [B,T,Hv]; h0 [N,Hv,Dk,Dv].

    Arrays may be numpy or torch (CPU); they are widened to fp32 values.
    Returns (o fp64 [B,T,Hv,Dv], ht fp64 [N,Hv,Dk,Dv]) and, with
    ``record_states``, (codes u8 [n_chunks,Hv,Dk,Dv], scales [n_chunks,Hv,Dv/block_v])
    of the quantized state entering every chunk, chunks numbered densely.
    """
    f = lambda a: None if a is None else np.ascontiguousarray(_np(a), dtype=np.float32)
    q, k, v, beta, g, h0 = f(q), f(k), f(v), f(beta), f(g), f(h0)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(_np(cu_seqlens), dtype=np.int32)
        N = cu.size - 1
        lengths = np.diff(cu.astype(np.int64))
    else:
        cu = None
        N = B
        lengths = np.full(B, T, dtype=np.int64)
    o = np.zeros((B, T, Hv, Dv), dtype=np.float64)
    ht = np.zeros((N, Hv, Dk, Dv), dtype=np.float64)
    codes = scales = base = None
    if record_states and _mode(state_mode) != QDQ_NONE:
        base, nc = dense_chunk_base(lengths, chunk)
        codes = np.zeros((nc, Hv, Dk, Dv), dtype=np.uint8)
        scales = np.zeros((nc, Hv, Dv // block_v), dtype=np.float32)
    rc = lib().oracle_gdn_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                    _ptr(cu), B, T, Hk, Hv, Dk, Dv, N, float(scale),
                                    _mode(state_mode), block_v, chunk, _ptr(o), _ptr(ht),
                                    _ptr(codes), _ptr(scales), _ptr(base), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_gdn_recurrent: bad arguments")
    if record_states:
        return o, ht, codes, scales
    return o, ht


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _np(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.float()
        return a.numpy()
    return np.asarray(a)
