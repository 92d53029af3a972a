"""fp64 CPU oracle for absorbed-MLA verify attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The CUDA library never loads
or calls anything here, and this package imports nothing from it.

The C source (``mla_oracle.c``) states the computation row by row from the
pages' definition; this wrapper only marshals numpy arrays.  The shared
library is compiled with gcc on first use (or by ``build()``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_HDR = os.path.join(_HERE, "mla_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C, -O2, pthreads)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or
             os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MLA_ORACLE_LIB lets the oracle's own mutation test load a
            # deliberately broken build; nothing else sets it.
            lib = ctypes.CDLL(os.environ.get("MLA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            D = ctypes.c_double
            lib.mla_oracle_verify_attn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, P, P, I]
            lib.mla_oracle_verify_attn_rows.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, L, L,
                                                        P, P, I]
            lib.mla_oracle_partial.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, P, P, P, P, P, I]
            lib.mla_oracle_combine.argtypes = [P, P, P, I, L, I, P, P]
            lib.mla_oracle_combine.restype = None
            lib.mla_oracle_row_weights.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, I, I, I, P]
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _inputs(q_nope, q_rope, kv, seq_lens, mask):
    qn, pqn = _c(q_nope, np.uint16)
    qr, pqr = _c(q_rope, np.uint16)
    k, pk = _c(kv, np.uint16)
    s, ps = _c(seq_lens, np.int32)
    m, pm = _c(mask, np.uint32)
    B, q, H, Dl = qn.shape
    Dr = qr.shape[3]
    assert qr.shape[:3] == (B, q, H) and k.shape[0] == B and k.shape[2] == Dl + Dr
    assert m.shape == (B, q, (q + 31) // 32) and s.shape == (B,)
    return (qn, qr, k, s, m), (pqn, pqr, pk, ps, pm), (B, q, H, k.shape[1], Dl, Dr)


def _threads(nthreads):
    return nthreads if nthreads else (os.cpu_count() or 1)


def verify_attn(q_nope, q_rope, kv, seq_lens, mask, scale, nthreads: int = 0, rows=None):
    """Reference out [B,q,H,Dl] and lse [B,q,H] in float64.

    ``rows`` = (begin, count) restricts the work to those flattened (b, i, h)
    rows; the others are left as NaN.
    """
    keep, ptrs, (B, q, H, Smax, Dl, Dr) = _inputs(q_nope, q_rope, kv, seq_lens, mask)
    out = np.full((B, q, H, Dl), np.nan)
    lse = np.full((B, q, H), np.nan)
    lib = _load()
    if rows is None:
        rc = lib.mla_oracle_verify_attn(*ptrs, B, q, H, Smax, Dl, Dr, float(scale),
                                        out.ctypes.data, lse.ctypes.data, _threads(nthreads))
    else:
        rc = lib.mla_oracle_verify_attn_rows(*ptrs, B, q, H, Smax, Dl, Dr, float(scale),
                                             int(rows[0]), int(rows[1]), out.ctypes.data,
                                             lse.ctypes.data, _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (code %d)" % rc)
    return out, lse


def partial(q_nope, q_rope, kv, seq_lens, mask, scale, k0, k1, nthreads: int = 0):
    """Unnormalised (acc, m, l) over keys [k0[b], k1[b]) of each stream."""
    keep, ptrs, (B, q, H, Smax, Dl, Dr) = _inputs(q_nope, q_rope, kv, seq_lens, mask)
    a0, p0 = _c(k0, np.int32)
    a1, p1 = _c(k1, np.int32)
    acc = np.zeros((B * q * H, Dl))
    m = np.zeros(B * q * H)
    l = np.zeros(B * q * H)
    rc = _load().mla_oracle_partial(*ptrs, B, q, H, Smax, Dl, Dr, float(scale), p0, p1,
                                    acc.ctypes.data, m.ctypes.data, l.ctypes.data,
                                    _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (code %d)" % rc)
    return acc, m, l


def combine(acc, m, l):
    """Merge partial states acc [ns, rows, Dl], m/l [ns, rows] -> (out, lse)."""
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    ns, nrows, Dl = acc.shape
    out = np.zeros((nrows, Dl))
    lse = np.zeros(nrows)
    _load().mla_oracle_combine(acc.ctypes.data, m.ctypes.data, l.ctypes.data, ns, nrows, Dl,
                               out.ctypes.data, lse.ctypes.data)
    return out, lse


def row_weights(q_nope, q_rope, kv, seq_lens, mask, scale, b, i, h):
    """Normalised weights of row (b, i, h) over all Smax cache rows."""
    keep, ptrs, (B, q, H, Smax, Dl, Dr) = _inputs(q_nope, q_rope, kv, seq_lens, mask)
    w = np.zeros(Smax)
    rc = _load().mla_oracle_row_weights(*ptrs, B, q, H, Smax, Dl, Dr, float(scale), b, i, h,
                                        w.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the inputs (code %d)" % rc)
    return w


def case_reference(case, nthreads: int = 0, rows=None):
    """Oracle on an ``inputs.Case``."""
    return verify_attn(case.q_nope, case.q_rope, case.kv, case.seq_lens, case.mask, case.scale,
                       nthreads, rows)
