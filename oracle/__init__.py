"""fp64 CPU oracle for the Mixture-of-Depths Attention (MoDA) forward.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``sequence_depth_attention_gb300``) never imports it and shares no code with
it; the two meet only through the seeded input generator, which holds none of
the method's arithmetic.

The arithmetic lives in ``moda_oracle.c`` (plain C, double precision, one
query row at a time, the joint score row [sequence scores <= t | L depth
scores] materialised and softmaxed once). This module compiles it with gcc
and marshals numpy arrays to it. Definitions and citations are in the C
file's header; in short (Mixture-of-Depths Attention, Sec. 2.1 Eq. (2) and
Sec. 2.2 "MoDA"):

    o[t,h]   = softmax([scale*q.k_j (j<=t) | scale*q.kd_l (l<L)]) . [v_j | vd_l]
    lse[t,h] = ln sum exp(joint row)

Inputs are bf16 bit patterns as ``numpy.uint16`` arrays in the layouts
q[T,Hq,d], k/v[T,Hk,d] and the UNPACKED depth stream kd/vd[L,T,Hk,d].

``Oracle.kv_proj`` is the depth K/V of an FFN layer, a linear map of the
FFN's input (reading notes Sec. 二.3; summary Sec. 2.2, the "write" step):
out[t, n] = sum_c x[t, c] * w[n, c] in fp64.

``Oracle.depth_mass`` is the utility of the bounded depth cache (summary
Sec. 6.2): the probability mass the joint softmax gives each depth slot,
summed over the rows of each KV head; ``oracle.depth_cache`` is the cache's
slot choice in plain Python.

Pins (what ties this oracle to the pages and the mathematics rather than to
itself) are in ``tests/test_oracle_pins.py``, ``tests/test_oracle_bwd.py``,
``tests/test_oracle_kvproj.py`` and ``tests/test_oracle_cache.py``; every
function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoda_oracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (fp contraction off, so x86 and Arm agree)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out)) or (os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, src, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _u16(a, name):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(q, k, v, kd, vd):
    T, Hq, d = q.shape
    if k.shape[0] != T or k.shape[2] != d or v.shape != k.shape:
        raise ValueError("k/v must be [T,Hk,d] matching q[T,Hq,d]")
    Hk = k.shape[1]
    if kd is None or kd.size == 0:
        L = 0
    else:
        L = kd.shape[0]
        if kd.shape != (L, T, Hk, d) or vd is None or vd.shape != kd.shape:
            raise ValueError("kd/vd must be [L,T,Hk,d]")
    return T, Hq, Hk, d, L


class Oracle:
    """ctypes front end of one compiled copy of ``moda_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i = ctypes.c_int
        lib.moda_oracle_row.argtypes = [u16p] * 5 + [i] * 5 + [
            ctypes.c_double, i, i, f64p, f64p, f64p]
        lib.moda_oracle_row.restype = ctypes.c_int
        lib.moda_oracle_rows.argtypes = [u16p] * 5 + [i] * 5 + [
            ctypes.c_double, i64p, i64p, ctypes.c_int64, f64p, f64p, i]
        lib.moda_oracle_rows.restype = ctypes.c_int
        lib.moda_oracle_bwd.argtypes = [u16p] * 6 + [i] * 5 + [ctypes.c_double] + [f64p] * 5 + [i]
        lib.moda_oracle_bwd.restype = ctypes.c_int
        lib.moda_oracle_bwd_rows.argtypes = [u16p] * 6 + [i] * 5 + [ctypes.c_double, i64p,
                                              ctypes.c_int64, i] + [f64p] * 5 + [i]
        lib.moda_oracle_bwd_rows.restype = ctypes.c_int
        lib.moda_oracle_kv_proj.argtypes = [u16p, u16p, i, i, i, i64p, ctypes.c_int64, f64p]
        lib.moda_oracle_kv_proj.restype = ctypes.c_int
        lib.moda_oracle_depth_mass.argtypes = [u16p] * 5 + [i] * 5 + [
            ctypes.c_double, i64p, i64p, ctypes.c_int64, f64p, i]
        lib.moda_oracle_depth_mass.restype = ctypes.c_int
        self._lib = lib

    @staticmethod
    def _prep(q, k, v, kd, vd):
        q, k, v, kd, vd = (_u16(x, n) for x, n in
                           zip((q, k, v, kd, vd), ("q", "k", "v", "kd", "vd")))
        T, Hq, Hk, d, L = _shapes(q, k, v, kd, vd)
        return (q, k, v, kd if L else None, vd if L else None), (T, Hq, Hk, d, L)

    def row(self, q, k, v, kd, vd, scale, t, h):
        """One query row (t, h): returns (o[d] float64, lse float, p[t+1+L]).

        ``p`` is the joint probability row [sequence keys 0..t | depth slots
        0..L-1]; it is exported so tests can check that it sums to one and
        can read the depth mass.
        """
        arrs, (T, Hq, Hk, d, L) = self._prep(q, k, v, kd, vd)
        o = np.zeros(d, np.float64)
        lse = np.zeros(1, np.float64)
        p = np.zeros(int(t) + 1 + L, np.float64)
        rc = self._lib.moda_oracle_row(
            *(_ptr(a, ctypes.c_uint16) for a in arrs), T, Hq, Hk, d, L,
            float(scale), int(t), int(h),
            _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(p, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"moda_oracle_row failed with {rc}")
        return o, float(lse[0]), p

    def rows(self, q, k, v, kd, vd, scale, ts, hs, nthreads: int = 1):
        """Rows (ts[i], hs[i]): returns (o[n,d] float64, lse[n] float64)."""
        arrs, (T, Hq, Hk, d, L) = self._prep(q, k, v, kd, vd)
        ts = np.ascontiguousarray(ts, dtype=np.int64).reshape(-1)
        hs = np.ascontiguousarray(hs, dtype=np.int64).reshape(-1)
        if ts.shape != hs.shape:
            raise ValueError("ts and hs must have the same length")
        n = ts.shape[0]
        o = np.zeros((n, d), np.float64)
        lse = np.zeros(n, np.float64)
        rc = self._lib.moda_oracle_rows(
            *(_ptr(a, ctypes.c_uint16) for a in arrs), T, Hq, Hk, d, L, float(scale),
            _ptr(ts, ctypes.c_int64), _ptr(hs, ctypes.c_int64), n,
            _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
        if rc != 0:
            raise ValueError(f"moda_oracle_rows failed with {rc}")
        return o, lse

    def forward(self, q, k, v, kd, vd, scale, nthreads: int = 1):
        """Every row: returns (o[T,Hq,d] float64, lse[T,Hq] float64)."""
        T, Hq, d = np.asarray(q).shape
        tt, hh = np.meshgrid(np.arange(T), np.arange(Hq), indexing="ij")
        o, lse = self.rows(q, k, v, kd, vd, scale, tt.reshape(-1), hh.reshape(-1), nthreads)
        return o.reshape(T, Hq, d), lse.reshape(T, Hq)


    def backward(self, q, k, v, kd, vd, dO, scale, nthreads: int = 1):
        """All gradients of the forward for upstream gradient dO[T,Hq,d]
        (bf16 bits). Returns float64 (dq[T,Hq,d], dk[T,Hk,d], dv[T,Hk,d],
        dkd[L,T,Hk,d], dvd[L,T,Hk,d]); the depth gradients are in the
        unpacked append layout."""
        arrs, (T, Hq, Hk, d, L) = self._prep(q, k, v, kd, vd)
        dO = _u16(dO, "dO")
        if dO.shape != (T, Hq, d):
            raise ValueError("dO must be [T,Hq,d]")
        dq = np.zeros((T, Hq, d))
        dk = np.zeros((T, Hk, d))
        dv = np.zeros((T, Hk, d))
        dkd = np.zeros((L, T, Hk, d))
        dvd = np.zeros((L, T, Hk, d))
        p = lambda a: _ptr(a, ctypes.c_double) if a.size else None
        rc = self._lib.moda_oracle_bwd(
            *(_ptr(a, ctypes.c_uint16) for a in arrs), _ptr(dO, ctypes.c_uint16),
            T, Hq, Hk, d, L, float(scale), p(dq), p(dk), p(dv), p(dkd), p(dvd), int(nthreads))
        if rc != 0:
            raise ValueError(f"moda_oracle_bwd failed with {rc}")
        return dq, dk, dv, dkd, dvd


    def backward_rows(self, q, k, v, kd, vd, dO, scale, rows, k_lo, nthreads: int = 1):
        """Gradient contributions of the rows listed (row = t*Hq + h): returns
        (dq_rows[n,d], dk_tail[T-k_lo,Hk,d], dv_tail, dkd_rows[n,L,d], dvd_rows)."""
        arrs, (T, Hq, Hk, d, L) = self._prep(q, k, v, kd, vd)
        dO = _u16(dO, "dO")
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        n = rows.shape[0]
        dq = np.zeros((n, d))
        dk = np.zeros((T - k_lo, Hk, d))
        dv = np.zeros((T - k_lo, Hk, d))
        dkd = np.zeros((n, L, d))
        dvd = np.zeros((n, L, d))
        p = lambda a: _ptr(a, ctypes.c_double) if a.size else None
        rc = self._lib.moda_oracle_bwd_rows(
            *(_ptr(a, ctypes.c_uint16) for a in arrs), _ptr(dO, ctypes.c_uint16),
            T, Hq, Hk, d, L, float(scale), _ptr(rows, ctypes.c_int64), n, int(k_lo),
            p(dq), p(dk), p(dv), p(dkd), p(dvd), int(nthreads))
        if rc != 0:
            raise ValueError(f"moda_oracle_bwd_rows failed with {rc}")
        return dq, dk, dv, dkd, dvd


    def depth_mass(self, q, k, v, kd, vd, scale, ts=None, hs=None, nthreads: int = 1):
        """Depth probability mass [Hk, L] float64: entry (hk, l) sums p(slot l)
        over the rows (ts[i], hs[i]) of KV head hk (every row when ts is None)."""
        arrs, (T, Hq, Hk, d, L) = self._prep(q, k, v, kd, vd)
        if L < 1:
            raise ValueError("depth_mass needs L >= 1")
        if ts is None:
            tt, hh = np.meshgrid(np.arange(T), np.arange(Hq), indexing="ij")
            ts, hs = tt.reshape(-1), hh.reshape(-1)
        ts = np.ascontiguousarray(ts, dtype=np.int64).reshape(-1)
        hs = np.ascontiguousarray(hs, dtype=np.int64).reshape(-1)
        if ts.shape != hs.shape:
            raise ValueError("ts and hs must have the same length")
        mass = np.zeros((Hk, L), np.float64)
        rc = self._lib.moda_oracle_depth_mass(
            *(_ptr(a, ctypes.c_uint16) for a in arrs), T, Hq, Hk, d, L, float(scale),
            _ptr(ts, ctypes.c_int64), _ptr(hs, ctypes.c_int64), ts.shape[0],
            _ptr(mass, ctypes.c_double), int(nthreads))
        if rc != 0:
            raise ValueError(f"moda_oracle_depth_mass failed with {rc}")
        return mass

    def kv_proj(self, x, w, rows=None):
        """Linear depth-KV projection of an FFN layer's input: x [T,Dm] and
        w [N,Dm] (bf16 bits, one weight row per output feature). Returns
        float64 out [len(rows), N] (all T rows when rows is None), unrounded."""
        x, w = _u16(x, "x"), _u16(w, "w")
        if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
            raise ValueError("x must be [T,Dm] and w [N,Dm]")
        T, Dm = x.shape
        N = w.shape[0]
        if rows is None:
            rows = np.arange(T, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        out = np.zeros((rows.shape[0], N), np.float64)
        rc = self._lib.moda_oracle_kv_proj(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                                           T, Dm, N, _ptr(rows, ctypes.c_int64), rows.shape[0],
                                           _ptr(out, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"moda_oracle_kv_proj failed with {rc}")
        return out


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def row(*args, **kw):
    return default().row(*args, **kw)


def rows(*args, **kw):
    return default().rows(*args, **kw)


def forward(*args, **kw):
    return default().forward(*args, **kw)


def backward(*args, **kw):
    return default().backward(*args, **kw)


def kv_proj(*args, **kw):
    return default().kv_proj(*args, **kw)


def depth_mass(*args, **kw):
    return default().depth_mass(*args, **kw)
