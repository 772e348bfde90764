"""fp64 CPU oracle for OAL causal attention (ctypes wrapper around oal_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA path; only the seeded input generator
(``grouped_quadratic_gb300.inputs``, which holds none of the method's
arithmetic) feeds both.

Method: "Not All Dimensions Are Equal: Outlier-Aware Attention
Linearization with Grouped Quadratic Kernels" (arXiv:2610.13674).
  direct()        -- the definition: kappa = eps + s_bar^T L L^T s_bar
                     (Sec. 4.3, Eq. 7) and the normalised inclusive causal
                     average (Sec. 2, Eq. 1; App. D, Eq. 25), pair by pair.
  recurrent()     -- Algorithm 1's causal-evaluation stage: prefix states
                     H0/H1/H2 (Sec. 4.1, Eq. 5) and readout (Eq. 6).
  expand_coeffs() -- the fp32 coefficient tables of Sec. 4.3 (a, b_r, C_rt)
                     under the rounding rule stated in oal_oracle.c.
  full_to_packed_state() -- re-indexes an ordered-pair state into the packed
                     symmetric layout of App. D (indexing only, no arithmetic).

Parity status of each function (what pins it) is listed in the test module
``tests/test_oracle_pins.py``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        ip = ctypes.POINTER(ctypes.c_int32)
        lp = ctypes.POINTER(ctypes.c_int64)
        ci = ctypes.c_int
        lib.oal_oracle_direct.argtypes = [dp, dp, dp, ci, ci, ci, ci, ci, ci,
                                          dp, ip, ci, ctypes.c_double, lp,
                                          ctypes.c_int64, dp, dp, ci]
        lib.oal_oracle_direct.restype = ci
        lib.oal_oracle_recurrent.argtypes = [dp, dp, dp, ci, ci, ci, ci, ci, ci,
                                             dp, ip, ci, ctypes.c_double, dp,
                                             dp, dp]
        lib.oal_oracle_recurrent.restype = ci
        lib.oal_oracle_expand_coeffs.argtypes = [fp, ip, ci, ci, ci,
                                                 ctypes.c_float, ci, fp, fp, fp]
        lib.oal_oracle_expand_coeffs.restype = ci
        lib.oal_oracle_max_threads.argtypes = []
        lib.oal_oracle_max_threads.restype = ci
        _lib = lib
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def max_threads() -> int:
    return int(_load().oal_oracle_max_threads())


def direct(Q, K, V, L, group, eps, rows=None, nthreads=0, return_min_kappa=False):
    """Direct O(T^2 d) evaluation.

    Q [B,Hq,T,d], K [B,Hkv,T,d], V [B,Hkv,T,dv] (any real dtype, widened
    exactly to fp64), L [Hq,G+1,G+1], group [Hq,d] (values 1..G), eps scalar.
    rows: optional int64 array of flat row ids (b*Hq+h)*T+i.
    Returns Y [B,Hq,T,dv] (or [len(rows),dv]) in fp64.
    """
    lib = _load()
    Q, K, V, L = _f64(Q), _f64(K), _f64(V), _f64(L)
    group = np.ascontiguousarray(np.asarray(group, dtype=np.int32))
    B, Hq, T, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    G = L.shape[1] - 1
    assert K.shape == (B, Hkv, T, d) and V.shape == (B, Hkv, T, dv)
    assert L.shape == (Hq, G + 1, G + 1) and group.shape == (Hq, d)
    if rows is None:
        rows_arr, nrows, Y = None, 0, np.empty((B, Hq, T, dv), np.float64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        Y = np.empty((nrows, dv), np.float64)
    mk = np.empty(1, np.float64)
    st = lib.oal_oracle_direct(
        _ptr(Q, ctypes.c_double), _ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double),
        B, Hq, Hkv, T, d, dv, _ptr(L, ctypes.c_double), _ptr(group, ctypes.c_int32),
        G, float(eps),
        None if rows_arr is None else _ptr(rows_arr, ctypes.c_int64), nrows,
        _ptr(Y, ctypes.c_double), _ptr(mk, ctypes.c_double), int(nthreads))
    if st != 0:
        raise ValueError("oal_oracle_direct failed with status %d" % st)
    return (Y, float(mk[0])) if return_min_kappa else Y


def full_rows(d: int) -> int:
    return 1 + d + d * d


def packed_rows(d: int) -> int:
    return 1 + d + d * (d + 1) // 2


def recurrent(Q, K, V, L, group, eps, S0=None):
    """Algorithm 1 in fp64.  Returns (Y [B,Hq,T,dv], S [B,Hkv,1+d+d*d,dv+1]).

    S0: optional initial state in the same ordered-pair layout.
    """
    lib = _load()
    Q, K, V, L = _f64(Q), _f64(K), _f64(V), _f64(L)
    group = np.ascontiguousarray(np.asarray(group, dtype=np.int32))
    B, Hq, T, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    G = L.shape[1] - 1
    Y = np.empty((B, Hq, T, dv), np.float64)
    S = np.empty((B, Hkv, full_rows(d), dv + 1), np.float64)
    if S0 is not None:
        S0 = _f64(S0)
        assert S0.shape == S.shape
    st = lib.oal_oracle_recurrent(
        _ptr(Q, ctypes.c_double), _ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double),
        B, Hq, Hkv, T, d, dv, _ptr(L, ctypes.c_double), _ptr(group, ctypes.c_int32),
        G, float(eps), None if S0 is None else _ptr(S0, ctypes.c_double),
        _ptr(Y, ctypes.c_double), _ptr(S, ctypes.c_double))
    if st != 0:
        raise ValueError("oal_oracle_recurrent failed with status %d" % st)
    return Y, S


def expand_coeffs(L, group, eps, packed=False):
    """fp32 tables (a [Hq], b [Hq,d], C [Hq,d*d] or [Hq,d(d+1)/2])."""
    lib = _load()
    L = np.ascontiguousarray(np.asarray(L, dtype=np.float32))
    group = np.ascontiguousarray(np.asarray(group, dtype=np.int32))
    Hq, G1, _ = L.shape
    d = group.shape[1]
    a = np.empty(Hq, np.float32)
    b = np.empty((Hq, d), np.float32)
    C = np.empty((Hq, d * (d + 1) // 2 if packed else d * d), np.float32)
    st = lib.oal_oracle_expand_coeffs(
        _ptr(L, ctypes.c_float), _ptr(group, ctypes.c_int32), Hq, G1 - 1, d,
        np.float32(eps), int(bool(packed)), _ptr(a, ctypes.c_float),
        _ptr(b, ctypes.c_float), _ptr(C, ctypes.c_float))
    if st != 0:
        raise ValueError("oal_oracle_expand_coeffs failed with status %d" % st)
    return a, b, C


def packed_index(d: int):
    """Row-major upper-triangle pair list: idx(r,t) = r*d - r(r-1)/2 + (t-r)."""
    r, t = np.triu_indices(d)
    return r, t


def full_to_packed_state(S_full, d: int):
    """Re-index an ordered-pair state [..., 1+d+d*d, U] into the packed layout
    [..., 1+d+d(d+1)/2, U] (H0, H1, then H2_rt for r <= t).  Indexing only."""
    r, t = packed_index(d)
    head = S_full[..., : 1 + d, :]
    h2 = S_full[..., 1 + d + r * d + t, :]
    return np.concatenate([head, h2], axis=-2)
