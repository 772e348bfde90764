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
  contribution_scores() -- the per-prompt contribution score of Sec. 3.1,
                     Eq. (2), pair by pair over the causal pair set.
  bootstrap_groups() -- the dimension grouping of App. B, Eqs. (16)-(19), for
                     one query head, step by step in the appendix's order.
  backward()      -- gradients of the causal output with respect to Q, K, V
                     and L (the derivative of the definition above; the
                     calibration of App. B, Eq. (20), and the LoRA adaptation
                     of Sec. 5 differentiate through it), pair by pair.

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


def contribution_scores(Q, K, lengths=None):
    """Eq. (2) for every prompt: chi[p, h, r] = 1/|Omega_p| * sum over the
    causal pairs (i, j), j <= i < N_p, of |q_{p,i,r} k_{p,j,r} / sqrt(d)|,
    with |Omega_p| = N_p (N_p + 1) / 2 (chi = 0 for an empty prompt).

    Q [P,Hq,T,d], K [P,Hkv,T,d]; query head h pairs with KV head h // (Hq/Hkv)
    (the model's GQA map, App. B).  lengths [P] (default: T for every prompt).
    Pair by pair, in fp64: O(N^2 d) per head, for small cases.
    """
    Q, K = _f64(Q), _f64(K)
    P, Hq, T, d = Q.shape
    Hkv = K.shape[1]
    rho = Hq // Hkv
    if lengths is None:
        lengths = [T] * P
    chi = np.zeros((P, Hq, d), np.float64)
    for p in range(P):
        n = int(lengths[p])
        if n == 0:
            continue
        omega = n * (n + 1) / 2.0
        causal = np.tril(np.ones((n, n), dtype=bool))   # [i, j] with j <= i
        for h in range(Hq):
            q, k = Q[p, h, :n], K[p, h // rho, :n]
            for r in range(d):
                pair = np.abs(np.outer(q[:, r], k[:, r]) / np.sqrt(d))
                chi[p, h, r] = pair[causal].sum() / omega
    return chi


def bootstrap_groups(chi_p, boot_idx, alpha, tau, gamma, g_min, eps=1e-12):
    """App. B grouping of one query head.  Returns (group [d] int32 in 1..G, G).

    chi_p [P, d] per-prompt scores (Eq. (2) before the average over prompts);
    boot_idx [nboot, P] the prompt indices of each bootstrap replicate.
    fp64 throughout; every average is a sum in index order, then one division.
    """
    chi_p = np.asarray(chi_p, dtype=np.float64)
    boot_idx = np.asarray(boot_idx)
    P, d = chi_p.shape
    nboot = boot_idx.shape[0]

    def average(rows):
        acc = np.zeros(d, np.float64)
        for t in rows:
            acc = acc + chi_p[t]
        return acc / len(rows)

    chi = average(range(P))
    # increasing contribution, stable: pi[0] is pi_1 of the appendix
    pi = sorted(range(d), key=lambda r: chi[r])
    m = int(np.ceil(alpha * d))
    cands = list(range(max(1, d - m), d))          # k: L_k = pi[:k], U_k = pi[k:]
    # Eq. (16): the adjacent gap across cut k
    rho_gap = {k: chi[pi[k]] / max(chi[pi[k - 1]], eps) for k in cands}
    # Eqs. (17)-(18): the bootstrap support of each cut, ordering pi kept fixed
    hits = {k: 0 for k in cands}
    for b in range(nboot):
        chi_b = average(boot_idx[b])
        for k in cands:
            lo = max(chi_b[r] for r in pi[:k])
            hi = min(chi_b[r] for r in pi[k:])
            if hi / max(lo, eps) >= tau:
                hits[k] += 1
    support = {k: hits[k] / nboot for k in cands}
    # natural cuts; then fallback cuts by descending (support, gap) until
    # g_min groups (ties keep the candidate order)
    cuts = [k for k in cands if rho_gap[k] >= tau and support[k] >= gamma]
    if len(cuts) + 1 < g_min:
        rest = [k for k in cands if k not in cuts]
        rest = sorted(rest, key=lambda k: (-support[k], -rho_gap[k]))
        for k in rest:
            if len(cuts) + 1 >= g_min:
                break
            cuts.append(k)
    bounds = [0] + sorted(cuts) + [d]
    group = np.zeros(d, np.int32)
    for g in range(1, len(bounds)):                # Eq. (19)
        for r in pi[bounds[g - 1]:bounds[g]]:
            group[r] = g
    return group, len(bounds) - 1


def backward(Q, K, V, L, group, eps, dY):
    """Gradients of <dY, Y> for Y = direct(Q, K, V, L, group, eps).

    Returns (dQ, dK, dV, dL) in fp64, shaped like Q, K, V, L; dL is zero
    above the diagonal (the upper triangle of L is not a parameter).  With
    y_i = N_i / D_i, N_i = sum_{j<=i} kappa_ij v_j, D_i = sum_{j<=i} kappa_ij:
        d/d kappa_ij = dY_i . (v_j - y_i) / D_i =: g_ij,
        dV_j = sum_{i>=j} kappa_ij dY_i / D_i,
        kappa_ij = eps + s_bar^T M s_bar, M = L L^T:
            d kappa / d s_g = 2 (M s_bar)_g,  d kappa / d M = s_bar s_bar^T,
        s_g = sum_{r in G_g} q_ir k_jr / sqrt(d),
        dL = (dM + dM^T) L restricted to the lower triangle.
    Key/value gradients are summed over the query heads of a KV head.  Every
    pair is formed explicitly: O(T^2 d) memory per head, for small cases.
    """
    Q, K, V, L, dY = _f64(Q), _f64(K), _f64(V), _f64(L), _f64(dY)
    group = np.asarray(group)
    B, Hq, T, d = Q.shape
    Hkv = K.shape[1]
    rho = Hq // Hkv
    G = L.shape[1] - 1
    sd = np.sqrt(d)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dL = np.zeros_like(L)
    causal = np.tril(np.ones((T, T)))
    for h in range(Hq):
        kv = h // rho
        Lh = np.tril(L[h])
        M = Lh @ Lh.T
        member = np.zeros((d, G + 1))                     # dim r -> its group column
        member[np.arange(d), group[h]] = 1.0
        for b in range(B):
            q, k, v, dy = Q[b, h], K[b, kv], V[b, kv], dY[b, h]
            x = q[:, None, :] * k[None, :, :] / sd        # [i, j, r]
            sbar = x @ member                             # [i, j, g]
            sbar[..., 0] = 1.0
            kap = (eps + np.einsum("ija,ab,ijb->ij", sbar, M, sbar)) * causal
            D = kap.sum(axis=1)
            y = (kap @ v) / D[:, None]
            g = (dy @ v.T - (dy * y).sum(axis=1)[:, None]) / D[:, None] * causal
            dV[b, kv] += (kap / D[:, None]).T @ dy
            dx = (2.0 * g[..., None] * (sbar @ M)) @ member.T   # d/dx_ijr = d/ds_{g(r)}
            dQ[b, h] += (dx * k[None, :, :]).sum(axis=1) / sd
            dK[b, kv] += (dx * q[:, None, :]).sum(axis=0) / sd
            dM = np.einsum("ij,ija,ijb->ab", g, sbar, sbar)
            dL[h] += np.tril((dM + dM.T) @ Lh)
    return dQ, dK, dV, dL
