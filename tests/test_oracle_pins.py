"""Pins for the fp64 CPU oracle against facts the pages and mathematics fix.

Each test ties the oracle to something other than itself (paper: "Not All
Dimensions Are Equal: Outlier-Aware Attention Linearization with Grouped
Quadratic Kernels", arXiv:2610.13674):

  direct == recurrent        App. D, Eqs. (24)-(25): the H0/H1/H2 recurrence
                             (Algorithm 1) equals the pairwise kernel sum.
                             Two independent formulations must agree to 1e-12.
  hand example               tests/golden/hand_example.json, derived by hand.
  running mean               L = diag(L00, 0, ...) makes kappa constant, so
                             y_i is the causal running mean of v (Eq. 7 with
                             Eq. 1); pins causality, normalisation and GQA.
  Taylor, G = 1              App. D Eq. (23) with M = [[1,1/2],[1/2,1/2]] is
                             the second-order Taylor polynomial 1+s+s^2/2
                             (Sec. 2); compared with a brute-force textbook sum.
  global embedding           App. D: M_0g = m01, M_gh = m11 for all groups gives
                             the global quadratic for ANY partition.
  kappa >= eps               Sec. 4.3: L L^T is PSD.
  coefficient map            Sec. 4.3 (a = eps + M00, b_r = 2 M_0g(r),
                             C_rt = M_g(r)g(t)) in exact rational arithmetic on
                             dyadic inputs; packed multiplicity of App. D.
  packed == full readout     App. D "Exact state and parameter counts".
  continuation               the state after T1 tokens resumes to the same
                             outputs as one pass over T1 + T2 tokens.
  empty groups               App. B (groups partition the dims) with L lower-
                             triangular: empty groups give the kernel of the
                             truncated L, whatever their rows of L hold.
  backward                   every gradient entry against central differences
                             of the forward oracle (the C pair sum); the
                             constant kernel's closed form (dQ = dK = 0, dV of
                             a running mean, no gradient on L00).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from grouped_quadratic_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_case(seed, B=2, Hq=4, Hkv=2, T=24, d=8, dv=5, G=3, outlier=6.0):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, Hq, T, d))
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, dv))
    Q[..., 1] *= outlier
    K[..., 1] *= outlier
    L = np.stack([inputs.random_L(rng, G) for _ in range(Hq)]).astype(np.float64)
    group = rng.integers(1, G + 1, size=(Hq, d)).astype(np.int32)
    return Q, K, V, L, group


def rel_err(a, b):
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


@pytest.mark.parametrize("seed,shape", [
    (1, dict()),
    (2, dict(B=1, Hq=3, Hkv=3, T=17, d=6, dv=3, G=1)),
    (3, dict(B=1, Hq=6, Hkv=2, T=40, d=10, dv=4, G=5)),
    (4, dict(B=1, Hq=2, Hkv=1, T=12, d=64, dv=64, G=4)),
])
def test_direct_equals_recurrent(seed, shape):
    Q, K, V, L, group = small_case(seed, **shape)
    eps = 1e-3
    yd = oracle.direct(Q, K, V, L, group, eps)
    yr, _ = oracle.recurrent(Q, K, V, L, group, eps)
    assert np.all(np.isfinite(yd))
    assert rel_err(yr, yd) <= 1e-12
    assert np.max(np.abs(yr - yd)) <= 1e-10 * max(1.0, np.max(np.abs(yd)))


def test_hand_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    Q = np.array(g["Q"], np.float64)[None, None]
    K = np.array(g["K"], np.float64)[None, None]
    V = np.array(g["V"], np.float64)[None, None]
    L = np.array(g["L"], np.float64)[None]
    group = np.array(g["group"], np.int32)[None]
    want = np.array(g["Y"], np.float64)[None, None]
    yd = oracle.direct(Q, K, V, L, group, g["eps"])
    yr, _ = oracle.recurrent(Q, K, V, L, group, g["eps"])
    np.testing.assert_allclose(yd, want, rtol=0, atol=1e-14)
    np.testing.assert_allclose(yr, want, rtol=0, atol=1e-13)
    a, b, C = oracle.expand_coeffs(np.array(g["L"], np.float32)[None], group, g["eps"])
    assert a[0] == g["coeffs"]["a"]
    assert list(b[0]) == g["coeffs"]["b"]
    Cm = C[0].reshape(4, 4)
    assert np.all(Cm[:3, :3] == 2) and np.all(Cm[:3, 3] == 1) and np.all(Cm[3, :3] == 1)
    assert Cm[3, 3] == 2


@pytest.mark.parametrize("fn", ["direct", "recurrent"])
def test_constant_kernel_gives_running_mean(fn):
    Q, K, V, L, group = small_case(7, B=2, Hq=6, Hkv=3, T=20, d=8, dv=4, G=3)
    L[:] = 0.0
    L[:, 0, 0] = 0.7
    eps = 1e-6
    if fn == "direct":
        y = oracle.direct(Q, K, V, L, group, eps)
    else:
        y, _ = oracle.recurrent(Q, K, V, L, group, eps)
    T = Q.shape[2]
    mean = np.cumsum(V, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    rho = Q.shape[1] // K.shape[1]
    want = np.repeat(mean, rho, axis=1)        # query head h reads KV head h // rho
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


def textbook_global(Q, K, V, d, poly):
    """Brute-force normalised causal average with weights poly(q.k/sqrt(d))."""
    B, Hq, T, _ = Q.shape
    Hkv = K.shape[1]
    rho = Hq // Hkv
    Y = np.empty(Q.shape[:3] + (V.shape[3],))
    for b in range(B):
        for h in range(Hq):
            s = Q[b, h] @ K[b, h // rho].T / np.sqrt(d)
            w = np.tril(poly(s))
            Y[b, h] = (w @ V[b, h // rho]) / w.sum(axis=1, keepdims=True)
    return Y


def test_taylor_special_case():
    Q, K, V, _, _ = small_case(11, B=1, Hq=2, Hkv=1, T=30, d=16, dv=3, G=1, outlier=1.0)
    L = np.array([[[1.0, 0.0], [0.5, 0.5]]] * 2)
    group = np.ones((2, 16), np.int32)
    eps = 1e-9
    want = textbook_global(Q, K, V, 16, lambda s: eps + 1.0 + s + 0.5 * s * s)
    y = oracle.direct(Q, K, V, L, group, eps)
    np.testing.assert_allclose(y, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("G", [2, 3, 5])
def test_global_embedding_invariant_to_partition(G):
    Q, K, V, _, _ = small_case(20 + G, B=1, Hq=2, Hkv=1, T=25, d=12, dv=3, G=G)
    l00, l10, l11, eps = 0.8, 0.45, 0.6, 1e-4
    L = np.zeros((2, G + 1, G + 1))
    L[:, 0, 0] = l00
    L[:, 1:, 0] = l10
    L[:, 1:, 1] = l11
    m00, m01, m11 = l00 * l00, l00 * l10, l10 * l10 + l11 * l11
    want = textbook_global(Q, K, V, 12, lambda s: eps + m00 + 2 * m01 * s + m11 * s * s)
    rng = np.random.default_rng(G)
    for _ in range(3):
        group = rng.integers(1, G + 1, size=(2, 12)).astype(np.int32)
        y = oracle.direct(Q, K, V, L, group, eps)
        np.testing.assert_allclose(y, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("gh", [1, 2, 3])
def test_empty_groups_equal_fewer_groups(gh):
    # App. B: the groups partition the dims.  A group with no dims has group
    # sum 0, and L is lower-triangular, so the kernel of a head whose groups
    # above gh are empty is the one of the leading (gh + 1) x (gh + 1) block
    # of L with gh groups: heads of different group counts share one G.
    Q, K, V, L, group = small_case(60 + gh, B=2, Hq=2, Hkv=1, T=30, d=10, dv=4, G=4)
    group[group > gh] = 1
    eps = 1e-3
    y = oracle.direct(Q, K, V, L, group, eps)
    y_trunc = oracle.direct(Q, K, V, np.ascontiguousarray(L[:, :gh + 1, :gh + 1]), group, eps)
    np.testing.assert_allclose(y, y_trunc, rtol=1e-12, atol=1e-13)
    # and the L entries of the empty groups do not matter
    L2 = L.copy()
    L2[:, gh + 1:, :] = 7.0 * np.tril(np.ones_like(L2[:, gh + 1:, :]), gh + 1)
    np.testing.assert_allclose(oracle.direct(Q, K, V, L2, group, eps), y, rtol=1e-12, atol=1e-13)


def test_kappa_at_least_eps():
    w = inputs.make_workload("pin", B=1, Hq=2, Hkv=1, T=64, G=4, dtype="f32", seed=5)
    rows = np.arange(0, 2 * 64, 7)
    _, mk = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps, rows=rows,
                          return_min_kappa=True)
    assert mk >= w.eps


def exact_M(L):
    G1 = len(L)
    return [[sum(Fraction(L[g][c]) * Fraction(L[h][c]) for c in range(min(g, h) + 1))
             for h in range(G1)] for g in range(G1)]


def test_coefficient_map_exact_on_dyadic_inputs():
    rng = np.random.default_rng(3)
    G, d, Hq = 4, 10, 3
    # dyadic entries (k/8, |k| <= 16): every fp64 and fp32 value below is exact
    L = (rng.integers(-16, 17, size=(Hq, G + 1, G + 1)) / 8.0).astype(np.float32)
    L[:, np.triu_indices(G + 1, 1)[0], np.triu_indices(G + 1, 1)[1]] = 5.0  # ignored
    group = rng.integers(1, G + 1, size=(Hq, d)).astype(np.int32)
    eps = 0.25
    a, b, C = oracle.expand_coeffs(L, group, eps)
    ap, bp, Cp = oracle.expand_coeffs(L, group, eps, packed=True)
    r_idx, t_idx = oracle.packed_index(d)
    for h in range(Hq):
        M = exact_M(L[h].astype(np.float64).tolist())
        assert Fraction(float(a[h])) == Fraction(eps) + M[0][0]
        for r in range(d):
            assert Fraction(float(b[h, r])) == 2 * M[0][group[h, r]]
            for t in range(d):
                assert Fraction(float(C[h, r * d + t])) == M[group[h, r]][group[h, t]]
        for n, (r, t) in enumerate(zip(r_idx, t_idx)):
            mult = 1 if r == t else 2
            assert Fraction(float(Cp[h, n])) == mult * M[group[h, r]][group[h, t]]
        assert n == d * (d + 1) // 2 - 1
    assert np.array_equal(a, ap) and np.array_equal(b, bp)


def test_coefficient_rounding_rule_single_rounding():
    # M00 = (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24: exact in fp64, a tie in fp32
    # that rounds to even (1 + 2^-11); eps = 2^-30 then breaks the tie upward.
    L = np.array([[[1 + 2.0 ** -12, 0.0], [0.0, 1.0]]], np.float32)
    group = np.ones((1, 4), np.int32)
    a, _, _ = oracle.expand_coeffs(L, group, 0.0)
    assert float(a[0]) == 1 + 2.0 ** -11
    a, _, _ = oracle.expand_coeffs(L, group, 2.0 ** -30)
    assert float(a[0]) == 1 + 2.0 ** -11 + 2.0 ** -23


def test_packed_readout_equals_full_readout():
    Q, K, V, L, group = small_case(9, B=1, Hq=2, Hkv=1, T=15, d=8, dv=3, G=3)
    eps = 1e-3
    _, S = oracle.recurrent(Q, K, V, L, group, eps)
    d = 8
    Sp = oracle.full_to_packed_state(S, d)
    assert Sp.shape[-2] == oracle.packed_rows(d)
    a, b, C = oracle.expand_coeffs(L.astype(np.float32), group, eps)
    _, _, Cp = oracle.expand_coeffs(L.astype(np.float32), group, eps, packed=True)
    r_idx, t_idx = oracle.packed_index(d)
    q = Q[0, 0, -1]
    full = sum(C[0, r * d + t] * q[r] * q[t] * S[0, 0, 1 + d + r * d + t]
               for r in range(d) for t in range(d))
    packed = sum(Cp[0, n] * q[r] * q[t] * Sp[0, 0, 1 + d + n]
                 for n, (r, t) in enumerate(zip(r_idx, t_idx)))
    np.testing.assert_allclose(packed, full, rtol=1e-12)
    # H2 of the full layout is symmetric in (r, t)
    H2 = S[0, 0, 1 + d:].reshape(d, d, -1)
    np.testing.assert_allclose(H2, H2.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_state_continuation():
    Q, K, V, L, group = small_case(13, B=1, Hq=4, Hkv=2, T=30, d=8, dv=3, G=2)
    eps = 1e-3
    y_all, s_all = oracle.recurrent(Q, K, V, L, group, eps)
    _, s1 = oracle.recurrent(Q[:, :, :18], K[:, :, :18], V[:, :, :18], L, group, eps)
    y2, s2 = oracle.recurrent(Q[:, :, 18:], K[:, :, 18:], V[:, :, 18:], L, group, eps, S0=s1)
    np.testing.assert_allclose(y2, y_all[:, :, 18:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s2, s_all, rtol=1e-12, atol=1e-11)
    # the H0 denominator entry counts the tokens seen (u = [v; 1])
    assert np.all(s_all[:, :, 0, -1] == 30)


def test_direct_rows_subset_matches_full():
    Q, K, V, L, group = small_case(17, B=2, Hq=4, Hkv=2, T=21, d=8, dv=3, G=3)
    full = oracle.direct(Q, K, V, L, group, 1e-3)
    rows = np.array([0, 5, 20, 21, 63, 100, 167])
    sub = oracle.direct(Q, K, V, L, group, 1e-3, rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, 3)[rows])


def test_invalid_group_rejected():
    Q, K, V, L, group = small_case(1)
    group[0, 0] = 0
    with pytest.raises(ValueError):
        oracle.direct(Q, K, V, L, group, 1e-3)


def test_named_workloads_shapes_and_structure():
    w = inputs.config(0)
    assert w.Q.shape == (1, 1, 256, 64) and w.dtype == "f32"
    g = w.group[0]
    assert set(np.flatnonzero(g == 2)) == {3, 17} and list(np.flatnonzero(g == 3)) == [40]
    assert list(np.flatnonzero(g == 4)) == [58] and np.sum(g == 1) == 60
    assert np.all(np.triu(w.L[0], 1) == 0) and np.all(np.diag(w.L[0]) >= 0.5)
    w1 = inputs.config(1, T=64)
    assert w1.Q.shape == (1, 14, 64, 64) and w1.K.shape == (1, 2, 64, 64)
    # bf16 workloads carry bf16-representable values
    assert np.array_equal(inputs.round_to_bf16(w1.Q), w1.Q)
    for h in range(14):
        assert set(np.unique(w1.group[h])) == {1, 2, 3, 4}


# ---------------------------------------------------------------- backward
def _loss(Q, K, V, L, group, eps, dY):
    return float((oracle.direct(Q, K, V, L, group, eps) * dY).sum())


def test_backward_matches_central_differences():
    # every gradient entry of a small GQA case against central differences of
    # the forward oracle (an independent code path: the C pair sum)
    Q, K, V, L, group = small_case(70, B=1, Hq=2, Hkv=1, T=6, d=5, dv=3, G=2)
    eps = 1e-2
    dY = np.random.default_rng(71).standard_normal((1, 2, 6, 3))
    dQ, dK, dV, dL = oracle.backward(Q, K, V, L, group, eps, dY)
    h = 1e-6
    for name, X, dX in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV), ("L", L, dL)):
        for idx in np.ndindex(X.shape):
            if name == "L" and idx[2] > idx[1]:
                assert dX[idx] == 0.0          # the upper triangle is not a parameter
                continue
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args = {"Q": Q, "K": K, "V": V, "L": L}
            args[name] = Xp
            fp = _loss(args["Q"], args["K"], args["V"], args["L"], group, eps, dY)
            args[name] = Xm
            fm = _loss(args["Q"], args["K"], args["V"], args["L"], group, eps, dY)
            fd = (fp - fm) / (2 * h)
            assert abs(fd - dX[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, dX[idx])


def test_backward_constant_kernel():
    # L = diag(L00, 0, ...): kappa is the constant eps + L00^2, y_i is the
    # causal running mean of v, so dQ = dK = 0 and dV_j = sum_{i >= j} dY_i / (i + 1)
    Q, K, V, _, group = small_case(72, B=2, Hq=4, Hkv=2, T=9, d=6, dv=4, G=3)
    L = np.zeros((4, 4, 4))
    L[:, 0, 0] = 0.7
    dY = np.random.default_rng(73).standard_normal((2, 4, 9, 4))
    dQ, dK, dV, dL = oracle.backward(Q, K, V, L, group, 1e-3, dY)
    assert not dQ.any() and not dK.any()
    want = np.zeros_like(V)
    for i in range(9):
        for h in range(4):
            want[:, h // 2, : i + 1] += dY[:, h, i][:, None, :] / (i + 1)
    np.testing.assert_allclose(dV, want, rtol=1e-12, atol=1e-13)
    # L00 only moves the constant, which the normalisation cancels
    np.testing.assert_allclose(dL[:, 0, 0], 0.0, atol=1e-12)
