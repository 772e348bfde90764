"""Calibration step before the path: contribution scores and dimension groups.

Paper: "Not All Dimensions Are Equal: Outlier-Aware Attention Linearization
with Grouped Quadratic Kernels" -- Sec. 3.1, Eq. (2) (contribution score)
and App. B, Eqs. (16)-(19) (bootstrap grouping).

  oracle pins (CPU)   Eq. (2) against closed forms (constant magnitudes, a
                      single non-zero key, per-KV-head magnitudes for the GQA
                      map), a pure-Python double loop, and prompt lengths;
                      the grouping against hand-built profiles whose groups
                      follow from the appendix's rules by inspection.
  host grouping (CPU) the library's oal_group_dims, through the C ABI, equal
                      to the oracle group for group on random profiles.
  GPU parity          oal_contribution_scores against the oracle (bf16 and
                      fp32 inputs, GQA, ragged and empty prompts).
"""
import math

import numpy as np
import pytest

import oracle
from grouped_quadratic_gb300 import inputs


# ---------------------------------------------------------------- Eq. (2) pins
def test_chi_constant_magnitudes():
    # |q_{i,r}| = a_r and |k_{j,r}| = b_r for every token: every causal pair
    # contributes a_r b_r / sqrt(d), so the average is exactly that
    rng = np.random.default_rng(1)
    P, Hq, T, d = 2, 2, 9, 6
    a = rng.uniform(0.5, 3.0, size=d)
    b = rng.uniform(0.5, 3.0, size=d)
    Q = a * rng.choice([-1.0, 1.0], size=(P, Hq, T, d))
    K = b * rng.choice([-1.0, 1.0], size=(P, 1, T, d))
    chi = oracle.contribution_scores(Q, K)
    np.testing.assert_allclose(chi, np.broadcast_to(a * b / math.sqrt(d), chi.shape),
                               rtol=1e-13)


def test_chi_single_key_is_causal():
    # only key 0 is non-zero: every query i >= 0 pairs with it, so
    # chi_r = |k_{0,r}| sum_i |q_{i,r}| / sqrt(d) / (T (T + 1) / 2); with the
    # pair order reversed (j >= i) only query 0 would
    rng = np.random.default_rng(2)
    T, d = 11, 4
    Q = rng.standard_normal((1, 1, T, d))
    K = np.zeros((1, 1, T, d))
    K[0, 0, 0] = rng.standard_normal(d)
    want = np.abs(K[0, 0, 0]) * np.abs(Q[0, 0]).sum(axis=0) / math.sqrt(d) / (T * (T + 1) / 2)
    np.testing.assert_allclose(oracle.contribution_scores(Q, K)[0, 0], want, rtol=1e-13)


def test_chi_against_double_loop():
    rng = np.random.default_rng(3)
    P, Hq, Hkv, T, d = 2, 4, 2, 7, 5
    Q = rng.standard_normal((P, Hq, T, d))
    K = rng.standard_normal((P, Hkv, T, d))
    lengths = [7, 4]
    want = np.zeros((P, Hq, d))
    for p in range(P):
        n = lengths[p]
        for h in range(Hq):
            for r in range(d):
                acc = 0.0
                for i in range(n):
                    for j in range(i + 1):
                        acc += abs(Q[p, h, i, r] * K[p, h // 2, j, r] / math.sqrt(d))
                want[p, h, r] = acc / (n * (n + 1) / 2)
    np.testing.assert_allclose(oracle.contribution_scores(Q, K, lengths), want, rtol=1e-12)


def test_chi_gqa_map_and_lengths():
    # KV head kv has key magnitude kv + 1 in every dim: query head h must see
    # that of h // (Hq / Hkv); a prompt cut to N tokens equals the cut arrays;
    # an empty prompt scores 0
    P, Hq, Hkv, T, d = 3, 6, 3, 8, 4
    Q = np.ones((P, Hq, T, d))
    K = np.ones((P, Hkv, T, d)) * (np.arange(Hkv) + 1.0)[None, :, None, None]
    chi = oracle.contribution_scores(Q, K, lengths=[8, 5, 0])
    for h in range(Hq):
        np.testing.assert_allclose(chi[:2, h], (h // 2 + 1) / math.sqrt(d), rtol=1e-13)
    assert not chi[2].any()
    rng = np.random.default_rng(4)
    Q2, K2 = rng.standard_normal((1, 2, T, d)), rng.standard_normal((1, 1, T, d))
    np.testing.assert_allclose(oracle.contribution_scores(Q2, K2, lengths=[5]),
                               oracle.contribution_scores(Q2[:, :, :5], K2[:, :, :5]),
                               rtol=1e-13)


# ---------------------------------------------------------------- App. B pins
def flat_profile(P, d, value=1.0):
    return np.full((P, d), value)


def test_groups_two_level_tail():
    # bulk 1, dim 6 at 5, dim 7 at 20, identical in every prompt: both gaps
    # (5 and 4) pass tau = 1.5 with full support -> cuts at k = 6 and 7
    chi = flat_profile(3, 8)
    chi[:, 6], chi[:, 7] = 5.0, 20.0
    g, G = oracle.bootstrap_groups(chi, inputs.bootstrap_indices(40, 3, 1), 0.5, 1.5, 0.9, 2)
    assert G == 3 and list(g) == [1, 1, 1, 1, 1, 1, 2, 3]


def test_groups_alpha_limits_candidates():
    # the only gap sits below the tail fraction: not a candidate, so the
    # fallback takes the first candidate (all tie at support 0, gap 1)
    d = 8
    chi = flat_profile(2, d)
    chi[:, 4:] = 10.0                              # gap at k = 4, tail m = 2 -> k in {6, 7}
    g, G = oracle.bootstrap_groups(chi, inputs.bootstrap_indices(20, 2, 2), 0.25, 1.5, 0.9, 2)
    assert G == 2 and list(g) == [1] * 6 + [2] * 2


def test_groups_fallback_prefers_support_then_gap():
    # no natural cut (gamma = 1.01 is out of reach); the fallback adds cuts by
    # (support, gap) descending: k = 7 (gap 3) before k = 6 (gap 2) when
    # both have full support
    d = 8
    chi = flat_profile(2, d)
    chi[:, 6], chi[:, 7] = 2.0, 6.0
    bi = inputs.bootstrap_indices(10, 2, 3)
    g, G = oracle.bootstrap_groups(chi, bi, 0.25, 1.5, 1.01, 2)
    assert G == 2 and list(g) == [1] * 7 + [2]
    g, G = oracle.bootstrap_groups(chi, bi, 0.25, 1.5, 1.01, 3)
    assert G == 3 and list(g) == [1] * 6 + [2, 3]


def test_groups_unstable_tail_needs_support():
    # dim 7 is large in one prompt of four only: its full-sample gap passes
    # tau, but replicates that miss that prompt do not -> support < gamma, no
    # natural cut; with g_min = 1 the head stays one group
    P, d = 4, 8
    chi = flat_profile(P, d)
    chi[0, 7] = 40.0
    bi = inputs.bootstrap_indices(200, P, 4)
    g, G = oracle.bootstrap_groups(chi, bi, 0.25, 1.5, 0.9, 1)
    assert G == 1 and not (g - 1).any()
    # the replicates without prompt 0 are the ones that fail
    frac_without = np.mean([0 not in row for row in bi])
    assert 0.2 < frac_without < 0.45          # (3/4)^4 ~ 0.32


def test_groups_order_and_ties():
    # equal scores keep index order (stable sort); the groups follow the sort
    d = 6
    chi = np.array([[3.0, 1.0, 3.0, 1.0, 9.0, 1.0]])
    g, G = oracle.bootstrap_groups(chi, np.zeros((5, 1), np.int32), 0.5, 1.5, 0.5, 2)
    # sorted: dims 1,3,5 (1.0), 0,2 (3.0), 4 (9.0); candidates k in {3,4,5}:
    # gaps 3, 1, 3 -> cuts at 3 and 5
    assert G == 3 and list(g) == [2, 1, 2, 1, 3, 1]


# ---------------------------------------------------------------- host grouping
@pytest.fixture(scope="module")
def lib_binding():
    from grouped_quadratic_gb300 import build, oal as binding
    build.build()
    binding.load_library()
    return binding


@pytest.mark.parametrize("seed", range(24))
def test_host_grouping_equals_oracle(lib_binding, seed):
    rng = np.random.default_rng(100 + seed)
    P, d = int(rng.integers(1, 9)), int(rng.choice([8, 16, 64]))
    # a bulk with a few heavy dims of varying stability across prompts
    chi = rng.uniform(0.5, 1.5, size=(P, d))
    heavy = rng.choice(d, size=int(rng.integers(0, 5)), replace=False)
    chi[:, heavy] *= rng.uniform(1.0, 30.0, size=(P, heavy.size))
    chi = chi.astype(np.float32)
    nboot = int(rng.integers(1, 60))
    bi = inputs.bootstrap_indices(nboot, P, seed)
    alpha = float(rng.choice([0.125, 0.25, 0.5, 1.0]))
    tau, gamma = float(rng.choice([1.2, 1.5, 3.0])), float(rng.choice([0.5, 0.9, 1.0]))
    g_min = int(rng.integers(1, 4))
    want, G_want = oracle.bootstrap_groups(chi, bi, alpha, tau, gamma, g_min)
    got, G = lib_binding.oal_group_dims(chi, bi, alpha, tau, gamma, g_min)
    assert G == G_want and np.array_equal(got, want)


def test_host_grouping_hand_case_and_errors(lib_binding):
    chi = np.ones((3, 8), np.float32)
    chi[:, 6], chi[:, 7] = 5.0, 20.0
    g, G = lib_binding.oal_group_dims(chi, inputs.bootstrap_indices(40, 3, 1), 0.5, 1.5, 0.9, 2)
    assert G == 3 and list(g) == [1, 1, 1, 1, 1, 1, 2, 3]
    bad = np.full((4, 3), 3, np.int32)             # index 3 is outside 0..2
    with pytest.raises(lib_binding.OALError):
        lib_binding.oal_group_dims(chi, bad, 0.5, 1.5, 0.9, 2)
    with pytest.raises(lib_binding.OALError):
        lib_binding.oal_group_dims(chi, inputs.bootstrap_indices(4, 3, 1), 0.0, 1.5, 0.9, 2)


# ---------------------------------------------------------------- GPU parity
@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gpu_contribution_scores(lib_binding, dtype):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(7)
    P, Hq, Hkv, T, d = 5, 6, 2, 300, 64
    Q = rng.standard_normal((P, Hq, T, d)).astype(np.float32)
    K = rng.standard_normal((P, Hkv, T, d)).astype(np.float32)
    Q[..., 5] *= 12.0
    K[..., 5] *= 9.0
    if dtype == "bf16":
        Q, K = inputs.round_to_bf16(Q), inputs.round_to_bf16(K)
    lengths = np.array([300, 129, 128, 1, 0], np.int32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    chi = lib_binding.oal_contribution_scores(
        torch.from_numpy(Q).to(tdt).cuda(), torch.from_numpy(K).to(tdt).cuda(),
        torch.from_numpy(lengths).cuda())
    lib_binding.oal_sync_status()
    got = chi.cpu().numpy().astype(np.float64)
    want = oracle.contribution_scores(Q, K, lengths)
    assert not got[4].any()
    err = np.abs(got - want) / np.maximum(np.abs(want), 1e-30)
    assert float(err[:4].max()) <= 1e-5
    # and every prompt at full length (no length array)
    chi = lib_binding.oal_contribution_scores(torch.from_numpy(Q).to(tdt).cuda(),
                                              torch.from_numpy(K).to(tdt).cuda())
    want = oracle.contribution_scores(Q, K)
    np.testing.assert_allclose(chi.cpu().numpy(), want, rtol=1e-5)
