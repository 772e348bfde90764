"""GPU parity of the prefill backward (dQ, dK, dV, dL) through the C ABI.

Small cases compare every gradient entry with the fp64 oracle's backward
(itself pinned by central differences of the forward definition).  The
tolerance, rel-L2 <= 1e-4 per gradient, follows from the arithmetic: the
kernels work in fp32 (bf16 inputs are exact in fp32) and each gradient entry
is a sum over at most T pairs, so its rounding error grows like
sqrt(T) * 2^-24 relative to the magnitude of the terms, with some
cancellation between them.

At the Qwen-shaped size (T = 4096, Hq = 14, Hkv = 2) the oracle's backward
does not fit in memory, so the test checks the property that defines a
gradient: for a random direction, <dQ, dq> + <dK, dk> + <dV, dv> equals the
derivative of f = <dY, Y> along (dq, dk, dv), taken by central differences of
the fp64 oracle forward; likewise <dL, dl> along a direction in L.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_quadratic_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def oal():
    from grouped_quadratic_gb300 import build, oal as binding
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load_library()
    return binding


def rel_l2(got, want):
    return float(np.linalg.norm((got - want).ravel()) / np.linalg.norm(want.ravel()))


def run_backward(oal, w, dY):
    Q, K, V = w.torch_inputs("cuda")
    dYt = torch.from_numpy(np.ascontiguousarray(dY, dtype=np.float32)).to("cuda", Q.dtype)
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    grads = oal.oal_prefill_backward(Q, K, V, dYt, L, group, w.eps)
    oal.oal_sync_status()
    return [g.cpu().numpy() for g in grads]


def dY_for(w, seed, dtype):
    dY = np.random.default_rng(seed).standard_normal(w.Q.shape).astype(np.float32)
    return inputs.round_to_bf16(dY) if dtype == "bf16" else dY


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,Hq,Hkv,T,G", [(2, 4, 2, 150, 3), (1, 6, 3, 70, 5), (1, 4, 1, 97, 1),
                                          (1, 2, 2, 129, 7)])
def test_backward_matches_oracle(oal, dtype, B, Hq, Hkv, T, G):
    w = inputs.make_workload("bw", B=B, Hq=Hq, Hkv=Hkv, T=T, G=G, dtype=dtype, seed=500 + T + G)
    dY = dY_for(w, 7 + T, dtype)
    got = run_backward(oal, w, dY)
    want = oracle.backward(w.Q, w.K, w.V, w.L, w.group, w.eps, dY)
    for name, g, r in zip(("dQ", "dK", "dV", "dL"), got, want):
        assert np.all(np.isfinite(g)), name
        assert rel_l2(g, r) <= TOL, (name, rel_l2(g, r))


def test_backward_wide_groups_and_bulk_not_first(oal):
    # a tail group of three dims and the bulk (largest) group numbered 3
    w = inputs.make_workload("bw-wide", B=1, Hq=4, Hkv=2, T=120, G=3, dtype="f32", seed=560,
                             fixed_outliers=([3, 17, 40, 58], 12.0),
                             fixed_groups=[[3, 17, 40], [58]])
    w.group[w.group == 1] = 4
    w.group[w.group == 3] = 1
    w.group[w.group == 4] = 3
    dY = dY_for(w, 9, "f32")
    got = run_backward(oal, w, dY)
    want = oracle.backward(w.Q, w.K, w.V, w.L, w.group, w.eps, dY)
    for name, g, r in zip(("dQ", "dK", "dV", "dL"), got, want):
        assert rel_l2(g, r) <= TOL, (name, rel_l2(g, r))


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65])
def test_backward_short_sequences(oal, T):
    w = inputs.make_workload("bw-T", B=2, Hq=2, Hkv=1, T=T, G=4, dtype="f32", seed=570 + T)
    dY = dY_for(w, 11, "f32")
    got = run_backward(oal, w, dY)
    want = oracle.backward(w.Q, w.K, w.V, w.L, w.group, w.eps, dY)
    for name, g, r in zip(("dQ", "dK", "dV", "dL"), got, want):
        # (T = 1: g = dY . (v_0 - y_0) / D = 0 up to rounding, so dQ and dK
        # are zero; the scale of the inputs bounds the error instead)
        scale = max(np.linalg.norm(r), 1.0)
        assert np.linalg.norm(g - r) / scale <= TOL, name


def test_backward_empty_sequence_zeroes_dL(oal):
    w = inputs.make_workload("bw-0", B=1, Hq=2, Hkv=1, T=4, G=2, dtype="f32", seed=580)
    Q, K, V = (t[:, :, :0].contiguous() for t in w.torch_inputs("cuda"))
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    dL = torch.full((2, 3, 3), 5.0, device="cuda")
    oal.oal_prefill_backward(Q, K, V, Q.clone(), L, group, w.eps, dL=dL)
    oal.oal_sync_status()
    assert torch.all(dL == 0)


def test_backward_qwen_shape_directional_derivatives(oal):
    """T = 4096, Hq = 14, Hkv = 2, G = 4 (fp32 inputs): the gradients against
    central differences of the fp64 oracle forward along random directions."""
    w = inputs.config(1, dtype="f32")
    rng = np.random.default_rng(33)
    dY = rng.standard_normal(w.Q.shape).astype(np.float32)
    dQ, dK, dV, dL = (g.astype(np.float64) for g in run_backward(oal, w, dY))

    def f(Q, K, V, L):
        return float(np.sum(oracle.direct(Q, K, V, L, w.group, w.eps) * dY))

    Q, K, V, L = (x.astype(np.float64) for x in (w.Q, w.K, w.V, w.L))
    dq, dk, dv = (rng.standard_normal(x.shape) for x in (Q, K, V))
    h = 1e-3
    fd = (f(Q + h * dq, K + h * dk, V + h * dv, L) - f(Q - h * dq, K - h * dk, V - h * dv, L)) / (2 * h)
    got = float(np.sum(dQ * dq) + np.sum(dK * dk) + np.sum(dV * dv))
    assert abs(got - fd) <= 1e-3 * abs(fd), (got, fd)
    dl = np.tril(rng.standard_normal(L.shape))
    fd = (f(Q, K, V, L + h * dl) - f(Q, K, V, L - h * dl)) / (2 * h)
    got = float(np.sum(dL * dl))
    assert abs(got - fd) <= 1e-3 * abs(fd), (got, fd)
