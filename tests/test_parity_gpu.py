"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Tolerances (rel-L2 over the whole output tensor): 1e-5 for fp32 inputs,
2e-2 for bf16 inputs with fp32 states; coefficient tables bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_quadratic_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
FULL, PACKED = 0, 1


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


def dev_params(oal, w, layout):
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, layout)
    return L, group, a, b, C


def run_prefill(oal, w, layout=FULL, chunk=0, T=None):
    T = w.T if T is None else T
    Q, K, V = (t[:, :, :T].contiguous() for t in w.torch_inputs("cuda"))
    L, group, a, b, C = dev_params(oal, w, layout)
    Y, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout, chunk=chunk)
    oal.oal_sync_status()
    return Y.float().cpu().numpy(), S.cpu().numpy()


# ---------------------------------------------------------------- coefficients
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("layout", [FULL, PACKED])
def test_expand_coeffs_bit_exact(oal, cfg, layout):
    w = inputs.config(cfg, T=8) if cfg else inputs.config(0)
    _, _, a, b, C = dev_params(oal, w, layout)
    ra, rb, rC = oracle.expand_coeffs(w.L, w.group, w.eps, packed=layout == PACKED)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ra.view(np.uint32))
    assert np.array_equal(b.cpu().numpy().view(np.uint32), rb.view(np.uint32))
    assert np.array_equal(C.cpu().numpy().view(np.uint32), rC.view(np.uint32))


def test_bad_group_reported_by_status(oal):
    w = inputs.config(0)
    L = torch.from_numpy(w.L).cuda()
    g = w.group.copy()
    g[0, 5] = 9
    with pytest.raises(oal.OALError) as e:
        oal.oal_expand_coeffs(L, torch.from_numpy(g).cuda(), w.eps)
        oal.oal_sync_status()
    assert e.value.status == oal.OAL_ERR_INVALID_ARG
    oal.oal_sync_status()  # cleared


# ---------------------------------------------------------------- prefill, fp32
@pytest.mark.parametrize("layout", [FULL, PACKED])
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_prefill_fp32_tiny_config(oal, layout, chunk):
    w = inputs.config(0)
    Y, S = run_prefill(oal, w, layout, chunk)
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(Y, want) <= TOL["f32"]
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    if layout == PACKED:
        S_ref = oracle.full_to_packed_state(S_ref, 64)
    assert rel_l2(S, S_ref) <= 1e-6


@pytest.mark.parametrize("T", [1, 2, 63, 65, 200])
def test_prefill_fp32_ragged(oal, T):
    w = inputs.make_workload("ragged", B=2, Hq=4, Hkv=2, T=T, G=3, dtype="f32", seed=31 + T)
    Y, _ = run_prefill(oal, w, PACKED, 64)
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(Y, want) <= TOL["f32"]


# ---------------------------------------------------------------- prefill, bf16
@pytest.mark.parametrize("layout", [FULL, PACKED])
def test_prefill_bf16_gqa_ragged(oal, layout):
    w = inputs.make_workload("bf16-small", B=2, Hq=14, Hkv=2, T=333, G=4, seed=77)
    Y, S = run_prefill(oal, w, layout)
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(Y, want) <= TOL["bf16"]
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    if layout == PACKED:
        S_ref = oracle.full_to_packed_state(S_ref, 64)
    assert rel_l2(S, S_ref) <= 1e-5


def sampled_rows(w, n_first=64, n_rand=64, n_last=16, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        for h in range(w.Hq):
            base = (b * w.Hq + h) * w.T
            idx = np.unique(np.concatenate([
                np.arange(min(n_first, w.T)), rng.integers(0, w.T, n_rand),
                np.arange(max(0, w.T - n_last), w.T)]))
            rows.append(base + idx)
    return np.concatenate(rows)


@pytest.mark.parametrize("cfg,layout,chunk", [(1, FULL, 0), (1, PACKED, 0), (2, PACKED, 0),
                                              (4, PACKED, 0), (4, PACKED, 64),
                                              (4, PACKED, 256)])
def test_prefill_full_size_sampled(oal, cfg, layout, chunk):
    """Full-size workloads (the long-context one at every chunk size), output
    rows sampled at the start, at random and at the end of every head."""
    w = inputs.config(cfg)
    Y, _ = run_prefill(oal, w, layout, chunk)
    rows = sampled_rows(w, n_rand=32 if cfg == 2 else 64, n_last=8 if cfg == 2 else 16)
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps, rows=rows)
    got = Y.reshape(-1, w.dv)[rows]
    assert np.all(np.isfinite(Y))
    assert rel_l2(got, want) <= TOL["bf16"]


# ---------------------------------------------------------------- invariants
def test_running_mean_when_kernel_constant(oal):
    w = inputs.make_workload("const", B=2, Hq=6, Hkv=3, T=190, G=3, dtype="f32", seed=5)
    w.L[:] = 0
    w.L[:, 0, 0] = 0.9
    Y, _ = run_prefill(oal, w, PACKED)
    V = w.V.astype(np.float64)
    mean = np.cumsum(V, axis=2) / np.arange(1, w.T + 1)[None, None, :, None]
    want = np.repeat(mean, 2, axis=1)
    assert rel_l2(Y, want) <= TOL["f32"]


def test_affine_equivariance_in_v(oal):
    w = inputs.make_workload("affine", B=1, Hq=4, Hkv=2, T=150, G=4, dtype="f32", seed=8)
    Y1, _ = run_prefill(oal, w)
    w.V = (2.0 * w.V + 0.5).astype(np.float32)
    Y2, _ = run_prefill(oal, w)
    assert rel_l2(Y2, 2.0 * Y1 + 0.5) <= 1e-5


def test_packed_equals_full_and_chunk_invariance(oal):
    w = inputs.make_workload("inv", B=1, Hq=4, Hkv=1, T=300, G=4, seed=12)
    ref, _ = run_prefill(oal, w, FULL, 64)
    for layout, chunk in [(PACKED, 64), (FULL, 128), (PACKED, 256)]:
        Y, _ = run_prefill(oal, w, layout, chunk)
        assert rel_l2(Y, ref) <= 1e-2


def test_prefill_continuation(oal):
    w = inputs.make_workload("cont", B=2, Hq=4, Hkv=2, T=260, G=3, dtype="f32", seed=21)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = dev_params(oal, w, PACKED)
    T1 = 131
    Y1, S = oal.oal_prefill(Q[:, :, :T1].contiguous(), K[:, :, :T1].contiguous(),
                            V[:, :, :T1].contiguous(), L, group, w.eps, a, b, C, PACKED)
    Y2, S = oal.oal_prefill(Q[:, :, T1:].contiguous(), K[:, :, T1:].contiguous(),
                            V[:, :, T1:].contiguous(), L, group, w.eps, a, b, C, PACKED,
                            state=S, continue_from_state=True)
    oal.oal_sync_status()
    got = torch.cat([Y1, Y2], 2).cpu().numpy()
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(got, want) <= TOL["f32"]


def test_empty_inputs(oal):
    w = inputs.make_workload("empty", B=1, Hq=2, Hkv=1, T=4, G=2, dtype="f32", seed=3)
    Q, K, V = (t[:, :, :0].contiguous() for t in w.torch_inputs("cuda"))
    L, group, a, b, C = dev_params(oal, w, FULL)
    S = torch.full((1, 1, 4161, 65), 7.0, device="cuda")
    _, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, FULL, state=S,
                           continue_from_state=True)
    oal.oal_sync_status()
    assert torch.all(S == 7.0)
    _, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, FULL, state=S)
    oal.oal_sync_status()
    assert torch.all(S == 0.0)


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("layout,dtype", [(FULL, "f32"), (PACKED, "f32"), (FULL, "bf16"),
                                          (PACKED, "bf16")])
def test_decode_matches_oracle(oal, layout, dtype):
    w = inputs.make_workload("dec", B=3, Hq=14, Hkv=2, T=100 + 6, G=4, dtype=dtype,
                             seed=40, decode_steps=6)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = dev_params(oal, w, layout)
    Tp = w.T_prefill
    Y, S = oal.oal_prefill(Q[:, :, :Tp].contiguous(), K[:, :, :Tp].contiguous(),
                           V[:, :, :Tp].contiguous(), L, group, w.eps, a, b, C, layout)
    ys = [oal.oal_decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(),
                              V[:, :, t].contiguous(), a, b, C, S, layout)
          for t in range(Tp, w.T)]
    oal.oal_sync_status()
    got = torch.stack(ys, 2).float().cpu().numpy()
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)[:, :, Tp:]
    assert rel_l2(got, want) <= TOL[dtype]
    # the state after decoding equals the oracle's recurrence over all tokens
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    if layout == PACKED:
        S_ref = oracle.full_to_packed_state(S_ref, 64)
    assert rel_l2(S.cpu().numpy(), S_ref) <= 1e-5


def test_decode_equals_longer_prefill(oal):
    w = inputs.make_workload("dec2", B=2, Hq=4, Hkv=2, T=70, G=3, dtype="f32", seed=41)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = dev_params(oal, w, FULL)
    Yfull, Sfull = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, FULL)
    _, S = oal.oal_prefill(Q[:, :, :67].contiguous(), K[:, :, :67].contiguous(),
                           V[:, :, :67].contiguous(), L, group, w.eps, a, b, C, FULL)
    ys = [oal.oal_decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(),
                              V[:, :, t].contiguous(), a, b, C, S, FULL) for t in range(67, 70)]
    oal.oal_sync_status()
    got = torch.stack(ys, 2).cpu().numpy()
    assert rel_l2(got, Yfull[:, :, 67:].cpu().numpy()) <= 1e-5
    assert rel_l2(S.cpu().numpy(), Sfull.cpu().numpy()) <= 1e-6


def test_decode_config3_all_steps(oal):
    """Decode workload (B=64, Hq=14, Hkv=2, G=4, full fp32 state): a 2048-token
    prefill, then all 1024 decode steps.  Every step's output of 8 of the 64
    sequences (all 14 heads) is compared with the oracle's direct sum over
    all tokens up to that step, and the states of those sequences after the
    last step with the oracle's recurrence over all 3072 tokens, so drift in
    the long fp32 accumulation would show."""
    w = inputs.config(3)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = dev_params(oal, w, FULL)
    Tp, steps = w.T_prefill, w.decode_steps
    _, S = oal.oal_prefill(Q[:, :, :Tp].contiguous(), K[:, :, :Tp].contiguous(),
                           V[:, :, :Tp].contiguous(), L, group, w.eps, a, b, C, FULL)
    qd, kd, vd = (t[:, :, Tp:].permute(2, 0, 1, 3).contiguous() for t in (Q, K, V))
    del Q, K, V
    y = torch.empty(steps, w.B, w.Hq, 64, dtype=qd.dtype, device="cuda")
    ws = torch.empty(oal.oal_decode_workspace_bytes(w.B, w.Hq, w.Hkv, layout=FULL),
                     dtype=torch.uint8, device="cuda")
    for t in range(steps):
        oal.oal_decode_step(qd[t], kd[t], vd[t], a, b, C, S, FULL, y=y[t], workspace=ws)
    oal.oal_sync_status()
    got = y.float().permute(1, 2, 0, 3).cpu().numpy()           # [B, Hq, steps, 64]
    bsel = np.sort(np.random.default_rng(2).choice(w.B, 8, replace=False))
    rows = np.concatenate([((b * w.Hq + h) * w.T + Tp + np.arange(steps))
                           for b in bsel for h in range(w.Hq)])
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps, rows=rows)
    assert np.all(np.isfinite(got))
    assert rel_l2(got[bsel].reshape(-1, 64), want) <= TOL["bf16"]
    # the states depend on K and V only: one query head per KV head suffices
    rho = w.Hq // w.Hkv
    _, S_ref = oracle.recurrent(w.Q[bsel][:, ::rho], w.K[bsel], w.V[bsel], w.L[::rho],
                                w.group[::rho], w.eps)
    assert rel_l2(S.cpu().numpy()[bsel], S_ref) <= 1e-5


def test_decode_config3_sampled(oal):
    """Decode workload shape (B=64, Hq=14, Hkv=2): prefill 2048, then decode;
    the full 1024-step run is the benchmark, here 16 steps are checked."""
    w = inputs.config(3)
    steps = 16
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = dev_params(oal, w, FULL)
    Tp = w.T_prefill
    _, S = oal.oal_prefill(Q[:, :, :Tp].contiguous(), K[:, :, :Tp].contiguous(),
                           V[:, :, :Tp].contiguous(), L, group, w.eps, a, b, C, FULL)
    ys = [oal.oal_decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(),
                              V[:, :, t].contiguous(), a, b, C, S, FULL)
          for t in range(Tp, Tp + steps)]
    oal.oal_sync_status()
    got = torch.stack(ys, 2).float().cpu().numpy()            # [B, Hq, steps, 64]
    rng = np.random.default_rng(1)
    bsel = rng.choice(w.B, 6, replace=False)
    rows = np.concatenate([((b * w.Hq + h) * w.T + Tp + np.arange(steps))
                           for b in bsel for h in range(w.Hq)])
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps, rows=rows)
    assert rel_l2(got[bsel].reshape(-1, 64), want) <= TOL["bf16"]
