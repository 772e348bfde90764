"""oal_prefill_noalloc against oal_prefill, through the C ABI.

oal_prefill_noalloc serves callers that cannot allocate device memory when
they run a prefill (a host framework that owns all device memory, a runtime
that forbids allocation after start-up): it uses the library's own fixed
scratch array instead of a caller workspace.  Each check first fills that
array with NaN (a call on all-NaN inputs), then runs calls in a row with
different inputs, sizes and chunk sizes, so a result that leaned on what an
earlier call left in the shared array would show up, and compares each with
oal_prefill on the same inputs at the parity tolerances of the other GPU
tests (rel-L2 2e-2 for bf16 outputs, 1e-5 for fp32 outputs and for states).

The file sorts last so that a run stopping at its first failure has already
run every other test; it also passes when run alone.
"""
import numpy as np
import pytest
import torch

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


def both_ways(oal, w, layout, chunk=0):
    Q, K, V = w.torch_inputs("cuda")
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, layout)
    Y_ref, S_ref = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout, chunk=chunk)
    oal.oal_sync_status()
    # caller-owned outputs, filled with garbage so that unwritten entries show
    S = torch.full_like(S_ref, float("nan"))
    Y = torch.full_like(Y_ref, float("nan"))
    oal.oal_prefill_noalloc(Q, K, V, L, group, w.eps, a, b, C, S, Y, layout, chunk=chunk)
    oal.oal_sync_status()
    return (Y.float().cpu().numpy(), S.cpu().numpy(),
            Y_ref.float().cpu().numpy(), S_ref.cpu().numpy())


def poison_scratch(oal):
    """One call whose inputs are all NaN: every scratch byte it writes holds
    NaN afterwards (its outputs are ignored), so a later call that read
    scratch it had not written first would produce non-finite or wrong values.
    Its second half uses the fp32 kernels, whose scratch layout differs."""
    for dtype in ("bf16", "f32"):
        w = inputs.make_workload("noalloc-poison", B=2, Hq=8, Hkv=2, T=520, G=4, seed=70,
                                 dtype=dtype)
        Q, K, V = (torch.full_like(t, float("nan")) for t in w.torch_inputs("cuda"))
        L = torch.from_numpy(w.L).cuda()
        group = torch.from_numpy(w.group).cuda()
        a, b, C = oal.oal_expand_coeffs(L, group, w.eps, PACKED)
        S = torch.zeros(w.B, w.Hkv, oal.oal_state_rows(64, PACKED), 65, device="cuda")
        Y = torch.empty_like(Q)
        oal.oal_prefill_noalloc(Q, K, V, L, group, w.eps, a, b, C, S, Y, PACKED,
                                chunk=64 if dtype == "f32" else 0)
        oal.oal_sync_status()


@pytest.mark.parametrize("dtype,layout,chunk", [("bf16", PACKED, 0), ("f32", FULL, 0),
                                                ("f32", PACKED, 256), ("bf16", PACKED, 64)])
def test_noalloc_matches_prefill_on_two_calls(oal, dtype, layout, chunk):
    poison_scratch(oal)
    first = inputs.make_workload("noalloc-a", B=2, Hq=8, Hkv=2, T=333, G=4, seed=71,
                                 dtype=dtype)
    second = inputs.make_workload("noalloc-b", B=1, Hq=4, Hkv=1, T=200, G=3, seed=72,
                                  dtype=dtype)
    for w in (first, second):
        Y, S, Y_ref, S_ref = both_ways(oal, w, layout, chunk)
        assert np.isfinite(Y).all() and np.isfinite(S).all()
        assert rel_l2(Y, Y_ref) <= TOL[dtype]
        assert rel_l2(S, S_ref) <= 1e-5


def test_noalloc_continuation_matches_prefill(oal):
    """A prefill in two calls, the second continuing from the first's state."""
    poison_scratch(oal)
    w = inputs.make_workload("noalloc-cont", B=2, Hq=4, Hkv=2, T=300, G=3, seed=73)
    Q, K, V = w.torch_inputs("cuda")
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, PACKED)
    T1 = 170
    parts = [(t[:, :, :T1].contiguous(), t[:, :, T1:].contiguous()) for t in (Q, K, V)]
    Y_ref, S_ref = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, PACKED)
    S = torch.zeros_like(S_ref)
    Y1 = torch.empty_like(parts[0][0])
    Y2 = torch.empty_like(parts[0][1])
    oal.oal_prefill_noalloc(parts[0][0], parts[1][0], parts[2][0], L, group, w.eps, a, b, C,
                            S, Y1, PACKED)
    oal.oal_prefill_noalloc(parts[0][1], parts[1][1], parts[2][1], L, group, w.eps, a, b, C,
                            S, Y2, PACKED, continue_from_state=True)
    oal.oal_sync_status()
    got = torch.cat([Y1, Y2], 2).float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, Y_ref.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_l2(S.cpu().numpy(), S_ref.cpu().numpy()) <= 1e-5


def test_noalloc_rejects_problems_above_its_scratch(oal):
    B, Hq, Hkv = 1, 14, 2
    # the shortest sequence whose scratch need is above the fixed array
    T = 128
    while oal.oal_prefill_workspace_bytes(B, Hq, Hkv, T, dtype=oal.OAL_BF16,
                                          layout=PACKED) <= oal.oal_prefill_noalloc_scratch_bytes():
        T += 128
    need = oal.oal_prefill_workspace_bytes(B, Hq, Hkv, T, dtype=oal.OAL_BF16, layout=PACKED)
    z = lambda *shape, dt=torch.bfloat16: torch.zeros(*shape, dtype=dt, device="cuda")
    Q, K, V = z(B, Hq, T, 64), z(B, Hkv, T, 64), z(B, Hkv, T, 64)
    L = torch.eye(5, dtype=torch.float32, device="cuda")[None].repeat(Hq, 1, 1)
    group = torch.ones(Hq, 64, dtype=torch.int32, device="cuda")
    a, b, C = oal.oal_expand_coeffs(L, group, 1.0, PACKED)
    S = z(B, Hkv, oal.oal_state_rows(64, PACKED), 65, dt=torch.float32)
    Y = z(B, Hq, T, 64)
    with pytest.raises(oal.OALError) as e:
        oal.oal_prefill_noalloc(Q, K, V, L, group, 1.0, a, b, C, S, Y, PACKED)
    assert e.value.status == oal.OAL_ERR_INVALID_ARG
    assert str(need) in str(e.value)
