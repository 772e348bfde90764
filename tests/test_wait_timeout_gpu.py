"""The failure path of the bounded waits, on the GPU, without a fault.

Every mbarrier wait in the library's kernels gives up after a limit: the
block raises its abort flag, records OAL_ERR_TIMEOUT in the device status
word, drains the copies and tensor-core products it has in flight, frees its
tensor memory and returns.  Here the UMMA issuer of one prefill kernel
(readout, state or intra-chunk) is made to wait on a barrier that nothing
arrives on, with a short limit (2^22 cycles, about 2 ms), so its wait runs
out while the block's other warps are mid-pipeline.  The call must end, the
status must read OAL_ERR_TIMEOUT, and the next ordinary call on the same
context must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_quadratic_gb300 import inputs

pytestmark = pytest.mark.gpu

PACKED = 1


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


@pytest.mark.parametrize("starve,name", [(1, "readout"), (2, "state"), (3, "intra")])
def test_starved_wait_times_out_and_the_context_stays_usable(oal, starve, name):
    w = inputs.make_workload("timeout", B=1, Hq=4, Hkv=2, T=300, G=3, seed=90)
    Q, K, V = w.torch_inputs("cuda")
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, PACKED)
    oal.oal_sync_status()
    oal.oal_debug_wait_test(1 << 22, starve)
    try:
        oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, PACKED)
        with pytest.raises(oal.OALError) as e:
            oal.oal_sync_status()
        assert e.value.status == oal.OAL_ERR_TIMEOUT, name
    finally:
        oal.oal_debug_wait_test(0, 0)
    oal.oal_sync_status()   # the status word was cleared
    Y, _ = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, PACKED)
    oal.oal_sync_status()
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(Y.float().cpu().numpy(), want) <= 2e-2
