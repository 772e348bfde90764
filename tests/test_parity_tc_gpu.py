"""GPU parity of the tensor-core prefill and the decode paths across shapes.

Each case runs through the C ABI and is compared with the fp64 oracle:
outputs at rel-L2 <= 2e-2 (bf16 inputs, fp32 states), states at <= 1e-5 (the
state contraction is exact up to fp32 accumulation).  The cases cover what the
Qwen/Llama-shaped workloads do not: every group count the library accepts
(G = 1 is the single global embedding) at every chunk size (64, 128, 256),
wide tail groups, readout weights without the rank-one form or with exception
words at the first and last rows (the general and the patched builder paths),
GQA ratios 1 to 8, sequences split into many parts, continuation through the
tensor-core path, lengths around every chunk and tile boundary, heads of
different group counts in one launch (empty groups), and both decode
reductions (thread-block clusters for few sequences, persistent streaming
blocks and a finishing kernel for many).
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_quadratic_gb300 import inputs

pytestmark = pytest.mark.gpu

FULL, PACKED = 0, 1
TOL_Y, TOL_S = 2e-2, 1e-5


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


def params(oal, w, layout):
    L = torch.from_numpy(w.L).cuda()
    group = torch.from_numpy(w.group).cuda()
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, layout)
    return L, group, a, b, C


def check_prefill(oal, w, layout=PACKED, chunk=128):
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = params(oal, w, layout)
    Y, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout, chunk=chunk)
    oal.oal_sync_status()
    Yh = Y.float().cpu().numpy()
    assert np.isfinite(Yh).all()
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(Yh, want) <= TOL_Y
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    if layout == PACKED:
        S_ref = oracle.full_to_packed_state(S_ref, 64)
    assert rel_l2(S.cpu().numpy(), S_ref) <= TOL_S


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7])
def test_tc_prefill_every_group_count(oal, G, chunk):
    w = inputs.make_workload("tc-G%d" % G, B=1, Hq=4, Hkv=2, T=300, G=G, seed=300 + G)
    check_prefill(oal, w, chunk=chunk)


@pytest.mark.parametrize("chunk", [64, 256])
def test_tc_prefill_wide_tail_group(oal, chunk):
    # tail group {3, 17, 40} has three dims, the bulk group is not group 1
    w = inputs.make_workload("tc-wide", B=1, Hq=4, Hkv=2, T=260, G=3, seed=311,
                             fixed_outliers=([3, 17, 40, 58], 12.0),
                             fixed_groups=[[3, 17, 40], [58]])
    w.group[w.group == 1] = 4
    w.group[w.group == 3] = 1
    w.group[w.group == 4] = 3
    check_prefill(oal, w, chunk=chunk)


@pytest.mark.parametrize("chunk", [64, 128])
def test_tc_prefill_many_tail_dims_of_two(oal, chunk):
    # five tail groups of two dims each: ten tail dims, every group within the
    # fast form but more tail dims than the tensor-core kappa has features for
    # (the intra-chunk kernel evaluates these heads from the Q and K tiles);
    # then nine (still too many) and eight (the largest tensor-core case)
    ten = [[1, 7], [12, 20], [33, 41], [47, 52], [58, 63]]
    w = inputs.make_workload("tc-10", B=1, Hq=4, Hkv=2, T=300, G=6, seed=318,
                             fixed_outliers=([7, 20, 41, 63], 9.0), fixed_groups=ten)
    check_prefill(oal, w, chunk=chunk)
    nine = [[1, 7], [12, 20], [33, 41], [47, 52], [58]]
    w = inputs.make_workload("tc-9", B=1, Hq=4, Hkv=2, T=300, G=6, seed=319,
                             fixed_outliers=([7, 20, 41, 58], 9.0), fixed_groups=nine)
    check_prefill(oal, w, chunk=chunk)
    eight = [[1, 7], [12, 20], [33, 41], [47, 52]]
    w = inputs.make_workload("tc-8", B=1, Hq=4, Hkv=2, T=300, G=5, seed=320,
                             fixed_outliers=([7, 20, 41, 52], 9.0), fixed_groups=eight)
    check_prefill(oal, w, chunk=chunk)


def run_prefill(oal, w, chunk, layout=PACKED):
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = params(oal, w, layout)
    Y, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout, chunk=chunk)
    oal.oal_sync_status()
    return Y.view(torch.int16).cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("chunk", [64, 128])
def test_tc_intra_two_heads_per_block(oal, chunk):
    # the intra-chunk kernel's blocks of two query heads (the large-grid
    # choice) forced on small cases: odd GQA ratios (a last block of one
    # head), ragged lengths, heads of one KV head with different group counts
    # (one head on the generic kappa path, its neighbour on the tensor-core
    # path; different tail dims, so the key features are rebuilt): the same
    # bits as one head a block, and the oracle's values
    cases = []
    cases.append(inputs.make_workload("tc-2h-a", B=2, Hq=6, Hkv=2, T=333, G=4, seed=330))
    cases.append(inputs.make_workload("tc-2h-b", B=1, Hq=5, Hkv=1, T=129, G=6, seed=331))
    w = inputs.make_workload("tc-2h-c", B=1, Hq=4, Hkv=1, T=260, G=4, seed=332)
    # head 1: a tail group of three dims (generic kappa); head 2: G = 1
    w.group[1] = 1
    w.group[1, [3, 17, 40]] = 2
    w.group[1, [58]] = 3
    w.group[2] = 1
    cases.append(w)
    try:
        for w in cases:
            oal.oal_debug_intra_heads(1)
            y1, s1 = run_prefill(oal, w, chunk)
            oal.oal_debug_intra_heads(2)
            y2, s2 = run_prefill(oal, w, chunk)
            assert np.array_equal(y1, y2) and np.array_equal(s1, s2)
            check_prefill(oal, w, chunk=chunk)
    finally:
        oal.oal_debug_intra_heads(0)


def test_tc_prefill_readout_general_weights(oal):
    # heads 0 and 2: the bulk row of L is zero, so M_bb = 0 and the readout
    # weights have no rank-one form; those heads take the general builder
    # path while heads 1 and 3 (same kv heads) keep the rank-one path
    w = inputs.make_workload("tc-gen", B=1, Hq=4, Hkv=2, T=290, G=4, seed=315)
    w.L[0, 1, :] = 0.0
    w.L[2, 1, :] = 0.0
    check_prefill(oal, w)
    check_prefill(oal, w, FULL)


def test_tc_prefill_readout_many_exception_words(oal):
    # a tail group of nine dims: 45 pairs inside it on both sides, more
    # exception words than the rank-one record holds (general path)
    dims = [2, 9, 17, 23, 30, 38, 44, 51, 60]
    w = inputs.make_workload("tc-exc", B=1, Hq=2, Hkv=1, T=200, G=3, seed=316,
                             fixed_outliers=(dims[:4], 10.0), fixed_groups=[dims, [63]])
    check_prefill(oal, w)


def test_tc_prefill_readout_exception_words(oal):
    # six tail dims in three groups, one of them at dim 0 and one at dim 63:
    # exception words at the first and the last paired rows
    w = inputs.make_workload("tc-exc2", B=1, Hq=4, Hkv=1, T=257, G=4, seed=317,
                             fixed_outliers=([0, 31, 32, 63], 14.0),
                             fixed_groups=[[0, 31], [32, 62], [63, 1]])
    check_prefill(oal, w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_heterogeneous_group_counts(oal, dtype):
    # heads of 1 to 5 groups in one launch: G = 5 for all, head h keeps
    # groups 1 .. 1 + h % 5 and leaves the others empty (their dims join the
    # bulk group 1); bf16 runs the tensor-core path, f32 the CUDA-core one
    w = inputs.make_workload("het", B=1, Hq=10, Hkv=2, T=300, G=5, dtype=dtype, seed=330)
    for h in range(w.Hq):
        w.group[h][w.group[h] > 1 + h % 5] = 1
    check_prefill(oal, w)
    check_prefill(oal, w, FULL)
    if dtype == "bf16":
        check_prefill(oal, w, chunk=64)
        check_prefill(oal, w, FULL, chunk=256)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 3), (8, 2), (16, 2)])
def test_tc_prefill_gqa_ratios(oal, Hq, Hkv):
    w = inputs.make_workload("tc-rho", B=2, Hq=Hq, Hkv=Hkv, T=200, G=4, seed=320 + Hq)
    check_prefill(oal, w, FULL if Hq == 6 else PACKED)


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383])
def test_tc_prefill_chunk_boundaries(oal, T, chunk):
    w = inputs.make_workload("tc-T", B=1, Hq=2, Hkv=1, T=T, G=4, seed=330 + T)
    check_prefill(oal, w, chunk=chunk)


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_tc_prefill_many_parts(oal, chunk):
    # one (batch, KV head): the state walk splits 20 stages of 128 tokens
    # into parts of 3 (C = 64, 128) or 4 (C = 256) stages
    w = inputs.make_workload("tc-parts", B=1, Hq=2, Hkv=1, T=20 * 128 - 37, G=4, seed=340)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = params(oal, w, PACKED)
    Y, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, PACKED, chunk=chunk)
    oal.oal_sync_status()
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(S.cpu().numpy(), oracle.full_to_packed_state(S_ref, 64)) <= TOL_S
    rows = np.concatenate([h * w.T + np.arange(0, w.T, 7) for h in range(w.Hq)])
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps, rows=rows)
    got = Y.float().cpu().numpy().reshape(-1, 64)[rows]
    assert rel_l2(got, want) <= TOL_Y


@pytest.mark.parametrize("layout,chunk", [(FULL, 128), (PACKED, 128), (PACKED, 64),
                                          (FULL, 256)])
def test_tc_prefill_continuation(oal, layout, chunk):
    w = inputs.make_workload("tc-cont", B=2, Hq=4, Hkv=2, T=500, G=4, seed=350)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = params(oal, w, layout)
    T1 = 200
    Y1, S = oal.oal_prefill(Q[:, :, :T1].contiguous(), K[:, :, :T1].contiguous(),
                            V[:, :, :T1].contiguous(), L, group, w.eps, a, b, C, layout,
                            chunk=chunk)
    Y2, S = oal.oal_prefill(Q[:, :, T1:].contiguous(), K[:, :, T1:].contiguous(),
                            V[:, :, T1:].contiguous(), L, group, w.eps, a, b, C, layout,
                            state=S, continue_from_state=True, chunk=chunk)
    oal.oal_sync_status()
    got = torch.cat([Y1, Y2], 2).float().cpu().numpy()
    want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)
    assert rel_l2(got, want) <= TOL_Y
    _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
    if layout == PACKED:
        S_ref = oracle.full_to_packed_state(S_ref, 64)
    assert rel_l2(S.cpu().numpy(), S_ref) <= TOL_S


@pytest.mark.parametrize("B,Hq,Hkv", [(1, 16, 2), (2, 6, 3), (16, 8, 2), (20, 4, 2),
                                      (24, 16, 2)])
def test_decode_reductions(oal, B, Hq, Hkv):
    # B * Hkv <= 19: slices meet in a thread-block cluster of 16 blocks; 32:
    # clusters of 8; 40 and 48: the
    # streaming kernel (runs of slices crossing (batch, KV head) boundaries,
    # eight query heads per KV head in the last case) and its finishing kernel
    w = inputs.make_workload("dec-red", B=B, Hq=Hq, Hkv=Hkv, T=40 + 3, G=4, seed=360 + B,
                             decode_steps=3)
    Q, K, V = w.torch_inputs("cuda")
    for layout in (FULL, PACKED):
        L, group, a, b, C = params(oal, w, layout)
        Tp = w.T_prefill
        _, S = oal.oal_prefill(Q[:, :, :Tp].contiguous(), K[:, :, :Tp].contiguous(),
                               V[:, :, :Tp].contiguous(), L, group, w.eps, a, b, C, layout)
        ys = [oal.oal_decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(),
                                  V[:, :, t].contiguous(), a, b, C, S, layout)
              for t in range(Tp, w.T)]
        oal.oal_sync_status()
        got = torch.stack(ys, 2).float().cpu().numpy()
        want = oracle.direct(w.Q, w.K, w.V, w.L, w.group, w.eps)[:, :, Tp:]
        assert rel_l2(got, want) <= TOL_Y
        _, S_ref = oracle.recurrent(w.Q, w.K, w.V, w.L, w.group, w.eps)
        if layout == PACKED:
            S_ref = oracle.full_to_packed_state(S_ref, 64)
        assert rel_l2(S.cpu().numpy(), S_ref) <= TOL_S


@pytest.mark.parametrize("layout", [FULL, PACKED])
def test_prefill_slices_equal_one_call(oal, layout):
    # every (batch, KV head) unit is independent: calls on slices of one
    # sequence and four KV heads (with their query heads, the coefficient rows
    # and the state slice) give the single call's outputs bit for bit (the
    # end-to-end pipeline of bench.py runs the prefill this way)
    w = inputs.make_workload("slices", B=2, Hq=16, Hkv=8, T=300, G=5, seed=340)
    Q, K, V = w.torch_inputs("cuda")
    L, group, a, b, C = params(oal, w, layout)
    Y, S = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout)
    Y2, S2 = torch.empty_like(Y), torch.empty_like(S)
    nk, nq = 4, 8
    for bb in range(w.B):
        for g in range(w.Hkv // nk):
            hs, ks = slice(g * nq, (g + 1) * nq), slice(g * nk, (g + 1) * nk)
            oal.oal_prefill(Q[bb:bb + 1, hs], K[bb:bb + 1, ks], V[bb:bb + 1, ks], L[hs], group[hs],
                            w.eps, a[hs], b[hs], C[hs], layout, state=S2[bb:bb + 1, ks],
                            Y=Y2[bb:bb + 1, hs])
    oal.oal_sync_status()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(S, S2)
