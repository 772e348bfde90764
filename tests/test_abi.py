"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/oal.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oal.h")


@pytest.fixture(scope="module")
def lib():
    from grouped_quadratic_gb300 import build, oal
    build.build()
    return oal.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(oal_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["oal_expand_coeffs", "oal_prefill", "oal_prefill_workspace_bytes",
                     "oal_decode_step", "oal_decode_workspace_bytes", "oal_state_rows",
                     "oal_state_elems", "oal_sync_status", "oal_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_state_sizes(lib):
    from grouped_quadratic_gb300 import oal
    assert oal.oal_state_rows(64, oal.OAL_STATE_FULL) == 4161
    assert oal.oal_state_rows(64, oal.OAL_STATE_PACKED) == 2145
    assert oal.oal_state_elems(64, 64, oal.OAL_STATE_FULL) * 4 == 1081860
    assert oal.oal_state_elems(64, 64, oal.OAL_STATE_PACKED) * 4 == 557700
    assert oal.oal_coeff_table_elems(64, oal.OAL_STATE_PACKED) == 2080
    assert oal.oal_state_rows(64, 7) == 0
    assert oal.oal_version()


def _prefill_raw(lib, **kw):
    from grouped_quadratic_gb300 import oal
    p = ctypes.c_void_p(4096)  # a fake, aligned address; never dereferenced
    args = dict(Q=p, K=p, V=p, dtype=oal.OAL_BF16, B=1, Hq=4, Hkv=2, T=8, d=64, dv=64,
                L=p, group=p, G=3, eps=1e-6, a=p, b=p, C=p, layout=oal.OAL_STATE_FULL,
                state=p, cont=0, Y=p, chunk=0, ws=p, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.oal_prefill(*args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(d=32), 2), (dict(dv=128), 2), (dict(G=0), 2), (dict(G=8), 2),
    (dict(Hq=5), 1), (dict(Hkv=0), 1), (dict(dtype=7), 1), (dict(layout=3), 1),
    (dict(chunk=96), 1), (dict(eps=0.0), 1), (dict(T=-1), 1),
    (dict(Q=ctypes.c_void_p(0)), 1), (dict(K=ctypes.c_void_p(4100)), 1),
    (dict(ws_bytes=16), 1),
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, status):
    assert _prefill_raw(lib, **kw) == status
    assert lib.oal_last_error().decode() != ""


def _contrib_raw(lib, **kw):
    from grouped_quadratic_gb300 import oal
    p = ctypes.c_void_p(4096)  # a fake, aligned address; never dereferenced
    args = dict(Q=p, K=p, dtype=oal.OAL_BF16, P=2, Hq=4, Hkv=2, T=8, d=64, lengths=None,
                chi=p, ws=p, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.oal_contribution_scores(*args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(d=32), 2), (dict(Hq=3), 1), (dict(Hkv=0), 1), (dict(dtype=5), 1), (dict(P=-1), 1),
    (dict(T=-2), 1), (dict(chi=ctypes.c_void_p(0)), 1), (dict(Q=ctypes.c_void_p(4100)), 1),
    (dict(lengths=ctypes.c_void_p(4098)), 1), (dict(ws=ctypes.c_void_p(4096 + 16)), 1),
    (dict(ws_bytes=8), 1),
])
def test_contribution_scores_reject_bad_arguments_on_host(lib, kw, status):
    assert _contrib_raw(lib, **kw) == status
    assert lib.oal_last_error().decode() != ""


def test_workspace_queries(lib):
    from grouped_quadratic_gb300 import oal
    n = oal.oal_prefill_workspace_bytes(1, 14, 2, 4096, layout=oal.OAL_STATE_PACKED)
    assert n > 0
    assert oal.oal_prefill_workspace_bytes(1, 14, 2, 4096, chunk=96) == 0
    assert oal.oal_decode_workspace_bytes(64, 14, 2) > 0
    n = oal.oal_contribution_workspace_bytes(40, 14, 2, 4096)
    assert n == 40 * 32 * 64 * 4 * (2 + 2 * 14)
    assert oal.oal_contribution_workspace_bytes(40, 14, 2, 4096, d=32) == 0


def test_intra_heads_hook_validates_on_host(lib):
    # the test hook for the intra-chunk kernel's block shape takes 0, 1 or 2
    for bad in (-1, 3):
        assert lib.oal_debug_intra_heads(bad) == 1   # OAL_ERR_INVALID_ARG
    for good in (1, 2, 0):
        assert lib.oal_debug_intra_heads(good) == 0


def test_missing_library_fails_loudly(tmp_path):
    from grouped_quadratic_gb300 import oal
    saved = oal._lib
    oal._lib = None
    try:
        with pytest.raises(oal.OALError):
            oal.load_library(str(tmp_path / "nope.so"))
    finally:
        oal._lib = saved
