"""ctypes binding of liboal.so (include/oal.h), same entry-point names.

Argument marshalling only: every step of OAL runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library is missing or fails to load, every call raises ``OALError`` -- there
is no CPU fallback.

Tensor layouts (row-major, contiguous, CUDA):
  Q [B,Hq,T,64], K/V [B,Hkv,T,64] (float32 or bfloat16)
  L [Hq,G+1,G+1] float32 (lower triangle), group [Hq,64] int32 in 1..G
  state [B,Hkv,F,65] float32 (F = 4161 FULL, 2145 PACKED)
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboal.so")

OAL_OK, OAL_ERR_INVALID_ARG, OAL_ERR_UNSUPPORTED, OAL_ERR_CUDA, OAL_ERR_TIMEOUT = range(5)
OAL_F32, OAL_BF16 = 0, 1
OAL_STATE_FULL, OAL_STATE_PACKED = 0, 1
_STATUS_NAMES = {0: "OAL_OK", 1: "OAL_ERR_INVALID_ARG", 2: "OAL_ERR_UNSUPPORTED",
                 3: "OAL_ERR_CUDA", 4: "OAL_ERR_TIMEOUT"}


class OALError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, status), msg))
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load liboal.so (raises OALError if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OALError(OAL_ERR_CUDA, "liboal.so not found at %s; run "
                       "`python -m grouped_quadratic_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    vp, sz, ci, cf = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    lib.oal_state_rows.argtypes = [ci, ci]
    lib.oal_state_rows.restype = sz
    lib.oal_state_elems.argtypes = [ci, ci, ci]
    lib.oal_state_elems.restype = sz
    lib.oal_coeff_table_elems.argtypes = [ci, ci]
    lib.oal_coeff_table_elems.restype = sz
    lib.oal_expand_coeffs.argtypes = [vp, vp, ci, ci, ci, cf, ci, vp, vp, vp, vp]
    lib.oal_expand_coeffs.restype = ci
    lib.oal_prefill_workspace_bytes.argtypes = [ci] * 6 + [ci, ci, ci]
    lib.oal_prefill_workspace_bytes.restype = sz
    lib.oal_prefill.argtypes = ([vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp, vp, ci, cf,
                                 vp, vp, vp, ci, vp, ci, vp, ci, vp, sz, vp])
    lib.oal_prefill.restype = ci
    lib.oal_prefill_noalloc.argtypes = ([vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp, vp, ci,
                                         cf, vp, vp, vp, ci, vp, ci, vp, ci, vp])
    lib.oal_prefill_noalloc.restype = ci
    lib.oal_prefill_backward_workspace_bytes.argtypes = [ci] * 6
    lib.oal_prefill_backward_workspace_bytes.restype = sz
    lib.oal_prefill_backward.argtypes = ([vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp, vp, ci,
                                          cf, vp, vp, vp, vp, vp, sz, vp])
    lib.oal_prefill_backward.restype = ci
    lib.oal_decode_workspace_bytes.argtypes = [ci] * 5 + [ci]
    lib.oal_decode_workspace_bytes.restype = sz
    lib.oal_decode_step.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, ci,
                                    vp, vp, vp, sz, vp]
    lib.oal_decode_step.restype = ci
    lib.oal_contribution_workspace_bytes.argtypes = [ci] * 5
    lib.oal_contribution_workspace_bytes.restype = sz
    lib.oal_contribution_scores.argtypes = [vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, sz, vp]
    lib.oal_contribution_scores.restype = ci
    cd = ctypes.c_double
    lib.oal_group_dims.argtypes = [vp, ci, ci, vp, ci, cd, cd, cd, ci, cd, vp, vp]
    lib.oal_group_dims.restype = ci
    lib.oal_sync_status.argtypes = [vp]
    lib.oal_sync_status.restype = ci
    lib.oal_debug_wait_test.argtypes = [ctypes.c_uint64, ci]
    lib.oal_debug_wait_test.restype = ci
    lib.oal_debug_intra_heads.argtypes = [ci]
    lib.oal_debug_intra_heads.restype = ci
    lib.oal_prefill_noalloc_scratch_bytes.argtypes = []
    lib.oal_prefill_noalloc_scratch_bytes.restype = sz
    lib.oal_last_error.argtypes = []
    lib.oal_last_error.restype = ctypes.c_char_p
    lib.oal_version.argtypes = []
    lib.oal_version.restype = ctypes.c_char_p
    lib.oal_launch_counter.argtypes = []
    lib.oal_launch_counter.restype = ctypes.c_uint64
    lib.oal_set_launch_events.argtypes = [vp, ci]
    lib.oal_set_launch_events.restype = ci
    lib.oal_last_call_launches.argtypes = []
    lib.oal_last_call_launches.restype = ci
    lib.oal_last_call_launch_name.argtypes = [ci]
    lib.oal_last_call_launch_name.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status):
    if status != OAL_OK:
        raise OALError(status, _lib.oal_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return OAL_F32
    if t.dtype == torch.bfloat16:
        return OAL_BF16
    raise OALError(OAL_ERR_INVALID_ARG, "unsupported dtype %s" % t.dtype)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise OALError(OAL_ERR_INVALID_ARG, "tensors must be contiguous CUDA tensors")


def oal_version():
    return load_library().oal_version().decode()


def oal_state_rows(d=64, layout=OAL_STATE_FULL):
    return int(load_library().oal_state_rows(d, layout))


def oal_state_elems(d=64, dv=64, layout=OAL_STATE_FULL):
    return int(load_library().oal_state_elems(d, dv, layout))


def oal_coeff_table_elems(d=64, layout=OAL_STATE_FULL):
    return int(load_library().oal_coeff_table_elems(d, layout))


def oal_expand_coeffs(L, group, eps, layout=OAL_STATE_FULL, a=None, b=None, C=None,
                      stream=None):
    """Coefficient tables (a [Hq], b [Hq,64], C [Hq, 4096 or 2080]) on the device."""
    lib = load_library()
    Hq, G1, _ = L.shape
    d = group.shape[1]
    dev = L.device
    if a is None:
        a = torch.empty(Hq, dtype=torch.float32, device=dev)
    if b is None:
        b = torch.empty(Hq, d, dtype=torch.float32, device=dev)
    if C is None:
        C = torch.empty(Hq, lib.oal_coeff_table_elems(d, layout), dtype=torch.float32,
                        device=dev)
    _need_cuda(L, group, a, b, C)
    _check(lib.oal_expand_coeffs(_ptr(L), _ptr(group), Hq, G1 - 1, d, float(eps), layout,
                                 _ptr(a), _ptr(b), _ptr(C), _stream(stream)))
    return a, b, C


def oal_prefill_workspace_bytes(B, Hq, Hkv, T, d=64, dv=64, dtype=OAL_BF16,
                                layout=OAL_STATE_FULL, chunk=0):
    return int(load_library().oal_prefill_workspace_bytes(B, Hq, Hkv, T, d, dv, dtype,
                                                          layout, chunk))


def oal_prefill(Q, K, V, L, group, eps, a, b, C, layout=OAL_STATE_FULL, state=None,
                continue_from_state=False, Y=None, chunk=0, workspace=None, stream=None):
    """Causal OAL prefill.  Returns (Y, state)."""
    lib = load_library()
    B, Hq, T, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    G = L.shape[1] - 1
    dt = _dtype_code(Q)
    dev = Q.device
    if state is None:
        state = torch.empty(B, Hkv, lib.oal_state_rows(d, layout), dv + 1,
                            dtype=torch.float32, device=dev)
    if Y is None:
        Y = torch.empty(B, Hq, T, dv, dtype=Q.dtype, device=dev)
    need = lib.oal_prefill_workspace_bytes(B, Hq, Hkv, T, d, dv, dt, layout, chunk)
    if workspace is None:
        workspace = torch.empty(max(int(need), 256), dtype=torch.uint8, device=dev)
    _need_cuda(Q, K, V, L, group, a, b, C, state, Y, workspace)
    _check(lib.oal_prefill(_ptr(Q), _ptr(K), _ptr(V), dt, B, Hq, Hkv, T, d, dv, _ptr(L),
                           _ptr(group), G, float(eps), _ptr(a), _ptr(b), _ptr(C), layout,
                           _ptr(state), int(bool(continue_from_state)), _ptr(Y), chunk,
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream)))
    return Y, state


def oal_prefill_noalloc_scratch_bytes():
    """Size of the library's fixed prefill scratch array, read from the library."""
    return int(load_library().oal_prefill_noalloc_scratch_bytes())


def oal_prefill_noalloc(Q, K, V, L, group, eps, a, b, C, state, Y, layout=OAL_STATE_FULL,
                        continue_from_state=False, chunk=0, stream=None):
    """oal_prefill with the library's fixed scratch instead of a workspace.

    For callers that cannot allocate device memory: `state` and `Y` must be
    passed in, and this wrapper allocates nothing either.  Problems whose
    workspace would exceed oal_prefill_noalloc_scratch_bytes() are rejected.
    """
    lib = load_library()
    B, Hq, T, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    G = L.shape[1] - 1
    _need_cuda(Q, K, V, L, group, a, b, C, state, Y)
    _check(lib.oal_prefill_noalloc(_ptr(Q), _ptr(K), _ptr(V), _dtype_code(Q), B, Hq, Hkv, T,
                                   d, dv, _ptr(L), _ptr(group), G, float(eps), _ptr(a),
                                   _ptr(b), _ptr(C), layout, _ptr(state),
                                   int(bool(continue_from_state)), _ptr(Y), chunk,
                                   _stream(stream)))
    return Y, state


def oal_prefill_backward_workspace_bytes(B, Hq, Hkv, T, d=64, dv=64):
    return int(load_library().oal_prefill_backward_workspace_bytes(B, Hq, Hkv, T, d, dv))


def oal_prefill_backward(Q, K, V, dY, L, group, eps, dQ=None, dK=None, dV=None, dL=None,
                         workspace=None, stream=None):
    """Gradients of <dY, Y> for Y = oal_prefill(Q, K, V, L, group, eps).
    Returns (dQ, dK, dV, dL), fp32."""
    lib = load_library()
    B, Hq, T, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    G = L.shape[1] - 1
    dev = Q.device
    f32 = torch.float32
    dQ = torch.empty(B, Hq, T, d, dtype=f32, device=dev) if dQ is None else dQ
    dK = torch.empty(B, Hkv, T, d, dtype=f32, device=dev) if dK is None else dK
    dV = torch.empty(B, Hkv, T, dv, dtype=f32, device=dev) if dV is None else dV
    dL = torch.empty(Hq, G + 1, G + 1, dtype=f32, device=dev) if dL is None else dL
    if workspace is None:
        need = lib.oal_prefill_backward_workspace_bytes(B, Hq, Hkv, T, d, dv)
        workspace = torch.empty(max(int(need), 256), dtype=torch.uint8, device=dev)
    if dY.dtype != Q.dtype:
        raise OALError(OAL_ERR_INVALID_ARG, "dY must have the dtype of Q")
    _need_cuda(Q, K, V, dY, L, group, dQ, dK, dV, dL, workspace)
    _check(lib.oal_prefill_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dY), _dtype_code(Q), B, Hq,
                                    Hkv, T, d, dv, _ptr(L), _ptr(group), G, float(eps), _ptr(dQ),
                                    _ptr(dK), _ptr(dV), _ptr(dL), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream)))
    return dQ, dK, dV, dL


def oal_decode_workspace_bytes(B, Hq, Hkv, d=64, dv=64, layout=OAL_STATE_FULL):
    return int(load_library().oal_decode_workspace_bytes(B, Hq, Hkv, d, dv, layout))


def oal_decode_step(q, k, v, a, b, C, state, layout=OAL_STATE_FULL, y=None,
                    workspace=None, stream=None):
    """One decode token for all sequences: q [B,Hq,64], k/v [B,Hkv,64]. Returns y."""
    lib = load_library()
    B, Hq, d = q.shape
    Hkv, dv = k.shape[1], v.shape[2]
    dt = _dtype_code(q)
    if y is None:
        y = torch.empty(B, Hq, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        need = lib.oal_decode_workspace_bytes(B, Hq, Hkv, d, dv, layout)
        workspace = torch.empty(max(int(need), 256), dtype=torch.uint8, device=q.device)
    _need_cuda(q, k, v, a, b, C, state, y, workspace)
    _check(lib.oal_decode_step(_ptr(q), _ptr(k), _ptr(v), dt, B, Hq, Hkv, d, dv, _ptr(a),
                               _ptr(b), _ptr(C), layout, _ptr(state), _ptr(y),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream)))
    return y


def oal_contribution_workspace_bytes(P, Hq, Hkv, T, d=64):
    return int(load_library().oal_contribution_workspace_bytes(P, Hq, Hkv, T, d))


def oal_contribution_scores(Q, K, lengths=None, chi=None, workspace=None, stream=None):
    """Per-prompt contribution scores: Q [P,Hq,T,64], K [P,Hkv,T,64], lengths
    [P] int32 (CUDA) or None for T tokens each.  Returns chi [P,Hq,64] float32."""
    lib = load_library()
    P, Hq, T, d = Q.shape
    Hkv = K.shape[1]
    if chi is None:
        chi = torch.empty(P, Hq, d, dtype=torch.float32, device=Q.device)
    if workspace is None:
        need = lib.oal_contribution_workspace_bytes(P, Hq, Hkv, T, d)
        workspace = torch.empty(max(int(need), 256), dtype=torch.uint8, device=Q.device)
    _need_cuda(Q, K, lengths, chi, workspace)
    _check(lib.oal_contribution_scores(_ptr(Q), _ptr(K), _dtype_code(Q), P, Hq, Hkv, T, d,
                                       _ptr(lengths), _ptr(chi), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
    return chi


def oal_group_dims(chi_p, boot_idx, alpha, tau, gamma, g_min, eps=1e-12):
    """Dimension groups of one query head (host arrays, no GPU): chi_p [P, d]
    per-prompt scores, boot_idx [nboot, P] bootstrap prompt indices.
    Returns (group [d] int32 in 1..G, G)."""
    import numpy as np
    lib = load_library()
    chi_p = np.ascontiguousarray(np.asarray(chi_p, dtype=np.float32))
    boot_idx = np.ascontiguousarray(np.asarray(boot_idx, dtype=np.int32))
    if chi_p.ndim != 2 or boot_idx.ndim != 2 or boot_idx.shape[1] != chi_p.shape[0]:
        raise OALError(OAL_ERR_INVALID_ARG, "chi_p must be [P, d] and boot_idx [nboot, P]")
    P, d = chi_p.shape
    group = np.zeros(d, np.int32)
    G = ctypes.c_int(0)
    _check(lib.oal_group_dims(chi_p.ctypes.data, P, d, boot_idx.ctypes.data, boot_idx.shape[0],
                              float(alpha), float(tau), float(gamma), int(g_min), float(eps),
                              group.ctypes.data, ctypes.byref(G)))
    return group, G.value


def oal_sync_status(stream=None):
    lib = load_library()
    _check(lib.oal_sync_status(_stream(stream)))


def oal_debug_wait_test(wait_limit_cycles=0, starve=0):
    """Test-only: the limit of the kernels' bounded waits in SM cycles (0: the
    built-in limit) and the prefill kernel whose UMMA issuer waits on a barrier
    nothing arrives on (0 none, 1 readout, 2 state, 3 intra-chunk), for kernels
    launched afterwards on the current device.  (0, 0) restores normal operation."""
    _check(load_library().oal_debug_wait_test(int(wait_limit_cycles), int(starve)))


def oal_debug_intra_heads(heads=0):
    """Test-only: query heads per block of the bf16 prefill's intra-chunk kernel
    at chunk sizes 64 and 128 (1 or 2; 0 restores the automatic choice)."""
    _check(load_library().oal_debug_intra_heads(int(heads)))


def oal_last_error():
    return load_library().oal_last_error().decode()
