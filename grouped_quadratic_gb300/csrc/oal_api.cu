// oal_api.cu -- the extern "C" entry points of liboal.so (include/oal.h):
// argument validation, workspace sizing, dispatch to the kernels, error
// reporting.  No allocation happens here; all memory is the caller's.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>

#include "oal_internal.cuh"

namespace oal {
oal_status launch_expand_coeffs(const float *L, const int32_t *group, int Hq, int G,
                                float eps, int packed, float *a, float *b, float *C,
                                cudaStream_t stream);
size_t simt_prefill_workspace_bytes(int B, int Hkv, int T, int packed, int chunk);
oal_status launch_prefill_simt(const void *Q, const void *K, const void *V, int is_bf16,
                               int B, int Hq, int Hkv, int T, const float *L,
                               const int32_t *group, int G, float eps, const float *a,
                               const float *b, const float *C, int packed, float *state,
                               int cont, void *Y, int chunk, void *ws, cudaStream_t stream);
size_t tc_prefill_workspace_bytes(int B, int Hq, int Hkv, int T, int chunk);
void set_intra_heads(int heads);
oal_status launch_prefill_tc(const void *Q, const void *K, const void *V, int B, int Hq,
                             int Hkv, int T, const float *L, const int32_t *group, int G,
                             float eps, const float *a, const float *b, const float *C,
                             int packed, float *state, int cont, void *Y, int chunk, void *ws,
                             cudaStream_t stream);
size_t decode_workspace_bytes(int B, int Hkv, int packed);
int decode_max_rho();
oal_status launch_decode(const void *q, const void *k, const void *v, int is_bf16, int B,
                         int Hq, int Hkv, const float *a, const float *b, const float *C,
                         int packed, float *state, void *y, void *ws, cudaStream_t stream);

size_t backward_workspace_bytes(int B, int Hq, int Hkv, int T);
oal_status launch_backward(const void *Q, const void *K, const void *V, const void *dY, int is_bf16,
                           int B, int Hq, int Hkv, int T, const float *L, const int32_t *group,
                           int G, float eps, float *dQ, float *dK, float *dV, float *dL, void *ws,
                           cudaStream_t stream);

size_t contrib_workspace_bytes(int P, int Hq, int Hkv, int T);
oal_status launch_contrib(const void *Q, const void *K, int is_bf16, int P, int Hq, int Hkv,
                          int T, const int32_t *lengths, float *chi, void *ws,
                          cudaStream_t stream);
oal_status group_dims_host(const float *chi_p, int P, int d, const int32_t *boot_idx,
                           int nboot, double alpha, double tau, double gamma, int g_min,
                           double eps, int32_t *group, int *G);

// Device control block (one per device the library runs on): the status
// word kernels record errors in; then, for tests of the failure path, the
// kernel whose UMMA issuer is to wait on a barrier nothing arrives on
// (0 = none), and the limit of the bounded waits in SM cycles (0 = the
// built-in limit).
struct DeviceControl {
  int status;
  int starve;
  unsigned long long wait_limit;
};
__device__ DeviceControl g_control;
}  // namespace oal

static thread_local char t_msg[512] = "";

oal_status oal_fail(oal_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
  return st;
}

oal_status oal_check_launch(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return oal_fail(OAL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return OAL_OK;
}

// ---- launch accounting and the timing hook
#include <atomic>
static std::atomic<unsigned long long> g_launches{0};
static thread_local cudaEvent_t *t_events = nullptr;
static thread_local int t_nevents = 0;
static thread_local int t_call_launches = 0;
static thread_local const char *t_call_names[32];

void oal_begin_call(cudaStream_t stream) {
  t_call_launches = 0;
  if (t_events && t_nevents > 0) cudaEventRecord(t_events[0], stream);
}

oal_status oal_after_launch(const char *name, cudaStream_t stream) {
  const oal_status st = oal_check_launch(name);
  if (st != OAL_OK) return st;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  const int k = ++t_call_launches;
  if (k <= 32) t_call_names[k - 1] = name;
  if (t_events && k < t_nevents) cudaEventRecord(t_events[k], stream);
  return OAL_OK;
}

#include <mutex>
static std::mutex g_control_mutex;
static int *g_control_addr[oal::kMaxDevices] = {nullptr};

int *oal_device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= oal::kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_control_mutex);
  if (!g_control_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, oal::g_control) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_control_addr[dev] = &static_cast<oal::DeviceControl *>(p)->status;
  }
  return g_control_addr[dev];
}

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

oal_status check_ptr(const void *p, const char *name) {
  if (!p) return oal_fail(OAL_ERR_INVALID_ARG, "%s is null", name);
  if (!aligned16(p)) return oal_fail(OAL_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return OAL_OK;
}

oal_status check_common(int B, int Hq, int Hkv, int d, int dv, oal_dtype dtype,
                        oal_state_layout layout) {
  if (B < 0 || Hq <= 0 || Hkv <= 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d", B, Hq, Hkv);
  if (Hq % Hkv != 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (dtype != OAL_F32 && dtype != OAL_BF16)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
  if (layout != OAL_STATE_FULL && layout != OAL_STATE_PACKED)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad state layout %d", (int)layout);
  if (d != oal::kD || dv != oal::kDv)
    return oal_fail(OAL_ERR_UNSUPPORTED, "only d = dv = 64 is supported (d=%d dv=%d)", d, dv);
  return OAL_OK;
}

#define OAL_TRY(x)                        \
  do {                                    \
    const oal_status _s = (x);            \
    if (_s != OAL_OK) return _s;          \
  } while (0)

}  // namespace

extern "C" {

const char *oal_version(void) { return "0.1.0"; }

uint64_t oal_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

oal_status oal_set_launch_events(cudaEvent_t *events, int n) {
  if (n < 0) return oal_fail(OAL_ERR_INVALID_ARG, "n=%d", n);
  t_events = (events && n > 0) ? events : nullptr;
  t_nevents = t_events ? n : 0;
  return OAL_OK;
}

int oal_last_call_launches(void) { return t_call_launches; }

const char *oal_last_call_launch_name(int k) {
  if (k < 0 || k >= t_call_launches || k >= 32) return "";
  return t_call_names[k];
}

const char *oal_last_error(void) { return t_msg; }

size_t oal_state_rows(int d, oal_state_layout layout) {
  if (d <= 0) return 0;
  const size_t dd = (size_t)d;
  if (layout == OAL_STATE_FULL) return 1 + dd + dd * dd;
  if (layout == OAL_STATE_PACKED) return 1 + dd + dd * (dd + 1) / 2;
  return 0;
}

size_t oal_state_elems(int d, int dv, oal_state_layout layout) {
  if (dv <= 0) return 0;
  return oal_state_rows(d, layout) * (size_t)(dv + 1);
}

size_t oal_coeff_table_elems(int d, oal_state_layout layout) {
  if (d <= 0) return 0;
  if (layout == OAL_STATE_FULL) return (size_t)d * d;
  if (layout == OAL_STATE_PACKED) return (size_t)d * (d + 1) / 2;
  return 0;
}

oal_status oal_expand_coeffs(const float *L, const int32_t *group, int Hq, int G, int d,
                             float eps, oal_state_layout layout, float *a, float *b,
                             float *C, cudaStream_t stream) {
  t_msg[0] = 0;
  if (Hq <= 0) return oal_fail(OAL_ERR_INVALID_ARG, "Hq=%d", Hq);
  if (layout != OAL_STATE_FULL && layout != OAL_STATE_PACKED)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad state layout %d", (int)layout);
  if (d != oal::kD) return oal_fail(OAL_ERR_UNSUPPORTED, "only d = 64 is supported (d=%d)", d);
  if (G < 1 || G > oal::kMaxG)
    return oal_fail(OAL_ERR_UNSUPPORTED, "G=%d outside 1..%d", G, oal::kMaxG);
  if (!(eps > 0.f)) return oal_fail(OAL_ERR_INVALID_ARG, "eps must be > 0 (got %g)", eps);
  OAL_TRY(check_ptr(L, "L"));
  OAL_TRY(check_ptr(group, "group"));
  OAL_TRY(check_ptr(a, "a"));
  OAL_TRY(check_ptr(b, "b"));
  OAL_TRY(check_ptr(C, "C"));
  oal_begin_call(stream);
  return oal::launch_expand_coeffs(L, group, Hq, G, eps, layout == OAL_STATE_PACKED, a, b,
                                   C, stream);
}

static int default_chunk(oal_dtype dtype) { return dtype == OAL_BF16 ? 128 : 64; }

// bf16 inputs run on the tensor cores (tcgen05) at every chunk size; fp32
// inputs run the fp32 CUDA-core kernels.
static bool use_tc(oal_dtype dtype) { return dtype == OAL_BF16; }

size_t oal_prefill_workspace_bytes(int B, int Hq, int Hkv, int T, int d, int dv,
                                   oal_dtype dtype, oal_state_layout layout, int chunk) {
  if (check_common(B, Hq, Hkv, d, dv, dtype, layout) != OAL_OK || T < 0) return 0;
  if (chunk == 0) chunk = default_chunk(dtype);
  if (chunk != 64 && chunk != 128 && chunk != 256) return 0;
  if (T == 0 || B == 0) return 256;
  if (use_tc(dtype)) return oal::tc_prefill_workspace_bytes(B, Hq, Hkv, T, chunk);
  return oal::simt_prefill_workspace_bytes(B, Hkv, T, layout == OAL_STATE_PACKED, chunk);
}

oal_status oal_prefill(const void *Q, const void *K, const void *V, oal_dtype dtype, int B,
                       int Hq, int Hkv, int T, int d, int dv, const float *L,
                       const int32_t *group, int G, float eps, const float *a,
                       const float *b, const float *C, oal_state_layout layout,
                       float *state, int continue_from_state, void *Y, int chunk,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  t_msg[0] = 0;
  OAL_TRY(check_common(B, Hq, Hkv, d, dv, dtype, layout));
  if (T < 0) return oal_fail(OAL_ERR_INVALID_ARG, "T=%d", T);
  if (G < 1 || G > oal::kMaxG)
    return oal_fail(OAL_ERR_UNSUPPORTED, "G=%d outside 1..%d", G, oal::kMaxG);
  if (!(eps > 0.f)) return oal_fail(OAL_ERR_INVALID_ARG, "eps must be > 0 (got %g)", eps);
  if (chunk == 0) chunk = default_chunk(dtype);
  if (chunk != 64 && chunk != 128 && chunk != 256)
    return oal_fail(OAL_ERR_INVALID_ARG, "chunk=%d (allowed: 0, 64, 128, 256)", chunk);
  t_call_launches = 0;
  if (B == 0) return OAL_OK;
  OAL_TRY(check_ptr(state, "state"));
  const int packed = layout == OAL_STATE_PACKED;
  if (T == 0) {
    if (!continue_from_state) {
      const size_t bytes = (size_t)B * Hkv * oal_state_elems(d, dv, layout) * sizeof(float);
      if (cudaMemsetAsync(state, 0, bytes, stream) != cudaSuccess)
        return oal_check_launch("state reset");
    }
    return OAL_OK;
  }
  OAL_TRY(check_ptr(Q, "Q"));
  OAL_TRY(check_ptr(K, "K"));
  OAL_TRY(check_ptr(V, "V"));
  OAL_TRY(check_ptr(Y, "Y"));
  OAL_TRY(check_ptr(L, "L"));
  OAL_TRY(check_ptr(group, "group"));
  OAL_TRY(check_ptr(a, "a"));
  OAL_TRY(check_ptr(b, "b"));
  OAL_TRY(check_ptr(C, "C"));
  OAL_TRY(check_ptr(workspace, "workspace"));
  if (((uintptr_t)workspace & 255u) != 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need =
      oal_prefill_workspace_bytes(B, Hq, Hkv, T, d, dv, dtype, layout, chunk);
  if (workspace_bytes < need)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                    workspace_bytes, need);
  if ((long long)T * Hq * B > (1LL << 40))
    return oal_fail(OAL_ERR_UNSUPPORTED, "problem too large");
  oal_begin_call(stream);
  if (use_tc(dtype))
    return oal::launch_prefill_tc(Q, K, V, B, Hq, Hkv, T, L, group, G, eps, a, b, C, packed,
                                  state, continue_from_state != 0, Y, chunk, workspace, stream);
  return oal::launch_prefill_simt(Q, K, V, dtype == OAL_BF16, B, Hq, Hkv, T, L, group, G,
                                  eps, a, b, C, packed, state, continue_from_state != 0,
                                  Y, chunk, workspace, stream);
}

size_t oal_prefill_backward_workspace_bytes(int B, int Hq, int Hkv, int T, int d, int dv) {
  if (check_common(B, Hq, Hkv, d, dv, OAL_F32, OAL_STATE_FULL) != OAL_OK || T < 0) return 0;
  if (B == 0 || T == 0) return 256;
  return oal::backward_workspace_bytes(B, Hq, Hkv, T);
}

oal_status oal_prefill_backward(const void *Q, const void *K, const void *V, const void *dY,
                                oal_dtype dtype, int B, int Hq, int Hkv, int T, int d, int dv,
                                const float *L, const int32_t *group, int G, float eps, float *dQ,
                                float *dK, float *dV, float *dL, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  t_msg[0] = 0;
  OAL_TRY(check_common(B, Hq, Hkv, d, dv, dtype, OAL_STATE_FULL));
  if (T < 0) return oal_fail(OAL_ERR_INVALID_ARG, "T=%d", T);
  if (G < 1 || G > oal::kMaxG)
    return oal_fail(OAL_ERR_UNSUPPORTED, "G=%d outside 1..%d", G, oal::kMaxG);
  if (!(eps > 0.f)) return oal_fail(OAL_ERR_INVALID_ARG, "eps must be > 0 (got %g)", eps);
  OAL_TRY(check_ptr(L, "L"));
  OAL_TRY(check_ptr(group, "group"));
  OAL_TRY(check_ptr(dL, "dL"));
  t_call_launches = 0;
  if (B == 0 || T == 0) {   // no pairs: every gradient is zero (dQ, dK, dV are empty)
    const size_t bytes = (size_t)Hq * (G + 1) * (G + 1) * sizeof(float);
    if (cudaMemsetAsync(dL, 0, bytes, stream) != cudaSuccess) return oal_check_launch("dL reset");
    return OAL_OK;
  }
  OAL_TRY(check_ptr(Q, "Q"));
  OAL_TRY(check_ptr(K, "K"));
  OAL_TRY(check_ptr(V, "V"));
  OAL_TRY(check_ptr(dY, "dY"));
  OAL_TRY(check_ptr(dQ, "dQ"));
  OAL_TRY(check_ptr(dK, "dK"));
  OAL_TRY(check_ptr(dV, "dV"));
  OAL_TRY(check_ptr(workspace, "workspace"));
  if (((uintptr_t)workspace & 255u) != 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = oal_prefill_backward_workspace_bytes(B, Hq, Hkv, T, d, dv);
  if (workspace_bytes < need)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                    workspace_bytes, need);
  oal_begin_call(stream);
  return oal::launch_backward(Q, K, V, dY, dtype == OAL_BF16, B, Hq, Hkv, T, L, group, G, eps, dQ,
                              dK, dV, dL, workspace, stream);
}

size_t oal_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int dv,
                                  oal_state_layout layout) {
  if (check_common(B, Hq, Hkv, d, dv, OAL_F32, layout) != OAL_OK) return 0;
  if (B == 0) return 256;
  return oal::decode_workspace_bytes(B, Hkv, layout == OAL_STATE_PACKED);
}

oal_status oal_decode_step(const void *q, const void *k, const void *v, oal_dtype dtype,
                           int B, int Hq, int Hkv, int d, int dv, const float *a,
                           const float *b, const float *C, oal_state_layout layout,
                           float *state, void *y, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  t_msg[0] = 0;
  OAL_TRY(check_common(B, Hq, Hkv, d, dv, dtype, layout));
  if (Hq / Hkv > oal::decode_max_rho())
    return oal_fail(OAL_ERR_UNSUPPORTED, "Hq/Hkv=%d exceeds %d", Hq / Hkv,
                    oal::decode_max_rho());
  if (B == 0) return OAL_OK;
  OAL_TRY(check_ptr(q, "q"));
  OAL_TRY(check_ptr(k, "k"));
  OAL_TRY(check_ptr(v, "v"));
  OAL_TRY(check_ptr(y, "y"));
  OAL_TRY(check_ptr(a, "a"));
  OAL_TRY(check_ptr(b, "b"));
  OAL_TRY(check_ptr(C, "C"));
  OAL_TRY(check_ptr(state, "state"));
  OAL_TRY(check_ptr(workspace, "workspace"));
  if (((uintptr_t)workspace & 255u) != 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = oal_decode_workspace_bytes(B, Hq, Hkv, d, dv, layout);
  if (workspace_bytes < need)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                    workspace_bytes, need);
  oal_begin_call(stream);
  return oal::launch_decode(q, k, v, dtype == OAL_BF16, B, Hq, Hkv, a, b, C,
                            layout == OAL_STATE_PACKED, state, y, workspace, stream);
}

size_t oal_contribution_workspace_bytes(int P, int Hq, int Hkv, int T, int d) {
  if (P < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || d != oal::kD) return 0;
  return std::max<size_t>(256, oal::contrib_workspace_bytes(P, Hq, Hkv, T));
}

oal_status oal_contribution_scores(const void *Q, const void *K, oal_dtype dtype, int P,
                                   int Hq, int Hkv, int T, int d, const int32_t *lengths,
                                   float *chi, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  t_msg[0] = 0;
  OAL_TRY(check_common(P, Hq, Hkv, d, d, dtype, OAL_STATE_FULL));
  if (T < 0) return oal_fail(OAL_ERR_INVALID_ARG, "bad T=%d", T);
  if (P == 0) return OAL_OK;
  if (P > 65535) return oal_fail(OAL_ERR_UNSUPPORTED, "P=%d above 65535", P);
  OAL_TRY(check_ptr(chi, "chi"));
  OAL_TRY(check_ptr(workspace, "workspace"));
  if (T > 0) {
    OAL_TRY(check_ptr(Q, "Q"));
    OAL_TRY(check_ptr(K, "K"));
    if ((T + 127) / 128 > 65535) return oal_fail(OAL_ERR_UNSUPPORTED, "T=%d too long", T);
  }
  if (lengths) OAL_TRY(check_ptr(lengths, "lengths"));
  if (((uintptr_t)workspace & 255u) != 0)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = oal_contribution_workspace_bytes(P, Hq, Hkv, T, d);
  if (workspace_bytes < need)
    return oal_fail(OAL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                    workspace_bytes, need);
  oal_begin_call(stream);
  return oal::launch_contrib(Q, K, dtype == OAL_BF16, P, Hq, Hkv, T, lengths, chi, workspace,
                             stream);
}

oal_status oal_group_dims(const float *chi_p, int P, int d, const int32_t *boot_idx, int nboot,
                          double alpha, double tau, double gamma, int g_min, double eps,
                          int32_t *group, int *G) {
  t_msg[0] = 0;
  if (!chi_p || !boot_idx || !group || !G)
    return oal_fail(OAL_ERR_INVALID_ARG, "null pointer");
  if (P < 1 || d < 2 || nboot < 1)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad sizes P=%d d=%d nboot=%d", P, d, nboot);
  if (!(alpha > 0.0 && alpha <= 1.0) || !(eps > 0.0) || !(tau > 0.0) || !(gamma >= 0.0) ||
      g_min < 1)
    return oal_fail(OAL_ERR_INVALID_ARG, "bad parameters alpha=%g tau=%g gamma=%g g_min=%d "
                    "eps=%g", alpha, tau, gamma, g_min, eps);
  for (size_t i = 0; i < (size_t)nboot * P; ++i)
    if (boot_idx[i] < 0 || boot_idx[i] >= P)
      return oal_fail(OAL_ERR_INVALID_ARG, "bootstrap index %d outside 0..%d", boot_idx[i],
                      P - 1);
  for (size_t i = 0; i < (size_t)P * d; ++i)
    if (!isfinite(chi_p[i]) || chi_p[i] < 0.f)
      return oal_fail(OAL_ERR_INVALID_ARG, "score %zu is negative or not finite", i);
  return oal::group_dims_host(chi_p, P, d, boot_idx, nboot, alpha, tau, gamma, g_min, eps,
                              group, G);
}

oal_status oal_debug_wait_test(uint64_t wait_limit_cycles, int starve) {
  t_msg[0] = 0;
  if (starve < 0 || starve > 3) return oal_fail(OAL_ERR_INVALID_ARG, "starve=%d", starve);
  int *w = oal_device_status_word();
  if (!w) return oal_fail(OAL_ERR_CUDA, "device control block unavailable");
  oal::DeviceControl c;
  cudaError_t e = cudaMemcpy(&c, w, sizeof c, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) {
    c.starve = starve;
    c.wait_limit = wait_limit_cycles;
    e = cudaMemcpy(w, &c, sizeof c, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess)
    return oal_fail(OAL_ERR_CUDA, "setting the wait test: %s", cudaGetErrorString(e));
  return OAL_OK;
}

oal_status oal_debug_intra_heads(int heads) {
  t_msg[0] = 0;
  if (heads < 0 || heads > 2) return oal_fail(OAL_ERR_INVALID_ARG, "heads=%d", heads);
  oal::set_intra_heads(heads);
  return OAL_OK;
}

oal_status oal_sync_status(cudaStream_t stream) {
  t_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess)
    return oal_fail(OAL_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int *w = oal_device_status_word();
  if (!w) return oal_fail(OAL_ERR_CUDA, "status word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return oal_fail(OAL_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    const char *what = v == OAL_ERR_INVALID_ARG ? "a group id outside 1..G or a prompt "
                                                  "length outside 0..T"
                       : v == OAL_ERR_TIMEOUT   ? "a device-side wait timed out"
                                                : "device error";
    return oal_fail((oal_status)v, "device status %d: %s", v, what);
  }
  return OAL_OK;
}

}  // extern "C"
