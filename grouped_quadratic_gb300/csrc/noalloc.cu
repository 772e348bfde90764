// noalloc.cu -- oal_prefill_noalloc: the prefill for callers that cannot
// allocate device memory.  Its scratch is one fixed array owned by the
// library; the kernels and their arithmetic are those of oal_prefill.
#include <mutex>

#include "oal_internal.cuh"

namespace {

constexpr size_t kScratchBytes = OAL_PREFILL_NOALLOC_SCRATCH_BYTES;

// One copy per device, reserved when the library's device code is loaded on
// that device and kept until the process exits.  In host code this name is
// only a host-side stand-in: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[oal::kMaxDevices] = {};

// Device address of g_prefill_scratch on the current device, looked up once
// per device (with that device current) and cached.
oal_status scratch_for_current_device(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return oal_fail(OAL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= oal::kMaxDevices)
    return oal_fail(OAL_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, oal::kMaxDevices - 1);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess || p == nullptr)
      return oal_fail(OAL_ERR_CUDA, "cudaGetSymbolAddress of the prefill scratch on device %d: %s",
                      dev, cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return OAL_OK;
}

}  // namespace

size_t oal_prefill_noalloc_scratch_bytes(void) { return kScratchBytes; }

oal_status oal_prefill_noalloc(const void *Q, const void *K, const void *V, oal_dtype dtype,
                               int B, int Hq, int Hkv, int T, int d, int dv, const float *L,
                               const int32_t *group, int G, float eps, const float *a,
                               const float *b, const float *C, oal_state_layout layout,
                               float *state, int continue_from_state, void *Y, int chunk,
                               cudaStream_t stream) {
  const size_t need = oal_prefill_workspace_bytes(B, Hq, Hkv, T, d, dv, dtype, layout, chunk);
  if (need > kScratchBytes)
    return oal_fail(OAL_ERR_INVALID_ARG,
                    "oal_prefill_noalloc: this problem needs %zu bytes of scratch, above the "
                    "fixed %zu bytes of the library's array; call oal_prefill with a workspace",
                    need, kScratchBytes);
  // need == 0 means invalid arguments: oal_prefill reports which.
  void *scratch = nullptr;
  if (need > 0 && B > 0 && T > 0) {
    const oal_status st = scratch_for_current_device(&scratch);
    if (st != OAL_OK) return st;
  }
  return oal_prefill(Q, K, V, dtype, B, Hq, Hkv, T, d, dv, L, group, G, eps, a, b, C, layout,
                     state, continue_from_state, Y, chunk, scratch, kScratchBytes, stream);
}
