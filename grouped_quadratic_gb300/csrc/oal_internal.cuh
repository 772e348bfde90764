// oal_internal.cuh -- helpers shared by the CUDA sources of liboal.so.
//
// Feature order of the prefix states ([OAL] = "Not All Dimensions Are Equal:
// Outlier-Aware Attention Linearization with Grouped Quadratic Kernels",
// Eq. (5); packed symmetric layout of App. D):
//   row 0: H0;  rows 1..64: H1_r;  rows 65..: H2_rt
//   FULL:   H2 row index r*64 + t
//   PACKED: H2 row index r*64 - r(r-1)/2 + (t - r), r <= t
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/oal.h"

namespace oal {

constexpr int kD = 64;                          // d_h (only size supported)
constexpr int kDv = 64;                         // d_v
constexpr int kU = kDv + 1;                     // u = [v; 1]
constexpr int kH2Full = kD * kD;                // 4096
constexpr int kH2Packed = kD * (kD + 1) / 2;    // 2080
constexpr int kFFull = 1 + kD + kH2Full;        // 4161
constexpr int kFPacked = 1 + kD + kH2Packed;    // 2145
constexpr int kMaxG = 7;
// Per-device caches of the library (symbol addresses, function attributes)
// cover device ordinals 0 .. kMaxDevices - 1.
constexpr int kMaxDevices = 256;

// Device status word values (written by kernels, read by oal_sync_status).
constexpr int kStatusOk = 0;

__host__ __device__ constexpr int state_rows(int packed) {
  return packed ? kFPacked : kFFull;
}

// (r, t) of packed H2 entry n, r <= t, row-major upper triangle.
struct PairTable {
  uint16_t rt[kH2Packed];  // r << 8 | t
};

__host__ __device__ constexpr PairTable make_pair_table() {
  PairTable p{};
  int n = 0;
  for (int r = 0; r < kD; ++r)
    for (int t = r; t < kD; ++t) p.rt[n++] = (uint16_t)((r << 8) | t);
  return p;
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization: it signals at entry that the next
// kernel on the stream may be scheduled (pdl_trigger), and waits for the
// previous kernel's completion and memory (pdl_wait) before it reads or
// writes global memory that kernel may touch.  Every kernel calls pdl_wait,
// so the completion order along the stream stays transitive.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace oal

// Host-side error reporting (oal_api.cu).
oal_status oal_fail(oal_status st, const char *fmt, ...);
oal_status oal_check_launch(const char *what);
// After every kernel launch: checks the launch, counts it and records the
// timing-hook event if one is installed.
oal_status oal_after_launch(const char *name, cudaStream_t stream);
// At the start of every entry point that may launch kernels.
void oal_begin_call(cudaStream_t stream);
// Device address of the status word of the current device, or null.  For
// tests of the failure path, the int after it names a kernel whose UMMA
// issuer is to wait on a barrier nothing arrives on (kStarve*; 0 = none) and
// the 64-bit word 8 bytes after it holds the limit of the bounded waits in SM
// cycles (0: the built-in limit); kernels read both through the status
// pointer they are given.
int *oal_device_status_word();
namespace oal {
constexpr int kStarveReadout = 1, kStarveState = 2, kStarveIntra = 3;
}
