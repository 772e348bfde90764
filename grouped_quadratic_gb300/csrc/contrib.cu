// contrib.cu -- the calibration step before the path: per-prompt contribution
// scores on the GPU ([OAL] Sec. 3.1, Eq. (2)) and the bootstrap dimension
// grouping on the host ([OAL] App. B, Eqs. (16)-(19)).
//
// Eq. (2) is separable: |q_{i,r} k_{j,r}| = |q_{i,r}| |k_{j,r}|, so
//     sum_{j <= i} |q_{i,r} k_{j,r}| = sum_i |q_{i,r}| Kbar_{i,r},
//     Kbar_{i,r} = sum_{j <= i} |k_{j,r}|,
// a prefix sum over the tokens instead of the O(N^2) pair set.  One pass over
// Q and K: HBM-bound.
//   contrib_chunk_kernel   per (query head, 128-token chunk, prompt): the
//                          chunk's |k| total A_c (written by the first head
//                          of each KV head), Qs_c = sum_{i in c} |q_i| and
//                          W_c = sum_{i in c} |q_i| (inclusive |k| prefix
//                          inside the chunk), per dim.  Thread = 8 dims x a
//                          run of 4 tokens, 16-byte loads; the run totals are
//                          scanned across the chunk's 32 runs in shared memory
//   contrib_finish_kernel  per (prompt, query head), thread = dim: walks the
//                          chunks, sum_c W_c + Qs_c sum_{c' < c} A_c', and
//                          divides by |Omega_p| sqrt(d)
#include <math.h>

#include <algorithm>
#include <vector>

#include "oal_internal.cuh"

namespace oal {
namespace {

constexpr int kCC = 128;               // tokens per chunk
constexpr int kCThreads = 256;         // 8 dim groups x 32 runs
constexpr int kRun = 4;                // tokens of a thread's run
constexpr int kRuns = kCC / kRun;
constexpr int kRunPitch = kRuns + 1;   // [dim][run] in shared memory: conflict-free per dim

// |x| of dims 8g .. 8g + 7 of one token row: one 16-byte load (bf16) or two (fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, bool ok, uint4 (&raw)[2]) {
  raw[0] = ok ? __ldg(reinterpret_cast<const uint4 *>(p)) : make_uint4(0u, 0u, 0u, 0u);
  raw[1] = make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void load8(const float *p, bool ok, uint4 (&raw)[2]) {
  raw[0] = ok ? __ldg(reinterpret_cast<const uint4 *>(p)) : make_uint4(0u, 0u, 0u, 0u);
  raw[1] = ok ? __ldg(reinterpret_cast<const uint4 *>(p) + 1) : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void abs8(const uint4 (&raw)[2], __nv_bfloat16, float (&o)[8]) {
  const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    o[2 * e] = __uint_as_float((w[e] << 16) & 0x7FFFFFFFu);
    o[2 * e + 1] = __uint_as_float(w[e] & 0x7FFF0000u);
  }
}
__device__ __forceinline__ void abs8(const uint4 (&raw)[2], float, float (&o)[8]) {
  const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w,
                         raw[1].x, raw[1].y, raw[1].z, raw[1].w};
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(w[e] & 0x7FFFFFFFu);
}

// Prompt length, clamped to 0..T; a length outside records OAL_ERR_INVALID_ARG.
__device__ __forceinline__ int prompt_len(const int32_t *lengths, int p, int T, int *status) {
  if (!lengths) return T;
  const int n = lengths[p];
  if (n < 0 || n > T) {
    atomicCAS(status, kStatusOk, (int)OAL_ERR_INVALID_ARG);
    return n < 0 ? 0 : T;
  }
  return n;
}

// Query heads vary fastest in the grid, so the rho blocks that read one K
// chunk run close together and share it through L2.
template <typename Tin>
__global__ void __launch_bounds__(kCThreads)
contrib_chunk_kernel(const Tin *__restrict__ Q, const Tin *__restrict__ K,
                     const int32_t *__restrict__ lengths, int Hq, int Hkv, int T, int nC,
                     float *__restrict__ A, float *__restrict__ Qs, float *__restrict__ W,
                     int *status) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, c = blockIdx.y, p = blockIdx.z;
  const int rho = Hq / Hkv, kv = h / rho;
  const int tid = threadIdx.x, g = tid & 7, run = tid >> 3;   // a warp: 8 groups x 4 runs
  const int n = prompt_len(lengths, p, T, status);
  const int t0 = c * kCC + run * kRun;   // first token of the run
  __shared__ float s_off[64 * kRunPitch];             // run totals of |k|, then their prefixes
  __shared__ float s_q[64 * kRunPitch], s_w[64 * kRunPitch];
  const Tin *kp = K + (((size_t)p * Hkv + kv) * T + t0) * 64 + 8 * g;
  const Tin *qp = Q + (((size_t)p * Hq + h) * T + t0) * 64 + 8 * g;
  uint4 kr[kRun][2], qr[kRun][2];
#pragma unroll
  for (int i = 0; i < kRun; ++i) {   // every load of the thread in flight at once
    load8(kp + (size_t)i * 64, t0 + i < n, kr[i]);
    load8(qp + (size_t)i * 64, t0 + i < n, qr[i]);
  }
  // inclusive |k| prefix inside the run
  float pk[kRun][8];
#pragma unroll
  for (int i = 0; i < kRun; ++i) {
    float a[8];
    abs8(kr[i], Tin(), a);
#pragma unroll
    for (int e = 0; e < 8; ++e) pk[i][e] = (i ? pk[i - 1][e] : 0.f) + a[e];
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_off[(8 * g + e) * kRunPitch + run] = pk[kRun - 1][e];
  __syncthreads();
  if (tid < 64) {
    // exclusive prefix over the runs of dim tid; the total is the chunk's A_c
    float acc = 0.f;
    for (int j = 0; j < kRuns; ++j) {
      const float v = s_off[tid * kRunPitch + j];
      s_off[tid * kRunPitch + j] = acc;
      acc += v;
    }
    if (h % rho == 0) A[(((size_t)p * Hkv + kv) * nC + c) * 64 + tid] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float off = s_off[(8 * g + e) * kRunPitch + run];
    float qs = 0.f, w = 0.f;
#pragma unroll
    for (int i = 0; i < kRun; ++i) {
      float a[8];
      abs8(qr[i], Tin(), a);
      qs += a[e];
      w = fmaf(a[e], off + pk[i][e], w);
    }
    s_q[(8 * g + e) * kRunPitch + run] = qs;
    s_w[(8 * g + e) * kRunPitch + run] = w;
  }
  __syncthreads();
  if (tid < 128) {
    // the runs' sums per dim, in run order
    const int r = tid & 63;
    const float *src = (tid < 64 ? s_q : s_w) + r * kRunPitch;
    float sum = 0.f;
    for (int j = 0; j < kRuns; ++j) sum += src[j];
    const size_t ch = (((size_t)p * Hq + h) * nC + c) * 64 + r;
    if (tid < 64) Qs[ch] = sum;
    else W[ch] = sum;
  }
}

__global__ void __launch_bounds__(64)
contrib_finish_kernel(const int32_t *__restrict__ lengths, int Hq, int Hkv, int T, int nC,
                      const float *__restrict__ A, const float *__restrict__ Qs,
                      const float *__restrict__ W, float *__restrict__ chi, int *status) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, p = blockIdx.y, r = threadIdx.x;
  const int kv = h / (Hq / Hkv);
  const int n = prompt_len(lengths, p, T, status);
  const float *a = A + ((size_t)p * Hkv + kv) * nC * 64 + r;
  const float *qs = Qs + ((size_t)p * Hq + h) * nC * 64 + r;
  const float *w = W + ((size_t)p * Hq + h) * nC * 64 + r;
  // across chunks in fp64 (a few values per chunk; the chunk sums stay fp32)
  double acc = 0.0, kbefore = 0.0;
  for (int c = 0; c < nC; ++c) {
    acc += (double)w[(size_t)c * 64] + (double)qs[(size_t)c * 64] * kbefore;
    kbefore += (double)a[(size_t)c * 64];
  }
  const double omega = 0.5 * (double)n * (double)(n + 1);
  chi[((size_t)p * Hq + h) * 64 + r] = n > 0 ? (float)(acc / (omega * 8.0)) : 0.f;   // sqrt(64) = 8
}

}  // namespace

size_t contrib_workspace_bytes(int P, int Hq, int Hkv, int T) {
  const size_t nC = (size_t)(T + kCC - 1) / kCC;
  return (size_t)P * nC * 64 * sizeof(float) * ((size_t)Hkv + 2 * (size_t)Hq);
}

oal_status launch_contrib(const void *Q, const void *K, int is_bf16, int P, int Hq, int Hkv,
                          int T, const int32_t *lengths, float *chi, void *ws,
                          cudaStream_t stream) {
  int *status = oal_device_status_word();
  if (!status) return oal_fail(OAL_ERR_CUDA, "no device status word");
  const int nC = (T + kCC - 1) / kCC;
  float *A = static_cast<float *>(ws);
  float *Qs = A + (size_t)P * Hkv * nC * 64;
  float *W = Qs + (size_t)P * Hq * nC * 64;
  if (nC > 0) {
    const dim3 grid(Hq, nC, P);
    if (is_bf16)
      launch_pdl(contrib_chunk_kernel<__nv_bfloat16>, grid, dim3(kCThreads), 0, stream,
                 static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(K),
                 lengths, Hq, Hkv, T, nC, A, Qs, W, status);
    else
      launch_pdl(contrib_chunk_kernel<float>, grid, dim3(kCThreads), 0, stream,
                 static_cast<const float *>(Q), static_cast<const float *>(K), lengths, Hq,
                 Hkv, T, nC, A, Qs, W, status);
    const oal_status st = oal_after_launch("contrib_chunk_kernel", stream);
    if (st != OAL_OK) return st;
  }
  launch_pdl(contrib_finish_kernel, dim3(Hq, P), dim3(64), 0, stream, lengths, Hq, Hkv, T, nC,
             A, Qs, W, chi, status);
  return oal_after_launch("contrib_finish_kernel", stream);
}

// ---------------------------------------------------------------- host grouping
// [OAL] App. B for one query head, in the appendix's order.  fp64; every
// average is a sum in index order followed by one division, so the result
// does not depend on the compiler's contraction of multiply-adds.
oal_status group_dims_host(const float *chi_p, int P, int d, const int32_t *boot_idx,
                           int nboot, double alpha, double tau, double gamma, int g_min,
                           double eps, int32_t *group, int *G) {
  std::vector<double> chi(d, 0.0), chib(d);
  for (int p = 0; p < P; ++p)
    for (int r = 0; r < d; ++r) chi[r] += (double)chi_p[(size_t)p * d + r];
  for (int r = 0; r < d; ++r) chi[r] /= (double)P;
  // increasing contribution, stable (pi[0] is pi_1 of the appendix)
  std::vector<int> pi(d);
  for (int r = 0; r < d; ++r) pi[r] = r;
  std::stable_sort(pi.begin(), pi.end(), [&](int x, int y) { return chi[x] < chi[y]; });
  const int m = (int)ceil(alpha * (double)d);
  const int k0 = std::max(1, d - m);
  const int nk = d - k0;                       // candidates k0 .. d-1
  std::vector<double> gap(nk), support(nk);
  std::vector<int> hits(nk, 0);
  // Eq. (16): adjacent gap across cut k (L_k = pi[0, k), U_k = pi[k, d))
  for (int e = 0; e < nk; ++e) {
    const int k = k0 + e;
    gap[e] = chi[pi[k]] / std::max(chi[pi[k - 1]], eps);
  }
  // Eqs. (17)-(18): bootstrap support, the ordering pi kept fixed
  std::vector<double> lo(d), hi(d);
  for (int b = 0; b < nboot; ++b) {
    std::fill(chib.begin(), chib.end(), 0.0);
    for (int t = 0; t < P; ++t) {
      const int ip = boot_idx[(size_t)b * P + t];
      for (int r = 0; r < d; ++r) chib[r] += (double)chi_p[(size_t)ip * d + r];
    }
    for (int r = 0; r < d; ++r) chib[r] /= (double)P;
    // max over L_k and min over U_k for every k, by a prefix max and a suffix min
    for (int k = 0; k < d; ++k) lo[k] = k ? std::max(lo[k - 1], chib[pi[k]]) : chib[pi[k]];
    for (int k = d - 1; k >= 0; --k)
      hi[k] = k < d - 1 ? std::min(hi[k + 1], chib[pi[k]]) : chib[pi[k]];
    for (int e = 0; e < nk; ++e) {
      const int k = k0 + e;
      if (hi[k] / std::max(lo[k - 1], eps) >= tau) ++hits[e];
    }
  }
  for (int e = 0; e < nk; ++e) support[e] = (double)hits[e] / (double)nboot;
  // natural cuts, then fallback cuts by descending (support, gap), ties in
  // candidate order, until g_min groups
  std::vector<int> cuts, rest;
  for (int e = 0; e < nk; ++e) {
    if (gap[e] >= tau && support[e] >= gamma)
      cuts.push_back(k0 + e);
    else
      rest.push_back(e);
  }
  std::stable_sort(rest.begin(), rest.end(), [&](int x, int y) {
    return support[x] > support[y] || (support[x] == support[y] && gap[x] > gap[y]);
  });
  for (size_t i = 0; i < rest.size() && (int)cuts.size() + 1 < g_min; ++i)
    cuts.push_back(k0 + rest[i]);
  std::sort(cuts.begin(), cuts.end());
  // Eq. (19): group g holds pi[k_{g-1}, k_g)
  int start = 0, g = 1;
  for (size_t i = 0; i <= cuts.size(); ++i, ++g) {
    const int end = i < cuts.size() ? cuts[i] : d;
    for (int k = start; k < end; ++k) group[pi[k]] = g;
    start = end;
  }
  *G = (int)cuts.size() + 1;
  return OAL_OK;
}

}  // namespace oal
