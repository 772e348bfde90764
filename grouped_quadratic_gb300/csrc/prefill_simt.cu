// prefill_simt.cu -- chunked causal OAL prefill on fp32 CUDA cores.
//
// [OAL] = "Not All Dimensions Are Equal: Outlier-Aware Attention
// Linearization with Grouped Quadratic Kernels".  Tokens are cut into chunks
// of C; for token i of chunk c
//     u~_i = Phi~(q_i)^T S_{c-1}  +  sum_{j in chunk c, j <= i} kappa(q_i,k_j) u_j
// where S_{c-1} holds the prefix states H0/H1/H2 of Eq. (5) over all tokens
// before the chunk, Phi~ is the readout weight vector of Eq. (6), and kappa
// is Eq. (7).  App. D, Eq. (25) shows both terms are the same kernel sum, so
// the split is exact.  Three launches:
//   chunk_delta_kernel  per chunk: Delta S_c = sum_{j in c} phi(k_j) u_j^T
//   chunk_scan_kernel   exclusive prefix over chunks (in place), final state
//   readout_kernel      inter-chunk readout + intra-chunk pair sums, Eq. (6)
// This path serves fp32 inputs (fp32 FMA everywhere).
#include "oal_internal.cuh"

namespace oal {
namespace {

// In global memory, not __constant__: threads read different entries, which
// the constant cache would serialize.
static __device__ const PairTable c_pairs = make_pair_table();

constexpr int kThreads = 256;
constexpr int kTile = 64;     // feature rows / query rows per block
constexpr int kP = 65;        // padded row pitch (floats) of 64-wide tiles
constexpr int kFB = 32;       // features per readout step

// phi_f(k): key feature of state row f (Eq. 5 with u factored out).
__device__ __forceinline__ float key_feature(int f, int F, int packed,
                                             const float *k /* smem, 64 */) {
  if (f == 0) return 1.f;
  if (f <= kD) return k[f - 1];
  if (f >= F) return 0.f;
  const int n = f - 1 - kD;
  int r, t;
  if (packed) {
    r = c_pairs.rt[n] >> 8;
    t = c_pairs.rt[n] & 0xff;
  } else {
    r = n >> 6;
    t = n & 63;
  }
  return k[r] * k[t];
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
chunk_delta_kernel(const Tin *__restrict__ K, const Tin *__restrict__ V, int T,
                   int C, int nC, int F, int packed, float *__restrict__ ws) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm[];
  float *ks = sm;                     // [64 tokens][kP]
  float *us = ks + kTile * kP;        // [64 tokens][kP]  (u = [v; 1])
  float *ph = us + kTile * kP;        // [64 features][kP] phi_f(k_j)
  const int f0 = blockIdx.x * kTile;
  const int c = blockIdx.y;
  const size_t unit = blockIdx.z;
  const int tid = threadIdx.x;
  const int fr = tid >> 2, cq = tid & 3;
  float acc[17];
#pragma unroll
  for (int m = 0; m < 17; ++m) acc[m] = 0.f;

  const int t_begin = c * C;
  const int t_end = min(T, t_begin + C);
  for (int jb = t_begin; jb < t_end; jb += kTile) {
    __syncthreads();
    for (int n = tid; n < kTile * kD; n += kThreads) {
      const int j = n >> 6, r = n & 63;
      const int tok = jb + j;
      const bool ok = tok < t_end;
      ks[j * kP + r] = ok ? to_f32(K[(unit * T + tok) * kD + r]) : 0.f;
      us[j * kP + r] = ok ? to_f32(V[(unit * T + tok) * kDv + r]) : 0.f;
      if (r == 0) us[j * kP + kDv] = ok ? 1.f : 0.f;
    }
    __syncthreads();
    for (int n = tid; n < kTile * kTile; n += kThreads) {
      const int f = n >> 6, j = n & 63;
      ph[f * kP + j] = key_feature(f0 + f, F, packed, ks + j * kP);
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kTile; ++j) {
      const float p = ph[fr * kP + j];
#pragma unroll
      for (int m = 0; m < 17; ++m) {
        const int col = cq + 4 * m;
        if (col < kU) acc[m] = fmaf(p, us[j * kP + col], acc[m]);
      }
    }
  }
  const int f = f0 + fr;
  if (f < F) {
    float *out = ws + ((unit * nC + c) * (size_t)F + f) * kU;
#pragma unroll
    for (int m = 0; m < 17; ++m) {
      const int col = cq + 4 * m;
      if (col < kU) out[col] = acc[m];
    }
  }
}

// Exclusive prefix over chunks, in place: ws[c] <- S0 + sum_{c' < c} Delta S_c'.
__global__ void chunk_scan_kernel(float *__restrict__ ws, int nC, size_t FU,
                                  float *__restrict__ state, int cont) {
  pdl_trigger();
  pdl_wait();
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t unit = blockIdx.y;
  if (e >= FU) return;
  float prev = cont ? state[unit * FU + e] : 0.f;
  float *p = ws + unit * (size_t)nC * FU + e;
  for (int c = 0; c < nC; ++c) {
    const float x = p[(size_t)c * FU];
    p[(size_t)c * FU] = prev;
    prev += x;
  }
  state[unit * FU + e] = prev;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
readout_kernel(const Tin *__restrict__ Q, const Tin *__restrict__ K,
               const Tin *__restrict__ V, Tin *__restrict__ Y,
               const float *__restrict__ ws, const float *__restrict__ a,
               const float *__restrict__ b, const float *__restrict__ Ctab,
               const float *__restrict__ L, const int32_t *__restrict__ group,
               int G, float eps, int Hq, int Hkv, int T, int C, int nC, int F,
               int packed, int *status) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm[];
  float *qs = sm;                        // [64 rows][kP]  q (natural order)
  float *qp = qs + kTile * kP;           // [64 rows][kP]  q (group order)
  float *work = qp + kTile * kP;         // phase-dependent
  __shared__ float s_b[kD];
  __shared__ float s_L[(kMaxG + 1) * (kMaxG + 1)];
  __shared__ int s_perm[kD];
  __shared__ int s_off[kMaxG + 2];
  __shared__ float s_den[kTile];

  const int tiles_per_chunk = C / kTile;
  const int chunk = blockIdx.x / tiles_per_chunk;
  const int i0 = blockIdx.x * kTile;     // first query row of this tile
  const int bh = blockIdx.y;
  const int h = bh % Hq;
  const int bidx = bh / Hq;
  const int kv = h / (Hq / Hkv);
  const size_t unit = (size_t)bidx * Hkv + kv;
  const int tid = threadIdx.x;
  const int row = tid >> 2, cq = tid & 3;
  if (i0 >= T) return;
  const int G1 = G + 1;

  // per-head constants: b, L, and the dims sorted by group (counting sort)
  for (int r = tid; r < kD; r += kThreads) s_b[r] = b[(size_t)h * kD + r];
  for (int n = tid; n < G1 * G1; n += kThreads) s_L[n] = L[(size_t)h * G1 * G1 + n];
  if (tid == 0) {
    int cnt[kMaxG + 2] = {0};
    const int32_t *gh = group + (size_t)h * kD;
    for (int r = 0; r < kD; ++r) {
      int g = gh[r];
      if (g < 1 || g > G) { atomicCAS(status, kStatusOk, (int)OAL_ERR_INVALID_ARG); g = 1; }
      cnt[g]++;
    }
    s_off[1] = 0;
    for (int g = 1; g <= G; ++g) s_off[g + 1] = s_off[g] + cnt[g];
    int pos[kMaxG + 2];
    for (int g = 1; g <= G + 1; ++g) pos[g] = s_off[g];
    for (int r = 0; r < kD; ++r) {
      int g = gh[r];
      if (g < 1 || g > G) g = 1;
      s_perm[pos[g]++] = r;
    }
  }
  for (int n = tid; n < kTile * kD; n += kThreads) {
    const int i = n >> 6, r = n & 63;
    const int tok = i0 + i;
    qs[i * kP + r] = tok < T ? to_f32(Q[(((size_t)bidx * Hq + h) * T + tok) * kD + r]) : 0.f;
  }
  __syncthreads();
  for (int n = tid; n < kTile * kD; n += kThreads) {
    const int i = n >> 6, r = n & 63;
    qp[i * kP + r] = qs[i * kP + s_perm[r]];
  }

  float acc[17];
#pragma unroll
  for (int m = 0; m < 17; ++m) acc[m] = 0.f;

  // ---- inter-chunk readout: Phi~(q_i)^T S_{chunk-1}   (Eq. 6)
  {
    float *ph = work;                     // [64 rows][kFB + 1]
    float *Ss = ph + kTile * (kFB + 1);   // [kFB rows][kU]
    const float *S = ws + (unit * nC + chunk) * (size_t)F * kU;
    const float ah = a[h];
    const float *Ch = Ctab + (size_t)h * (packed ? kH2Packed : kH2Full);
    for (int fb = 0; fb < F; fb += kFB) {
      __syncthreads();
      const int nrows = min(kFB, F - fb);
      for (int n = tid; n < kFB * kU; n += kThreads)
        Ss[n] = n < nrows * kU ? S[(size_t)fb * kU + n] : 0.f;
      for (int n = tid; n < kTile * kFB; n += kThreads) {
        const int i = n / kFB, jf = n % kFB;
        const int f = fb + jf;
        const float *q = qs + i * kP;
        float w;
        if (f == 0) {
          w = ah;
        } else if (f <= kD) {
          w = s_b[f - 1] * q[f - 1] * 0.125f;           // b_r q_r / sqrt(64)
        } else if (f < F) {
          const int nn = f - 1 - kD;
          int r, t;
          if (packed) { r = c_pairs.rt[nn] >> 8; t = c_pairs.rt[nn] & 0xff; }
          else { r = nn >> 6; t = nn & 63; }
          w = Ch[nn] * q[r] * q[t] * 0.015625f;          // C_rt q_r q_t / 64
        } else {
          w = 0.f;
        }
        ph[i * (kFB + 1) + jf] = w;
      }
      __syncthreads();
#pragma unroll 4
      for (int j = 0; j < kFB; ++j) {
        const float p = ph[row * (kFB + 1) + j];
#pragma unroll
        for (int m = 0; m < 17; ++m) {
          const int col = cq + 4 * m;
          if (col < kU) acc[m] = fmaf(p, Ss[j * kU + col], acc[m]);
        }
      }
    }
  }

  // ---- intra-chunk pairs: kappa(q_i, k_j) u_j for chunk start <= j <= i   (Eq. 7)
  {
    float *kp = work;                  // [64 tokens][kP] k (group order)
    float *us = kp + kTile * kP;       // [64 tokens][kP] u = [v; 1]
    float *kap = us + kTile * kP;      // [64 rows][kP]
    const int cs = chunk * C;
    const int i_last = min(T, i0 + kTile) - 1;
    for (int jb = cs; jb <= i_last; jb += kTile) {
      __syncthreads();
      for (int n = tid; n < kTile * kD; n += kThreads) {
        const int j = n >> 6, r = n & 63;
        const int tok = jb + j;
        const bool ok = tok < T;
        kp[j * kP + r] = ok ? to_f32(K[(unit * T + tok) * kD + s_perm[r]]) : 0.f;
        us[j * kP + r] = ok ? to_f32(V[(unit * T + tok) * kDv + r]) : 0.f;
        if (r == 0) us[j * kP + kDv] = ok ? 1.f : 0.f;
      }
      __syncthreads();
      for (int n = tid; n < kTile * kTile; n += kThreads) {
        const int i = n >> 6, j = n & 63;
        float kapv = 0.f;
        if (jb + j <= i0 + i) {
          const float *q = qp + i * kP;
          const float *k = kp + j * kP;
          float sbar[kMaxG + 1];
          sbar[0] = 1.f;
#pragma unroll
          for (int g = 1; g <= kMaxG; ++g) {
            float s = 0.f;
            if (g <= G)
              for (int r = s_off[g]; r < s_off[g + 1]; ++r) s = fmaf(q[r], k[r], s);
            sbar[g] = s * 0.125f;                      // x_r = q_r k_r / sqrt(64)
          }
          float quad = 0.f;
#pragma unroll
          for (int cc = 0; cc <= kMaxG; ++cc) {
            if (cc <= G) {
              float w = 0.f;                           // (L^T s_bar)_cc
#pragma unroll
              for (int g = cc; g <= kMaxG; ++g)
                if (g <= G) w = fmaf(s_L[g * G1 + cc], sbar[g], w);
              quad = fmaf(w, w, quad);
            }
          }
          kapv = eps + quad;
        }
        kap[i * kP + j] = kapv;
      }
      __syncthreads();
#pragma unroll 4
      for (int j = 0; j < kTile; ++j) {
        const float p = kap[row * kP + j];
#pragma unroll
        for (int m = 0; m < 17; ++m) {
          const int col = cq + 4 * m;
          if (col < kU) acc[m] = fmaf(p, us[j * kP + col], acc[m]);
        }
      }
    }
  }

  // ---- normalise: y = u~[0:64] / u~[64]
  if (cq == 0) s_den[row] = acc[16];
  __syncthreads();
  const int tok = i0 + row;
  if (tok < T) {
    const float den = s_den[row];
    Tin *y = Y + (((size_t)bidx * Hq + h) * T + tok) * kDv;
#pragma unroll
    for (int m = 0; m < 16; ++m) y[cq + 4 * m] = from_f32<Tin>(acc[m] / den);
  }
}

constexpr size_t delta_smem() { return sizeof(float) * 3 * kTile * kP; }
constexpr size_t readout_smem() {
  return sizeof(float) * (2 * kTile * kP + 3 * kTile * kP);
}

}  // namespace

size_t simt_prefill_workspace_bytes(int B, int Hkv, int T, int packed, int chunk) {
  const size_t nC = (size_t)(T + chunk - 1) / chunk;
  return nC * B * Hkv * (size_t)state_rows(packed) * kU * sizeof(float);
}

template <typename Tin>
static oal_status launch_simt(const Tin *Q, const Tin *K, const Tin *V, int B,
                              int Hq, int Hkv, int T, const float *L,
                              const int32_t *group, int G, float eps,
                              const float *a, const float *b, const float *C,
                              int packed, float *state, int cont, Tin *Y,
                              int chunk, float *ws, cudaStream_t stream) {
  const int F = state_rows(packed);
  const int nC = (T + chunk - 1) / chunk;
  // shared-memory limits above 48 KB: a function attribute of each device
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return oal_fail(OAL_ERR_CUDA, "prefill: no current device");
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(chunk_delta_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)delta_smem()) != cudaSuccess ||
        cudaFuncSetAttribute(readout_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)readout_smem()) != cudaSuccess) {
      cudaGetLastError();   // reported here, not by the next launch
      return oal_fail(OAL_ERR_CUDA, "prefill: setting the shared memory limit failed");
    }
    attr_set[dev] = true;
  }
  dim3 g1((F + kTile - 1) / kTile, nC, B * Hkv);
  launch_pdl(chunk_delta_kernel<Tin>, g1, dim3(kThreads), delta_smem(), stream, K, V, T, chunk,
             nC, F, packed, ws);
  oal_status st = oal_after_launch("chunk_delta_kernel", stream);
  if (st != OAL_OK) return st;
  const size_t FU = (size_t)F * kU;
  dim3 g2((unsigned)((FU + 255) / 256), B * Hkv);
  launch_pdl(chunk_scan_kernel, g2, dim3(256), 0, stream, ws, nC, FU, state, cont);
  st = oal_after_launch("chunk_scan_kernel", stream);
  if (st != OAL_OK) return st;
  dim3 g3(nC * (chunk / kTile), B * Hq);
  launch_pdl(readout_kernel<Tin>, g3, dim3(kThreads), readout_smem(), stream, Q, K, V, Y, ws, a, b,
             C, L, group, G, eps, Hq, Hkv, T, chunk, nC, F, packed, oal_device_status_word());
  return oal_after_launch("readout_kernel", stream);
}

oal_status launch_prefill_simt(const void *Q, const void *K, const void *V,
                               int is_bf16, int B, int Hq, int Hkv, int T,
                               const float *L, const int32_t *group, int G,
                               float eps, const float *a, const float *b,
                               const float *C, int packed, float *state, int cont,
                               void *Y, int chunk, void *ws, cudaStream_t stream) {
  if (is_bf16)
    return launch_simt<__nv_bfloat16>(
        (const __nv_bfloat16 *)Q, (const __nv_bfloat16 *)K, (const __nv_bfloat16 *)V, B,
        Hq, Hkv, T, L, group, G, eps, a, b, C, packed, state, cont, (__nv_bfloat16 *)Y,
        chunk, (float *)ws, stream);
  return launch_simt<float>((const float *)Q, (const float *)K, (const float *)V, B, Hq,
                            Hkv, T, L, group, G, eps, a, b, C, packed, state, cont,
                            (float *)Y, chunk, (float *)ws, stream);
}

}  // namespace oal
