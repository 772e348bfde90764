// backward.cu -- gradients of the causal OAL output with respect to Q, K, V
// and L ([OAL] = "Not All Dimensions Are Equal: Outlier-Aware Attention
// Linearization with Grouped Quadratic Kernels"; the calibration of App. B,
// Eq. (20), and the LoRA adaptation of Sec. 5 differentiate through this
// operator).
//
// Forward (Sec. 2, Eq. (1); Sec. 4.3, Eq. (7)): for query row i and key j <= i,
//     s_bar = [1, s_1 .. s_G],  s_g = sum_{r in group g} q_r k_r / sqrt(d),
//     kappa_ij = eps + s_bar^T M s_bar,  M = L L^T,
//     D_i = sum_j kappa_ij,  y_i = sum_j kappa_ij v_j / D_i.
// Backward of <dY, Y>:
//     g_ij  = dY_i . (v_j - y_i) / D_i                  (d / d kappa_ij)
//     dV_j  = sum_{i >= j} kappa_ij dY_i / D_i
//     u_ij,g = 2 g_ij (M s_bar)_g / sqrt(d)             (d kappa / d s_g, scaled)
//     dQ_ir = sum_j u_ij,g(r) k_jr,   dK_jr = sum_i u_ij,g(r) q_ir
//     dM    = sum_ij g_ij s_bar s_bar^T,  dL = lower((dM + dM^T) L).
// The pairs are evaluated explicitly, O(T^2 d) per head, in fp32 on the CUDA
// cores: a query-major pass (D_i, y_i, c_i = dY_i . y_i, then dQ), a
// key-major pass per query head (its parts of dK, dV and dM), a kernel that
// sums the heads' parts of dK and dV in head order, and one that sums the dM
// partials in a fixed order and forms dL.  No atomics: the results are
// reproducible bit for bit.
//
// Group sums: the largest group (the bulk) is s - sum of the other groups,
// s = q . k over all 64 dims; the other groups' dims are read from a per-head
// list, so any partition works and the common case (a bulk group and a few
// small outlier groups) costs one 64-dim dot product per pair.  Two threads
// share a row (or key), 32 dims each.
#include <algorithm>
#include <mutex>

#include "oal_internal.cuh"

namespace oal {
namespace bw {

constexpr int kRowsPB = 64;                 // rows (or keys) of a block: two threads each
constexpr int kThreads = 2 * kRowsPB;
constexpr int kTile = 32;                   // streamed keys (or rows) per shared-memory tile
constexpr int kPitch = kD + 4;              // rows stay 16-byte aligned; own-row reads at most 2-way conflicted

// One head's constants, in shared memory.
struct HeadPlan {
  float M[8][8];       // L L^T from the lower triangle of L
  int gstar;           // the bulk group: the largest (the first of equals)
  int goff[9];         // dims of group g != gstar at tdims[goff[g] .. goff[g + 1])
  int tdims[kD];
};

// Thread 0 builds the plan of query head h (the block synchronises after).
template <int G>
__device__ void build_plan(HeadPlan &P, const float *__restrict__ L,
                           const int32_t *__restrict__ group, int h, int *status) {
  constexpr int G1 = G + 1;
  if (threadIdx.x < G1 * G1) {
    const int g = threadIdx.x / G1, c2 = threadIdx.x % G1;
    const float *Lh = L + (size_t)h * G1 * G1;
    float m = 0.f;
    for (int c = 0; c <= (g < c2 ? g : c2); ++c) m = fmaf(Lh[g * G1 + c], Lh[c2 * G1 + c], m);
    P.M[g][c2] = m;
  }
  if (threadIdx.x == 0) {
    int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int gid[kD];
    for (int r = 0; r < kD; ++r) {
      int g = group[(size_t)h * kD + r];
      if (g < 1 || g > G) {
        atomicCAS(status, kStatusOk, (int)OAL_ERR_INVALID_ARG);
        g = 1;
      }
      gid[r] = g;
      ++cnt[g];
    }
    int gs = 1;
    for (int g = 2; g <= G; ++g)
      if (cnt[g] > cnt[gs]) gs = g;
    P.gstar = gs;
    int o = 0;
    for (int g = 0; g <= G; ++g) {
      P.goff[g] = o;
      if (g >= 1 && g != gs)
        for (int r = 0; r < kD; ++r)
          if (gid[r] == g) P.tdims[o++] = r;
    }
    for (int g = G + 1; g <= 8; ++g) P.goff[g] = o;
  }
}

// sum_r a[r] b[r] over this thread's half, b 16-byte aligned in shared memory.
__device__ __forceinline__ float dot32(const float (&a)[32], const float *b) {
  const float4 *b4 = reinterpret_cast<const float4 *>(b);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 x = b4[v];
    s0 = fmaf(a[4 * v], x.x, s0);
    s1 = fmaf(a[4 * v + 1], x.y, s1);
    s0 = fmaf(a[4 * v + 2], x.z, s0);
    s1 = fmaf(a[4 * v + 3], x.w, s1);
  }
  return s0 + s1;
}
// acc[r] += w b[r] over this thread's half, b 16-byte aligned in shared memory.
__device__ __forceinline__ void axpy32(float w, const float *b, float (&acc)[32]) {
  const float4 *b4 = reinterpret_cast<const float4 *>(b);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 x = b4[v];
    acc[4 * v] = fmaf(w, x.x, acc[4 * v]);
    acc[4 * v + 1] = fmaf(w, x.y, acc[4 * v + 1]);
    acc[4 * v + 2] = fmaf(w, x.z, acc[4 * v + 2]);
    acc[4 * v + 3] = fmaf(w, x.w, acc[4 * v + 3]);
  }
}

// s_bar of one pair.  `a` is this thread's half (dims 32 hf ..) of its own
// vector, `arow` the whole own vector and `b` the streamed one, both in
// shared memory.  Both threads of the pair return the same values.
template <int G>
__device__ __forceinline__ void pair_sbar(const float (&a)[32], const float *arow, const float *b,
                                          const HeadPlan &P, int hf, float (&sb)[G + 1]) {
  const float sp = dot32(a, b + 32 * hf);
  const float s = sp + __shfl_xor_sync(0xffffffffu, sp, 1);
  float tot = 0.f;
#pragma unroll
  for (int g = 1; g <= G; ++g) {
    float acc = 0.f;
    for (int e = P.goff[g]; e < P.goff[g + 1]; ++e) {
      const int r = P.tdims[e];
      acc = fmaf(arow[r], b[r], acc);
    }
    sb[g] = acc * 0.125f;
    tot += acc;
  }
  sb[0] = 1.f;
#pragma unroll
  for (int g = 1; g <= G; ++g)
    if (g == P.gstar) sb[g] = (s - tot) * 0.125f;
}

// m = M s_bar and kappa = eps + s_bar . m.
template <int G>
__device__ __forceinline__ float pair_kappa(const HeadPlan &P, const float (&sb)[G + 1], float eps,
                                            float (&m)[G + 1]) {
  float kap = eps;
#pragma unroll
  for (int g = 0; g <= G; ++g) {
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h <= G; ++h) acc = fmaf(P.M[g][h], sb[h], acc);
    m[g] = acc;
    kap = fmaf(sb[g], acc, kap);
  }
  return kap;
}

// Add u_{g(r)} b_r to this thread's half of the gradient (registers: the
// bulk group's u for every dim) and the difference for the other groups'
// dims (shared memory, indexed by dim; the thread owning the dim's half).
template <int G>
__device__ __forceinline__ void add_grad(const HeadPlan &P, const float (&u)[G + 1], const float *b,
                                         int hf, float (&acc)[32], float *corr) {
  float ub = 0.f;
#pragma unroll
  for (int g = 1; g <= G; ++g)
    if (g == P.gstar) ub = u[g];
  axpy32(ub, b + 32 * hf, acc);
#pragma unroll
  for (int g = 1; g <= G; ++g) {
    const float du = u[g] - ub;
    for (int e = P.goff[g]; e < P.goff[g + 1]; ++e) {
      const int r = P.tdims[e];
      if ((r >> 5) == hf) corr[r] = fmaf(du, b[r], corr[r]);
    }
  }
}

struct BwArgs {
  const void *Q, *K, *V, *dY;
  int is_bf16;
  int B, Hq, Hkv, T, rho, ntiles;   // ntiles = ceil(T / kRowsPB)
  const float *L;
  const int32_t *group;
  float eps;
  float *dQ, *dK, *dV, *dL;
  float *Dn, *Cn;   // [B][Hq][T]: D_i and c_i = dY_i . y_i
  float *dMp;       // [B * Hkv][ntiles][rho][8][8]: partial dM of each key-major block
  float *dKp, *dVp; // [rho][B][Hkv][T][64]: each query head's part of dK, dV (dK, dV if rho = 1)
  int *status;
};

__device__ __forceinline__ float ld_in(const void *p, size_t idx, int is_bf16) {
  return is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[idx])
                 : static_cast<const float *>(p)[idx];
}

// Rows [64 t, 64 t + 64) of `src` (tokens of one head, 64 dims) into `dst`
// (pitch kPitch), zero past T.
__device__ __forceinline__ void load_rows(float *dst, int nrows, const void *src, size_t row_base,
                                          int first, int T, int is_bf16) {
  for (int e = threadIdx.x; e < nrows * kD; e += kThreads) {
    const int r = e / kD, c = e % kD, tok = first + r;
    dst[r * kPitch + c] = tok < T ? ld_in(src, (row_base + tok) * kD + c, is_bf16) : 0.f;
  }
}

constexpr size_t kRowsSmem = (size_t)(2 * kRowsPB + 2 * kTile) * kPitch * sizeof(float);

// Query-major pass: one block per (64 query rows, batch x query head).
// Pass A over the keys j <= i: D_i and the numerator, hence y_i and
// c_i = dY_i . y_i; pass B: g_ij and dQ_i.
template <int G>
__global__ void __launch_bounds__(kThreads) bw_rows_kernel(BwArgs a) {
  extern __shared__ float smf[];
  float *qS = smf;                          // the block's query rows
  float *corr = qS + kRowsPB * kPitch;      // dQ of the non-bulk dims
  float *kS = corr + kRowsPB * kPitch;      // key tile
  float *vS = kS + kTile * kPitch;          // value tile
  __shared__ HeadPlan P;
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int bidx = bh / a.Hq, h = bh % a.Hq, kv = h / a.rho;
  const int tid = threadIdx.x, row = tid >> 1, hf = tid & 1;
  const int row0 = tile * kRowsPB, i = row0 + row;
  const bool vi = i < a.T;
  pdl_trigger();
  pdl_wait();
  build_plan<G>(P, a.L, a.group, h, a.status);
  const size_t qbase = ((size_t)bidx * a.Hq + h) * a.T;
  const size_t kbase = ((size_t)bidx * a.Hkv + kv) * a.T;
  load_rows(qS, kRowsPB, a.Q, qbase, row0, a.T, a.is_bf16);
  for (int e = tid; e < kRowsPB * kPitch; e += kThreads) corr[e] = 0.f;
  __syncthreads();
  const float *arow = qS + row * kPitch;
  float q[32], dy[32], acc[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    q[r] = arow[32 * hf + r];
    dy[r] = vi ? ld_in(a.dY, (qbase + i) * kD + 32 * hf + r, a.is_bf16) : 0.f;
    acc[r] = 0.f;
  }
  const int jend = min(a.T, row0 + kRowsPB);   // keys 0 .. jend - 1
  float D = 0.f;
  for (int jt = 0; jt < jend; jt += kTile) {
    __syncthreads();
    load_rows(kS, kTile, a.K, kbase, jt, a.T, a.is_bf16);
    load_rows(vS, kTile, a.V, kbase, jt, a.T, a.is_bf16);
    __syncthreads();
    const int nj = min(kTile, jend - jt);
    for (int jj = 0; jj < nj; ++jj) {
      float sb[G + 1], m[G + 1];
      pair_sbar<G>(q, arow, kS + jj * kPitch, P, hf, sb);
      const float kap = pair_kappa<G>(P, sb, a.eps, m);
      const float w = (vi && jt + jj <= i) ? kap : 0.f;
      D += w;
      axpy32(w, vS + jj * kPitch + 32 * hf, acc);
    }
  }
  const float invD = vi ? 1.f / D : 0.f;
  float cp = 0.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) cp = fmaf(dy[r], acc[r] * invD, cp);
  const float c = cp + __shfl_xor_sync(0xffffffffu, cp, 1);
#pragma unroll
  for (int r = 0; r < 32; ++r) acc[r] = 0.f;
  for (int jt = 0; jt < jend; jt += kTile) {
    __syncthreads();
    load_rows(kS, kTile, a.K, kbase, jt, a.T, a.is_bf16);
    load_rows(vS, kTile, a.V, kbase, jt, a.T, a.is_bf16);
    __syncthreads();
    const int nj = min(kTile, jend - jt);
    for (int jj = 0; jj < nj; ++jj) {
      float sb[G + 1], m[G + 1];
      pair_sbar<G>(q, arow, kS + jj * kPitch, P, hf, sb);
      pair_kappa<G>(P, sb, a.eps, m);
      const float dp = dot32(dy, vS + jj * kPitch + 32 * hf);
      const float dyv = dp + __shfl_xor_sync(0xffffffffu, dp, 1);
      const float g = (vi && jt + jj <= i) ? (dyv - c) * invD : 0.f;
      float u[G + 1];
#pragma unroll
      for (int gg = 0; gg <= G; ++gg) u[gg] = 0.25f * g * m[gg];   // 2 g m_g / sqrt(64)
      add_grad<G>(P, u, kS + jj * kPitch, hf, acc, corr + row * kPitch);
    }
  }
  if (vi) {
    float *dst = a.dQ + (qbase + i) * kD + 32 * hf;
    const float *cr = corr + row * kPitch + 32 * hf;
#pragma unroll
    for (int r = 0; r < 32; ++r) dst[r] = acc[r] + cr[r];
    if (hf == 0) {
      a.Dn[qbase + i] = D;
      a.Cn[qbase + i] = c;
    }
  }
}

constexpr size_t kColsSmem =
    (size_t)(2 * kRowsPB + 2 * kTile) * kPitch * sizeof(float) + 2 * kTile * sizeof(float);

// Key-major pass: one block per (64 keys, batch x KV head, query head of the
// KV head), over the query rows i >= j: that head's part of dV_j and dK_j and
// this block's part of the head's dM.
template <int G>
__global__ void __launch_bounds__(kThreads) bw_cols_kernel(BwArgs a) {
  constexpr int NE = (G + 1) * (G + 2) / 2;   // entries of the symmetric dM
  extern __shared__ float smf[];
  float *kOwn = smf;                        // the block's keys
  float *corr = kOwn + kRowsPB * kPitch;    // dK of the non-bulk dims
  float *qS = corr + kRowsPB * kPitch;      // query tile
  float *dyS = qS + kTile * kPitch;         // dY tile
  float *Dt = dyS + kTile * kPitch;         // D_i of the tile's rows
  float *Ct = Dt + kTile;                   // c_i of the tile's rows
  __shared__ HeadPlan P;
  __shared__ float red[kThreads / 32][NE];
  const int tile = blockIdx.x, bkv = blockIdx.y;
  const int bidx = bkv / a.Hkv, kv = bkv % a.Hkv;
  const int tid = threadIdx.x, row = tid >> 1, hf = tid & 1, lane = tid & 31, warp = tid >> 5;
  const int row0 = tile * kRowsPB, j = row0 + row;
  const bool vj = j < a.T;
  pdl_trigger();
  pdl_wait();   // D_i and c_i of the query-major pass
  const size_t kbase = ((size_t)bidx * a.Hkv + kv) * a.T;
  load_rows(kOwn, kRowsPB, a.K, kbase, row0, a.T, a.is_bf16);
  for (int e = tid; e < kRowsPB * kPitch; e += kThreads) corr[e] = 0.f;
  __syncthreads();
  const float *krow = kOwn + row * kPitch;
  float k[32], v[32], dk[32], dv[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    k[r] = krow[32 * hf + r];
    v[r] = vj ? ld_in(a.V, (kbase + j) * kD + 32 * hf + r, a.is_bf16) : 0.f;
    dk[r] = 0.f;
    dv[r] = 0.f;
  }
  {
    const int hh = blockIdx.z;
    const int h = kv * a.rho + hh;
    const size_t qbase = ((size_t)bidx * a.Hq + h) * a.T;
    __syncthreads();
    build_plan<G>(P, a.L, a.group, h, a.status);
    float dm[(NE + 1) / 2];
#pragma unroll
    for (int e = 0; e < (NE + 1) / 2; ++e) dm[e] = 0.f;
    for (int it = row0; it < a.T; it += kTile) {
      __syncthreads();
      load_rows(qS, kTile, a.Q, qbase, it, a.T, a.is_bf16);
      load_rows(dyS, kTile, a.dY, qbase, it, a.T, a.is_bf16);
      if (tid < kTile) {
        const int i = it + tid;
        Dt[tid] = i < a.T ? a.Dn[qbase + i] : 1.f;
        Ct[tid] = i < a.T ? a.Cn[qbase + i] : 0.f;
      }
      __syncthreads();
      const int ni = min(kTile, a.T - it);
      for (int ii = 0; ii < ni; ++ii) {
        float sb[G + 1], m[G + 1];
        pair_sbar<G>(k, krow, qS + ii * kPitch, P, hf, sb);
        const float kap = pair_kappa<G>(P, sb, a.eps, m);
        const bool ok = vj && it + ii >= j;
        const float invD = 1.f / Dt[ii];
        const float *dyr = dyS + ii * kPitch + 32 * hf;
        const float dp = dot32(v, dyr);
        const float dyv = dp + __shfl_xor_sync(0xffffffffu, dp, 1);
        const float g = ok ? (dyv - Ct[ii]) * invD : 0.f;
        const float pv = ok ? kap * invD : 0.f;
        axpy32(pv, dyr, dv);
        float u[G + 1];
#pragma unroll
        for (int gg = 0; gg <= G; ++gg) u[gg] = 0.25f * g * m[gg];   // 2 g m_g / sqrt(64)
        add_grad<G>(P, u, qS + ii * kPitch, hf, dk, corr + row * kPitch);
        // this thread's half of the dM entries (x, y >= x): those of parity hf
        int e = 0;
#pragma unroll
        for (int x = 0; x <= G; ++x)
#pragma unroll
          for (int y = x; y <= G; ++y, ++e)
            if ((e & 1) == hf) dm[e >> 1] = fmaf(g * sb[x], sb[y], dm[e >> 1]);
      }
    }
    // the block's dM of head hh: sum over the lanes of each parity, then the warps
#pragma unroll
    for (int e2 = 0; e2 < (NE + 1) / 2; ++e2) {
      float x = dm[e2];
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      const int e = 2 * e2 + hf;
      if ((lane >> 1) == 0 && e < NE) red[warp][e] = x;
    }
    __syncthreads();
    if (tid < NE) {
      int x = 0, e = tid;
      while (e > G - x) {
        e -= G - x + 1;
        ++x;
      }
      const int y = x + e;
      float tot = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) tot += red[w][tid];
      float *dst = a.dMp + ((((size_t)bidx * a.Hkv + kv) * a.ntiles + tile) * a.rho + hh) * 64;
      dst[x * 8 + y] = tot;
      dst[y * 8 + x] = tot;
    }
  }
  if (vj) {
    const size_t part = (size_t)blockIdx.z * a.B * a.Hkv * a.T * kD;
    float *dkd = a.dKp + part + (kbase + j) * kD + 32 * hf;
    float *dvd = a.dVp + part + (kbase + j) * kD + 32 * hf;
    const float *cr = corr + row * kPitch + 32 * hf;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      dkd[r] = dk[r] + cr[r];
      dvd[r] = dv[r];
    }
  }
}

// dK and dV: the query heads' parts summed in head order (rho > 1).
__global__ void __launch_bounds__(256) bw_kv_reduce_kernel(BwArgs a) {
  pdl_trigger();
  pdl_wait();
  const size_t n4 = (size_t)a.B * a.Hkv * a.T * kD / 4;
  const float4 *kp = reinterpret_cast<const float4 *>(a.dKp);
  const float4 *vp = reinterpret_cast<const float4 *>(a.dVp);
  for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < n4;
       x += (size_t)gridDim.x * blockDim.x) {
    float4 sk = kp[x], sv = vp[x];
    for (int hh = 1; hh < a.rho; ++hh) {
      const float4 k4 = kp[hh * n4 + x], v4 = vp[hh * n4 + x];
      sk.x += k4.x; sk.y += k4.y; sk.z += k4.z; sk.w += k4.w;
      sv.x += v4.x; sv.y += v4.y; sv.z += v4.z; sv.w += v4.w;
    }
    reinterpret_cast<float4 *>(a.dK)[x] = sk;
    reinterpret_cast<float4 *>(a.dV)[x] = sv;
  }
}

// dL of one query head: its dM partials summed in a fixed order (batch, key
// tile), then dL = lower((dM + dM^T) L).
template <int G>
__global__ void __launch_bounds__(64) bw_dl_kernel(BwArgs a) {
  constexpr int G1 = G + 1;
  __shared__ float dM[8][8];
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, kv = h / a.rho, hh = h % a.rho, t = threadIdx.x;
  if (t < G1 * G1) {
    const int x = t / G1, y = t % G1;
    float tot = 0.f;
    for (int b = 0; b < a.B; ++b)
      for (int tile = 0; tile < a.ntiles; ++tile)
        tot += a.dMp[((((size_t)b * a.Hkv + kv) * a.ntiles + tile) * a.rho + hh) * 64 + x * 8 + y];
    dM[x][y] = tot;
  }
  __syncthreads();
  if (t < G1 * G1) {
    const int x = t / G1, c = t % G1;
    const float *Lh = a.L + (size_t)h * G1 * G1;
    float acc = 0.f;
    if (c <= x)
      for (int z = c; z <= G; ++z) acc = fmaf(dM[x][z] + dM[z][x], Lh[z * G1 + c], acc);
    a.dL[(size_t)h * G1 * G1 + t] = acc;
  }
}

struct BwLayout {
  size_t dn_off, cn_off, dm_off, kp_off, vp_off, total;
};
static BwLayout bw_layout(int B, int Hq, int Hkv, int T) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwLayout l;
  const int ntiles = (T + kRowsPB - 1) / kRowsPB;
  size_t o = 0;
  l.dn_off = o; o = al(o + (size_t)B * Hq * T * sizeof(float));
  l.cn_off = o; o = al(o + (size_t)B * Hq * T * sizeof(float));
  l.dm_off = o; o = al(o + (size_t)B * Hkv * ntiles * (Hq / Hkv) * 64 * sizeof(float));
  const size_t parts = Hq / Hkv > 1 ? (size_t)Hq / Hkv * B * Hkv * T * kD * sizeof(float) : 0;
  l.kp_off = o; o = al(o + parts);
  l.vp_off = o; o = al(o + parts);
  l.total = o < 256 ? 256 : o;
  return l;
}

template <int G>
static oal_status launch_bw_g(const BwArgs &a, cudaStream_t stream) {
  static std::mutex mu;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return oal_fail(OAL_ERR_CUDA, "backward: no current device below ordinal %d", kMaxDevices);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(bw_rows_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kRowsSmem) != cudaSuccess ||
          cudaFuncSetAttribute(bw_cols_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kColsSmem) != cudaSuccess) {
        cudaGetLastError();
        return oal_fail(OAL_ERR_CUDA, "backward: setting the shared memory limit failed");
      }
      attr_set[dev] = true;
    }
  }
  launch_pdl(bw_rows_kernel<G>, dim3(a.ntiles, a.B * a.Hq), dim3(kThreads), kRowsSmem, stream, a);
  oal_status st = oal_after_launch("bw_rows_kernel", stream);
  if (st != OAL_OK) return st;
  launch_pdl(bw_cols_kernel<G>, dim3(a.ntiles, a.B * a.Hkv, a.rho), dim3(kThreads), kColsSmem,
             stream, a);
  st = oal_after_launch("bw_cols_kernel", stream);
  if (st != OAL_OK) return st;
  if (a.rho > 1) {
    const size_t n4 = (size_t)a.B * a.Hkv * a.T * kD / 4;
    const unsigned nb = (unsigned)std::min<size_t>((n4 + 255) / 256, 4 * 152);
    launch_pdl(bw_kv_reduce_kernel, dim3(nb), dim3(256), 0, stream, a);
    st = oal_after_launch("bw_kv_reduce_kernel", stream);
    if (st != OAL_OK) return st;
  }
  launch_pdl(bw_dl_kernel<G>, dim3(a.Hq), dim3(64), 0, stream, a);
  return oal_after_launch("bw_dl_kernel", stream);
}

}  // namespace bw

size_t backward_workspace_bytes(int B, int Hq, int Hkv, int T) {
  return bw::bw_layout(B, Hq, Hkv, T).total;
}

oal_status launch_backward(const void *Q, const void *K, const void *V, const void *dY, int is_bf16,
                           int B, int Hq, int Hkv, int T, const float *L, const int32_t *group,
                           int G, float eps, float *dQ, float *dK, float *dV, float *dL, void *ws,
                           cudaStream_t stream) {
  using namespace bw;
  const BwLayout lay = bw_layout(B, Hq, Hkv, T);
  BwArgs a;
  a.Q = Q; a.K = K; a.V = V; a.dY = dY; a.is_bf16 = is_bf16;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.T = T; a.rho = Hq / Hkv;
  a.ntiles = (T + kRowsPB - 1) / kRowsPB;
  a.L = L; a.group = group; a.eps = eps;
  a.dQ = dQ; a.dK = dK; a.dV = dV; a.dL = dL;
  uint8_t *w = static_cast<uint8_t *>(ws);
  a.Dn = reinterpret_cast<float *>(w + lay.dn_off);
  a.Cn = reinterpret_cast<float *>(w + lay.cn_off);
  a.dMp = reinterpret_cast<float *>(w + lay.dm_off);
  a.dKp = a.rho > 1 ? reinterpret_cast<float *>(w + lay.kp_off) : dK;
  a.dVp = a.rho > 1 ? reinterpret_cast<float *>(w + lay.vp_off) : dV;
  a.status = oal_device_status_word();
  if (!a.status) return oal_fail(OAL_ERR_CUDA, "backward: device status word unavailable");
  switch (G) {
    case 1: return launch_bw_g<1>(a, stream);
    case 2: return launch_bw_g<2>(a, stream);
    case 3: return launch_bw_g<3>(a, stream);
    case 4: return launch_bw_g<4>(a, stream);
    case 5: return launch_bw_g<5>(a, stream);
    case 6: return launch_bw_g<6>(a, stream);
    default: return launch_bw_g<7>(a, stream);
  }
}

}  // namespace oal
