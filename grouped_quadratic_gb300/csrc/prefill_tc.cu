// prefill_tc.cu -- chunked causal OAL prefill on the Blackwell tensor cores
// (tcgen05 UMMA, tensor memory, TMA), bf16 inputs, fp32 states.
//
// [OAL] = "Not All Dimensions Are Equal: Outlier-Aware Attention
// Linearization with Grouped Quadratic Kernels".  For token i of chunk c
// (C = 64, 128 or 256 tokens)
//     u~_i = Phi~(q_i)^T S_{c-1}  +  sum_{j in c, j <= i} kappa(q_i, k_j) u_j,
// S_{c-1} = the Eq. (5) prefix states over all tokens before the chunk,
// Phi~ = the Eq. (6) readout weights, kappa = Eq. (7).  The split is exact
// (App. D, Eq. (25)).  The kernels work on 128-token stages and 128-row
// tiles whatever C is: a tile is one chunk (C = 128), half of one (C = 256)
// or two (C = 64).
//
// Internal feature order (K of every contraction, 2192 = 35 x 64 - 48):
//   [0, 2112)     H2_rt in "paired" rows: for r = 0..63, t = (r & ~1) .. 63.
//                 Every row has even length, so bf16 pairs never straddle a
//                 row; the entry (r, r-1) of an odd row r duplicates
//                 (r-1, r) (H2 is symmetric) and carries readout weight 0.
//   [2112, 2176)  H1_r
//   2176          H0, then 15 zero features (the state's and the snapshots'
//                 row length; the readout's contraction stops at 2176 and
//                 adds the H0 term a S0 in its epilogue)
// Readout weights per head (from the oal_expand_coeffs tables):
//   H2: C_rt q_r q_t / 64 with multiplicity 2 for t > r (App. D packed
//   readout), H1: b_r q_r / 8, H0: a.
//
// Launches per call:
//   tc_prep_kernel      per query head: readout weights in the feature order
//                       above (bf16) and their rank-one record, the plan of
//                       the intra-chunk kappa (its quadratic form and the
//                       tensor-core feature table); K^T for the state kernel.
//   tc_state_kernel     mode 0 (only when the sequence is split into parts):
//                       per (feature tile, part): the part's total
//                       Delta S = sum phi(k_j) u_j^T.
//                       mode 1: per (feature tile, part): walk the part's
//                       stages with the fp32 running state in registers;
//                       before each chunk write its bf16 snapshot S_{c-1};
//                       the last part writes the final fp32 state.
//   tc_intra_tk_kernel  per (one or two query heads, 128-row tile):
//                       intra-chunk kappa from three UMMA products per
//                       32-key block (s = Q K^T and the tail-dim feature
//                       contractions T, U), three FMAs a pair, P.V by UMMA;
//                       numerators and denominators to the workspace.  The
//                       second half of a 256-token chunk has 256 keys: its
//                       second 128-key tile reloads K and V.
//   tc_readout_kernel   per (query head, 128-row tile, batch x KV head):
//                       inter-chunk readout Phi~(Q) S_{c-1} as a
//                       128 x 80 x 2176 UMMA (128 x 160 for C = 64: the
//                       snapshots of the tile's two chunks side by side;
//                       A = Phi~ built by threads straight into tensor
//                       memory, B = snapshots streamed by TMA), plus the
//                       intra-chunk rows, then normalisation.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>

#include "oal_internal.cuh"
#include "tc_ptx.cuh"

namespace oal {
namespace tcp {

using namespace oal::tc;

constexpr int kC = 128;          // tokens per chunk
constexpr int kKP = 2192;        // internal features
constexpr int kH2P = 2112;       // paired H2 features
constexpr int kNKB = 34;         // readout K blocks of 64: 33 of paired H2 features, 1 of H1
constexpr int kH0Feat = 2176;    // the H0 feature (constant term): added in the readout epilogue
constexpr int kTiles = 18;       // 128-feature tiles of the state kernel
constexpr int kN = 80;           // UMMA N of [v | 1]: 64 value columns, the "1" column, 15 zeros
constexpr int kMaxNH = 1;        // query heads per readout block (four blocks per SM)
constexpr int kMaxTailG = 6;     // tail groups (G - 1 <= 6)
// Snapshot rows: the 64 value columns and the "1" column; the readout's TMA box
// is kN = 80 rows high and reads rows 65..79 as zero (out of range).
constexpr int kSnapRows = kU;
constexpr size_t kSnapBytes = (size_t)kSnapRows * kKP * 2;   // 284,960 B per (unit, chunk)
// Rank-one form of the H2 readout weights of one query head.  With
// C_rt = M_{g(r) g(t)}, w(r, t) = alpha_r pw_t for every pair that is not
// inside the tail groups on both sides (alpha_r = M_{g(r) b} / M_bb, pw_t =
// 2 M_{b g(t)} / d, b the bulk group; the diagonal carries half of it).  The
// readout builds such a word as bf16(alpha_r q_r) * bf16(pw_t q_t), one
// multiply, and overwrites the few other words ("exceptions") with
// q_r q_t w(r, t).  Heads whose table does not have this form (or has too many
// exceptions) take the general path with the weights of the table.
constexpr int kExcMax = 32;
constexpr int kH2Words = kH2P / 2;        // 1056 bf16 pairs
constexpr int kH2Halves = kH2Words / 16;  // 66 half blocks of 16 words
struct RFactor {
  float pw[64];
  float alpha[64];
  float exc_wlo[kExcMax];      // weights of the low / high feature of each exception word
  float exc_whi[kExcMax];
  uint16_t exc_word[kExcMax];  // word index in the paired H2 order, ascending
  uint16_t exc_rt[kExcMax];    // its row r and low feature t (r << 8 | t): features (r, t), (r, t + 1)
  uint8_t exc_start[72];       // exceptions of half block hb: [exc_start[hb], exc_start[hb + 1])
  int factored;
  int nexc;
  int pad[4];
};
static_assert(sizeof(RFactor) % 16 == 0, "factor record alignment");
// Per query head: kKP bf16 readout weights, then the RFactor record.
constexpr int kCoefRow = kKP + (int)sizeof(RFactor) / 2;
static_assert((kCoefRow * 2) % 16 == 0 && (kKP * 2) % 16 == 0, "coef row alignment");

__host__ __device__ constexpr int row_len(int r) { return 64 - (r & ~1); }
__host__ __device__ constexpr int row_off(int r) {
  int o = 0;
  for (int i = 0; i < r; ++i) o += row_len(i);
  return o;
}
__host__ __device__ constexpr int feat_r(int f) {
  int r = 0;
  while (r < 63 && row_off(r + 1) <= f) ++r;
  return r;
}
__host__ __device__ constexpr int feat_t(int f) { return (feat_r(f) & ~1) + (f - row_off(feat_r(f))); }

static_assert(row_off(64) == kH2P, "paired H2 size");

// code: H2 -> r << 8 | t ; H1 -> 0x8000 | r ; H0 -> 0xC000 ; padding -> 0xFFFF
struct FeatTable {
  uint16_t code[kKP];
};
__host__ __device__ constexpr FeatTable make_feat_table() {
  FeatTable ft{};
  int f = 0;
  for (int r = 0; r < 64; ++r)
    for (int t = r & ~1; t < 64; ++t) ft.code[f++] = (uint16_t)((r << 8) | t);
  for (int r = 0; r < 64; ++r) ft.code[f++] = (uint16_t)(0x8000 | r);
  ft.code[f++] = 0xC000;
  while (f < kKP) ft.code[f++] = 0xFFFF;
  return ft;
}
static __device__ const FeatTable g_feat = make_feat_table();

// Row of the external state (FULL or PACKED layout) holding feature `code`;
// -1 for padding.  `mirror` (FULL only) receives the (t, r) row or -1.
__device__ __forceinline__ int ext_row(uint16_t code, int packed, int *mirror) {
  *mirror = -1;
  if (code == 0xFFFF) return -1;
  if (code == 0xC000) return 0;
  if (code & 0x8000) return 1 + (code & 0xff);
  int r = code >> 8, t = code & 0xff;
  if (t < r) { const int x = r; r = t; t = x; }   // duplicate of (r-1, r)
  if (packed) return 1 + kD + r * kD - r * (r - 1) / 2 + (t - r);
  if (t != r) *mirror = 1 + kD + t * kD + r;
  return 1 + kD + r * kD + t;
}

// H2 entry (r, r-1) of an odd row: a copy of (r-1, r), not exported.
__device__ __forceinline__ bool is_duplicate(uint16_t code) {
  return !(code & 0x8000) && (code >> 8) > (code & 0xff);
}

// Constants of the intra-chunk kernel evaluation for one query head.
//   w_c = L00 [c == 0] + alpha_c s + sum_g' beta[g'][c] s_g',
//   kappa = eps + sum_c w_c^2,
// where s = q.k (unscaled) and s_g' = sum over the dims of tail group g' of
// q_r k_r.  The bulk group g* (largest) is eliminated through
// s_{g*} = s - sum_{g != g*} s_g; alpha/beta carry the 1/sqrt(64) scale.
// Features of the tensor-core kappa of tc_intra_tk_kernel in a 64-column row:
// T's linear feature of tail dim i at column i (i < kTkMaxLin), its pair
// (i, j), i <= j, at kTkMaxLin + tk_pair(i, j) (44 columns, zero up to 48),
// then U's linear feature of tail dim i at column kTkU0 + i.
constexpr int kTkMaxLin = 8;
constexpr int kTkFeat = kTkMaxLin + kTkMaxLin * (kTkMaxLin + 1) / 2;
constexpr int kTkU0 = 48;
__host__ __device__ constexpr int tk_pair(int i, int j) {
  return i * kTkMaxLin - i * (i - 1) / 2 + (j - i);
}
static_assert(kTkFeat <= kTkU0 && kTkU0 % 16 == 0 && kTkU0 + kTkMaxLin <= 64,
              "T over K = 48 and U over K = 16 of one 64-column feature row");

struct KPlan {
  float alpha[8];
  float beta[kMaxTailG][8];
  float L00, eps;
  // kappa as a quadratic form in z = (s, tail sums), Horner order:
  // kappa = max(eps, c0 + sum_v z_v (lin_v + sum_{w >= v} quad[v, w] z_w))
  float c0;
  float lin[8];
  float quad[36];
  int ntg;                     // tail groups (G - 1)
  int nd[kMaxTailG];           // dims per tail group
  int dims[kMaxTailG][2];      // the dims when nd <= 2 (fast path)
  int fast;                    // every tail group has <= 2 dims
  int goff[kMaxTailG + 1];     // generic path: dims of tail group g' in gdims[goff[g']..]
  int gdims[64];
  int G;
  // tensor-core kappa (tc_intra_tk_kernel): 1 when every tail dim has a
  // feature (a fast plan with at most kTkMaxLin tail dims); the dims in slot
  // order; the coefficients of each feature for T and for U (zero past nlin)
  int tk_mode, tk_nlin;
  int tk_dim[kTkMaxLin];
  float tk_cT[kTkFeat];
  float tk_cU[kTkMaxLin];
  int pad_[3];                 // (a multiple of 16 bytes: copied by bulk copy)
};
static_assert(sizeof(KPlan) % 16 == 0, "plan size");

// The dynamic shared memory rounded up to a 1024-byte boundary (swizzled
// tiles need it), by pointer arithmetic on the shared array itself so the
// compiler keeps the shared address space (shared loads, not generic ones).
__device__ __forceinline__ uint8_t *smem_align1024(uint8_t *raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// ---------------------------------------------------------------- prep
struct KtArgs {
  const __nv_bfloat16 *K;    // [U][T][64]
  __nv_bfloat16 *Kt;         // [U][64][Tpad]
  int T, Tpad, U, nC;
};

constexpr int kPrepThreads = 256;
static_assert(kPrepThreads == 256, "the K^T tiles and the coefficient rows assume 256 threads");

__global__ void __launch_bounds__(kPrepThreads)
tc_prep_kernel(const float *__restrict__ a, const float *__restrict__ b,
               const float *__restrict__ Ctab, const float *__restrict__ L,
               const int32_t *__restrict__ group, int G, float eps, int packed,
               __nv_bfloat16 *__restrict__ coef, KPlan *__restrict__ plans, int *status,
               KtArgs kt) {
  pdl_trigger();
  pdl_wait();
  const int ncoef = (kKP + 255) / 256;
  if ((int)blockIdx.y > ncoef + 1) {
    // ---- K^T for the state kernel: [unit][64 dims][nC * 128 tokens], zero past T
    __shared__ __nv_bfloat16 ks[kC][64 + 2];      // padded: column reads hit distinct banks
    const int ntr = (gridDim.y - ncoef - 2) * gridDim.x;
    for (int tile = blockIdx.x + gridDim.x * (blockIdx.y - ncoef - 2); tile < kt.U * kt.nC;
         tile += ntr) {
      const int u = tile / kt.nC, c = tile % kt.nC;
      __syncthreads();
      // 16-byte loads, all in flight before any is stored (blockDim.x == 256)
      uint4 v[kC * 8 / 256];
#pragma unroll
      for (int k = 0; k < kC * 8 / 256; ++k) {   // token j, 8-dim chunk
        const int e = threadIdx.x + 256 * k, j = e >> 3, d8 = e & 7, tok = c * kC + j;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (tok < kt.T)
          v[k] = *reinterpret_cast<const uint4 *>(kt.K + ((size_t)u * kt.T + tok) * 64 + 8 * d8);
      }
#pragma unroll
      for (int k = 0; k < kC * 8 / 256; ++k) {
        const int e = threadIdx.x + 256 * k, j = e >> 3, d8 = e & 7;
        uint32_t *row = reinterpret_cast<uint32_t *>(&ks[j][8 * d8]);
        row[0] = v[k].x; row[1] = v[k].y; row[2] = v[k].z; row[3] = v[k].w;
      }
      __syncthreads();
      __nv_bfloat16 *dst = kt.Kt + (size_t)u * 64 * kt.Tpad + (size_t)c * kC;
      for (int e = threadIdx.x; e < 64 * (kC / 2); e += blockDim.x) {   // dim d, token pair
        const int d = e / (kC / 2), jp = e % (kC / 2);
        const uint32_t lo = *reinterpret_cast<const uint16_t *>(&ks[2 * jp][d]);
        const uint32_t hi = *reinterpret_cast<const uint16_t *>(&ks[2 * jp + 1][d]);
        *reinterpret_cast<uint32_t *>(dst + (size_t)d * kt.Tpad + 2 * jp) = lo | (hi << 16);
      }
    }
    return;
  }
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const int G1 = G + 1;
  __shared__ int sgrp[kD];
  __shared__ float sL[64];
  __shared__ int scnt[8];
  if (tid < 8) scnt[tid] = 0;
  if (tid < G1 * G1) sL[tid] = L[(size_t)h * G1 * G1 + tid];
  __syncthreads();
  if (tid < kD) {
    int g = group[(size_t)h * kD + tid];
    if (g < 1 || g > G) { atomicCAS(status, kStatusOk, (int)OAL_ERR_INVALID_ARG); g = 1; }
    sgrp[tid] = g;
    atomicAdd(&scnt[g], 1);
  }
  // readout weights in the internal feature order (blockIdx.y < ncoef split
  // the rows); meanwhile block row ncoef forms the kappa plan and block row
  // ncoef + 1 the rank-one record of the weights
  const float *Ch = Ctab + (size_t)h * (packed ? kH2Packed : kH2Full);
  // weight of H2 entry (r, t), t >= r: C_rt / d with multiplicity two off the diagonal
  auto h2w = [&](int r, int t) -> float {
    if (packed) return Ch[r * kD - r * (r - 1) / 2 + (t - r)] * 0.015625f;
    return Ch[r * kD + t] * (t == r ? 0.015625f : 0.03125f);
  };
  for (int f = blockIdx.y * blockDim.x + tid; blockIdx.y < ncoef && f < kKP;
       f += blockDim.x * ncoef) {
    const uint16_t code = g_feat.code[f];
    float w = 0.f;
    if (code == 0xC000) {
      w = a[h];
    } else if (code == 0xFFFF) {
      w = 0.f;
    } else if (code & 0x8000) {
      w = b[(size_t)h * kD + (code & 0xff)] * 0.125f;
    } else {
      const int r = code >> 8, t = code & 0xff;
      w = t < r ? 0.f : h2w(r, t);
    }
    coef[(size_t)h * kCoefRow + f] = __float2bfloat16_rn(w);
  }
  __syncthreads();
  if (blockIdx.y != ncoef && blockIdx.y != ncoef + 1) return;
  // kappa constants: the bulk group g* is the largest; the others are tail groups
  int gstar = 1;
  for (int g = 2; g <= G; ++g)
    if (scnt[g] > scnt[gstar]) gstar = g;
  if (blockIdx.y == ncoef + 1) {
    // Rank-one form of the H2 weights (RFactor): b = g*, its first dim r*.
    __shared__ float spw[kD], salpha[kD];
    __shared__ uint8_t sexc[kH2Words];
    __shared__ uint16_t slist[kExcMax];
    __shared__ int sbad, snexc;
    // this head's C table and the feature codes in shared memory: every
    // check below reads them many times
    __shared__ __align__(16) float sC[kH2Full];
    __shared__ uint16_t scode[kH2P];
    const int nCt = packed ? kH2Packed : kH2Full;
    for (int i = tid; i < nCt / 4; i += blockDim.x)
      reinterpret_cast<float4 *>(sC)[i] = reinterpret_cast<const float4 *>(Ch)[i];
    for (int i = tid; i < kH2P; i += blockDim.x) scode[i] = g_feat.code[i];
    RFactor *F = reinterpret_cast<RFactor *>(coef + (size_t)h * kCoefRow + kKP);
    int rstar = 0;
    while (rstar < kD - 1 && sgrp[rstar] != gstar) ++rstar;
    if (tid == 0) sbad = 0;
    __syncthreads();
    auto h2ws = [&](int r, int t) -> float {   // h2w from the staged table
      if (packed) return sC[r * kD - r * (r - 1) / 2 + (t - r)] * 0.015625f;
      return sC[r * kD + t] * (t == r ? 0.015625f : 0.03125f);
    };
    if (tid < kD) {
      const int t = tid;
      spw[t] = t == rstar ? 2.f * h2ws(rstar, rstar) : h2ws(min(t, rstar), max(t, rstar));
    }
    __syncthreads();
    if (tid < kD) {
      const int r = tid;
      float al = 1.f;
      if (sgrp[r] != gstar) {
        if (spw[rstar] != 0.f) al = h2ws(min(r, rstar), max(r, rstar)) / spw[rstar];
        else sbad = 1;
      }
      salpha[r] = al;
    }
    __syncthreads();
    // exception words: a feature inside the tail groups on both sides, or one
    // whose table weight the rank-one form does not reproduce to fp32 rounding
    auto tail = [&](int d) { return sgrp[d] != gstar; };
    auto feat_exc = [&](int f) -> bool {
      const uint16_t code = scode[f];
      const int r = code >> 8, t = code & 0xff;
      if (t < r) return false;   // duplicate entry: weight 0 on both forms
      if (tail(r) && tail(t)) return true;
      const float want = h2ws(r, t);
      const float got = t == r ? 0.5f * salpha[r] * spw[r] : salpha[r] * spw[t];
      return !(fabsf(want - got) <= 4e-6f * fmaxf(fabsf(want), fabsf(got)));
    };
    for (int w = tid; w < kH2Words; w += blockDim.x)
      sexc[w] = (feat_exc(2 * w) || feat_exc(2 * w + 1)) ? 1 : 0;
    __syncthreads();
    {
      // ascending list, every thread: thread t scans words [kPer t, kPer t + kPer)
      constexpr int kPer = (kH2Words + kPrepThreads - 1) / kPrepThreads;
      __shared__ int swarp[kPrepThreads / 32];
      const int w0 = kPer * tid, lane = tid & 31;
      int cnt = 0;
      for (int i = 0; i < kPer; ++i) cnt += (w0 + i < kH2Words) ? sexc[w0 + i] : 0;
      int pre = cnt;
  #pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += v;
      }
      if (lane == 31) swarp[tid >> 5] = pre;
      __syncthreads();
      int base = 0, total = 0;
      for (int i = 0; i < kPrepThreads / 32; ++i) {
        base += i < (tid >> 5) ? swarp[i] : 0;
        total += swarp[i];
      }
      int pos = base + pre - cnt;
      for (int i = 0; i < kPer; ++i)
        if (w0 + i < kH2Words && sexc[w0 + i]) {
          if (pos < kExcMax) slist[pos] = (uint16_t)(w0 + i);
          ++pos;
        }
      if (tid == 0) snexc = total;
    }
    __syncthreads();
    const int nexc = snexc;
    const int nlist = nexc < kExcMax ? nexc : kExcMax;
    if (tid < kD) F->pw[tid] = spw[tid];
    if (tid >= 64 && tid < 128) F->alpha[tid - 64] = salpha[tid - 64];
    if (tid >= 128 && tid < 128 + kExcMax) {
      const int i = tid - 128;
      float wl = 0.f, wh = 0.f;
      uint16_t wd = 0, rt = 0;
      if (i < nlist) {
        wd = slist[i];
        const uint16_t cl = scode[2 * wd], ch = scode[2 * wd + 1];
        const int r = cl >> 8, tl = cl & 0xff, th = ch & 0xff;
        wl = tl < r ? 0.f : h2ws(r, tl);
        wh = th < r ? 0.f : h2ws(r, th);
        rt = cl;
      }
      F->exc_wlo[i] = wl;
      F->exc_whi[i] = wh;
      F->exc_word[i] = wd;
      F->exc_rt[i] = rt;
    }
    if (tid >= 160 && tid < 160 + 72) {
      const int hb = tid - 160;
      int n = 0;
      for (int i = 0; i < nlist; ++i) n += slist[i] < 16 * hb ? 1 : 0;
      F->exc_start[hb] = (uint8_t)(hb <= kH2Halves ? n : nlist);
    }
    if (tid == 0) {
      F->factored = (!sbad && nexc <= kExcMax) ? 1 : 0;
      F->nexc = nexc;
      for (int i = 0; i < 4; ++i) F->pad[i] = 0;
    }
    return;
  }
  auto Lat = [&](int g, int c) { return c <= g ? sL[g * G1 + c] : 0.f; };
  KPlan *P = plans + h;
  // tail slots: the non-empty groups other than g*, in group order.  An empty
  // group's sum is zero for every pair, so it takes no slot and the head's
  // kappa is a quadratic form in 1 + (its non-empty tail groups) variables.
  __shared__ int sslot[kMaxG + 1], sntg;
  if (tid == 0) {
    int n = 0;
    for (int g = 1; g <= G; ++g) sslot[g] = (g != gstar && scnt[g] > 0) ? n++ : -1;
    sntg = n;
  }
  // first dims of each tail group, one thread per dim: its rank in its group
  // from the groups' ballots over the 64 dims
  __shared__ uint32_t sball[2][kMaxG + 1];
  auto tail_off = [&](int g) {   // dims of the tail groups before g
    int off = 0;
    for (int gg = 1; gg < g; ++gg)
      if (gg != gstar) off += scnt[gg];
    return off;
  };
  if (tid < kD) {
    for (int gg = 1; gg <= G; ++gg) {
      const uint32_t m = __ballot_sync(0xffffffffu, sgrp[tid] == gg);
      if ((tid & 31) == 0) sball[tid >> 5][gg] = m;
    }
  }
  __syncthreads();
  if (tid < kD && sgrp[tid] != gstar) {
    const int r = tid, g = sgrp[r];
    const int slot = sslot[g];
    const int k = (r < 32 ? 0 : __popc(sball[0][g])) +
                  __popc(sball[r >> 5][g] & ((1u << (r & 31)) - 1u));
    P->gdims[tail_off(g) + k] = r;
    if (k < 2) P->dims[slot][k] = r;
  }
  if (tid >= 1 && tid <= G && sslot[tid] >= 0) {
    const int g = tid;
    const int slot = sslot[g];
    P->goff[slot] = tail_off(g);
    P->nd[slot] = scnt[g];
    if (scnt[g] < 2) P->dims[slot][1] = 0;
    if (scnt[g] < 1) P->dims[slot][0] = 0;
    for (int c = 0; c < 8; ++c) P->beta[slot][c] = c <= G ? (Lat(g, c) - Lat(gstar, c)) * 0.125f : 0.f;
  }
  if (tid == 0) {
    int fast = 1, tot = 0;
    for (int g = 1; g <= G; ++g)
      if (g != gstar) { fast &= scnt[g] <= 2; tot += scnt[g]; }
    for (int slot = sntg; slot < kMaxTailG; ++slot) {
      for (int c = 0; c < 8; ++c) P->beta[slot][c] = 0.f;
      P->nd[slot] = 0;
      P->dims[slot][0] = P->dims[slot][1] = 0;
      P->goff[slot] = tot;
    }
    P->goff[kMaxTailG] = tot;
    for (int c = 0; c < 8; ++c) P->alpha[c] = c <= G ? Lat(gstar, c) * 0.125f : 0.f;
    P->ntg = sntg;
    P->fast = fast;
    P->L00 = sL[0];
    P->eps = eps;
    P->G = G;
  }
  // quadratic form, one entry per thread: sbar_g = sum_v A[g][v] z_v with
  // z_0 = s, z_i = tail sum i; sbar_{g*} = (z_0 - sum_i z_i) / 8,
  // sbar_{g_i} = z_i / 8; M = L L^T.  A[g][v] has at most two non-zero
  // rows per column, so every entry is a sum of at most four terms of M.
  __shared__ int slot_group[8];     // tail slot -> group
  __shared__ float sM[8][8];        // M = L L^T, one entry per thread
  if (tid == 0) {
    int slot = 0;
    for (int g = 1; g <= G; ++g)
      if (sslot[g] >= 0) slot_group[++slot] = g;   // z index slot (1-based)
  }
  if (tid < G1 * G1) {
    const int g = tid / G1, h2 = tid % G1;
    float m = 0.f;
    for (int c = 0; c <= (g < h2 ? g : h2); ++c) m = fmaf(Lat(g, c), Lat(h2, c), m);
    sM[g][h2] = m;
  }
  __syncthreads();
  // the (at most two) groups g with d sbar_g / d z_v != 0, and those values
  auto deps = [&](int v, int (&gs)[2], float (&as)[2]) -> int {
    if (v == 0) { gs[0] = gstar; as[0] = 0.125f; return 1; }
    gs[0] = gstar; as[0] = -0.125f;
    gs[1] = slot_group[v]; as[1] = 0.125f;
    return 2;
  };
  const int Ge = sntg + 1;   // variables of the quadratic form: s and the tail sums
  const int nq = Ge * (Ge + 1) / 2;
  if (tid < nq) {
    int v = 0, rem = tid;
    while (rem >= Ge - v) { rem -= Ge - v; ++v; }
    const int w2 = v + rem;
    int gv[2], gw[2];
    float av[2], aw[2];
    const int nv = deps(v, gv, av), nw = deps(w2, gw, aw);
    float q = 0.f;   // the coefficients are +-1/8: the products are exact
    for (int i = 0; i < nv; ++i)
      for (int j = 0; j < nw; ++j) q += av[i] * sM[gv[i]][gw[j]] * aw[j];
    P->quad[tid] = w2 == v ? q : 2.f * q;
  } else if (tid < 36) {
    P->quad[tid] = 0.f;
  } else if (tid >= 64 && tid < 72) {
    const int v = tid - 64;
    float l = 0.f;
    if (v < Ge) {
      int gv[2];
      float av[2];
      const int nv = deps(v, gv, av);
      for (int i = 0; i < nv; ++i) l += 2.f * sM[0][gv[i]] * av[i];
    }
    P->lin[v] = l;
  } else if (tid == 96) {
    P->c0 = eps + sM[0][0];
  }
  __syncthreads();   // every field of the plan above is written
  if (tid == 0) {
    // the tail dims in slot order, then the coefficients of kappa's terms in
    // them: U = sum_r quad[0][1+a(r)] q_r k_r; T = sum_r lin[1+a(r)] q_r k_r +
    // sum_{r <= r'} w q_r q_r' k_r k_r' (w = quad[v][w], doubled for two dims
    // of one group)
    int nlin = 0, slot[kTkMaxLin];
    bool ok = P->fast != 0;
    for (int a2 = 0; a2 < P->ntg && ok; ++a2)
      for (int d = 0; d < P->nd[a2]; ++d) {
        if (nlin == kTkMaxLin) { ok = false; break; }
        P->tk_dim[nlin] = P->dims[a2][d];
        slot[nlin++] = a2;
      }
    auto qi = [&](int v, int w) { return v * Ge - v * (v - 1) / 2 + (w - v); };
    for (int f = 0; f < kTkFeat; ++f) P->tk_cT[f] = 0.f;
    for (int i = 0; i < kTkMaxLin; ++i) {
      P->tk_cU[i] = 0.f;
      if (i >= nlin) P->tk_dim[i] = 0;
    }
    if (ok) {
      for (int i = 0; i < nlin; ++i) {
        P->tk_cT[i] = P->lin[1 + slot[i]];
        P->tk_cU[i] = P->quad[qi(0, 1 + slot[i])];
        for (int j = i; j < nlin; ++j) {
          const int v = 1 + slot[i], w = 1 + slot[j];
          const float qvw = P->quad[qi(v, w)];
          P->tk_cT[kTkMaxLin + tk_pair(i, j)] = v == w && i != j ? 2.f * qvw : qvw;
        }
      }
    }
    P->tk_mode = ok ? 1 : 0;
    P->tk_nlin = ok ? nlin : 0;
  }
}

// ---------------------------------------------------------------- swizzle helpers
// Byte offset of 16-byte chunk `c` of row `m` in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int m, int c) {
  return (uint32_t)(m * 128 + ((c ^ (m & 7)) << 4));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int warp, int col) {
  return base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col;
}
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ================================================================= state kernel
// One block per (128-feature tile, part of the sequence, batch x KV head).
// Per chunk c of the part: Delta S_c = phi(K_c)^T [V_c | 1] by UMMA into one of two
// tensor-memory accumulators; phi is split exactly into two bf16 terms
// (hi = bf16(k_r k_t), lo = k_r k_t - hi; the product of two bf16 values has
// at most 16 significant bits), so the fp32 state is exact up to fp32
// accumulation.  B = [V_c | 1] is MN-major with N = 80: the V tile as loaded
// by TMA is its first 128-byte atom and one constant tile whose column 0 is 1
// its second (the descriptor's atom stride differs per stage).  The epilogue
// warps keep the running fp32 state of their
// feature row in registers, add each Delta S_c, and (mode 1) write the bf16
// snapshot S_{c-1} that the readout of chunk c consumes.
constexpr int kStateStages = 3;

struct __align__(1024) StateSmem {
  // [stage][K^T | V]: K^T as two [64 dims][64 tokens] halves, V as [128 tokens][64
  // dims]; every tile 128B-swizzled (16-byte chunk c of row r at c ^ (r & 7))
  __nv_bfloat16 kv[kStateStages][2][kC * 64];
  __nv_bfloat16 ones[kC * 64];                  // second atom of B: column 0 is 1
  // walk: the part's starting state, then (last part) the final state, one
  // row per feature of the tile (odd pitch: row reads are conflict-free)
  float rows[128][kU];
  uint64_t kv_full[kStateStages], kv_empty[kStateStages];
  uint64_t a_full[2], a_empty[2], d_full[2], d_empty[2];
  uint64_t drain;                               // every MMA of the block complete
  uint64_t never;                               // failure-path tests: nothing arrives
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(StateSmem) + 1024 <= 227 * 1024, "state shared memory");

struct StateArgs {
  int T;
  int nS;                    // 128-token stages: ceil(T / 128)
  int chunk;                 // snapshot period C: 64, 128 or 256 tokens
  int nC;                    // chunks: ceil(T / C)
  int spp;                   // stages per part (a multiple of C / 128 when C = 256)
  int U, nparts, packed, cont, mode;
  const float *state_in;     // external state (continue) or null
  float *state_out;          // external state (mode 1, last part)
  float *ptot;               // [U][nparts][kTiles][128][kN] fp32 part totals
  __nv_bfloat16 *snap;       // [U*nC][kSnapRows][kKP]
  int *status;
};

constexpr int kStateThreads = 512;
constexpr int kStateD = 0;          // accumulators at cols 0 and 128 (80 wide)
constexpr int kStateA = 256;        // A slots at 256 and 384: [hi 64 | lo 64]

__device__ __forceinline__ float bf16lo_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {   // a * b + c, two lanes
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_bf16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__global__ void __launch_bounds__(kStateThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                StateArgs args) {
  extern __shared__ uint8_t smem_raw[];
  StateSmem &s = *reinterpret_cast<StateSmem *>(smem_align1024(smem_raw));
  const int tile = blockIdx.x, part = blockIdx.y, unit = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the part's 128-token stages [s0, s1) and chunks [j0, j0 + nchunks)
  const int C = args.chunk;
  const int s0 = part * args.spp;
  const int s1 = min(args.nS, s0 + args.spp);
  const int nstages = s1 - s0;
  const int j0 = s0 * kC / C;
  const int nchunks = min(args.nC, (s1 * kC + C - 1) / C) - j0;
  const int mode = args.mode;
  // Mode 0 signals its dependents only after its own wait, so the walk
  // (mode 1) can never start before the prep kernel's K^T is complete; the
  // walk's part 0 needs no part totals and skips the wait, running on the SMs
  // mode 0 leaves idle.  Every other walk block waits, so the walk still
  // completes after mode 0.
  if (mode == 1) pdl_trigger();

  if (tid == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < kStateStages; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.a_full[i], 8);    // every builder warp
      mbar_init(&s.a_empty[i], 1);
      mbar_init(&s.d_full[i], 1);
      mbar_init(&s.d_empty[i], 4);
    }
    mbar_init(&s.drain, 1);
    mbar_init(&s.never, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp >= 4 && warp < 8) {
    // the constant atom of B: row j (token) holds 1 in column 0, 0 elsewhere
    const int j = tid - 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (c == 0) v.x = 0x3F80u;
      *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(s.ones) + sw128(j, c)) = v;
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  volatile int *abort_flag = &s.abort_flag;
  if (mode == 0 || part > 0 || args.nparts == 1) pdl_wait();   // see above
  if (mode == 0) pdl_trigger();
  if (mode == 1 && part > 0) {
    // Starting state of this part: the totals of parts 0 .. part-1 for this
    // tile, summed in part order.  Every thread owns fixed float4s of the
    // tile's [128][80] block and keeps up to four parts' loads in flight.
    constexpr int kV4 = 128 * kN / 4;                     // float4s per part and tile
    constexpr int kPer = (kV4 + kStateThreads - 1) / kStateThreads;
    float4 acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < part; p0 += 4) {
      float4 v[4][kPer];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int e = tid + kStateThreads * k;
          v[pp][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p0 + pp < part && e < kV4)
            v[pp][k] = reinterpret_cast<const float4 *>(
                args.ptot + (((size_t)unit * args.nparts + p0 + pp) * kTiles + tile) * 128 * kN)[e];
        }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          acc[k].x += v[pp][k].x; acc[k].y += v[pp][k].y;
          acc[k].z += v[pp][k].z; acc[k].w += v[pp][k].w;
        }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = tid + kStateThreads * k;
      if (e < kV4) {
        const int row = e / (kN / 4), c4 = 4 * (e % (kN / 4));
        const float a4[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c4 + j < kU) s.rows[row][c4 + j] = a4[j];
      }
    }
    __syncthreads();
  }

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      for (int i = 0; i < nstages; ++i) {
        const int st = i % kStateStages;
        if (!mbar_wait(&s.kv_empty[st], ((i / kStateStages) & 1) ^ 1, abort_flag, args.status))
          break;
        mbar_arrive_expect_tx(&s.kv_full[st], 2 * kC * 64 * 2);
        tma_load_3d(s.kv[st][0], &tmK, &s.kv_full[st], (s0 + i) * kC, 0, unit);
        tma_load_3d(s.kv[st][0] + 64 * 64, &tmK, &s.kv_full[st], (s0 + i) * kC + 64, 0, unit);
        tma_load_3d(s.kv[st][1], &tmV, &s.kv_full[st], 0, (s0 + i) * kC, unit);
        issued = i + 1;
      }
      // copies still in flight must land before the block exits
      for (int i = max(0, issued - kStateStages); i < issued; ++i)
        mbar_wait_teardown(&s.kv_full[i % kStateStages], (i / kStateStages) & 1, args.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp runs the loop with warp-uniform
    // operands; one elected lane issues): D[:, 0:80] += A x [V | 1] (N = 80),
    // A = phi(K)^T of one stage as hi | lo (K = 256 for its 128 tokens); B read
    // MN-major: the V atom straight from the TMA stage, the constant atom at
    // the stage's atom stride.  Accumulator slot j & 1 collects chunk j: a
    // stage is one chunk (C = 128), half of one (C = 256: the chunk's two
    // stages accumulate into one slot), or two (C = 64: one MMA group per
    // 64-token half, each into its own slot).
    const uint32_t idn = idesc_bf16_f32(128, kN, 1);
    const bool starve = args.status[1] == kStarveState;   // failure-path test only
    bool ok = true;
    for (int i = 0; i < nstages && ok; ++i) {
      const int sl = i & 1, st = i % kStateStages;
      if (!mbar_wait(starve && i == 0 ? &s.never : &s.a_full[sl], (i >> 1) & 1, abort_flag,
                     args.status))
        break;
      tc_fence_after();
      const uint64_t bd = sdesc_sw128(smem_u32(s.kv[st][1]),
                                      smem_u32(s.ones) - smem_u32(s.kv[st][1]), 1024);
      const uint32_t a0 = tb + kStateA + 128 * sl;
      const int ng = C == 64 ? 2 : 1;
      for (int g = 0; g < ng; ++g) {
        int j;               // local chunk of this MMA group
        bool first, last;    // the group opens / closes chunk j
        if (C == 64) { j = 2 * i + g; first = last = true; }
        else if (C == 128) { j = i; first = last = true; }
        else { j = i >> 1; first = (i & 1) == 0; last = (i & 1) == 1 || i == nstages - 1; }
        if (j >= nchunks) break;   // C = 64: the second half of a last stage lies past T
        if (first) {
          if (!mbar_wait(&s.d_empty[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t d = tb + kStateD + 128 * (j & 1);
        // 16-token k-steps k: A columns 8 k (k < 8: hi of tokens 16 k ..; k >= 8:
        // lo of tokens 16 (k - 8) ..), B token block k & 7
        const uint32_t acc0 = first ? 0u : 1u;
        if (C == 64) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {   // hi then lo of tokens 64 g .. 64 g + 63
            const int k = 4 * g + kk + (kk >= 4 ? 4 : 0);
            umma_ts_warp(d, a0 + 8 * k, bd + (uint64_t)(128 * (k & 7)), idn, kk > 0 ? 1u : acc0);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k)
            umma_ts_warp(d, a0 + 8 * k, bd + (uint64_t)(128 * (k & 7)), idn, k > 0 ? 1u : acc0);
        }
        if (last) umma_commit_warp(&s.d_full[j & 1]);
      }
      if (!ok) break;
      umma_commit_warp(&s.a_empty[sl]);
      umma_commit_warp(&s.kv_empty[st]);
    }
    // no MMA in flight at dealloc: one commit after every MMA issued
    umma_commit_warp(&s.drain);
    if (lane == 0) mbar_wait_teardown(&s.drain, 0, args.status);
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ---------------- builders: group bg builds tokens 64 bg .. 64 bg + 63 of
    // A = phi(K_c)^T (hi | lo) from the K^T half bg of the stage
    const int bg = (warp - 4) >> 2;
    const int l = 32 * (warp & 3) + lane;    // TMEM lane = feature row
    const int f = tile * 128 + l;
    const uint16_t code = f < kKP ? g_feat.code[f] : (uint16_t)0xFFFF;
    for (int i = 0; i < nstages; ++i) {
      const int sl = i & 1, st = i % kStateStages;
      if (!mbar_wait(&s.kv_full[st], (i / kStateStages) & 1, abort_flag, args.status)) break;
      // slot sl (A in tensor memory) is free once the UMMAs of stage i - 2 are done
      if (!mbar_wait(&s.a_empty[sl], ((i >> 1) & 1) ^ 1, abort_flag, args.status)) break;
      const int nvalid = min(kC, args.T - (s0 + i) * kC);
      const uint32_t abase = kStateA + 128 * sl;
      const uint8_t *kth = reinterpret_cast<const uint8_t *>(s.kv[st][0]) + bg * (64 * 128);
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int q = 2 * bg + qq;           // 32-token block
        uint32_t hi[16], lo[16];
        if (code == 0xFFFF) {
#pragma unroll
          for (int w = 0; w < 16; ++w) hi[w] = lo[w] = 0u;
        } else if (code == 0xC000) {
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const int j = 32 * q + 2 * w;
            hi[w] = (j < nvalid ? 0x3F80u : 0u) | (j + 1 < nvalid ? 0x3F800000u : 0u);
            lo[w] = 0u;
          }
        } else if (code & 0x8000) {
          const int rr = code & 0xff;
          const uint4 *kr = reinterpret_cast<const uint4 *>(kth + rr * 128);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 x = kr[(4 * qq + v) ^ (rr & 7)];
            hi[4 * v] = x.x; hi[4 * v + 1] = x.y; hi[4 * v + 2] = x.z; hi[4 * v + 3] = x.w;
            lo[4 * v] = lo[4 * v + 1] = lo[4 * v + 2] = lo[4 * v + 3] = 0u;
          }
        } else {
          const int rr = code >> 8, tt = code & 0xff;
          const uint4 *kr = reinterpret_cast<const uint4 *>(kth + rr * 128);
          const uint4 *kt = reinterpret_cast<const uint4 *>(kth + tt * 128);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 x = kr[(4 * qq + v) ^ (rr & 7)], y = kt[(4 * qq + v) ^ (tt & 7)];
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t h2 = hmul2(xs[e], ys[e]);
              hi[4 * v + e] = h2;
              lo[4 * v + e] = hfma2_bf16(xs[e], ys[e], h2 ^ 0x80008000u);   // exact residual
            }
          }
        }
        tmem_st16(tmem_lane_addr(tb, warp, abase + 16 * q), hi);
        tmem_st16(tmem_lane_addr(tb, warp, abase + 64 + 16 * q), lo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.a_full[sl]);
    }
  } else if (warp >= 12) {
    // ---------------- epilogue: running fp32 state of this feature row
    const int l = tid - 384;
    const int f = tile * 128 + l;
    const uint16_t code = f < kKP ? g_feat.code[f] : (uint16_t)0xFFFF;
    int mirror;
    const int erow = ext_row(code, args.packed, &mirror);
    const size_t FU = (size_t)state_rows(args.packed) * kU;
    float S[kU];   // columns 65..79 of the accumulators stay zero
#pragma unroll
    for (int n = 0; n < kU; ++n) S[n] = 0.f;
    if (mode == 1) {
      if (args.cont && erow >= 0) {
        const float *src = args.state_in + (size_t)unit * FU + (size_t)erow * kU;
#pragma unroll
        for (int n = 0; n < kU; ++n) S[n] = src[n];
      }
      if (part > 0) {
#pragma unroll
        for (int n = 0; n < kU; ++n) S[n] += s.rows[l][n];
      }
    }
    __nv_bfloat16 *snap_row =
        f < kKP ? args.snap + ((size_t)unit * args.nC + j0) * kSnapRows * kKP + f : nullptr;
    auto write_snapshot = [&](int cc) {   // S_{cc-1} for chunk cc of this part
      if (snap_row) {
        __nv_bfloat16 *dst = snap_row + (size_t)cc * kSnapRows * kKP;
#pragma unroll
        for (int n = 0; n < kSnapRows; ++n) dst[(size_t)n * kKP] = __float2bfloat16_rn(S[n]);
      }
    };
    if (mode == 1 && nchunks > 0) write_snapshot(0);
    bool ok = true;
    for (int i = 0; i < nchunks; ++i) {
      const int sl = i & 1;
      if (!mbar_wait(&s.d_full[sl], (i >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < kN / 16; ++q) {
        uint32_t r[16];
        tmem_ld16(tmem_lane_addr(tb, warp, kStateD + 128 * sl + 16 * q), r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (16 * q + e < kU) S[16 * q + e] += __uint_as_float(r[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.d_empty[sl]);
      if (mode == 1 && i + 1 < nchunks) write_snapshot(i + 1);
    }
    if (ok && !*abort_flag) {
      if (mode == 0) {
        float4 *dst = reinterpret_cast<float4 *>(
            args.ptot + ((((size_t)unit * args.nparts + part) * kTiles + tile) * 128 + l) * kN);
#pragma unroll
        for (int n4 = 0; n4 < 16; ++n4)
          dst[n4] = make_float4(S[4 * n4], S[4 * n4 + 1], S[4 * n4 + 2], S[4 * n4 + 3]);
        dst[16] = make_float4(S[64], 0.f, 0.f, 0.f);
#pragma unroll
        for (int n4 = 17; n4 < kN / 4; ++n4) dst[n4] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (part == args.nparts - 1) {
        // final state: this warp's 32 feature rows go through shared memory
        // and out as runs of consecutive external rows, each run written by
        // the whole warp with consecutive addresses
        const bool mine = erow >= 0 && !is_duplicate(code);
#pragma unroll
        for (int n = 0; n < kU; ++n) s.rows[l][n] = S[n];
        __syncwarp();
        const int prev = __shfl_up_sync(0xffffffffu, mine ? erow : -2, 1);
        const bool start = mine && (lane == 0 || prev != erow - 1);
        unsigned starts = __ballot_sync(0xffffffffu, start);
        const unsigned mask_mine = __ballot_sync(0xffffffffu, mine);
        while (starts) {
          const int a = __ffs(starts) - 1;
          starts &= starts - 1;
          // the run goes on while rows are mine and consecutive
          const unsigned after = ~((2u << a) - 1u);
          const unsigned breaks = (starts | ~mask_mine) & after;
          const int b = breaks ? __ffs(breaks) - 1 : 32;
          const int e0 = __shfl_sync(0xffffffffu, erow, a);
          float *dst = args.state_out + (size_t)unit * FU + (size_t)e0 * kU;
          const float *src = &s.rows[32 * (warp & 3) + a][0];
          for (int idx = lane; idx < (b - a) * kU; idx += 32) dst[idx] = src[idx];
        }
        if (mine && mirror >= 0) {
          float *dm = args.state_out + (size_t)unit * FU + (size_t)mirror * kU;
#pragma unroll
          for (int n = 0; n < kU; ++n) dm[n] = S[n];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ================================================================= readout kernel
constexpr int kNB = 3;           // snapshot K-block stages
constexpr int kNA = 3;           // A half slots (128 x 32 bf16, 16 columns) in tensor memory

// NS snapshots per 128-row tile: 1 (C = 128: the tile's chunk; C = 256: the
// chunk the tile is half of) or 2 (C = 64: rows 0..63 read S_{2t-1}, rows
// 64..127 read S_{2t}, as the two halves of one N = 160 operand).
template <int NS>
struct __align__(1024) ReadSmem {
  __nv_bfloat16 q[kMaxNH][kC * 64];    // 128B-swizzled [token][dim], then q^T [dim][token]
  __nv_bfloat16 b[kNB][NS * kN * 64];  // snapshot K blocks [n][64 features]
  __nv_bfloat16 coef[kMaxNH][kCoefRow];
  uint64_t qkv_full, b_full[kNB], a_full[kNA], a_empty[kNA], d_full;
  uint64_t never;                      // failure-path tests: nothing arrives
  uint32_t tmem_base;
  int abort_flag;
  int loaded;                          // snapshot K blocks whose load was issued
  float s0[NS][kU];                    // the snapshots' H0 rows (feature kH0Feat)
};
static_assert(4 * (sizeof(ReadSmem<1>) + 1024) <= 228 * 1024, "four readout blocks per SM");
static_assert(2 * (sizeof(ReadSmem<2>) + 2048) <= 228 * 1024, "two readout blocks per SM");

struct ReadArgs {
  int T, nC, chunk, Hq, Hkv, rho, nh_per_block;
  __nv_bfloat16 *Y;
  float *intra_num;            // intra-chunk numerators, per (B*Hq, 128-row tile) [16][128][4]
  float *intra_den;            // [B*Hq][T]     intra-chunk denominators
  const __nv_bfloat16 *coef;   // [Hq][kCoefRow]
  const KPlan *plans;          // [Hq]
  int *status;
  const __nv_bfloat16 *snap;   // [U*nC][kSnapRows][kKP] per-chunk snapshots
};

constexpr int kReadThreads = 160;   // 5 warps
constexpr int kTmemD = 0;         // D at [0, 80 NS)
template <int NS>
constexpr int kTmemA = 80 * NS;   // three A half slots of 16 columns
template <int NS>
constexpr uint32_t kReadTmemCols = NS == 1 ? 128 : 256;

// ---- readout A block builders (compile-time feature layout)
// The builder of token row m keeps p = bf16(pw * q) in registers and reads
// q from the transposed tile qT[dim][token] in shared memory, one
// conflict-free 16-bit load per value.  Rows r of the paired H2 order split
// into runs of words that share r; a word of a run is qs_r * p_t with
// qs_r = bf16(alpha_r q_r) formed once per run, the row's first word
// rescaled (the diagonal entry by 1/2, the duplicate (r, r - 1) by 0).
__device__ __forceinline__ uint32_t qt_ld(const __nv_bfloat16 *qcol, int r) {
  return *reinterpret_cast<const uint16_t *>(qcol + r * kC);
}

template <int KB, int H, int P0, int... I>
__device__ __forceinline__ void h2_run(uint32_t qr, const uint32_t (&p)[32], uint32_t (&out)[16],
                                       std::integer_sequence<int, I...>) {
  constexpr int r = feat_r(64 * KB + 2 * (16 * H + P0));
  constexpr uint32_t fix = (r & 1) ? 0x3F000000u : 0x3F803F00u;   // bf16x2 (0, 1/2) : (1/2, 1)
  ((out[P0 + I] = (64 * KB + 2 * (16 * H + P0 + I) == row_off(r))
                      ? hmul2(hmul2(qr, p[feat_t(64 * KB + 2 * (16 * H + P0 + I)) >> 1]), fix)
                      : hmul2(qr, p[feat_t(64 * KB + 2 * (16 * H + P0 + I)) >> 1])),
   ...);
}

template <int KB, int H, int P0>
__device__ __forceinline__ void h2_runs(const __nv_bfloat16 *qcol, const float *alpha,
                                        const uint32_t (&p)[32], uint32_t (&out)[16]) {
  constexpr int r = feat_r(64 * KB + 2 * (16 * H + P0));
  constexpr int end_w = row_off(r + 1) / 2 - 32 * KB - 16 * H;   // run end (word in half)
  constexpr int P1 = end_w < 16 ? end_w : 16;
  const float sr = alpha[r] * __uint_as_float(qt_ld(qcol, r) << 16);
  const uint32_t qr = pack_bf16x2(sr, sr);   // (bf16(alpha_r q_r), the same)
  h2_run<KB, H, P0>(qr, p, out, std::make_integer_sequence<int, P1 - P0>{});
  if constexpr (P1 < 16) h2_runs<KB, H, P1>(qcol, alpha, p, out);
}

// Words 16 H .. 16 H + 15 of K block KB of one A row (token row of Phi~(Q)),
// rank-one form; cw = this head's weights of block KB (the H1 block).
template <int KB, int H>
__device__ __forceinline__ void build_half(const __nv_bfloat16 *qcol, const float *alpha,
                                           const uint32_t (&p)[32], const uint32_t *cw,
                                           uint32_t (&out)[16]) {
  if constexpr (KB < 33) {
    h2_runs<KB, H, 0>(qcol, alpha, p, out);
  } else {
    static_assert(KB == kNKB - 1, "the H1 block is the last");
#pragma unroll
    for (int w = 0; w < 16; ++w) {
      const int t = 2 * (16 * H + w);
      out[w] = hmul2(qt_ld(qcol, t) | (qt_ld(qcol, t + 1) << 16), cw[16 * H + w]);
    }
  }
}

// General form of one half block (heads whose table is not rank-one plus
// exceptions): q_r q_t times the table weight, feature codes from the table.
__device__ __forceinline__ void build_half_general(int kb, int H, const __nv_bfloat16 *qcol,
                                                const uint32_t *cw, uint32_t (&out)[16]) {
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    const int f = 64 * kb + 2 * (16 * H + w);
    const uint16_t code = g_feat.code[f];
    uint32_t qa, qb;
    if (code == 0xFFFF) {
      qa = 0u; qb = 0u;
    } else if (code == 0xC000) {
      qa = 0x3F80u; qb = 0x3F80u;   // (1, 0) * (1, 0): the H0 feature
    } else if (code & 0x8000) {
      const int r = code & 0xff;
      qa = 0x3F803F80u; qb = qt_ld(qcol, r) | (qt_ld(qcol, r + 1) << 16);   // H1 pair (r, r + 1)
    } else {
      const int r = code >> 8, t = code & 0xff;
      qa = qt_ld(qcol, r) * 0x10001u;
      qb = qt_ld(qcol, t) | (qt_ld(qcol, t + 1) << 16);
    }
    out[w] = hmul2(hmul2(qa, qb), cw[16 * H + w]);
  }
}

// Exception words of half block hb: their exact value q_r q_t w(r, t), stored
// over the rank-one words already in tensor memory.
__device__ __forceinline__ void patch_exceptions(const RFactor &F, int hb, const __nv_bfloat16 *qcol,
                                              uint32_t taddr) {
  for (int e = F.exc_start[hb]; e < F.exc_start[hb + 1]; ++e) {
    const int wd = F.exc_word[e];
    const int r = F.exc_rt[e] >> 8, t = F.exc_rt[e] & 0xff;
    const float qr = __uint_as_float(qt_ld(qcol, r) << 16);
    const float lo = qr * __uint_as_float(qt_ld(qcol, t) << 16) * F.exc_wlo[e];
    const float hi = qr * __uint_as_float(qt_ld(qcol, t + 1) << 16) * F.exc_whi[e];
    tmem_st1(taddr + (uint32_t)(wd - 16 * hb), pack_bf16x2(lo, hi));
  }
}

#define OAL_BUILD_CASE(n)                     \
  case n:                                     \
    build_half<n, 0>(qcol, alpha, p, cw, out0); \
    build_half<n, 1>(qcol, alpha, p, cw, out1); \
    break;

// Both halves of K block kb (one dispatch per K block).
__device__ __forceinline__ void build_dispatch(int kb, const __nv_bfloat16 *qcol,
                                               const float *alpha, const uint32_t (&p)[32],
                                               const uint32_t *cw, uint32_t (&out0)[16],
                                               uint32_t (&out1)[16]) {
  switch (kb) {
    OAL_BUILD_CASE(0) OAL_BUILD_CASE(1) OAL_BUILD_CASE(2) OAL_BUILD_CASE(3)
    OAL_BUILD_CASE(4) OAL_BUILD_CASE(5) OAL_BUILD_CASE(6) OAL_BUILD_CASE(7)
    OAL_BUILD_CASE(8) OAL_BUILD_CASE(9) OAL_BUILD_CASE(10) OAL_BUILD_CASE(11)
    OAL_BUILD_CASE(12) OAL_BUILD_CASE(13) OAL_BUILD_CASE(14) OAL_BUILD_CASE(15)
    OAL_BUILD_CASE(16) OAL_BUILD_CASE(17) OAL_BUILD_CASE(18) OAL_BUILD_CASE(19)
    OAL_BUILD_CASE(20) OAL_BUILD_CASE(21) OAL_BUILD_CASE(22) OAL_BUILD_CASE(23)
    OAL_BUILD_CASE(24) OAL_BUILD_CASE(25) OAL_BUILD_CASE(26) OAL_BUILD_CASE(27)
    OAL_BUILD_CASE(28) OAL_BUILD_CASE(29) OAL_BUILD_CASE(30) OAL_BUILD_CASE(31)
    OAL_BUILD_CASE(32) OAL_BUILD_CASE(33)
    default: break;
  }
}
#undef OAL_BUILD_CASE

// ---------------------------------------------------------------- intra-chunk helpers
// Intra-chunk numerators in workspace: per (batch x query head, 128-row tile)
// one 32 KB block [16][128][4] fp32, the 16-byte chunk e of tile row m at
// [e][m], so the 32 rows of a warp write or read one chunk as 512 contiguous
// bytes.  Denominators: [batch x query head][T] fp32.
__device__ __forceinline__ uint4 *intra_tile(float *num, size_t bh, int T, int tile) {
  const int nS = (T + kC - 1) / kC;
  return reinterpret_cast<uint4 *>(num + (bh * nS + tile) * (size_t)(kC * 64));
}

struct IntraGeom {
  int row0;   // first query row of the tile
  int ks;     // first key: the start of row0's chunk
  int nkb;    // 32-key blocks: 4, or 8 for the second half of a 256-token chunk
};
__device__ __forceinline__ IntraGeom intra_geom(int t, int C) {
  IntraGeom g;
  g.row0 = t * kC;
  g.ks = (g.row0 / C) * C;
  g.nkb = (g.row0 + kC - g.ks) / 32;
  return g;
}

__device__ __forceinline__ float bf16_at(const __nv_bfloat16 *tile, int row, int col) {
  const uint8_t *base = reinterpret_cast<const uint8_t *>(tile);
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
      base + sw128(row, col >> 3) + (col & 7) * 2));
}

// Generic path (a tail group with more than 2 dims): sums straight from the
// Q and K tiles, constants from shared memory.
__device__ float kappa_generic(const KPlan &p, float s, const __nv_bfloat16 *qtile,
                               const __nv_bfloat16 *ktile, int m, int j) {
  float sg[kMaxTailG];
  for (int g = 0; g < kMaxTailG; ++g) {
    float acc = 0.f;
    if (g < p.ntg)
      for (int d = p.goff[g]; d < p.goff[g + 1]; ++d)
        acc = fmaf(bf16_at(qtile, m, p.gdims[d]), bf16_at(ktile, j, p.gdims[d]), acc);
    sg[g] = acc;
  }
  float kap = p.eps;
  for (int c = 0; c <= p.G; ++c) {
    float w = fmaf(p.alpha[c], s, c == 0 ? p.L00 : 0.f);
    for (int g = 0; g < p.ntg; ++g) w = fmaf(p.beta[g][c], sg[g], w);
    kap = fmaf(w, w, kap);
  }
  return kap;
}

// ---------------------------------------------------------------- intra kernel, tensor-core kappa
// With z_0 = s = q.k and z_g the tail-group sums, the quadratic form of
// kappa splits into
//     kappa = (c0 + T) + s (lin_0 + U + quad_00 s),
//     U = sum_g quad_0g z_g = sum_r quad_{0 g(r)} q_r k_r,
//     T = sum_g lin_g z_g + sum_{g <= h} quad_gh z_g z_h
//       = sum_r lin_{g(r)} q_r k_r + sum_{r <= r'} w_{r r'} q_r q_r' k_r k_r'
// over the tail dims r (w_{r r'} = quad_gh for dims of different groups,
// 2 quad_gg for two dims of one group, quad_gg for r = r').  T and U are
// contractions of per-query and per-key features, so they run on the tensor
// cores beside s: per 32-key block, S = Q K^T, T = A B^T over the feature
// columns 0..47 and U = A B^T over the columns 48..63 into tensor memory,
// with B = [k_r, k_r k_r' | k_r] (key side) and A the query rows times the
// coefficients of T, then of U.  The CUDA cores keep three FMAs per pair.
// Heads whose features do not fit (more than 8 tail dims, or a group of more
// than two dims) evaluate kappa from the Q and K tiles (kappa_generic).
//
// A block serves one or two query heads of one KV head (nh_per_block; two
// when the grid of one head a block would still fill the GPU several times),
// one after the other: K, V and the key features are loaded or built once,
// the query tiles arrive with them, and the second head's query features are
// built while the first head's last P V products run.
constexpr int kTkThreads = 192;          // warps 0-3: features, kappa, epilogue; 4: UMMA; 5: TMA
constexpr int kTkHeads = 2;              // query heads per block at most
constexpr int kTkS = 0;                  // s / P sub-tiles at 0 and 32
constexpr int kTkT = 64;                 // T sub-tiles at 64 and 96
constexpr int kTkU = 128;                // U sub-tiles at 128 and 160
constexpr int kTkI = 192;                // numerators at [192, 256)
constexpr uint32_t kTkTmemCols = 256;
constexpr int kTkKB = 4;                 // 32-key blocks per head (C <= 128)
struct __align__(1024) TkSmem {
  __nv_bfloat16 q[kTkHeads][kC * 64];  // 128B-swizzled [row][64] tiles
  __nv_bfloat16 k[kC * 64];
  __nv_bfloat16 v[kC * 64];
  __nv_bfloat16 a[kC * 64];            // query features, K-major: T at 0.., U at kTkU0..
  __nv_bfloat16 bk[kC * 64];           // key features
  KPlan plan[kTkHeads];
  uint64_t qkv_full, phi_full, s_full[2], p_full[2], s_free[2], d_full, i_free, drain;
  uint64_t kv2_full;          // (C = 256) the second 128-key tile of K and V
  uint64_t never;                      // failure-path tests: nothing arrives
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(2 * (sizeof(TkSmem) + 1024) <= 228 * 1024, "two intra blocks per SM");

// Pair (i, j) of feature position f >= kTkMaxLin (folded at compile time
// once the loops over f are unrolled).
__host__ __device__ constexpr int tk_pair_i(int f) {
  int i = 0;
  while (i + 1 < kTkMaxLin && kTkMaxLin + tk_pair(i + 1, i + 1) <= f) ++i;
  return i;
}
__host__ __device__ constexpr int tk_pair_j(int f) {
  return f - kTkMaxLin - tk_pair(tk_pair_i(f), tk_pair_i(f)) + tk_pair_i(f);
}
static_assert(tk_pair_i(kTkMaxLin + tk_pair(3, 7)) == 3 && tk_pair_j(kTkMaxLin + tk_pair(3, 7)) == 7,
              "feature position of a pair");

// Eight features starting at F0 of the query row (a) and of the key row (b)
// from the rows' tail values: T columns cT_f q_i (q_j) / k_i (k_j), U columns
// cU_i q_i / k_i, zero elsewhere.
template <int F0>
__device__ __forceinline__ void tk_row_chunk(const float (&qv)[kTkMaxLin], const float (&kv)[kTkMaxLin],
                                             const float *cT, const float *cU, uint4 &at, uint4 &bk) {
  float a[8], b[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int f = F0 + e;
    if (f < kTkMaxLin) {
      a[e] = cT[f] * qv[f];
      b[e] = kv[f];
    } else if (f < kTkFeat) {
      const int fi = tk_pair_i(f), fj = tk_pair_j(f);
      a[e] = cT[f] * qv[fi] * qv[fj];
      b[e] = kv[fi] * kv[fj];
    } else if (f >= kTkU0 && f < kTkU0 + kTkMaxLin) {
      a[e] = cU[f - kTkU0] * qv[f - kTkU0];
      b[e] = kv[f - kTkU0];
    } else {
      a[e] = 0.f;
      b[e] = 0.f;
    }
  }
  at = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                  pack_bf16x2(a[6], a[7]));
  bk = make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]), pack_bf16x2(b[4], b[5]),
                  pack_bf16x2(b[6], b[7]));
}

// Query (and, with keys, key) feature rows of row m for plan p.
__device__ __forceinline__ void tk_build_rows(TkSmem &s, const KPlan &p, const __nv_bfloat16 *qt,
                                              int m, bool keys) {
  float qv[kTkMaxLin], kv[kTkMaxLin];
#pragma unroll
  for (int i = 0; i < kTkMaxLin; ++i) {
    const bool in = i < p.tk_nlin;
    qv[i] = in ? bf16_at(qt, m, p.tk_dim[i]) : 0.f;
    kv[i] = in ? bf16_at(s.k, m, p.tk_dim[i]) : 0.f;
  }
  uint8_t *ra = reinterpret_cast<uint8_t *>(s.a), *rb = reinterpret_cast<uint8_t *>(s.bk);
  uint4 at, bk;
#define OAL_TK_CHUNK(c)                                                       \
  tk_row_chunk<8 * (c)>(qv, kv, p.tk_cT, p.tk_cU, at, bk);                   \
  *reinterpret_cast<uint4 *>(ra + sw128(m, c)) = at;                          \
  if (keys) *reinterpret_cast<uint4 *>(rb + sw128(m, c)) = bk;
  OAL_TK_CHUNK(0) OAL_TK_CHUNK(1) OAL_TK_CHUNK(2) OAL_TK_CHUNK(3)
  OAL_TK_CHUNK(4) OAL_TK_CHUNK(5) OAL_TK_CHUNK(6) OAL_TK_CHUNK(7)
#undef OAL_TK_CHUNK
}

template <bool kTwoTiles>
__global__ void __launch_bounds__(kTkThreads, 2)
tc_intra_tk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, ReadArgs args) {
  extern __shared__ uint8_t smem_raw[];
  TkSmem &s = *reinterpret_cast<TkSmem *>(smem_align1024(smem_raw));
  const int hg = blockIdx.x, t = blockIdx.y, unit = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bidx = unit / args.Hkv, kv = unit % args.Hkv;
  const int hpb = args.nh_per_block;               // 1 or 2 (<= kTkHeads)
  const int h0 = kv * args.rho + hg * hpb;
  const int nh = min(hpb, args.rho - hg * hpb);
  const IntraGeom geo = intra_geom(t, args.chunk);
  // 128-key tiles of K and V: one (C <= 128, and the first half of a 256-token
  // chunk) or two (the second half: the second tile reloads the buffers)
  const int ntile = kTwoTiles ? geo.nkb / kTkKB : 1;
  const int nkb = kTkKB * ntile;
  constexpr int kIss = 4, kTma = 5;
  pdl_trigger();

  if (tid == 0) {
    s.abort_flag = 0;
    mbar_init(&s.qkv_full, 1);
    mbar_init(&s.phi_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.s_free[i], 1);
    }
    mbar_init(&s.d_full, 1);
    mbar_init(&s.i_free, 4);
    mbar_init(&s.drain, 1);
    mbar_init(&s.kv2_full, 1);
    mbar_init(&s.never, 1);
    fence_mbar_init();
    // Q, K and V are inputs of the call that no kernel of it writes: their
    // loads start before the wait on the previous kernels
    tma_prefetch_desc(&tmQ);
    // Q, K and V now, the heads' plans (the prep kernel's) after the wait below
    mbar_arrive_expect_tx(&s.qkv_full, (uint32_t)((nh + 2) * kC * 64 * 2 + nh * sizeof(KPlan)));
    for (int hh = 0; hh < nh; ++hh)
      tma_load_3d(s.q[hh], &tmQ, &s.qkv_full, 0, geo.row0, bidx * args.Hq + h0 + hh);
    tma_load_3d(s.k, &tmK, &s.qkv_full, 0, geo.ks, unit);
    tma_load_3d(s.v, &tmV, &s.qkv_full, 0, geo.ks, unit);
  }
  if (warp == kIss) {
    tmem_alloc(&s.tmem_base, kTkTmemCols);
    tmem_relinquish();
  }
  pdl_wait();   // plans of the prep kernel; the intra rows of the previous call
  if (tid == 0) bulk_load(s.plan, args.plans + h0, (uint32_t)(nh * sizeof(KPlan)), &s.qkv_full);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  volatile int *abort_flag = &s.abort_flag;

  if (warp == kIss) {
    {
      // Key block g = kTkKB hh + kb of head hh uses s/P, T and U sub-tiles g & 1;
      // every barrier of a sub-tile completes once per key block, in order.
      const uint32_t id32k = idesc_bf16_f32(128, 32, 0);
      const uint32_t id64mn = idesc_bf16_f32(128, 64, 1);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(s.k), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(s.v), 16, 1024);
      const uint64_t adesc = sdesc_sw128(smem_u32(s.a), 16, 1024);
      const uint64_t bdesc0 = sdesc_sw128(smem_u32(s.bk), 16, 1024);
      const bool starve = args.status[1] == kStarveIntra;   // failure-path test only
      bool ok = mbar_wait(starve ? &s.never : &s.qkv_full, 0, abort_flag, args.status);
      bool kv2 = false;   // the second tile's loads were issued
      for (int hh = 0; hh < nh && ok; ++hh) {
        const KPlan &p = s.plan[hh];
        const bool tu = p.tk_mode && p.tk_nlin > 0;
        const uint64_t qdesc = sdesc_sw128(smem_u32(s.q[hh]), 16, 1024);
        const int g0 = nkb * hh;
        // S = Q K^T of key block kb, then (tu) T over K = 48 and U over K = 16
        // (kb & 3: the block's place in the current 128-key tile)
        auto issue_s = [&](int kb) {
          const uint64_t koff = (uint64_t)((32 * (kb & 3) * 128) >> 4);
          const uint32_t b = (g0 + kb) & 1;
          umma_ss_warp(tb + kTkS + 32 * b, qdesc, kdesc0 + koff, id32k, 0u);
          umma_ss_warp(tb + kTkS + 32 * b, qdesc + 2, kdesc0 + koff + 2, id32k, 1u);
          umma_ss_warp(tb + kTkS + 32 * b, qdesc + 4, kdesc0 + koff + 4, id32k, 1u);
          umma_ss_warp(tb + kTkS + 32 * b, qdesc + 6, kdesc0 + koff + 6, id32k, 1u);
        };
        auto issue_tu = [&](int kb) {
          const uint64_t koff = (uint64_t)((32 * (kb & 3) * 128) >> 4);
          const uint32_t b = (g0 + kb) & 1;
          if (tu) {
#pragma unroll
            for (int k2 = 0; k2 < kTkU0 / 16; ++k2)
              umma_ss_warp(tb + kTkT + 32 * b, adesc + 2 * k2, bdesc0 + koff + 2 * k2, id32k, k2 > 0 ? 1u : 0u);
            umma_ss_warp(tb + kTkU + 32 * b, adesc + kTkU0 / 8, bdesc0 + koff + kTkU0 / 8, id32k, 0u);
          }
          umma_commit_warp(&s.s_full[b]);
        };
        if (hh > 0) {
          // the previous head's last two P V products have read their P sub-tiles
          for (int g = g0 - 2; g < g0 && ok; ++g)
            ok = mbar_wait(&s.s_free[g & 1], (g >> 1) & 1, abort_flag, args.status);
          if (!ok) break;
        }
        for (int j = 0; j < ntile && ok; ++j) {
          if (kTwoTiles && j > 0) {
            // the first tile's last P V products have read V and their P
            // sub-tiles (its S, T, U products were read before): reload K
            // and V with the second tile
            for (int g = g0 + kTkKB * j - 2; g < g0 + kTkKB * j && ok; ++g)
              ok = mbar_wait(&s.s_free[g & 1], (g >> 1) & 1, abort_flag, args.status);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(&s.kv2_full, 2u * kC * 64 * 2);
              tma_load_3d(s.k, &tmK, &s.kv2_full, 0, geo.ks + kC, unit);
              tma_load_3d(s.v, &tmV, &s.kv2_full, 0, geo.ks + kC, unit);
            }
            kv2 = true;
            __syncwarp();
            if (!mbar_wait(&s.kv2_full, 0, abort_flag, args.status)) { ok = false; break; }
          }
          const int k0 = kTkKB * j;
          // the first two S blocks of the tile need only Q and K: they run
          // while the feature rows are built
          tc_fence_after();
          issue_s(k0);
          issue_s(k0 + 1);
          if (!mbar_wait(&s.phi_full, (hh * ntile + j) & 1, abort_flag, args.status)) { ok = false; break; }
          tc_fence_after();
          issue_tu(k0);
          issue_tu(k0 + 1);
          for (int kb = k0; kb < k0 + kTkKB && ok; ++kb) {
            const int g = g0 + kb;
            if (!mbar_wait(&s.p_full[g & 1], (g >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
            // the numerators of the previous head are read out of tensor memory
            if (kb == 0 && hh > 0 &&
                !mbar_wait(&s.i_free, (hh - 1) & 1, abort_flag, args.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t at = tb + kTkS + 32 * (g & 1);
            const uint64_t vd = vdesc0 + (uint64_t)((32 * (kb & 3) * 128) >> 4);
            umma_ts_warp(tb + kTkI, at, vd, id64mn, kb > 0 ? 1u : 0u);
            umma_ts_warp(tb + kTkI, at + 8, vd + (2048 >> 4), id64mn, 1u);
            umma_commit_warp(&s.s_free[g & 1]);
            if (kb + 2 < k0 + kTkKB) {
              if (!mbar_wait(&s.s_free[g & 1], (g >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
              tc_fence_after();
              issue_s(kb + 2);
              issue_tu(kb + 2);
            }
          }
        }
        if (!ok) break;
        umma_commit_warp(&s.d_full);
      }
      umma_commit_warp(&s.drain);
      if (lane == 0) mbar_wait_teardown(&s.drain, 0, args.status);   // no MMA in flight at exit
      if (kTwoTiles && kv2 && lane == 0) mbar_wait_teardown(&s.kv2_full, 0, args.status);
    }
    __syncwarp();
  } else if (warp == kTma) {
    // the loads issued at the start land before the block exits
    if (lane == 0) mbar_wait_teardown(&s.qkv_full, 0, args.status);
    __syncwarp();
  } else {
    // warps 0-3, thread = query row m and key row m of the tile
    const int m = tid;
    const int C = args.chunk;
    const int i_tok = geo.row0 + m;
    const int cs = (i_tok / C) * C;                  // this row's chunk starts here
    const int rw0 = geo.row0 + 32 * warp, rw1 = rw0 + 31;
    const int csw = (rw0 / C) * C;                   // the warp's rows share one chunk (C >= 64)
    bool ok = mbar_wait(&s.qkv_full, 0, abort_flag, args.status);
    // the feature rows of head hh (the key rows too unless the previous
    // head's tail dims are the same), then one arrival on phi_full
    auto build = [&](int hh) {
      const KPlan &p = s.plan[hh];
      if (p.tk_mode && p.tk_nlin > 0) {
        bool keys = hh == 0;
        if (!keys) {
          const KPlan &o = s.plan[hh - 1];
          keys = !o.tk_mode || o.tk_nlin != p.tk_nlin;
          for (int i = 0; i < kTkMaxLin; ++i) keys = keys || o.tk_dim[i] != p.tk_dim[i];
        }
        tk_build_rows(s, p, s.q[hh], m, keys);
        fence_proxy_async();   // the features are read by the tensor cores
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.phi_full);
    };
    if (ok) build(0);
    for (int hh = 0; hh < nh && ok; ++hh) {
      const KPlan &p = s.plan[hh];
      const int mode = p.tk_mode;
      const bool tu = mode && p.tk_nlin > 0;   // (no tail dims: T = U = 0)
      const __nv_bfloat16 *qt = s.q[hh];
      const float c0 = p.c0, lin0 = p.lin[0], q00 = p.quad[0], eps = p.eps;
      float dsum = 0.f;
      for (int kb = 0; kb < nkb; ++kb) {
        const int g = nkb * hh + kb, b = g & 1;
        if (kTwoTiles && kb == kTkKB) {
          // the second tile: its K rows land, then its key features (the
          // first tile's T and U products are complete: their s_full arrived)
          if (!mbar_wait(&s.kv2_full, 0, abort_flag, args.status)) { ok = false; break; }
          if (p.tk_mode && p.tk_nlin > 0) {
            tk_build_rows(s, p, qt, m, true);
            fence_proxy_async();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.phi_full);
        }
        if (!mbar_wait(&s.s_full[b], (g >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        const int jbase = 32 * kb, jg0 = geo.ks + jbase;
        uint32_t pk[16];
        if (jg0 + 31 >= csw && jg0 <= rw1) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t sv[16], tv[16], uv[16];
            tmem_ld16(tmem_lane_addr(tb, warp, kTkS + 32 * b + 16 * half), sv);
            if (tu) {
              tmem_ld16(tmem_lane_addr(tb, warp, kTkT + 32 * b + 16 * half), tv);
              tmem_ld16(tmem_lane_addr(tb, warp, kTkU + 32 * b + 16 * half), uv);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) tv[e] = uv[e] = 0u;
            }
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; jj += 2) {
              const int j0 = jbase + 16 * half + jj, jg = geo.ks + j0;
              float kap[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float sx = __uint_as_float(sv[jj + e]);
                if (mode) {
                  const float tx = __uint_as_float(tv[jj + e]), ux = __uint_as_float(uv[jj + e]);
                  kap[e] = fmaxf(fmaf(sx, fmaf(q00, sx, lin0 + ux), c0 + tx), eps);
                } else {
                  kap[e] = (jg + e >= cs && jg + e <= i_tok)
                               ? kappa_generic(p, sx, qt, s.k, m, (j0 + e) & (kC - 1)) : 0.f;
                }
              }
              pk[8 * half + (jj >> 1)] = pack_bf16x2((jg >= cs && jg <= i_tok) ? kap[0] : 0.f,
                                                     (jg + 1 >= cs && jg + 1 <= i_tok) ? kap[1] : 0.f);
            }
          }
          // denominator from the same rounded weights the P.V product uses
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 pb = *reinterpret_cast<const __nv_bfloat162 *>(&pk[e]);
            dsum += __low2float(pb) + __high2float(pb);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        tmem_st16(tmem_lane_addr(tb, warp, kTkS + 32 * b), pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[b]);
      }
      if (!ok) break;
      // the last T and U products of this head are complete (their s_full
      // arrived): the next head's features may overwrite the feature rows
      if (hh + 1 < nh) build(hh + 1);
      if (!mbar_wait(&s.d_full, hh & 1, abort_flag, args.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t d[64];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r[16];
        tmem_ld16(tmem_lane_addr(tb, warp, kTkI + 16 * q4), r);
#pragma unroll
        for (int e = 0; e < 16; ++e) d[16 * q4 + e] = r[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.i_free);
      if (i_tok < args.T) {
        const size_t bh = (size_t)bidx * args.Hq + h0 + hh;
        uint4 *dst = intra_tile(args.intra_num, bh, args.T, t) + m;
#pragma unroll
        for (int e = 0; e < 16; ++e)
          dst[kC * e] = make_uint4(d[4 * e], d[4 * e + 1], d[4 * e + 2], d[4 * e + 3]);
        args.intra_den[bh * args.T + i_tok] = dsum;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIss) {
    tc_fence_after();
    tmem_dealloc(tb, kTkTmemCols);
  }
}

// ---------------------------------------------------------------- readout kernel
// One block per (query head, chunk, batch x KV head), four blocks per SM
// (128 tensor-memory columns, ~52 KB of shared memory and 96 registers a
// thread each): blocks that run independently keep the tensor pipe fed from
// whichever block has a K block ready, and the builders of four blocks hide
// each other's latencies.  Warp roles (5 warps):
//   0-3  A builders (one token row per thread): setup (transposed Q tile),
//        every K block of Phi~(Q_c), then the epilogue; warp 0 also
//        refills the snapshot stages (3) by TMA as soon as the wait for an A
//        slot shows that the MMAs reading a stage are complete
//   4    UMMA issuer (warp-uniform loop, elected lane), tensor memory owner,
//        loads the first snapshot K blocks
template <int NS>
__global__ void __launch_bounds__(kReadThreads, NS == 1 ? 4 : 2)
tc_readout_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmS,
                  ReadArgs args) {
  extern __shared__ uint8_t smem_raw[];
  ReadSmem<NS> &s = *reinterpret_cast<ReadSmem<NS> *>(smem_align1024(smem_raw));
  const int hg = blockIdx.x, c = blockIdx.y, unit = blockIdx.z;   // c: 128-row tile
  // snapshot read by the tile: the state before its chunk (C = 64: the
  // states before each of its two chunks)
  const int snap0 = NS == 2 ? 2 * c : (args.chunk == 256 ? c >> 1 : c);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bidx = unit / args.Hkv, kv = unit % args.Hkv;
  const int h0 = kv * args.rho + hg * args.nh_per_block;
  const int nh = min(args.nh_per_block, args.rho - hg * args.nh_per_block);
  constexpr int kIss0 = 4;
  pdl_trigger();

  if (tid == 0) {
    s.abort_flag = 0;
    mbar_init(&s.qkv_full, 1);
    for (int i = 0; i < kNB; ++i) mbar_init(&s.b_full[i], 1);
    for (int i = 0; i < kNA; ++i) { mbar_init(&s.a_full[i], 4); mbar_init(&s.a_empty[i], 1); }
    s.loaded = min(kNB, kNKB);          // the issuer loads the first kNB K blocks

    mbar_init(&s.d_full, nh);           // every head's issuer done
    mbar_init(&s.never, 1);
    fence_mbar_init();
    // Q is an input of the call that no kernel of it writes: its load starts
    // before the wait on the previous kernels
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
    // Q now, the heads' weight rows (the prep kernel's) after the wait below
    mbar_arrive_expect_tx(&s.qkv_full, (uint32_t)nh * (kC * 64 * 2 + kCoefRow * 2));
    for (int h = 0; h < nh; ++h)
      tma_load_3d(s.q[h], &tmQ, &s.qkv_full, 0, c * kC, bidx * args.Hq + h0 + h);
  }
  if (warp == kIss0) {
    tmem_alloc(&s.tmem_base, kReadTmemCols<NS>);
    tmem_relinquish();
  }
  pdl_wait();   // weights, snapshots and intra rows of the previous kernels
  if (tid == 32) {
    // the intra-chunk rows the epilogue reads, into L2 while the contraction runs
    const int rows = min(kC, args.T - c * kC);
    for (int h = 0; h < nh; ++h) {
      const size_t bh = (size_t)bidx * args.Hq + h0 + h;
      const size_t row0 = bh * args.T + (size_t)c * kC;
      prefetch_l2(intra_tile(args.intra_num, bh, args.T, c), kC * 64 * 4);
      const uintptr_t d0 = (reinterpret_cast<uintptr_t>(args.intra_den + row0) + 15) & ~uintptr_t(15);
      const uintptr_t d1 = reinterpret_cast<uintptr_t>(args.intra_den + row0 + rows) & ~uintptr_t(15);
      if (d1 > d0) prefetch_l2(reinterpret_cast<const void *>(d0), (uint32_t)(d1 - d0));
    }
  }
  if (tid == 0)
    for (int h = 0; h < nh; ++h)
      bulk_load(s.coef[h], args.coef + (size_t)(h0 + h) * kCoefRow, kCoefRow * 2, &s.qkv_full);
  for (int e = tid; e < NS * kU; e += kReadThreads) {
    const int x = e / kU, n = e % kU;
    float v = 0.f;   // (past the last chunk: rows past T only)
    if (snap0 + x < args.nC)
      v = __bfloat162float(args.snap[((size_t)(unit * args.nC + snap0 + x) * kSnapRows + n) * kKP + kH0Feat]);
    s.s0[x][n] = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  volatile int *abort_flag = &s.abort_flag;
  // snapshot K block kb2 into its stage (one thread)
  auto load_block = [&](int kb2) {
    const int st2 = kb2 % kNB;
    mbar_arrive_expect_tx(&s.b_full[st2], NS * kN * 64 * 2);
#pragma unroll
    for (int x = 0; x < NS; ++x)   // (past the last chunk: another unit's rows or zero fill,
                                   //  read only for rows past T)
      tma_load_3d(s.b[st2] + x * kN * 64, &tmS, &s.b_full[st2], 64 * kb2, 0,
                  unit * args.nC + snap0 + x);
  };

  if (warp >= kIss0) {
    const int hh = warp - kIss0;
    if (hh < nh) {
      // ---------------- UMMA issuer of head hh: D^h = sum over K blocks of A_kb B_kb.
      // The whole warp runs the loop (warp-uniform; an elected lane issues:
      // an issuing loop under a one-lane branch is several times slower).
      // Head 0's warp also loads the first kNB snapshot K blocks by TMA.
      const uint32_t id80 = idesc_bf16_f32(128, NS * kN, 0);
      const uint64_t bdesc0 = sdesc_sw128(smem_u32(s.b[0]), 16, 1024);
      constexpr uint64_t kStageStep = (NS * kN * 64 * 2) >> 4;   // one snapshot stage
      const uint32_t dt = tb + kTmemD + 80 * hh;
      const bool tma = hh == 0;
      // the first kNB K blocks; the builders load the rest as stages free up
      if (tma && lane == 0)
        for (int kb2 = 0; kb2 < kNB && kb2 < kNKB; ++kb2) load_block(kb2);
      // this head owns half slots [hh * nhs, (hh + 1) * nhs), used in turn
      const int nhs = kNA / nh > 6 ? 6 : kNA / nh;
      const int a0 = hh * nhs;
      const int fper = (nhs & 1) ? nhs : nhs / 2;   // K blocks between two uses as a first half
      int st = 0, sph = 0;                       // snapshot stage and its phase
      int hs = 0;                                // first half slot of K block kb: (2 kb) % nhs
      int fk = 0, fph = 0;                       // kb % fper and the phase of (kb / fper)
      const bool starve = args.status[1] == kStarveReadout;   // failure-path test only
      for (int kb = 0; kb < kNKB; ++kb) {
        if (!mbar_wait(starve && kb == 0 ? &s.never : &s.b_full[st], sph, abort_flag, args.status))
          break;
        const uint64_t bd = bdesc0 + kStageStep * st;
        // K block kb: halves of K = 32 in half slots (2 kb) % nhs and
        // (2 kb + 1) % nhs of this head;
        // its builders arrive once, on the first half slot's barrier
        const int hs1 = hs + 1 == nhs ? 0 : hs + 1;
        if (!mbar_wait(&s.a_full[a0 + hs], fph, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t at0 = tb + kTmemA<NS> + 16 * (a0 + hs), at1 = tb + kTmemA<NS> + 16 * (a0 + hs1);
        umma_ts_warp(dt, at0, bd, id80, kb > 0 ? 1u : 0u);
        umma_ts_warp(dt, at0 + 8, bd + 2, id80, 1u);
        umma_ts_warp(dt, at1, bd + 4, id80, 1u);
        umma_ts_warp(dt, at1 + 8, bd + 6, id80, 1u);
        umma_commit_warp(&s.a_empty[a0 + hs]);
        umma_commit_warp(&s.a_empty[a0 + hs1]);
        hs = hs1 + 1 == nhs ? 0 : hs1 + 1;
        if (++fk == fper) { fk = 0; fph ^= 1; }
        if (++st == kNB) { st = 0; sph ^= 1; }
      }
      umma_commit_warp(&s.d_full);
      mbar_wait_teardown(&s.d_full, 0, args.status);   // no MMA in flight at exit
      if (tma) mbar_wait_teardown(&s.qkv_full, 0, args.status);   // no copy in flight at exit
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------- readout A builders: group hh builds head hh; thread = token row
    const int m = 32 * (warp & 3) + lane;
    const int hh = warp >> 2;
    // q^T [64 dims][128 tokens] replaces the swizzled Q tile of head hh
    __nv_bfloat16 *qT = s.q[hh];
    const __nv_bfloat16 *qcol = qT + m;
    const RFactor &F = *reinterpret_cast<const RFactor *>(s.coef[hh] + kKP);
    const bool ok = hh < nh && mbar_wait(&s.qkv_full, 0, abort_flag, args.status);
    uint32_t p[32], q[32];
    if (ok) {
      // p_t = bf16(pw_t q_t): the rank-one weights applied once per token row
      const uint8_t *qrow = reinterpret_cast<const uint8_t *>(qT) + m * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4 *>(qrow + ((cc ^ (m & 7)) << 4));
        q[4 * cc] = v.x; q[4 * cc + 1] = v.y; q[4 * cc + 2] = v.z; q[4 * cc + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i)
        p[i] = pack_bf16x2(F.pw[2 * i] * __uint_as_float(q[i] << 16),
                           F.pw[2 * i + 1] * __uint_as_float(q[i] & 0xffff0000u));
    }
    if (hh < nh) {   // all four warps of the group pass both barriers, ok or not
      named_bar(1 + hh, 128);   // every row of the tile read
      if (ok) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          reinterpret_cast<uint16_t *>(qT)[(2 * i) * kC + m] = (uint16_t)(q[i] & 0xffffu);
          reinterpret_cast<uint16_t *>(qT)[(2 * i + 1) * kC + m] = (uint16_t)(q[i] >> 16);
        }
      }
      named_bar(1 + hh, 128);   // q^T complete
    }
    if (ok) {
      const bool factored = F.factored != 0;
      const int nhs = kNA / nh > 6 ? 6 : kNA / nh;   // as the issuer
      const int a0 = hh * nhs;
      int hs = 0;                // first half slot of K block kb, (2 kb) % nhs, as the issuer
      uint32_t uph = 0;          // bit j: number of completed uses of half slot j, mod 2
      uint64_t em = 0;                               // H2 half blocks 0..63 with exception words
      uint32_t em2 = 0;                              // half blocks 64, 65
      if (factored)
        for (int hb = 0; hb < kH2Halves; ++hb)
          if (F.exc_start[hb] != F.exc_start[hb + 1]) {
            if (hb < 64) em |= 1ull << hb;
            else em2 |= 1u << (hb - 64);
          }
      for (int kb = 0; kb < kNKB; ++kb) {
        const uint32_t *cw = reinterpret_cast<const uint32_t *>(s.coef[hh] + 64 * kb);
        // p is loop-invariant: keep the compiler from hoisting the per-row
        // products of every K block out of the loop (they would spill)
#pragma unroll
        for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(p[i]));
        uint32_t out0[16], out1[16];
        if (factored) {
          build_dispatch(kb, qcol, F.alpha, p, cw, out0, out1);
        } else {
          build_half_general(kb, 0, qcol, cw, out0);
          build_half_general(kb, 1, qcol, cw, out1);
        }
        // half index hx = 2 kb + H goes to half slot hx % nhs, its (hx / nhs)-th
        // use: wait for the MMAs of its previous use, store, arrive once
        const uint32_t xb = 2 * kb < 64 ? (uint32_t)(em >> (2 * kb)) & 3u : (em2 >> (2 * kb - 64)) & 3u;
        const int hs1 = hs + 1 == nhs ? 0 : hs + 1;
        const uint32_t par0 = ((uph >> hs) & 1u) ^ 1u, par1 = ((uph >> hs1) & 1u) ^ 1u;
        uint64_t *e0 = &s.a_empty[a0 + hs], *e1 = &s.a_empty[a0 + hs1];
        if (!mbar_test(e0, par0) && !mbar_wait(e0, par0, abort_flag, args.status)) break;
        // the half slot's previous use was half 2 kb - nhs, of K block j: its
        // MMAs are complete, so j's snapshot stage takes K block j + kNB
        if (warp == 0 && 2 * kb >= nhs) {
          const int nxt = ((2 * kb - nhs) >> 1) + kNB;
          if (nxt < kNKB && lane == 0) {
            load_block(nxt);
            s.loaded = nxt + 1;
          }
        }
        const uint32_t ta0 = tmem_lane_addr(tb, warp, kTmemA<NS> + 16 * (a0 + hs));
        const uint32_t ta1 = tmem_lane_addr(tb, warp, kTmemA<NS> + 16 * (a0 + hs1));
        tmem_st16(ta0, out0);
        if (!mbar_test(e1, par1) && !mbar_wait(e1, par1, abort_flag, args.status)) break;
        tmem_st16(ta1, out1);
        if (xb) {
          tmem_wait_st();
          if (xb & 1u) patch_exceptions(F, 2 * kb, qcol, ta0);
          if (xb & 2u) patch_exceptions(F, 2 * kb + 1, qcol, ta1);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.a_full[a0 + hs]);
        uph ^= (1u << hs) | (1u << hs1);
        hs = hs1 + 1 == nhs ? 0 : hs1 + 1;
      }
      tmem_wait_st();   // (a loop left early may have a store in flight)
    }
    if (hh < nh) {
      // ---------------- epilogue of head hh: y = (u~ + intra)[0:64] / (u~ + intra)[64].
      // The row's intra-chunk numerators and denominator are loaded at once
      // (one memory latency, overlapping the last MMAs), then the
      // accumulator is read 16 columns at a time
      const int i_tok = c * kC + m;
      const bool row_ok = i_tok < args.T;
      const size_t bh = (size_t)bidx * args.Hq + h0 + hh;
      const size_t row = bh * args.T + i_tok;
      const float4 *src = reinterpret_cast<const float4 *>(intra_tile(args.intra_num, bh, args.T, c) + m);
      float4 nv[16];
      float iden = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        nv[e] = row_ok ? __ldg(src + kC * e) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (row_ok) iden = __ldg(args.intra_den + row);
      // this row's columns of D: the second snapshot's (80 ..) for rows 64..127 when NS = 2
      const int dcol = kTmemD + 80 * hh + ((NS == 2 && m >= 64) ? kN : 0);
      if (!*abort_flag && mbar_wait(&s.d_full, 0, abort_flag, args.status)) {
        tc_fence_after();
        uint32_t r[16];
        // the H0 term a S0 (one product: the MMA's last K block held it before)
        const float a0w = __bfloat162float(s.coef[hh][kH0Feat]);
        const float *s0 = s.s0[(NS == 2 && m >= 64) ? 1 : 0];
        tmem_ld16(tmem_lane_addr(tb, warp, dcol + 64), r);
        tmem_wait_ld();
        const float inv = 1.0f / (fmaf(a0w, s0[64], __uint_as_float(r[0])) + iden);
        uint4 *dst = reinterpret_cast<uint4 *>(args.Y + row * kDv);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          tmem_ld16(tmem_lane_addr(tb, warp, dcol + 16 * q4), r);
          tmem_wait_ld();
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 n4 = nv[4 * q4 + e];
            const int n = 16 * q4 + 4 * e;
            pk[2 * e] = pack_bf16x2((fmaf(a0w, s0[n], __uint_as_float(r[4 * e])) + n4.x) * inv,
                                    (fmaf(a0w, s0[n + 1], __uint_as_float(r[4 * e + 1])) + n4.y) * inv);
            pk[2 * e + 1] = pack_bf16x2((fmaf(a0w, s0[n + 2], __uint_as_float(r[4 * e + 2])) + n4.z) * inv,
                                        (fmaf(a0w, s0[n + 3], __uint_as_float(r[4 * e + 3])) + n4.w) * inv);
          }
          if (row_ok) {
            dst[2 * q4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[2 * q4 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIss0) {
    // snapshot copies still in flight (a block that gave up early) land
    // before the block exits
    if (lane == 0)
      for (int kb = max(0, s.loaded - kNB); kb < s.loaded; ++kb)
        mbar_wait_teardown(&s.b_full[kb % kNB], (kb / kNB) & 1, args.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tb, kReadTmemCols<NS>);
  }
}

// ================================================================= host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// 3-D bf16 tensor map: x (inner, contiguous) extent nx, y extent ny (row
// pitch ybytes), z extent nz (pitch zbytes); box {64, by, 1}, 128B swizzle.
static bool make_map3(CUtensorMap *m, const void *ptr, uint64_t nx, uint64_t ny, uint64_t nz,
                      uint64_t ybytes, uint64_t zbytes, uint32_t by) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {nx, ny, nz};
  cuuint64_t strides[2] = {ybytes, zbytes};
  cuuint32_t box[3] = {64, by, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Layout {
  int nS, nC, nparts, spp, U;
  size_t snap_off, ptot_off, coef_off, plan_off, inum_off, iden_off, kt_off, total;
};

// Workspace of one call: the sequence splits into parts of spp 128-token
// stages (whole chunks), as many as give one state block per SM.
static Layout plan_layout(int B, int Hq, int Hkv, int T, int chunk) {
  Layout L{};
  L.U = B * Hkv;
  L.nS = (T + kC - 1) / kC;
  L.nC = (T + chunk - 1) / chunk;
  const int spc = chunk == 256 ? 2 : 1;    // stages per chunk (at least one)
  int P = 152 / (kTiles * L.U);            // one wave: every CTA walks its part once
  P = P < 1 ? 1 : (P > L.nS ? L.nS : P);
  L.spp = (L.nS + P - 1) / P;
  L.spp = (L.spp + spc - 1) / spc * spc;
  L.nparts = (L.nS + L.spp - 1) / L.spp;
  auto al = [](size_t x) { return (x + 1023) & ~size_t(1023); };
  size_t o = 0;
  L.snap_off = o; o = al(o + (size_t)L.U * L.nC * kSnapBytes);
  L.ptot_off = o; o = al(o + (size_t)L.U * L.nparts * kTiles * 128 * kN * sizeof(float));
  L.coef_off = o; o = al(o + (size_t)Hq * kCoefRow * 2);
  L.plan_off = o; o = al(o + (size_t)Hq * sizeof(KPlan));
  L.inum_off = o; o = al(o + (size_t)B * Hq * L.nS * kC * 64 * sizeof(float));
  L.iden_off = o; o = al(o + (size_t)B * Hq * T * sizeof(float));
  L.kt_off = o; o = al(o + (size_t)L.U * 64 * L.nS * kC * 2);
  L.total = o;
  return L;
}

}  // namespace tcp

size_t tc_prefill_workspace_bytes(int B, int Hq, int Hkv, int T, int chunk) {
  return tcp::plan_layout(B, Hq, Hkv, T, chunk).total;
}

// Query heads per block of the tensor-core-kappa intra kernel: 0 = automatic.
static std::atomic<int> g_intra_heads{0};
void set_intra_heads(int heads) { g_intra_heads.store(heads); }

oal_status launch_prefill_tc(const void *Q, const void *K, const void *V, int B, int Hq,
                             int Hkv, int T, const float *L, const int32_t *group, int G,
                             float eps, const float *a, const float *b, const float *C,
                             int packed, float *state, int cont, void *Y, int chunk, void *ws,
                             cudaStream_t stream) {
  using namespace tcp;
  const Layout lay = plan_layout(B, Hq, Hkv, T, chunk);
  uint8_t *w = static_cast<uint8_t *>(ws);
  __nv_bfloat16 *snap = reinterpret_cast<__nv_bfloat16 *>(w + lay.snap_off);
  float *ptot = reinterpret_cast<float *>(w + lay.ptot_off);
  __nv_bfloat16 *coef = reinterpret_cast<__nv_bfloat16 *>(w + lay.coef_off);
  KPlan *plans = reinterpret_cast<KPlan *>(w + lay.plan_off);
  int *status = oal_device_status_word();
  if (!status) return oal_fail(OAL_ERR_CUDA, "prefill: device status word unavailable");

  CUtensorMap tmQ, tmK, tmKn, tmV, tmS;
  const int Tpad = lay.nS * kC;
  __nv_bfloat16 *Kt = reinterpret_cast<__nv_bfloat16 *>(w + lay.kt_off);
  const uint64_t rowb = 64 * 2;
  if (!make_map3(&tmQ, Q, 64, T, (uint64_t)B * Hq, rowb, rowb * T, kC) ||
      !make_map3(&tmKn, K, 64, T, (uint64_t)lay.U, rowb, rowb * T, kC) ||
      !make_map3(&tmK, Kt, (uint64_t)Tpad, 64, (uint64_t)lay.U, (uint64_t)Tpad * 2,
                 (uint64_t)Tpad * 2 * 64, 64) ||
      !make_map3(&tmV, V, 64, T, (uint64_t)lay.U, rowb, rowb * T, kC) ||
      !make_map3(&tmS, snap, kKP, kSnapRows, (uint64_t)lay.U * lay.nC, (uint64_t)kKP * 2, kSnapBytes,
                 kN))
    return oal_fail(OAL_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  KtArgs kta;
  kta.K = static_cast<const __nv_bfloat16 *>(K); kta.Kt = Kt;
  kta.T = T; kta.Tpad = Tpad; kta.U = lay.U; kta.nC = lay.nS;
  const int ntiles = lay.U * lay.nS;
  const int ntr = (std::min(ntiles, 4 * 152) + Hq - 1) / Hq;   // block rows of transposes
  launch_pdl(tc_prep_kernel, dim3(Hq, (kKP + 255) / 256 + 2 + ntr), dim3(kPrepThreads), 0, stream, a, b, C,
             L, group, G, eps, packed, coef, plans, status, kta);
  oal_status st = oal_after_launch("tc_prep_kernel", stream);
  if (st != OAL_OK) return st;

  const size_t ssmem = sizeof(StateSmem) + 1024;
  const size_t rsmem1 = sizeof(ReadSmem<1>) + 1024;
  const size_t rsmem2 = sizeof(ReadSmem<2>) + 1024;
  const size_t tksmem = sizeof(TkSmem) + 1024;
  // shared-memory limits above 48 KB: a function attribute of each device
  static std::mutex attr_mutex;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return oal_fail(OAL_ERR_CUDA, "prefill: no current device below ordinal %d", kMaxDevices);
  {
    std::lock_guard<std::mutex> lock(attr_mutex);
    if (!attr_set[dev]) {
      bool ok =
          cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)ssmem) == cudaSuccess &&
          cudaFuncSetAttribute(tc_readout_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)rsmem1) == cudaSuccess &&
          cudaFuncSetAttribute(tc_readout_kernel<1>,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100) ==
              cudaSuccess &&
          cudaFuncSetAttribute(tc_readout_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)rsmem2) == cudaSuccess &&
          cudaFuncSetAttribute(tc_readout_kernel<2>,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100) ==
              cudaSuccess &&
          cudaFuncSetAttribute(tc_intra_tk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tksmem) == cudaSuccess &&
          cudaFuncSetAttribute(tc_intra_tk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tksmem) == cudaSuccess;
      if (!ok) {
        cudaGetLastError();   // reported here, not by the next launch
        return oal_fail(OAL_ERR_CUDA, "prefill: setting the shared memory limit failed");
      }
      attr_set[dev] = true;
    }
  }
  StateArgs sa;
  sa.T = T; sa.nS = lay.nS; sa.chunk = chunk; sa.nC = lay.nC; sa.spp = lay.spp;
  sa.U = lay.U; sa.nparts = lay.nparts;
  sa.packed = packed; sa.cont = cont; sa.state_in = state; sa.state_out = state;
  sa.ptot = ptot; sa.snap = snap; sa.status = status;
  if (lay.nparts > 1) {
    sa.mode = 0;
    dim3 g0(kTiles, lay.nparts - 1, lay.U);
    launch_pdl(tc_state_kernel, g0, dim3(kStateThreads), ssmem, stream, tmK, tmV, sa);
    st = oal_after_launch("tc_state_kernel", stream);
    if (st != OAL_OK) return st;
  }
  sa.mode = 1;
  dim3 g1(kTiles, lay.nparts, lay.U);
  launch_pdl(tc_state_kernel, g1, dim3(kStateThreads), ssmem, stream, tmK, tmV, sa);
  st = oal_after_launch("tc_state_kernel", stream);
  if (st != OAL_OK) return st;

  ReadArgs ra;
  ra.T = T; ra.nC = lay.nC; ra.chunk = chunk; ra.Hq = Hq; ra.Hkv = Hkv; ra.rho = Hq / Hkv;
  ra.Y = static_cast<__nv_bfloat16 *>(Y);
  ra.coef = coef; ra.plans = plans; ra.status = status; ra.snap = snap;
  ra.intra_num = reinterpret_cast<float *>(w + lay.inum_off);
  ra.intra_den = reinterpret_cast<float *>(w + lay.iden_off);
  {
    // two heads a block once one head a block would make four waves of two
    // blocks per SM (chunks of 64 and 128; a 256-token chunk's second half
    // reloads K and V for its second 128-key tile, one head a block)
    const int forced = g_intra_heads.load();
    int hpb = forced ? forced
                     : ((size_t)ra.rho * lay.nS * lay.U >= (size_t)4 * 2 * 152 ? kTkHeads : 1);
    if (chunk == 256) hpb = 1;
    ReadArgs rt = ra;
    rt.nh_per_block = hpb;
    dim3 gtk((ra.rho + hpb - 1) / hpb, lay.nS, lay.U);
    if (chunk == 256)
      launch_pdl(tc_intra_tk_kernel<true>, gtk, dim3(kTkThreads), tksmem, stream, tmQ, tmKn, tmV, rt);
    else
      launch_pdl(tc_intra_tk_kernel<false>, gtk, dim3(kTkThreads), tksmem, stream, tmQ, tmKn, tmV, rt);
    st = oal_after_launch("tc_intra_tk_kernel", stream);
  }
  if (st != OAL_OK) return st;
  ra.nh_per_block = kMaxNH;
  dim3 g2((ra.rho + kMaxNH - 1) / kMaxNH, lay.nS, lay.U);
  if (chunk == 64)
    launch_pdl(tc_readout_kernel<2>, g2, dim3(kReadThreads), rsmem2, stream, tmQ, tmS, ra);
  else
    launch_pdl(tc_readout_kernel<1>, g2, dim3(kReadThreads), rsmem1, stream, tmQ, tmS, ra);
  return oal_after_launch("tc_readout_kernel", stream);
}

}  // namespace oal
