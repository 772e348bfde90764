// decode.cu -- one decode token of OAL ([OAL] = "Not All Dimensions Are
// Equal: Outlier-Aware Attention Linearization with Grouped Quadratic
// Kernels", Algorithm 1, its per-token state update and readout).
//
// For each (batch, KV head) the fp32 state S [F][65] is streamed once:
//     S[f][c] += phi_f(k) u_c              (Eq. 5 update, u = [v; 1])
//     u~^h[c] += Phi~^h_f(q^h) S[f][c]     (Eq. 6 readout, every query head
//                                           h sharing the KV head)
// and y^h = u~^h[0:64] / u~^h[64].  The kernel is bound by HBM: 8 bytes
// (read + write) per state element.  Rows of the state are split into
// slices, one block per (slice, batch x KV head); inside a block each warp
// walks rows (lane l owns columns l and l+32, lane 0 also column 64), so
// every load and store is a coalesced 128-byte warp access and the readout
// accumulators stay in registers.  Per-slice partial readouts go to the
// workspace; the last block of a (batch, KV head) to finish (atomic ticket)
// sums them in slice order and divides.
#include "oal_internal.cuh"

namespace oal {
namespace {

// In global memory, not __constant__: threads read different entries, which
// the constant cache would serialize.
static __device__ const PairTable c_pairs = make_pair_table();

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerBlock = 256;
constexpr int kMaxRho = 8;
constexpr int kUnroll = 4;

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
              const Tin *__restrict__ v, Tin *__restrict__ y,
              const float *__restrict__ a, const float *__restrict__ b,
              const float *__restrict__ Ctab, float *__restrict__ state, int Hq,
              int Hkv, int F, int packed, int nslices,
              float *__restrict__ partial, unsigned *__restrict__ tickets) {
  const int rho = Hq / Hkv;
  const int slice = blockIdx.x;
  const int unit = blockIdx.y;              // b * Hkv + kv
  const int bidx = unit / Hkv, kv = unit % Hkv;
  const int h0 = kv * rho;
  const int f0 = slice * kRowsPerBlock;
  const int nrows = min(kRowsPerBlock, F - f0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  __shared__ float s_k[kD];
  __shared__ float s_u[kU];
  __shared__ float s_q[kMaxRho][kD];
  __shared__ float s_wk[kRowsPerBlock];
  __shared__ float s_wq[kMaxRho][kRowsPerBlock];
  __shared__ float s_red[kWarps][kMaxRho][kU];
  __shared__ bool s_last;

  for (int n = tid; n < kD; n += kThreads) s_k[n] = to_f32(k[(size_t)unit * kD + n]);
  for (int n = tid; n < kU; n += kThreads)
    s_u[n] = n < kDv ? to_f32(v[(size_t)unit * kDv + n]) : 1.f;
  for (int n = tid; n < rho * kD; n += kThreads)
    s_q[n / kD][n % kD] = to_f32(q[((size_t)bidx * Hq + h0) * kD + n]);
  __syncthreads();

  // per-row weights: phi_f(k) and Phi~^h_f(q^h); the table loads of all
  // heads are issued before any is used
  const size_t ctab_len = packed ? kH2Packed : kH2Full;
  for (int n = tid; n < nrows; n += kThreads) {
    const int f = f0 + n;
    int r = 0, t = 0, kind;
    if (f == 0) kind = 0;
    else if (f <= kD) { kind = 1; r = f - 1; }
    else {
      kind = 2;
      const int nn = f - 1 - kD;
      if (packed) { r = c_pairs.rt[nn] >> 8; t = c_pairs.rt[nn] & 0xff; }
      else { r = nn >> 6; t = nn & 63; }
    }
    s_wk[n] = kind == 0 ? 1.f : (kind == 1 ? s_k[r] : s_k[r] * s_k[t]);
    float coef[kMaxRho];
#pragma unroll
    for (int hh = 0; hh < kMaxRho; ++hh) {
      coef[hh] = 0.f;
      if (hh < rho) {
        const int h = h0 + hh;
        coef[hh] = kind == 0 ? __ldg(a + h)
                 : (kind == 1 ? __ldg(b + (size_t)h * kD + r)
                              : __ldg(Ctab + (size_t)h * ctab_len + (f - 1 - kD)));
      }
    }
#pragma unroll
    for (int hh = 0; hh < kMaxRho; ++hh) {
      if (hh < rho) {
        float w;
        if (kind == 0) w = coef[hh];
        else if (kind == 1) w = coef[hh] * s_q[hh][r] * 0.125f;
        else w = coef[hh] * s_q[hh][r] * s_q[hh][t] * 0.015625f;
        s_wq[hh][n] = w;
      }
    }
  }
  __syncthreads();

  float acc[kMaxRho][3];
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) acc[hh][0] = acc[hh][1] = acc[hh][2] = 0.f;
  const float u0 = s_u[lane], u1 = s_u[lane + 32], u2 = s_u[64];
  float *S = state + ((size_t)unit * F + f0) * kU;

  for (int rb = warp * kUnroll; rb < nrows; rb += kWarps * kUnroll) {
    float x0[kUnroll], x1[kUnroll], x2[kUnroll];
#pragma unroll
    for (int uu = 0; uu < kUnroll; ++uu) {
      const int rr = rb + uu;
      if (rr < nrows) {
        const float *src = S + (size_t)rr * kU;
        x0[uu] = __ldcs(src + lane);
        x1[uu] = __ldcs(src + lane + 32);
        x2[uu] = lane == 0 ? __ldcs(src + 64) : 0.f;
      }
    }
#pragma unroll
    for (int uu = 0; uu < kUnroll; ++uu) {
      const int rr = rb + uu;
      if (rr < nrows) {
        const float wk = s_wk[rr];
        const float n0 = fmaf(wk, u0, x0[uu]);
        const float n1 = fmaf(wk, u1, x1[uu]);
        const float n2 = fmaf(wk, u2, x2[uu]);
        float *dst = S + (size_t)rr * kU;
        __stcs(dst + lane, n0);
        __stcs(dst + lane + 32, n1);
        if (lane == 0) __stcs(dst + 64, n2);
#pragma unroll
        for (int hh = 0; hh < kMaxRho; ++hh) {
          if (hh < rho) {
            const float wq = s_wq[hh][rr];
            acc[hh][0] = fmaf(wq, n0, acc[hh][0]);
            acc[hh][1] = fmaf(wq, n1, acc[hh][1]);
            acc[hh][2] = fmaf(wq, n2, acc[hh][2]);
          }
        }
      }
    }
  }

  // block reduction (fixed order) -> partial[unit][slice][rho][65]
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) {
    if (hh < rho) {
      s_red[warp][hh][lane] = acc[hh][0];
      s_red[warp][hh][lane + 32] = acc[hh][1];
      if (lane == 0) s_red[warp][hh][64] = acc[hh][2];
    }
  }
  __syncthreads();
  float *part = partial + ((size_t)unit * nslices + slice) * kMaxRho * kU;
  for (int n = tid; n < rho * kU; n += kThreads) {
    const int hh = n / kU, c = n % kU;
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += s_red[w][hh][c];
    part[hh * kU + c] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&tickets[unit], 1u);
    s_last = (ticket == (unsigned)nslices - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last block of this (batch, KV head): sum the slices in order, divide.
  __shared__ float s_tot[kMaxRho][kU];
  const float *pu = partial + (size_t)unit * nslices * kMaxRho * kU;
  for (int n = tid; n < rho * kU; n += kThreads) {
    const int hh = n / kU, c = n % kU;
    float s = 0.f;
    for (int sl = 0; sl < nslices; ++sl) s += __ldcg(pu + (size_t)sl * kMaxRho * kU + hh * kU + c);
    s_tot[hh][c] = s;
  }
  __syncthreads();
  for (int n = tid; n < rho * kDv; n += kThreads) {
    const int hh = n / kDv, c = n % kDv;
    y[((size_t)bidx * Hq + h0 + hh) * kDv + c] = from_f32<Tin>(s_tot[hh][c] / s_tot[hh][kDv]);
  }
  if (tid == 0) tickets[unit] = 0u;   // ready for the next call
}

}  // namespace

int decode_slices(int packed) {
  return (state_rows(packed) + kRowsPerBlock - 1) / kRowsPerBlock;
}

size_t decode_workspace_bytes(int B, int Hkv, int packed) {
  const size_t units = (size_t)B * Hkv;
  const size_t part = units * decode_slices(packed) * kMaxRho * kU * sizeof(float);
  const size_t tick = units * sizeof(unsigned);
  return ((part + 255) / 256) * 256 + ((tick + 255) / 256) * 256;
}

int decode_max_rho() { return kMaxRho; }

oal_status launch_decode(const void *q, const void *k, const void *v, int is_bf16,
                         int B, int Hq, int Hkv, const float *a, const float *b,
                         const float *C, int packed, float *state, void *y,
                         void *ws, cudaStream_t stream) {
  const int F = state_rows(packed);
  const int nslices = decode_slices(packed);
  const size_t units = (size_t)B * Hkv;
  const size_t part_bytes =
      ((units * nslices * kMaxRho * kU * sizeof(float) + 255) / 256) * 256;
  float *partial = (float *)ws;
  unsigned *tickets = (unsigned *)((char *)ws + part_bytes);
  if (cudaMemsetAsync(tickets, 0, units * sizeof(unsigned), stream) != cudaSuccess)
    return oal_check_launch("decode ticket reset");
  dim3 grid(nslices, (unsigned)units);
  if (is_bf16)
    decode_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
        (__nv_bfloat16 *)y, a, b, C, state, Hq, Hkv, F, packed, nslices, partial, tickets);
  else
    decode_kernel<float><<<grid, kThreads, 0, stream>>>(
        (const float *)q, (const float *)k, (const float *)v, (float *)y, a, b, C, state,
        Hq, Hkv, F, packed, nslices, partial, tickets);
  return oal_after_launch("decode_kernel", stream);
}

}  // namespace oal
