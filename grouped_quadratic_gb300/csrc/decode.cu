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
// slices, one block per (slice, batch x KV head).  A block first copies its
// whole slice into shared memory with bulk copies (rows of 65 floats are not
// 16-byte aligned: the ends are read with plain loads), forms the per-row
// weights meanwhile, then
// each warp walks rows (lane l owns columns l and l+32, lane 0 also column
// 64): coalesced 128-byte stores of the updated rows and readout accumulators
// in registers.  The partial readouts of the slices are combined in one of two
// ways.  Few sequences: the slices of one (batch, KV head) form a thread-block
// cluster and meet in distributed shared memory, where the first block sums
// them in rank order and divides (no scratch, no extra launch).  Many
// sequences: persistent blocks stream runs of 112-row slices with the next
// slice's copy in flight, sum their partials per (batch, KV head) in shared
// memory and write them to the workspace; a second small kernel adds them in
// a fixed order and divides.
#include <cooperative_groups.h>

#include <utility>

#include "oal_internal.cuh"
#include "tc_ptx.cuh"

namespace oal {
namespace {

// In global memory, not __constant__: threads read different entries, which
// the constant cache would serialize.
static __device__ const PairTable c_pairs = make_pair_table();

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kClusterRows = 528;       // rows of a slice, cluster kernel (state rows / 8)
constexpr int kMaxRho = 8;

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {   // a * b + c, two lanes
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

constexpr int kGroups = 4;             // row groups of a slice, each with its own bulk copy

// k, u = [v; 1] and the query rows of every head sharing the KV head of
// `unit`, as fp32 in shared memory.
template <typename Tin>
__device__ __forceinline__ void load_unit_vectors(const Tin *__restrict__ q, const Tin *__restrict__ k,
                                                  const Tin *__restrict__ v, int unit, int Hq,
                                                  int Hkv, float *s_k, float *s_u,
                                                  float (*s_q)[kD]) {
  const int rho = Hq / Hkv, bidx = unit / Hkv, h0 = (unit % Hkv) * rho;
  for (int n = threadIdx.x; n < kD; n += kThreads) s_k[n] = to_f32(k[(size_t)unit * kD + n]);
  for (int n = threadIdx.x; n < kU; n += kThreads)
    s_u[n] = n < kDv ? to_f32(v[(size_t)unit * kDv + n]) : 1.f;
  for (int n = threadIdx.x; n < rho * kD; n += kThreads)
    s_q[n / kD][n % kD] = to_f32(q[((size_t)bidx * Hq + h0) * kD + n]);
}

// Per-row weights, in two steps so the table loads can be issued early:
// weight_fetch reads the row's kind, dims and every head's table entry;
// weight_finish forms phi_f(k) into s_wk[n] and Phi~^h_f(q^h) into
// s_wq[h * stride + n] from the head's k and q in shared memory.
struct WeightRow {
  int kind, r, t;            // kind 0: H0, 1: H1 (dim r), 2: H2 (dims r, t)
  float coef[kMaxRho];
};

__device__ __forceinline__ WeightRow weight_fetch(const float *__restrict__ a,
                                                  const float *__restrict__ b,
                                                  const float *__restrict__ Ctab, int packed,
                                                  int h0, int rho, int f) {
  const size_t ctab_len = packed ? kH2Packed : kH2Full;
  WeightRow w;
  w.r = 0;
  w.t = 0;
  if (f == 0) w.kind = 0;
  else if (f <= kD) { w.kind = 1; w.r = f - 1; }
  else {
    w.kind = 2;
    const int nn = f - 1 - kD;
    if (packed) { w.r = c_pairs.rt[nn] >> 8; w.t = c_pairs.rt[nn] & 0xff; }
    else { w.r = nn >> 6; w.t = nn & 63; }
  }
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) {
    w.coef[hh] = 0.f;
    if (hh < rho) {
      const int h = h0 + hh;
      w.coef[hh] = w.kind == 0 ? __ldg(a + h)
                 : (w.kind == 1 ? __ldg(b + (size_t)h * kD + w.r)
                                : __ldg(Ctab + (size_t)h * ctab_len + (f - 1 - kD)));
    }
  }
  return w;
}

__device__ __forceinline__ void weight_finish(const WeightRow &w, int rho, int n, const float *s_k,
                                              const float (*s_q)[kD], float *s_wk, float *s_wq,
                                              int stride) {
  s_wk[n] = w.kind == 0 ? 1.f : (w.kind == 1 ? s_k[w.r] : s_k[w.r] * s_k[w.t]);
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) {
    if (hh < rho) {
      float x;
      if (w.kind == 0) x = w.coef[hh];
      else if (w.kind == 1) x = w.coef[hh] * s_q[hh][w.r] * 0.125f;
      else x = w.coef[hh] * s_q[hh][w.r] * s_q[hh][w.t] * 0.015625f;
      s_wq[hh * stride + n] = x;
    }
  }
}

// Rows nrows .. nrows rounded up to 4 get zero weights (the readout reads
// weights four rows at a time).
__device__ __forceinline__ void weight_pad(int n, float *s_wk, float *s_wq, int stride) {
  s_wk[n] = 0.f;
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) s_wq[hh * stride + n] = 0.f;
}

// Per-row weights of rows f0 .. f0 + nrows - 1 (and the padding rows).
__device__ __forceinline__ void slice_weights(const float *__restrict__ a,
                                              const float *__restrict__ b,
                                              const float *__restrict__ Ctab, int packed, int h0,
                                              int rho, int f0, int nrows, const float *s_k,
                                              const float (*s_q)[kD], float *s_wk, float *s_wq,
                                              int stride) {
  for (int n = threadIdx.x; n < ((nrows + 3) & ~3); n += kThreads) {
    if (n >= nrows) {
      weight_pad(n, s_wk, s_wq, stride);
      continue;
    }
    const WeightRow w = weight_fetch(a, b, Ctab, packed, h0, rho, f0 + n);
    weight_finish(w, rho, n, s_k, s_q, s_wk, s_wq, stride);
  }
}

// Value columns of rows r0 .. r1 - 1 (r0 a multiple of 4): each warp takes 4
// consecutive rows per step (lane l owns columns l and l + 32), writes the
// updated rows and accumulates the readout of every head.  The packed fp32
// FMAs pair two adjacent rows of one column, so the weight pairs come
// straight from a 16-byte shared load: acc[h][0] holds the partial sums of
// column l over even and odd rows, acc[h][1] those of column l + 32 (their
// two halves are added at the end).  s_rows[i] holds float i of the slice, S
// the slice in the state.  NH: heads the loops are unrolled for (rho <= NH).
template <int NH>
__device__ __forceinline__ void rows_step(const float *s_rows, float *S, int r0, int r1, int rho,
                                          const float *s_u, const float *s_wk, const float *s_wq,
                                          int stride, float2 (&acc)[NH][2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 ua = make_float2(s_u[lane], s_u[lane]);
  const float2 ub = make_float2(s_u[lane + 32], s_u[lane + 32]);
  for (int rb = r0 + 4 * warp; rb < r1; rb += 4 * kWarps) {
    const float4 wk4 = *reinterpret_cast<const float4 *>(&s_wk[rb]);
    // rows past r1 (zero weights) read as zero: they add nothing to the
    // readout and are not stored
    float va[4], vb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool in = rb + u < r1;
      va[u] = in ? s_rows[(rb + u) * kU + lane] : 0.f;
      vb[u] = in ? s_rows[(rb + u) * kU + lane + 32] : 0.f;
    }
    const float2 sa[2] = {make_float2(va[0], va[1]), make_float2(va[2], va[3])};
    const float2 sb[2] = {make_float2(vb[0], vb[1]), make_float2(vb[2], vb[3])};
    const float2 wk01 = make_float2(wk4.x, wk4.y), wk23 = make_float2(wk4.z, wk4.w);
    const float2 na0 = ffma2(wk01, ua, sa[0]), nb0 = ffma2(wk01, ub, sb[0]);
    const float2 na1 = ffma2(wk23, ua, sa[1]), nb1 = ffma2(wk23, ub, sb[1]);
    const float nvA[4] = {na0.x, na0.y, na1.x, na1.y}, nvB[4] = {nb0.x, nb0.y, nb1.x, nb1.y};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (rb + u < r1) {
        float *dst = S + (size_t)(rb + u) * kU;
        __stcs(dst + lane, nvA[u]);
        __stcs(dst + lane + 32, nvB[u]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      if (hh < rho) {
        const float4 wq = *reinterpret_cast<const float4 *>(&s_wq[hh * stride + rb]);
        const float2 w01 = make_float2(wq.x, wq.y), w23 = make_float2(wq.z, wq.w);
        acc[hh][0] = ffma2(w01, na0, acc[hh][0]);
        acc[hh][0] = ffma2(w23, na1, acc[hh][0]);
        acc[hh][1] = ffma2(w01, nb0, acc[hh][1]);
        acc[hh][1] = ffma2(w23, nb1, acc[hh][1]);
      }
    }
  }
}

// Column 64 (the normaliser, one row per thread), then the block's readout
// partial of every head in a fixed order: into s_out (accumulate: added to
// it).  s_red is a free buffer of kWarps * kMaxRho * kU floats; the block
// passes a barrier at the end.
template <int NH>
__device__ __forceinline__ void slice_reduce(const float *s_rows, float *S, int nrows, int rho,
                                             const float *s_wk, const float *s_wq, int stride,
                                             const float2 (&acc)[NH][2], float *s_red_buf,
                                             float (*s_out)[kU], bool accumulate) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float den[NH];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) den[hh] = 0.f;
  for (int rr = tid; rr < nrows; rr += kThreads) {
    const float n2 = s_rows[rr * kU + kDv] + s_wk[rr];   // u_64 = 1
    __stcs(S + (size_t)rr * kU + kDv, n2);
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
      if (hh < rho) den[hh] = fmaf(s_wq[hh * stride + rr], n2, den[hh]);
  }
#pragma unroll
  for (int hh = 0; hh < NH; ++hh)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den[hh] += __shfl_xor_sync(0xffffffffu, den[hh], o);
  __syncthreads();   // the slice buffer is reused for the block reduction
  float(*s_red)[kMaxRho][kU] = reinterpret_cast<float(*)[kMaxRho][kU]>(s_red_buf);
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) {
    if (hh < rho) {
      s_red[warp][hh][lane] = acc[hh][0].x + acc[hh][0].y;
      s_red[warp][hh][lane + 32] = acc[hh][1].x + acc[hh][1].y;
      if (lane == 0) s_red[warp][hh][64] = den[hh];
    }
  }
  __syncthreads();
  for (int n = tid; n < rho * kU; n += kThreads) {
    const int hh = n / kU, c = n % kU;
    float sum = 0.f;
    for (int w = 0; w < kWarps; ++w) sum += s_red[w][hh][c];
    s_out[hh][c] = accumulate ? s_out[hh][c] + sum : sum;
  }
  __syncthreads();
}

// One slice of rows of one (batch, KV head): state update in place and this
// block's partial readout of every head in s_part (rho x 65, fixed order).
template <typename Tin, int kRows>
__device__ __forceinline__ void decode_slice(const Tin *__restrict__ q, const Tin *__restrict__ k,
                                             const Tin *__restrict__ v,
                                             const float *__restrict__ a,
                                             const float *__restrict__ b,
                                             const float *__restrict__ Ctab,
                                             float *__restrict__ state, int Hq, int Hkv, int F,
                                             int packed, int rows_per_block, int slice, int unit,
                                             int *status, float (&s_part)[kMaxRho][kU]) {
  pdl_trigger();
  pdl_wait();
  const int rho = Hq / Hkv;
  const int h0 = (unit % Hkv) * rho;
  const int f0 = slice * rows_per_block;
  const int nrows = min(rows_per_block, F - f0);
  const int tid = threadIdx.x;

  extern __shared__ __align__(16) float s_buf[];   // decode_smem_floats(rows_per_block)
  __shared__ float s_k[kD];
  __shared__ float s_u[kU];
  __shared__ float s_q[kMaxRho][kD];
  __shared__ __align__(16) float s_wk[kRows];
  __shared__ __align__(16) float s_wq[kMaxRho][kRows];
  __shared__ __align__(8) uint64_t s_bar[kGroups];
  __shared__ int s_abort;

  // The slice (nrows rows of 65 floats) is contiguous in memory but not
  // 16-byte aligned in general.  Its aligned interior is fetched by kGroups
  // bulk copies (one per group of rows, boundaries rounded up to 16 bytes)
  // issued before anything else; the at most 3 + 3 floats outside it are
  // read with plain loads.  s_rows[i] holds float i of the slice.
  float *S = state + ((size_t)unit * F + f0) * kU;
  const size_t sf0 = ((size_t)unit * F + f0) * kU;     // float index of the slice
  const int nel = nrows * kU;
  const int head = (int)((4 - (sf0 & 3)) & 3);
  const int tail = (int)((sf0 + nel) & 3);
  float *s_rows = s_buf + ((4 - head) & 3);            // s_rows + head is 16-byte aligned
  const int rows_per_group = (((nrows + kGroups - 1) / kGroups) + 3) & ~3;   // whole steps of 4
  auto copy_begin = [&](int g) {                      // float offset where copy g starts
    if (g == 0) return min(head, nel - tail);
    const int x = min(nrows, g * rows_per_group) * kU;
    return min(nel - tail, head + ((x - head + 3) & ~3));
  };
  if (tid == 0) {
    s_abort = 0;
    for (int g = 0; g < kGroups; ++g) oal::tc::mbar_init(&s_bar[g], 1);
    oal::tc::fence_mbar_init();
    for (int g = 0; g < kGroups; ++g) {
      const int c0 = copy_begin(g), c1 = copy_begin(g + 1 < kGroups ? g + 1 : kGroups);
      const int n = (g + 1 < kGroups ? c1 : nel - tail) - c0;
      oal::tc::mbar_arrive_expect_tx(&s_bar[g], n > 0 ? (uint32_t)n * 4u : 0u);
      if (n > 0) oal::tc::bulk_load(s_rows + c0, S + c0, (uint32_t)n * 4u, &s_bar[g]);
    }
  }
  if (tid < head) s_rows[tid] = __ldcs(S + tid);
  if (tid >= 32 && tid < 32 + tail) s_rows[nel - tail + tid - 32] = __ldcs(S + nel - tail + tid - 32);

  load_unit_vectors(q, k, v, unit, Hq, Hkv, s_k, s_u, s_q);
  __syncthreads();
  slice_weights(a, b, Ctab, packed, h0, rho, f0, nrows, s_k, s_q, s_wk, &s_wq[0][0], kRows);
  __syncthreads();   // (also publishes the head and tail floats)

  float2 acc[kMaxRho][2];
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) acc[hh][0] = acc[hh][1] = make_float2(0.f, 0.f);
  for (int g = 0; g < kGroups; ++g) {
    if (!oal::tc::mbar_wait(&s_bar[g], 0, &s_abort, status)) break;
    rows_step<kMaxRho>(s_rows, S, g * rows_per_group, min(nrows, (g + 1) * rows_per_group), rho,
                       s_u, s_wk, &s_wq[0][0], kRows, acc);
  }
  // every copy has landed (or timed out) before the buffer is read again
  for (int g = 0; g < kGroups; ++g) oal::tc::mbar_wait_teardown(&s_bar[g], 0, status);
  slice_reduce<kMaxRho>(s_rows, S, nrows, rho, s_wk, &s_wq[0][0], kRows, acc, s_buf, s_part,
                        false);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
decode_cluster_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                      const Tin *__restrict__ v, Tin *__restrict__ y,
                      const float *__restrict__ a, const float *__restrict__ b,
                      const float *__restrict__ Ctab, float *__restrict__ state, int Hq,
                      int Hkv, int F, int packed, int rows_per_block, int *status) {
  __shared__ float s_part[kMaxRho][kU];
  const int unit = blockIdx.y, bidx = unit / Hkv, kv = unit % Hkv, rho = Hq / Hkv;
  const int h0 = kv * rho, tid = threadIdx.x;
  decode_slice<Tin, kClusterRows>(q, k, v, a, b, Ctab, state, Hq, Hkv, F, packed, rows_per_block,
                                  blockIdx.x, unit, status, s_part);
  // the first block sums every block's partial from distributed shared
  // memory, in rank order, and divides
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    __shared__ float s_tot[kMaxRho][kU];
    const int nblk = (int)cluster.num_blocks();
    for (int n = tid; n < rho * kU; n += kThreads) {
      const int hh = n / kU, c = n % kU;
      float sum = 0.f;
      for (int r = 0; r < nblk; ++r) sum += cluster.map_shared_rank(&s_part[hh][c], r)[0];
      s_tot[hh][c] = sum;
    }
    __syncthreads();
    for (int n = tid; n < rho * kDv; n += kThreads) {
      const int hh = n / kDv, c = n % kDv;
      y[((size_t)bidx * Hq + h0 + hh) * kDv + c] = from_f32<Tin>(s_tot[hh][c] / s_tot[hh][kDv]);
    }
  }
  cluster.sync();   // no block leaves while the first one reads its partial
}

// ---------------------------------------------------------------- many sequences
// Persistent blocks, each walking a contiguous run of (batch x KV head, slice)
// items with the next slice's bulk copy in flight while the current one is
// updated (two slice buffers), so the memory system always has loads queued.
// A block sums the partial readouts of the items of one (batch, KV head) in
// shared memory and writes one partial per (block, batch x KV head) it
// touched (at most two: a run is never longer than a head's slices);
// decode_finish_kernel adds them in block order and divides.
constexpr int kStreamRows = 192;                  // rows of a slice (one per thread at most)
constexpr int kStreamBuf = kStreamRows * kU + 8;  // floats of one slice buffer (16-byte multiple)
constexpr int kStreamBlocksPerSM = 2;
static_assert(kStreamRows <= kThreads && kStreamRows % 4 == 0, "one weight row per thread");

struct SliceGeom {
  float *S;          // first float of the slice in the state
  int nrows, nel;    // rows, floats
  int head, tail;    // floats before the first / after the last 16-byte boundary
  int f0;            // first row
};

__device__ __forceinline__ SliceGeom slice_geom(float *state, int F, int rows_per_slice, int unit,
                                                int slice) {
  SliceGeom g;
  g.f0 = slice * rows_per_slice;
  g.nrows = min(rows_per_slice, F - g.f0);
  const size_t sf0 = ((size_t)unit * F + g.f0) * kU;
  g.S = state + sf0;
  g.nel = g.nrows * kU;
  g.head = (int)((4 - (sf0 & 3)) & 3);
  g.tail = (int)((sf0 + g.nel) & 3);
  return g;
}

template <typename Tin, int RHO>
__global__ void __launch_bounds__(kThreads, kStreamBlocksPerSM)
decode_stream_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                     const Tin *__restrict__ v, const float *__restrict__ a,
                     const float *__restrict__ b, const float *__restrict__ Ctab,
                     float *__restrict__ state, int Hq, int Hkv, int F, int packed, int nslices,
                     int nitems, int per_block, float *__restrict__ partial, int *status) {
  extern __shared__ __align__(16) float s_dyn[];   // two slice buffers
  __shared__ float s_k[kD];
  __shared__ float s_u[kU];
  __shared__ float s_q[kMaxRho][kD];
  __shared__ __align__(16) float s_wk[kStreamRows];
  __shared__ __align__(16) float s_wq[kMaxRho][kStreamRows];
  __shared__ float s_acc[kMaxRho][kU];
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ int s_abort;
  const int tid = threadIdx.x;
  constexpr int rho = RHO;
  const int i0 = blockIdx.x * per_block, i1 = min(nitems, i0 + per_block);
  if (tid == 0) {
    s_abort = 0;
    oal::tc::mbar_init(&s_bar[0], 1);
    oal::tc::mbar_init(&s_bar[1], 1);
    oal::tc::fence_mbar_init();
  }
  pdl_trigger();
  pdl_wait();   // the state rows the previous step wrote
  // bulk copy of the aligned interior of item x into buffer bb
  auto issue = [&](int x, int bb) {
    const SliceGeom g = slice_geom(state, F, kStreamRows, x / nslices, x % nslices);
    float *rows = s_dyn + bb * kStreamBuf + ((4 - g.head) & 3);
    const int n = g.nel - g.head - g.tail;
    oal::tc::mbar_arrive_expect_tx(&s_bar[bb], (uint32_t)n * 4u);
    oal::tc::bulk_load(rows + g.head, g.S + g.head, (uint32_t)n * 4u, &s_bar[bb]);
  };
  if (tid == 0 && i0 < i1) issue(i0, 0);
  // table entries of this thread's row of item x, loaded one item ahead
  auto fetch = [&](int x) {
    WeightRow w{};
    const int f = (x % nslices) * kStreamRows + tid;
    if (x < i1 && tid < kStreamRows && f < F)
      w = weight_fetch(a, b, Ctab, packed, (x / nslices) % Hkv * rho, rho, f);
    return w;
  };
  WeightRow wrow = fetch(i0);
  int cur_unit = -1, slot = -1, fail_at = -1;
  float *const pblk = partial + (size_t)blockIdx.x * 2 * kMaxRho * kU;
  for (int it = i0; it < i1; ++it) {
    const int j = it - i0, bb = j & 1;
    const int unit = it / nslices, slice = it % nslices;
    // buffer bb ^ 1 was released by the end of the previous item
    if (tid == 0 && it + 1 < i1) issue(it + 1, bb ^ 1);
    if (unit != cur_unit) {
      if (cur_unit >= 0)
        for (int n = tid; n < rho * kU; n += kThreads) pblk[slot * kMaxRho * kU + n] = s_acc[n / kU][n % kU];
      __syncthreads();
      ++slot;
      cur_unit = unit;
      for (int n = tid; n < rho * kU; n += kThreads) s_acc[n / kU][n % kU] = 0.f;
      load_unit_vectors(q, k, v, unit, Hq, Hkv, s_k, s_u, s_q);
      __syncthreads();
    }
    const SliceGeom g = slice_geom(state, F, kStreamRows, unit, slice);
    float *s_rows = s_dyn + bb * kStreamBuf + ((4 - g.head) & 3);
    if (tid < g.head) s_rows[tid] = __ldcs(g.S + tid);
    if (tid >= 32 && tid < 32 + g.tail)
      s_rows[g.nel - g.tail + tid - 32] = __ldcs(g.S + g.nel - g.tail + tid - 32);
    if (tid < g.nrows) weight_finish(wrow, rho, tid, s_k, s_q, s_wk, &s_wq[0][0], kStreamRows);
    else if (tid < ((g.nrows + 3) & ~3)) weight_pad(tid, s_wk, &s_wq[0][0], kStreamRows);
    wrow = fetch(it + 1);   // in flight while this item is processed
    __syncthreads();
    const bool landed = oal::tc::mbar_wait(&s_bar[bb], (j >> 1) & 1, &s_abort, status);
    if (__syncthreads_or(!landed)) { fail_at = it; break; }   // the same decision in every thread
    float2 acc[RHO][2];
#pragma unroll
    for (int hh = 0; hh < RHO; ++hh) acc[hh][0] = acc[hh][1] = make_float2(0.f, 0.f);
    rows_step<RHO>(s_rows, g.S, 0, g.nrows, RHO, s_u, s_wk, &s_wq[0][0], kStreamRows, acc);
    slice_reduce<RHO>(s_rows, g.S, g.nrows, RHO, s_wk, &s_wq[0][0], kStreamRows, acc,
                      s_dyn + bb * kStreamBuf, s_acc, true);
  }
  if (cur_unit >= 0 && fail_at < 0)
    for (int n = tid; n < rho * kU; n += kThreads) pblk[slot * kMaxRho * kU + n] = s_acc[n / kU][n % kU];
  if (fail_at >= 0 && tid == 0) {
    // the copies of the failed item and of the one after it must land before exit
    const int j = fail_at - i0;
    oal::tc::mbar_wait_teardown(&s_bar[j & 1], (j >> 1) & 1, status);
    if (fail_at + 1 < i1) oal::tc::mbar_wait_teardown(&s_bar[(j + 1) & 1], ((j + 1) >> 1) & 1, status);
  }
}

// y of every query head of (batch, KV head) blockIdx.x: the partials of the
// blocks whose runs touched it, in block order, then u~[0:64] / u~[64].
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
decode_finish_kernel(Tin *__restrict__ y, const float *__restrict__ partial, int Hq, int Hkv,
                     int nslices, int per_block) {
  pdl_trigger();
  pdl_wait();
  const int unit = blockIdx.x, bidx = unit / Hkv, kv = unit % Hkv, rho = Hq / Hkv;
  const int first = unit * nslices, last = first + nslices - 1;
  const int b0 = first / per_block, b1 = last / per_block;
  __shared__ float s_tot[kMaxRho][kU];
  for (int n = threadIdx.x; n < rho * kU; n += kThreads) {
    float sum = 0.f;
    for (int blk = b0; blk <= b1; ++blk) {
      const int slot = unit - (blk * per_block) / nslices;
      sum += __ldcg(partial + ((size_t)blk * 2 + slot) * kMaxRho * kU + n);
    }
    s_tot[n / kU][n % kU] = sum;
  }
  __syncthreads();
  for (int n = threadIdx.x; n < rho * kDv; n += kThreads) {
    const int hh = n / kDv, c = n % kDv;
    y[((size_t)bidx * Hq + kv * rho + hh) * kDv + c] = from_f32<Tin>(s_tot[hh][c] / s_tot[hh][kDv]);
  }
}

}  // namespace

// Dynamic shared memory of a block: the slice (+ alignment slack), reused
// afterwards for the per-warp readout partials.
static size_t decode_smem_floats(int rpb) {
  const size_t rows = (size_t)rpb * kU + 8, red = (size_t)kWarps * kMaxRho * kU;
  return rows > red ? rows : red;
}

// The cluster kernel serves batches whose clusters (one per batch x KV
// head, of 16 blocks or, for more than 19 units, 8) all fit the GPU at once.
static bool use_clusters(size_t units) { return units * 8 <= 2 * 152; }

// Work split of the streaming kernel: items (batch x KV head, slice), runs of
// per_block consecutive items, one run per block (a run never spans more than
// two heads: per_block <= nslices).
struct StreamPlan {
  int nslices, nitems, per_block, nblocks;
};
static StreamPlan stream_plan(size_t units, int packed) {
  StreamPlan p;
  p.nslices = (state_rows(packed) + kStreamRows - 1) / kStreamRows;
  p.nitems = (int)units * p.nslices;
  const int target = 152 * kStreamBlocksPerSM;
  p.per_block = (p.nitems + target - 1) / target;
  if (p.per_block > p.nslices) p.per_block = p.nslices;
  p.nblocks = (p.nitems + p.per_block - 1) / p.per_block;
  return p;
}

size_t decode_workspace_bytes(int B, int Hkv, int packed) {
  const size_t units = (size_t)B * Hkv;
  if (use_clusters(units)) return 256;
  const StreamPlan p = stream_plan(units, packed);
  const size_t part = (size_t)p.nblocks * 2 * kMaxRho * kU * sizeof(float);
  return ((part + 255) / 256) * 256;
}

int decode_max_rho() { return kMaxRho; }

// Blocks per (batch, KV head) of the cluster kernel: 16 where the device can
// schedule such clusters, else the portable 8.
template <typename Tin>
static int decode_cluster_size(int packed) {
  static int cs[2] = {0, 0};
  int &c = cs[packed != 0];
  if (c) return c;
  c = 8;
  if (cudaFuncSetAttribute(decode_cluster_kernel<Tin>,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    const int rpb = ((state_rows(packed) + 15) / 16 + 3) & ~3;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = decode_smem_floats(rpb) * sizeof(float);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<Tin>, &cfg) == cudaSuccess &&
        n > 0)
      c = 16;
  }
  cudaGetLastError();   // a refused query is not an error of the next launch
  return c;
}

// The streaming kernel of each query-head count 1..kMaxRho.
template <typename Tin, int... I>
static bool set_stream_smem(std::integer_sequence<int, I...>) {
  return ((cudaFuncSetAttribute(decode_stream_kernel<Tin, I + 1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(2 * kStreamBuf * sizeof(float))) == cudaSuccess) && ...);
}
template <typename Tin, int... I, typename... Args>
static oal_status launch_stream(std::integer_sequence<int, I...>, int rho, dim3 grid,
                                cudaStream_t stream, Args... args) {
  bool done = false;
  ((rho == I + 1 ? (launch_pdl(decode_stream_kernel<Tin, I + 1>, grid, dim3(kThreads),
                               2 * kStreamBuf * sizeof(float), stream, args...),
                    done = true)
                 : false),
   ...);
  if (!done) return oal_fail(OAL_ERR_UNSUPPORTED, "Hq/Hkv=%d", rho);
  return oal_after_launch("decode_stream_kernel", stream);
}

template <typename Tin>
static oal_status launch_decode_t(const Tin *q, const Tin *k, const Tin *v, int B, int Hq, int Hkv,
                                  const float *a, const float *b, const float *C, int packed,
                                  float *state, Tin *y, void *ws, cudaStream_t stream) {
  const int F = state_rows(packed);
  const size_t units = (size_t)B * Hkv;
  static bool attr_set[kMaxDevices] = {};   // per device: the slice buffers are above 48 KB
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return oal_check_launch("decode: cudaGetDevice");
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_cluster_kernel<Tin>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(decode_smem_floats(kClusterRows) * sizeof(float))) !=
            cudaSuccess ||
        !set_stream_smem<Tin>(std::make_integer_sequence<int, kMaxRho>{}))
      return oal_check_launch("decode: shared memory attribute");
    attr_set[dev] = true;
  }
  if (use_clusters(units)) {
    const int cs = units * 16 <= 2 * 152 ? decode_cluster_size<Tin>(packed) : 8;
    const int rpb = ((F + cs - 1) / cs + 3) & ~3;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, (unsigned)units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = decode_smem_floats(rpb) * sizeof(float);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaLaunchKernelEx(&cfg, decode_cluster_kernel<Tin>, q, k, v, y, a, b, C, state, Hq, Hkv, F,
                       packed, rpb, oal_device_status_word());
    return oal_after_launch("decode_cluster_kernel", stream);
  }
  const StreamPlan p = stream_plan(units, packed);
  float *partial = (float *)ws;
  oal_status st = launch_stream<Tin>(std::make_integer_sequence<int, kMaxRho>{}, Hq / Hkv,
                                     dim3(p.nblocks), stream, q, k, v, a, b, C, state, Hq, Hkv,
                                     F, packed, p.nslices, p.nitems, p.per_block, partial,
                                     oal_device_status_word());
  if (st != OAL_OK) return st;
  launch_pdl(decode_finish_kernel<Tin>, dim3((unsigned)units), dim3(kThreads), 0, stream, y,
             (const float *)partial, Hq, Hkv, p.nslices, p.per_block);
  return oal_after_launch("decode_finish_kernel", stream);
}

oal_status launch_decode(const void *q, const void *k, const void *v, int is_bf16,
                         int B, int Hq, int Hkv, const float *a, const float *b,
                         const float *C, int packed, float *state, void *y,
                         void *ws, cudaStream_t stream) {
  if (is_bf16)
    return launch_decode_t((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                           (const __nv_bfloat16 *)v, B, Hq, Hkv, a, b, C, packed, state,
                           (__nv_bfloat16 *)y, ws, stream);
  return launch_decode_t((const float *)q, (const float *)k, (const float *)v, B, Hq, Hkv, a, b, C,
                         packed, state, (float *)y, ws, stream);
}

}  // namespace oal
