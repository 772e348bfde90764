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
// sequences: 128-row slices, partials in the workspace, and the last block of
// a (batch, KV head) to finish (atomic ticket) sums them in a fixed order.
#include <cooperative_groups.h>

#include "oal_internal.cuh"
#include "tc_ptx.cuh"

namespace oal {
namespace {

// In global memory, not __constant__: threads read different entries, which
// the constant cache would serialize.
static __device__ const PairTable c_pairs = make_pair_table();

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTicketRows = 128;        // rows of a slice, many-sequence kernel
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
  const int bidx = unit / Hkv, kv = unit % Hkv;
  const int h0 = kv * rho;
  const int f0 = slice * rows_per_block;
  const int nrows = min(rows_per_block, F - f0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

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

  for (int n = tid; n < kD; n += kThreads) s_k[n] = to_f32(k[(size_t)unit * kD + n]);
  for (int n = tid; n < kU; n += kThreads)
    s_u[n] = n < kDv ? to_f32(v[(size_t)unit * kDv + n]) : 1.f;
  for (int n = tid; n < rho * kD; n += kThreads)
    s_q[n / kD][n % kD] = to_f32(q[((size_t)bidx * Hq + h0) * kD + n]);
  __syncthreads();

  // per-row weights: phi_f(k) and Phi~^h_f(q^h); the table loads of all
  // heads are issued before any is used
  const size_t ctab_len = packed ? kH2Packed : kH2Full;
  // (rows nrows .. nrows rounded up to 4 get zero weights: the readout reads
  // weights four rows at a time)
  for (int n = tid; n < ((nrows + 3) & ~3); n += kThreads) {
    if (n >= nrows) {
      s_wk[n] = 0.f;
#pragma unroll
      for (int hh = 0; hh < kMaxRho; ++hh) s_wq[hh][n] = 0.f;
      continue;
    }
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

  // Value columns: each warp takes 4 consecutive rows per step (lane l owns
  // columns l and l + 32) and accumulates the readout of every head with
  // packed fp32 FMAs.  Column 64 (the normaliser) follows, one row per thread.
  float2 acc[kMaxRho];
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) acc[hh] = make_float2(0.f, 0.f);
  const float2 u01 = make_float2(s_u[lane], s_u[lane + 32]);
  // (the __syncthreads above also publishes the head and tail floats)
  for (int g = 0; g < kGroups; ++g) {
    if (!oal::tc::mbar_wait(&s_bar[g], 0, &s_abort, status)) break;
    const int r1 = min(nrows, (g + 1) * rows_per_group);
    for (int rb = g * rows_per_group + 4 * warp; rb < r1; rb += 4 * kWarps) {
      const float4 wk4 = *reinterpret_cast<const float4 *>(&s_wk[rb]);
      const float wk[4] = {wk4.x, wk4.y, wk4.z, wk4.w};
      float2 nv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = rb + u;
        nv[u] = make_float2(0.f, 0.f);
        if (rr < r1) {
          const float *src = s_rows + rr * kU;
          nv[u] = make_float2(fmaf(wk[u], u01.x, src[lane]), fmaf(wk[u], u01.y, src[lane + 32]));
          float *dst = S + (size_t)rr * kU;
          __stcs(dst + lane, nv[u].x);
          __stcs(dst + lane + 32, nv[u].y);
        }
      }
#pragma unroll
      for (int hh = 0; hh < kMaxRho; ++hh) {
        if (hh < rho) {
          const float4 wq = *reinterpret_cast<const float4 *>(&s_wq[hh][rb]);
          acc[hh] = ffma2(make_float2(wq.x, wq.x), nv[0], acc[hh]);
          acc[hh] = ffma2(make_float2(wq.y, wq.y), nv[1], acc[hh]);
          acc[hh] = ffma2(make_float2(wq.z, wq.z), nv[2], acc[hh]);
          acc[hh] = ffma2(make_float2(wq.w, wq.w), nv[3], acc[hh]);
        }
      }
    }
  }
  // every copy has landed (or timed out) before the buffer is read again
  for (int g = 0; g < kGroups; ++g) oal::tc::mbar_wait_teardown(&s_bar[g], 0, status);
  float den[kMaxRho];
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) den[hh] = 0.f;
  for (int rr = tid; rr < nrows; rr += kThreads) {
    const float n2 = s_rows[rr * kU + kDv] + s_wk[rr];   // u_64 = 1
    __stcs(S + (size_t)rr * kU + kDv, n2);
#pragma unroll
    for (int hh = 0; hh < kMaxRho; ++hh)
      if (hh < rho) den[hh] = fmaf(s_wq[hh][rr], n2, den[hh]);
  }
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den[hh] += __shfl_xor_sync(0xffffffffu, den[hh], o);
  __syncthreads();   // the slice buffer is reused for the block reduction
  float(*s_red)[kMaxRho][kU] = reinterpret_cast<float(*)[kMaxRho][kU]>(s_buf);

  // block reduction (fixed order) -> this block's partial readout
#pragma unroll
  for (int hh = 0; hh < kMaxRho; ++hh) {
    if (hh < rho) {
      s_red[warp][hh][lane] = acc[hh].x;
      s_red[warp][hh][lane + 32] = acc[hh].y;
      if (lane == 0) s_red[warp][hh][64] = den[hh];
    }
  }
  __syncthreads();
  for (int n = tid; n < rho * kU; n += kThreads) {
    const int hh = n / kU, c = n % kU;
    float sum = 0.f;
    for (int w = 0; w < kWarps; ++w) sum += s_red[w][hh][c];
    s_part[hh][c] = sum;
  }
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

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
decode_ticket_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                     const Tin *__restrict__ v, Tin *__restrict__ y,
                     const float *__restrict__ a, const float *__restrict__ b,
                     const float *__restrict__ Ctab, float *__restrict__ state, int Hq, int Hkv,
                     int F, int packed, int rows_per_block, int nslices,
                     float *__restrict__ partial, unsigned *__restrict__ tickets, int *status) {
  __shared__ float s_part[kMaxRho][kU];
  __shared__ bool s_last;
  const int unit = blockIdx.y, slice = blockIdx.x, bidx = unit / Hkv, kv = unit % Hkv;
  const int rho = Hq / Hkv, h0 = kv * rho, tid = threadIdx.x;
  decode_slice<Tin, kTicketRows>(q, k, v, a, b, Ctab, state, Hq, Hkv, F, packed, rows_per_block,
                                 slice, unit, status, s_part);
  float *part = partial + ((size_t)unit * nslices + slice) * kMaxRho * kU;
  for (int n = tid; n < rho * kU; n += kThreads) part[(n / kU) * kU + n % kU] = s_part[n / kU][n % kU];
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&tickets[unit], 1u);
    s_last = (ticket == (unsigned)nslices - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last block of this (batch, KV head): sum the slices in a fixed order, divide
  __shared__ float s_tot[kMaxRho][kU];
  const float *pu = partial + (size_t)unit * nslices * kMaxRho * kU;
  for (int n = tid; n < rho * kU; n += kThreads) {
    const int hh = n / kU, c = n % kU;
    float p16[16];   // sixteen interleaved sums: the loads are in flight together
#pragma unroll
    for (int j = 0; j < 16; ++j) p16[j] = 0.f;
    for (int sl0 = 0; sl0 < nslices; sl0 += 16) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (sl0 + j < nslices) p16[j] += __ldcg(pu + (size_t)(sl0 + j) * kMaxRho * kU + hh * kU + c);
    }
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) p16[j] += p16[j + w];
    s_tot[hh][c] = p16[0];
  }
  __syncthreads();
  for (int n = tid; n < rho * kDv; n += kThreads) {
    const int hh = n / kDv, c = n % kDv;
    y[((size_t)bidx * Hq + h0 + hh) * kDv + c] = from_f32<Tin>(s_tot[hh][c] / s_tot[hh][kDv]);
  }
  if (tid == 0) tickets[unit] = 0u;   // ready for the next call
}

}  // namespace

// Dynamic shared memory of a block: the slice (+ alignment slack), reused
// afterwards for the per-warp readout partials.
static size_t decode_smem_floats(int rpb) {
  const size_t rows = (size_t)rpb * kU + 8, red = (size_t)kWarps * kMaxRho * kU;
  return rows > red ? rows : red;
}

// The cluster kernel serves batches whose clusters (one per batch x KV
// head) all fit the GPU at once.
static bool use_clusters(size_t units) { return units * 16 <= 2 * 152; }

static int ticket_slices(int packed) { return (state_rows(packed) + kTicketRows - 1) / kTicketRows; }

size_t decode_workspace_bytes(int B, int Hkv, int packed) {
  const size_t units = (size_t)B * Hkv;
  if (use_clusters(units)) return 256;
  const size_t part = units * ticket_slices(packed) * kMaxRho * kU * sizeof(float);
  const size_t tick = units * sizeof(unsigned);
  return ((part + 255) / 256) * 256 + ((tick + 255) / 256) * 256;
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

template <typename Tin>
static oal_status launch_decode_t(const Tin *q, const Tin *k, const Tin *v, int B, int Hq, int Hkv,
                                  const float *a, const float *b, const float *C, int packed,
                                  float *state, Tin *y, void *ws, cudaStream_t stream) {
  const int F = state_rows(packed);
  const size_t units = (size_t)B * Hkv;
  static bool attr_set[256] = {};   // per device: the slice buffers are above 48 KB
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
    return oal_check_launch("decode: cudaGetDevice");
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_cluster_kernel<Tin>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(decode_smem_floats(kClusterRows) * sizeof(float))) !=
            cudaSuccess ||
        cudaFuncSetAttribute(decode_ticket_kernel<Tin>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(decode_smem_floats(kTicketRows) * sizeof(float))) != cudaSuccess)
      return oal_check_launch("decode: shared memory attribute");
    attr_set[dev] = true;
  }
  if (use_clusters(units)) {
    const int cs = decode_cluster_size<Tin>(packed);
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
  const int nslices = ticket_slices(packed);
  const size_t part_bytes = ((units * nslices * kMaxRho * kU * sizeof(float) + 255) / 256) * 256;
  float *partial = (float *)ws;
  unsigned *tickets = (unsigned *)((char *)ws + part_bytes);
  if (cudaMemsetAsync(tickets, 0, units * sizeof(unsigned), stream) != cudaSuccess)
    return oal_check_launch("decode ticket reset");
  launch_pdl(decode_ticket_kernel<Tin>, dim3(nslices, (unsigned)units), dim3(kThreads),
             decode_smem_floats(kTicketRows) * sizeof(float), stream, q, k, v, y, a, b, C, state,
             Hq, Hkv, F, packed, (int)kTicketRows, nslices, partial, tickets,
             oal_device_status_word());
  return oal_after_launch("decode_ticket_kernel", stream);
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
