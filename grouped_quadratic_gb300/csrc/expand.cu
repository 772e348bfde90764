// expand.cu -- coefficient expansion of [OAL] Sec. 4.3 (Algorithm 1, the coefficient step).
//
//   M = L L^T,  a = eps + M_00,  b_r = 2 M_{0,g(r)},  C_rt = M_{g(r),g(t)}
//
// M is formed in fp64 with explicitly rounded multiplies and adds, c
// ascending, so the fp32 tables are reproducible bit for bit:
//   M_gh = sum_{c=0}^{min(g,h)} L[g][c] * L[h][c]   (each product exact)
//   a = fp32(fp64(eps) + M_00), b_r = fp32(2 M_0g), C = fp32(M) / fp32(2 M)
// The packed table holds the readout weight of pair r <= t, with
// multiplicity two off the diagonal ("Exact state and parameter counts",
// App. D).
#include "oal_internal.cuh"

namespace oal {

// In global memory, not __constant__: threads read different entries, which
// the constant cache would serialize.
static __device__ const PairTable c_pairs = make_pair_table();

__global__ void expand_coeffs_kernel(const float *__restrict__ L,
                                     const int32_t *__restrict__ group, int G,
                                     float eps, int packed, float *__restrict__ a,
                                     float *__restrict__ b, float *__restrict__ C,
                                     int *status) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x;
  const int G1 = G + 1;
  __shared__ double M[(kMaxG + 1) * (kMaxG + 1)];
  __shared__ int grp[kD];
  const float *Lh = L + (size_t)h * G1 * G1;
  for (int n = threadIdx.x; n < G1 * G1; n += blockDim.x) {
    const int g = n / G1, hh = n % G1;
    const int cmax = g < hh ? g : hh;
    double m = 0.0;
    for (int c = 0; c <= cmax; ++c)
      m = __dadd_rn(m, __dmul_rn((double)Lh[g * G1 + c], (double)Lh[hh * G1 + c]));
    M[n] = m;
  }
  for (int r = threadIdx.x; r < kD; r += blockDim.x) {
    int g = group[(size_t)h * kD + r];
    if (g < 1 || g > G) {
      atomicCAS(status, kStatusOk, (int)OAL_ERR_INVALID_ARG);
      g = 1;  // keep indexing in bounds; the tables are unspecified
    }
    grp[r] = g;
  }
  __syncthreads();
  // fp32 images of M and 2M (each conversion rounds once, to nearest even)
  __shared__ float Mf[(kMaxG + 1) * (kMaxG + 1)], M2f[(kMaxG + 1) * (kMaxG + 1)];
  for (int n = threadIdx.x; n < G1 * G1; n += blockDim.x) {
    Mf[n] = __double2float_rn(M[n]);
    M2f[n] = __double2float_rn(__dmul_rn(2.0, M[n]));
  }
  __syncthreads();
  // blockIdx.y splits the C table; block 0 also writes a and b
  const int n0 = blockIdx.y * blockDim.x + threadIdx.x, nstep = blockDim.x * gridDim.y;
  if (blockIdx.y == 0) {
    if (threadIdx.x == 0) a[h] = __double2float_rn(__dadd_rn((double)eps, M[0]));
    for (int r = threadIdx.x; r < kD; r += blockDim.x) b[(size_t)h * kD + r] = M2f[grp[r]];
  }
  if (!packed) {
    float *Ch = C + (size_t)h * kH2Full;
    for (int n = n0; n < kH2Full; n += nstep) {
      const int r = n / kD, t = n % kD;
      Ch[n] = Mf[grp[r] * G1 + grp[t]];
    }
  } else {
    float *Ch = C + (size_t)h * kH2Packed;
    for (int n = n0; n < kH2Packed; n += nstep) {
      const int r = c_pairs.rt[n] >> 8, t = c_pairs.rt[n] & 0xff;
      const int idx = grp[r] * G1 + grp[t];
      Ch[n] = r == t ? Mf[idx] : M2f[idx];
    }
  }
}

oal_status launch_expand_coeffs(const float *L, const int32_t *group, int Hq,
                                int G, float eps, int packed, float *a, float *b,
                                float *C, cudaStream_t stream) {
  launch_pdl(expand_coeffs_kernel, dim3(Hq, 4), dim3(256), 0, stream, L, group, G, eps, packed,
             a, b, C, oal_device_status_word());
  return oal_after_launch("expand_coeffs_kernel", stream);
}

}  // namespace oal
