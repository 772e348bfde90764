/*
 * oal.h -- C ABI of liboal.so: OAL causal attention on one GB300 (sm_103a).
 *
 * Method: "Not All Dimensions Are Equal: Outlier-Aware Attention
 * Linearization with Grouped Quadratic Kernels" (arXiv:2610.13674), cited as
 * [OAL].  With x_r = q_r k_r / sqrt(d), group sums s_g = sum_{r in G_g} x_r
 * and s_bar = [1, s_1..s_G], the kernel is
 *     kappa(q,k) = eps + s_bar^T L L^T s_bar                  [OAL] Eq. (7)
 * and the output is the normalised inclusive causal average
 *     y_i = sum_{j<=i} kappa(q_i,k_j) v_j / sum_{j<=i} kappa(q_i,k_j),
 * evaluated in linear time through the prefix states of Eq. (5),
 *     H0 = sum u_j,  H1_r = sum k_{j,r} u_j,  H2_rt = sum k_{j,r} k_{j,t} u_j,
 *     u_j = [v_j; 1],
 * and the readout of Eq. (6),
 *     u~_i = a H0 + (1/sqrt d) sum_r b_r q_r H1_r + (1/d) sum_rt C_rt q_r q_t H2_rt,
 *     y_i  = u~_i[0:dv] / u~_i[dv].
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *    in the stated row-major layout, and 16-byte aligned (oal_group_dims, a
 *    host function, takes host pointers).  The library keeps
 *    no allocation between calls; scratch memory is passed in `workspace`.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).
 *    Argument errors are detected on the host and returned synchronously,
 *    with nothing launched.  Errors found on the device (a group id out of
 *    range, a bounded wait that gave up) are recorded in a per-process device
 *    status word and returned by the next oal_sync_status().
 *  - Grouped-query attention: query head h reads key/value head
 *    h / (Hq / Hkv); Hq must be a multiple of Hkv.  L and the group map are
 *    per query head; the state is per (batch, key/value head).
 *  - Supported sizes: d == dv == 64, 1 <= G <= 7.  Other values return
 *    OAL_ERR_UNSUPPORTED.
 *  - On error, oal_last_error() returns a message for the calling thread.
 *  - Per device (ordinals 0..255) the library caches the addresses of its
 *    device globals and the function attributes it set; do not keep using
 *    the library on a device after cudaDeviceReset() on it.
 */
#ifndef OAL_H
#define OAL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OAL_OK = 0,
  OAL_ERR_INVALID_ARG = 1, /* null/unaligned pointer, bad size, bad enum */
  OAL_ERR_UNSUPPORTED = 2, /* valid but outside the supported sizes      */
  OAL_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed       */
  OAL_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up         */
} oal_status;

typedef enum { OAL_F32 = 0, OAL_BF16 = 1 } oal_dtype;

/*
 * State layouts ([OAL] Eq. (5); App. D "Exact state and parameter counts").
 * The state of one (batch, KV head) is F rows of dv+1 fp32 values
 * (the last value of a row belongs to the "1" of u = [v; 1]):
 *   row 0                 H0
 *   rows 1 .. d           H1_r,            r = row - 1
 *   FULL   (F = 1+d+d*d):        row 1+d + r*d + t            holds H2_rt
 *   PACKED (F = 1+d+d(d+1)/2):   row 1+d + r*d - r(r-1)/2 + (t-r) holds H2_rt,
 *                                r <= t (H2 is symmetric; App. D)
 * For d = dv = 64: FULL is 4161 x 65 fp32 (1,081,860 B), PACKED 2145 x 65
 * (557,700 B) per (batch, KV head).
 */
typedef enum { OAL_STATE_FULL = 0, OAL_STATE_PACKED = 1 } oal_state_layout;

/* Rows F of one state, and F*(dv+1), for the layout; 0 for a bad layout. */
size_t oal_state_rows(int d, oal_state_layout layout);
size_t oal_state_elems(int d, int dv, oal_state_layout layout);
/* Entries of one head's C table: d*d (FULL) or d(d+1)/2 (PACKED). */
size_t oal_coeff_table_elems(int d, oal_state_layout layout);

/*
 * oal_expand_coeffs -- coefficient map of [OAL] Sec. 4.3 ("Positive
 * group-aware kernel"), the coefficient step of Algorithm 1:  M = L L^T,
 *     a = eps + M_00,  b_r = 2 M_{0,g(r)},  C_rt = M_{g(r),g(t)}.
 *  L      [Hq][G+1][G+1] fp32, row-major; only the lower triangle is read.
 *  group  [Hq][d] int32, the group of each dimension, values 1..G.
 *  a [Hq], b [Hq][d] fp32.
 *  C [Hq][d*d] (FULL: C_rt at r*d+t) or [Hq][d(d+1)/2] (PACKED: the
 *    readout weight of pair r <= t at r*d - r(r-1)/2 + (t-r), which is
 *    C_rt on the diagonal and 2*C_rt off it -- App. D's multiplicity).
 * Rounding (the pages fix none): M_gh = sum_{c=0}^{min(g,h)} L[g][c]*L[h][c]
 * in fp64 with c ascending, then a = fp32(fp64(eps) + M_00),
 * b_r = fp32(2 M), C = fp32(M) or fp32(2 M), round to nearest even.  The
 * tables are therefore reproducible bit for bit.
 * A group id outside 1..G is reported by oal_sync_status() as
 * OAL_ERR_INVALID_ARG (the tables are then unspecified).
 */
oal_status oal_expand_coeffs(const float *L, const int32_t *group, int Hq,
                             int G, int d, float eps, oal_state_layout layout,
                             float *a, float *b, float *C, cudaStream_t stream);

/*
 * oal_prefill -- causal OAL attention over T tokens ([OAL] Algorithm 1,
 * causal-evaluation stage), evaluated in chunks of `chunk`
 * tokens: inter-chunk terms through the prefix states (Eqs. 5-6),
 * intra-chunk terms pair by pair from the group sums (Eq. 7).  Exact in
 * real arithmetic ([OAL] App. D, Eq. (25)).
 *  Q [B][Hq][T][d], K [B][Hkv][T][d], V [B][Hkv][T][dv] in `dtype`.
 *  L, group, G, eps: the kernel parameters (as for oal_expand_coeffs).
 *  a, b, C: the tables oal_expand_coeffs produced from the same
 *    (L, group, eps) in the same `layout` (not checked).
 *  state [B][Hkv][F][dv+1] fp32 in `layout`: on return, the states after
 *    token T-1.  continue_from_state != 0 starts from the values in `state`
 *    (resume after an earlier prefill or decode); 0 starts from zero.
 *  Y [B][Hq][T][dv] in `dtype` (bf16 outputs are rounded once from fp32).
 *  chunk: 0 (default: 128 for bf16, 64 for fp32) or one of 64, 128, 256
 *    tokens: the period of the inter-chunk states.
 *  workspace: device scratch of at least oal_prefill_workspace_bytes(...)
 *    bytes, 256-byte aligned; contents need not be initialised.
 * Arithmetic: OAL_F32 inputs use fp32 CUDA-core FMA throughout.  OAL_BF16
 * inputs, at every chunk size, use bf16 tensor-core products with fp32
 * accumulation and fp32 states (exact products phi(k) split into two bf16
 * terms; the state snapshots read by the readout and the intra-chunk
 * kernel values are rounded to bf16, the scaled queries of the intra-chunk
 * factors w_c too).
 * T == 0 leaves Y untouched and sets `state` to zero unless
 * continue_from_state != 0.
 */
size_t oal_prefill_workspace_bytes(int B, int Hq, int Hkv, int T, int d,
                                   int dv, oal_dtype dtype,
                                   oal_state_layout layout, int chunk);
oal_status oal_prefill(const void *Q, const void *K, const void *V,
                       oal_dtype dtype, int B, int Hq, int Hkv, int T, int d,
                       int dv, const float *L, const int32_t *group, int G,
                       float eps, const float *a, const float *b,
                       const float *C, oal_state_layout layout, float *state,
                       int continue_from_state, void *Y, int chunk,
                       void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/*
 * oal_prefill_noalloc -- oal_prefill without a caller workspace.  The paper
 * has no counterpart: this is a deployment convenience of this library.
 *
 * Some callers cannot allocate device memory at the point where they run a
 * prefill: code that must not call cudaMalloc or a caching allocator (for
 * instance inside a framework that owns all device memory, or a runtime that
 * forbids allocation after start-up), or code that has no allocator handle
 * at all.  This entry point takes the same arguments as oal_prefill minus
 * `workspace` / `workspace_bytes`; its scratch lives in one fixed array of
 * OAL_PREFILL_NOALLOC_SCRATCH_BYTES bytes inside the library, which every
 * GPU that loads the library keeps until the process exits.  It makes no
 * cudaMalloc / cudaFree call and calls no allocating library routine.
 *  Limit: a problem whose oal_prefill_workspace_bytes(...) exceeds
 *    OAL_PREFILL_NOALLOC_SCRATCH_BYTES is rejected with OAL_ERR_INVALID_ARG
 *    and a message giving both sizes (in this version bf16 with B = 1,
 *    Hq = 14, Hkv = 2 fits up to T = 7296); use oal_prefill with a
 *    workspace beyond that.
 *  First call on a device: looks up the array's device address with
 *    cudaGetSymbolAddress on the current device (this may load the
 *    library's device code on that device) and caches it per device.
 *    Make that first call before any stream capture begins.
 *  Sharing: all calls in the process share the one array per device.  Two
 *    calls whose kernels overlap on the GPU (different streams without an
 *    ordering between them, or different host threads) race on it and give
 *    wrong results; order them on one stream.  Nothing in the array needs to
 *    start at zero: each call writes every scratch byte before reading it.
 *  Everything else (arguments, layouts, errors, arithmetic) is as for
 *    oal_prefill.
 */
#define OAL_PREFILL_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
/* The size of that array in this build of the library, in bytes. */
size_t oal_prefill_noalloc_scratch_bytes(void);
oal_status oal_prefill_noalloc(const void *Q, const void *K, const void *V,
                               oal_dtype dtype, int B, int Hq, int Hkv, int T,
                               int d, int dv, const float *L,
                               const int32_t *group, int G, float eps,
                               const float *a, const float *b, const float *C,
                               oal_state_layout layout, float *state,
                               int continue_from_state, void *Y, int chunk,
                               cudaStream_t stream);

/*
 * oal_prefill_backward -- gradients of <dY, Y> for the causal prefill output
 * Y = oal_prefill(Q, K, V, L, group, eps): the step that the coefficient
 * calibration by output matching ([OAL] App. B, Eq. (20)) and the LoRA
 * adaptation ([OAL] Sec. 5.2) differentiate through.  With g_ij =
 * dY_i . (v_j - y_i) / D_i for j <= i (D_i the normaliser of row i):
 *     dV_j = sum_{i>=j} kappa_ij dY_i / D_i,
 *     dQ_ir = sum_j 2 g_ij (M s_bar_ij)_{g(r)} k_jr / sqrt(d),
 *     dK_jr = sum_i 2 g_ij (M s_bar_ij)_{g(r)} q_ir / sqrt(d),
 *     dL = lower((dM + dM^T) L),  dM = sum_ij g_ij s_bar_ij s_bar_ij^T,
 * key/value gradients summed over the query heads sharing the KV head.
 *  Q, K, V, dY: as for oal_prefill (dY [B][Hq][T][dv] in `dtype`).
 *  L, group, G, eps: the kernel parameters of the forward call.
 *  dQ [B][Hq][T][d], dK [B][Hkv][T][d], dV [B][Hkv][T][dv],
 *  dL [Hq][G+1][G+1] (zero above the diagonal): fp32 outputs.
 *  workspace: at least oal_prefill_backward_workspace_bytes(...) bytes,
 *    256-byte aligned, contents need not be initialised.
 * Arithmetic: fp32 on the CUDA cores, every pair formed explicitly
 * (O(T^2 d) per head); the forward normalisers are recomputed, so the call
 * needs no saved forward state.  Deterministic: no atomics on the outputs.
 * B == 0 or T == 0 writes dL = 0 and nothing else.
 */
size_t oal_prefill_backward_workspace_bytes(int B, int Hq, int Hkv, int T, int d, int dv);
oal_status oal_prefill_backward(const void *Q, const void *K, const void *V,
                                const void *dY, oal_dtype dtype, int B, int Hq,
                                int Hkv, int T, int d, int dv, const float *L,
                                const int32_t *group, int G, float eps,
                                float *dQ, float *dK, float *dV, float *dL,
                                void *workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * oal_decode_step -- one token of [OAL] Algorithm 1 (state update and readout) for every
 * sequence: u = [v; 1]; H0 += u; H1_r += k_r u; H2_rt += k_r k_t u; then the
 * Eq. (6) readout for each query head of the KV head (inclusive: the new
 * token attends to itself).
 *  q [B][Hq][d], k [B][Hkv][d], v [B][Hkv][dv] in `dtype`; y [B][Hq][dv].
 *  a, b, C, layout: as for oal_prefill.  state: in/out, fp32.
 *  workspace: at least oal_decode_workspace_bytes(...) bytes, 256-byte
 *    aligned, contents need not be initialised.
 * Arithmetic: fp32 state update and fp32 accumulation (CUDA cores).
 */
size_t oal_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int dv,
                                  oal_state_layout layout);
oal_status oal_decode_step(const void *q, const void *k, const void *v,
                           oal_dtype dtype, int B, int Hq, int Hkv, int d,
                           int dv, const float *a, const float *b,
                           const float *C, oal_state_layout layout,
                           float *state, void *y, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Calibration, the step before the path ([OAL] Sec. 3.1 and App. B "Dimension
 * grouping"): the groups of each query head follow from contribution scores.
 *
 * oal_contribution_scores -- [OAL] Eq. (2) for every prompt p of a batch:
 *     chi[p][h][r] = 1/|Omega_p| * sum_{0 <= j <= i < N_p} |q_{p,i,r} k_{p,j,r}| / sqrt(d),
 *     |Omega_p| = N_p (N_p + 1) / 2   (chi = 0 for N_p = 0),
 * query head h paired with key/value head h / (Hq / Hkv).  The average over
 * prompts (chi_r of Eq. (2)) and its bootstrap replicates belong to
 * oal_group_dims.  Evaluated through prefix sums of |k| (the pair set is
 * never formed); sums within a 128-token chunk in fp32, across chunks in fp64.
 *  Q        [P][Hq][T][d], K [P][Hkv][T][d] (device), dtype as oal_prefill.
 *  lengths  [P] int32 (device): N_p in 0..T; NULL = every prompt has T
 *           tokens.  A length outside 0..T is clamped and recorded in the
 *           device status word (OAL_ERR_INVALID_ARG at oal_sync_status).
 *  chi      [P][Hq][d] fp32 output (device).
 *  workspace  >= oal_contribution_workspace_bytes(P, Hq, Hkv, T, d) bytes,
 *           256-byte aligned (device); 0 from the size query means
 *           unsupported or invalid sizes.
 * Supported: d == 64, P <= 65535, T <= 8,388,480 (65,535 chunks of 128
 * tokens).  P == 0
 * launches nothing; T == 0 writes zeros.
 */
size_t oal_contribution_workspace_bytes(int P, int Hq, int Hkv, int T, int d);
oal_status oal_contribution_scores(const void *Q, const void *K, oal_dtype dtype, int P,
                                   int Hq, int Hkv, int T, int d, const int32_t *lengths,
                                   float *chi, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/*
 * oal_group_dims -- the dimension grouping of [OAL] App. B, Eqs. (16)-(19),
 * for one query head.  HOST function: every pointer is host memory, nothing
 * runs on the GPU, and the call is synchronous.
 *  chi_p     [P][d] fp32: this head's per-prompt scores (Eq. (2) before the
 *            average), finite and >= 0.
 *  boot_idx  [nboot][P] int32 in 0..P-1: the prompt indices of each
 *            bootstrap replicate (resampled with replacement by the caller).
 *  alpha     tail fraction: candidate cuts k in {max(1, d - ceil(alpha d)),
 *            ..., d - 1}; 0 < alpha <= 1.
 *  tau, gamma  gap threshold of Eq. (16) and minimum bootstrap support of
 *            Eq. (18) for a natural cut; g_min >= 1 the minimum group count,
 *            reached (as far as the candidates allow) by fallback cuts in
 *            descending (support, gap) order, ties in candidate order.
 *  eps       the small constant of Eqs. (16)-(17), > 0.
 *  group     [d] int32 output: 1..G in increasing contribution.
 *  G         output: the number of groups.  The pages set no upper bound;
 *            the prefill supports G <= 7.
 * Arithmetic in fp64; chi_r and every replicate's chi^(b) are sums in index
 * order followed by one division, so results are reproducible bit for bit.
 * Returns OAL_ERR_INVALID_ARG for null pointers, P < 1, d < 2, nboot < 1,
 * an index outside 0..P-1, a negative or non-finite score, or a parameter
 * outside its range.
 */
oal_status oal_group_dims(const float *chi_p, int P, int d, const int32_t *boot_idx, int nboot,
                          double alpha, double tau, double gamma, int g_min, double eps,
                          int32_t *group, int *G);

/*
 * oal_sync_status -- synchronises `stream`, then returns and clears the
 * device status word (OAL_OK if no kernel recorded an error), or
 * OAL_ERR_CUDA if the synchronisation itself failed.
 */
oal_status oal_sync_status(cudaStream_t stream);

/*
 * oal_debug_wait_test -- for tests of the failure path only (the paper has
 * no counterpart).  Every wait of the library's kernels on an mbarrier (a
 * copy landing, a tensor-core product completing, another warp's tile) is
 * bounded: past the limit the block raises its abort flag, records
 * OAL_ERR_TIMEOUT in the device status word, drains the copies and products
 * it has in flight, frees its tensor memory and returns.  For kernels
 * launched afterwards on the current device this call sets
 *  wait_limit_cycles  that limit in SM cycles (0: the built-in 2^32 cycles,
 *                     about 2 s; the limit is consulted once a wait has
 *                     lasted 2^20 cycles, so smaller values act as 2^20);
 *  starve             0: nothing; 1, 2, 3: the UMMA issuer of the prefill's
 *                     readout, state or intra-chunk kernel makes its first
 *                     wait on a barrier that nothing arrives on, so that wait
 *                     runs out after the limit and the other warps of the
 *                     block abort mid-pipeline.
 * A starved prefill leaves Y and the state unspecified, and the next
 * oal_sync_status() returns OAL_ERR_TIMEOUT.  (0, 0) restores normal
 * operation.  Synchronous; call it while none of the library's kernels runs.
 */
oal_status oal_debug_wait_test(uint64_t wait_limit_cycles, int starve);

/*
 * oal_debug_intra_heads -- for tests only.  The bf16 prefill's intra-chunk
 * kernel at chunk sizes 64 and 128 serves one or two query heads of a KV head
 * per block, two when one head a block would fill the GPU several times over.
 * heads = 1 or 2 forces that choice for later prefill calls of this process;
 * 0 restores the automatic one.  The results are the same bit for bit
 * whichever is used.  Returns OAL_ERR_INVALID_ARG for other values.
 */
oal_status oal_debug_intra_heads(int heads);

/*
 * Launch accounting and per-kernel timing, for benchmarks and tracing.
 *  oal_launch_counter: kernels this library has launched in this process.
 *  oal_set_launch_events: thread-local hook.  While `events` is non-null,
 *    each entry-point call made by the calling thread records events[0] on its
 *    stream before its first kernel and events[k] right after its k-th kernel
 *    (k = 1 .. n-1; launches beyond n-1 are not bracketed).  The events are
 *    caller-owned cudaEvent_t handles created on the current device.
 *    Pass NULL (or n = 0) to switch the hook off.
 *  oal_last_call_launches / oal_last_call_launch_name: number and names of
 *    the kernels launched by the calling thread's last entry-point call
 *    (memset nodes are not counted).
 */
uint64_t oal_launch_counter(void);
oal_status oal_set_launch_events(cudaEvent_t *events, int n);
int oal_last_call_launches(void);
const char *oal_last_call_launch_name(int k);

/* Message of the calling thread's last non-OK status ("" if none). */
const char *oal_last_error(void);

/* Library version, e.g. "0.1.0". */
const char *oal_version(void);

#ifdef __cplusplus
}
#endif
#endif /* OAL_H */
