/*
 * specoptim -- GB300 (sm_103a) kernels for the fast-circuit hot path of
 * "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"
 * (NeurIPS 2026, arXiv 2609.14339; papernotes.org notes):
 *
 *   * the spectral-correction optimizer step (key design 2: anchor EMA;
 *     key design 3: SVD of the anchor momentum, Tikhonov filter, two-sided
 *     projection, convex blend, AdamW), and
 *   * the in-graph activation mask (key design 1: keep K = round((1-p)H)
 *     dims per token chosen by a shared deterministic function g; only the K
 *     kept values are sent; the backward pass reuses the same indices).
 *
 * Conventions for every entry point below
 *   - Pointers named as device pointers must point to GPU memory of the
 *     current device; they are owned by the caller unless stated otherwise.
 *     Matrices are fp32, row-major, m x n with leading dimension n (as in
 *     torch.nn.Linear.weight: m = out_features, n = in_features), and must be
 *     16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream unless stated otherwise.
 *   - Every call returns a status code and never throws or aborts.  On a
 *     non-zero status, specoptim_last_error() gives a message (per thread).
 *   - A handle serves one weight matrix and is not thread-safe.
 *   - One device per process: the library's shared state (kernel launch
 *     limits, a scratch buffer, the flag of its bounded device-side waits)
 *     belongs to the device that is current at its first use.  Creating a
 *     handle, or a call that reaches that state, while another device is
 *     current returns SPECOPTIM_ERR_INVALID_ARG.
 */
#ifndef SPECOPTIM_H
#define SPECOPTIM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SPECOPTIM_OK                  0
#define SPECOPTIM_ERR_INVALID_ARG     1 /* null pointer, bad size or hyperparameter   */
#define SPECOPTIM_ERR_MISALIGNED      2 /* a pointer is not 16-byte aligned           */
#define SPECOPTIM_ERR_CUDA            3 /* a CUDA call failed (text in last_error)    */
#define SPECOPTIM_ERR_NOT_CONVERGED   4 /* SVD hit svd_max_sweeps; old factors kept   */
#define SPECOPTIM_ERR_NOT_IMPLEMENTED 5
#define SPECOPTIM_ERR_TIMEOUT         6 /* a bounded device-side wait gave up         */
#define SPECOPTIM_ERR_BOUNDS          7 /* an index check failed (checked build only) */

/* GEMM arithmetic of the projection (key design 3, projection equation) */
#define SPECOPTIM_PREC_TF32 0  /* tcgen05 kind::tf32 tensor cores, fp32 accumulate */
#define SPECOPTIM_PREC_FP32 1  /* fp32 FMA on the SIMT cores (slow, exact fp32)    */

typedef struct specoptim specoptim_t;

typedef struct {
    int32_t m, n;           /* weight shape, m = out_features, n = in_features (>= 1) */
    float beta_anc;         /* anchor EMA coefficient (default 0.9)                   */
    float tau_p;            /* Tikhonov threshold on raw singular values (1e-3), > 0  */
    float alpha;            /* blend weight of the masked gradient (0.3), in [0,1]    */
    float beta1, beta2;     /* AdamW moment coefficients (0.9, 0.999)                 */
    float eps;              /* AdamW epsilon (1e-8)                                   */
    float weight_decay;     /* AdamW decoupled weight decay (0.01)                    */
    int32_t precision;      /* SPECOPTIM_PREC_TF32 (default) or SPECOPTIM_PREC_FP32    */
    int32_t svd_max_sweeps; /* Jacobi sweep limit of the SVD refresh (default 20)      */
    float svd_tol;          /* off-diagonal / total Frobenius norm to stop at (1e-5)  */
    int32_t svd_inner_sweeps; /* Jacobi sweeps on each 64 x 64 subproblem per round (1) */
} specoptim_config;

/* Fills *cfg with the defaults above for an m x n weight.  The defaults are
 * the pages' recipe: tau_p = 1e-3, alpha = 0.3, beta_anc = 0.9 ("loss
 * function / training strategy"); AdamW betas / eps / weight decay are the
 * usual AdamW values the workloads state. */
int specoptim_config_default(specoptim_config *cfg, int32_t m, int32_t n);

/* Creates the optimizer state of one weight matrix.  Allocates on the current
 * device, zero-initialised on `stream`: anchor momentum M (m x n), SVD factors
 * U (m x r), s (r), V (n x r), filter d (r) with r = min(m, n), AdamW moments
 * (m x n) and a workspace.  The step counter starts at 0.  Before the first
 * svd_refresh all factors are zero, so the filtered gradient is 0 and a step
 * applies AdamW to alpha * G_mask.  *out receives the handle (owned by the
 * library until specoptim_destroy). */
int specoptim_create(specoptim_t **out, const specoptim_config *cfg, void *stream);

/* Frees the handle and its device memory (synchronises the device first). */
int specoptim_destroy(specoptim_t *h);

/* Anchor momentum update, key design 2, EMA equation:
 *   M <- beta_anc * M + (1 - beta_anc) * G_anc
 * G_anc: device, m x n fp32, read only.  No bias correction. */
int specoptim_anchor_update(specoptim_t *h, const float *G_anc, void *stream);

/* SVD refresh, key design 3: thin SVD M = U diag(s) V^T (r = min(m, n),
 * s descending) and the Tikhonov filter d_i = s_i / (s_i + tau_p).
 * Computed as the eigen-decomposition of the Gram matrix of M on its short
 * side (fp32) by block Jacobi, re-orthonormalised by Newton-Schulz; then
 * s_i = |M v_i| and the long-side factor M V / s (or M^T U / s).  Columns
 * with s_i = 0 are left zero (their d_i is 0).
 * The calling thread waits once per Jacobi sweep for its convergence test (an
 * event on the library's streams), and at the end synchronises `stream` once,
 * after the factor recovery, to read the device flag of the bounded waits.
 * sweeps_out (host pointer, may be NULL) receives the number of sweeps.
 * Returns SPECOPTIM_ERR_NOT_CONVERGED, keeping the previous factors, if the
 * off-diagonal norm is still above svd_tol after svd_max_sweeps sweeps. */
int specoptim_svd_refresh(specoptim_t *h, void *stream, int32_t *sweeps_out);

/* The same refresh for 1 to 16 handles at once (e.g. the 7 weights of one
 * decoder layer): their Jacobi rounds share kernel launches, so the GPU is
 * filled by the whole batch instead of one matrix at a time.  handles: host
 * array of distinct handles; sweeps_out: host array of `count` ints or NULL.
 * A handle that already holds factors starts its Jacobi from its previous
 * short-side factor (the anchor momentum moves slowly between anchors), which
 * shortens the iteration; the result is the same decomposition.  Matrices
 * that do not converge keep their previous factors and the call returns
 * SPECOPTIM_ERR_NOT_CONVERGED after finishing the others. */
int specoptim_svd_refresh_many(specoptim_t *const *handles, int32_t count, void *stream,
                               int32_t *sweeps_out);

/* The same batched refresh, split so that it runs beside the steps instead of
 * in front of them -- the anchor of key design 2 is asynchronous: its
 * momentum is decomposed off the fast replicas' critical path, and its
 * factors take effect once they are ready.
 *   begin: enqueues the Gram matrices and the Jacobi sweeps of the handles'
 *     current anchor momenta on two streams of the library's own (ordered
 *     after the work already on `stream`), and returns at once: a library
 *     thread runs the sweep loop and waits on each sweep's convergence test,
 *     so the calling thread never blocks.
 *   end: waits (on the host) until that loop has finished -- the GPU keeps
 *     running whatever the caller queued meanwhile -- then enqueues on
 *     `stream` the factor recovery (s, d, U, V) and the step's operand copies
 *     and projectors, and synchronises `stream` once to read the device flag
 *     of the bounded waits.  sweeps_out and the return value are those of
 *     specoptim_svd_refresh_many.
 * Steps of these handles enqueued between begin and end use the previous
 * factors; steps enqueued after end use the new ones, so the results do not
 * depend on timing.  end takes the same handles in the same order as begin.
 * Between the two calls anchor_update, set_state, svd_refresh(_many), begin
 * and destroy on these handles return SPECOPTIM_ERR_INVALID_ARG, and only one
 * refresh (of any form) may be in progress per process.  Every begin needs its
 * end before the process exits (the library thread must not outlive the CUDA
 * context). */
int specoptim_svd_refresh_begin(specoptim_t *const *handles, int32_t count, void *stream);
int specoptim_svd_refresh_end(specoptim_t *const *handles, int32_t count, void *stream,
                              int32_t *sweeps_out);

/* Spectral-corrected step, key design 3 (projection and blend equations)
 * followed by AdamW:
 *   X = U^T G V,  X_filt = diag(d) X diag(d),  G_filt = U X_filt V^T,
 *   G_proj = alpha G + (1 - alpha) G_filt,
 *   t += 1;  W <- W (1 - lr wd);  m1 <- b1 m1 + (1-b1) G_proj;
 *   m2 <- b2 m2 + (1-b2) G_proj^2;
 *   W <- W - lr (m1 / (1-b1^t)) / (sqrt(m2 / (1-b2^t)) + eps).
 * W: device m x n, updated in place.  G_mask: device m x n, read only.
 * lr: this step's learning rate (a schedule stays on the host).
 * G_filt_out, G_proj_out: optional device m x n outputs (NULL to skip).
 * G_filt is evaluated as P_L G P_R with the projectors P_L = U diag(d) U^T
 * and P_R = V diag(d) V^T (the same matrix, reassociated), formed at each
 * refresh for the side that needs one: m = n runs P_R G^T, then P_L T (two
 * products); m > n runs U^T G, then P_R (U^T G)^T diag(d), then U T2 (three);
 * m < n runs V^T G^T, then P_L (.) diag(d), then T2 V^T (three).  With
 * SPECOPTIM_PREC_TF32 the factors, the projectors and every intermediate are
 * rounded to TF32 (nearest); G enters the products as given.  The blend and
 * the AdamW update run in the epilogue of the last product. */
int specoptim_step(specoptim_t *h, float *W, const float *G_mask, float lr, void *stream,
                   float *G_filt_out, float *G_proj_out);

/* The same step for 1 to 16 handles at once (e.g. the 7 weights of one
 * decoder layer), all with learning rate lr: W[i] and G_mask[i] (host arrays
 * of device pointers) belong to handles[i].  The products are grouped by
 * their position in each handle's chain (first, middle, last, as listed for
 * specoptim_step): each position runs for all handles in persistent
 * tensor-core launches of up to 8 products (largest first), so small
 * matrices fill the SMs the large ones leave idle, and the transposes of G
 * that the m > n handles need share one launch.  Same results as calling
 * specoptim_step on each handle (without debug outputs). */
int specoptim_step_many(specoptim_t *const *handles, int32_t count, float *const *W,
                        const float *const *G_mask, float lr, void *stream);

/* Copies the current factors to caller device buffers (any may be NULL):
 * U m x r, s r, V n x r, d r (row-major fp32). */
int specoptim_get_factors(const specoptim_t *h, float *U, float *s, float *V, float *d,
                          void *stream);

/* Copies the state to caller device buffers (any may be NULL): anchor
 * momentum M, AdamW moments exp_avg / exp_avg_sq (m x n each); *t (host,
 * may be NULL) receives the step counter. */
int specoptim_get_state(const specoptim_t *h, float *M, float *exp_avg, float *exp_avg_sq,
                        int64_t *t, void *stream);

/* Restores a state saved by specoptim_get_state (checkpoint resume); the SVD
 * factors must be recomputed with specoptim_svd_refresh afterwards. */
int specoptim_set_state(specoptim_t *h, const float *M, const float *exp_avg,
                        const float *exp_avg_sq, int64_t t, void *stream);

/* Plain AdamW (same update as in specoptim_step, with G_proj replaced by g)
 * for tensors outside the spectral correction (embedding, norm vectors).
 * W, g, exp_avg, exp_avg_sq: device fp32 arrays of numel elements, 16-byte
 * aligned; t is the step number after increment (>= 1). */
int specoptim_adamw(float *W, const float *g, float *exp_avg, float *exp_avg_sq, int64_t numel,
                    int64_t t, float lr, float beta1, float beta2, float eps, float weight_decay,
                    void *stream);

/* C (M x N) = A (M x K) . B (N x K)^T, fp32 row-major with leading
 * dimensions lda, ldb, ldc (device pointers).  The building block of the
 * projection (key design 3, projection equation).  precision
 * SPECOPTIM_PREC_TF32 runs the tcgen05 tensor-core kernel and requires
 * lda, ldb multiples of 4 and 16-byte aligned A, B (else
 * SPECOPTIM_ERR_NOT_IMPLEMENTED); SPECOPTIM_PREC_FP32 runs the fp32 SIMT
 * kernel for any layout. */
int specoptim_gemm_nt(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, int32_t precision,
                      void *stream);

/* The filtered gradient alone, without allocating device memory.
 * The paper has no counterpart of this entry point; it exists for callers
 * that cannot call cudaMalloc -- code inside a framework that owns all device
 * memory through its own pool, or on a latency-critical path where the device
 * synchronisation of cudaMalloc / cudaFree is not acceptable.
 *   G_filt = U diag(d) U^T G V diag(d) V^T
 * U (m x r), V (n x r), d (r floats: exactly min(m, n) values, as
 * specoptim_get_factors returns them), G (m x n), G_filt (m x n, written)
 * with r = min(m, n): device pointers, fp32 row-major, U, V, G, G_filt
 * 16-byte aligned (d needs no alignment).  The products run in the literal
 * order of the projection equation (U^T G, then V, then U and V^T again),
 * not in specoptim_step's projector association, so the two agree to the
 * rounding of the products, not bit for bit.  precision SPECOPTIM_PREC_TF32
 * rounds U, V and every intermediate to TF32 (nearest) before the tensor
 * cores read them (G enters as given); SPECOPTIM_PREC_FP32 runs fp32 SIMT
 * products.
 * Intermediates live in one 16 MiB file-scope device array that every GPU
 * loading the library holds until exit; shapes whose intermediates do not fit
 * (2 r (m + n) + r (m + r) floats when m <= n, m n + 2 r (m + n) + r (n + r)
 * when m > n; e.g. 512 x 2048 and 2048 x 512 fit, 2048 x 2048 does not) are
 * rejected with SPECOPTIM_ERR_INVALID_ARG.  All calls share the array: calls
 * that overlap on the GPU race and give wrong results.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and should
 * come before any stream capture; the address is that of the device's primary
 * context, so after cudaDeviceReset this entry point must not be called again
 * in the process. */
int specoptim_filter_noalloc(const float *U, const float *V, const float *d, const float *G,
                             float *G_filt, int32_t m, int32_t n, int32_t precision, void *stream);

/* Tracing of the library's own kernels.  Every kernel launch is counted;
 * while tracing is enabled each launch is also bracketed by two CUDA events
 * recorded on its stream.  specoptim_trace_enable(1) synchronises the device,
 * clears earlier records and the launch counter, and starts recording;
 * specoptim_trace_enable(0) stops recording (records are kept).
 * specoptim_launch_count() returns the launches since the last reset.
 * specoptim_trace_reset() synchronises and clears records and counter.
 * specoptim_trace_report() synchronises the device and writes one line per
 * kernel name, "name launches total_ms\n", into buf (len bytes, NUL
 * terminated); SPECOPTIM_ERR_INVALID_ARG if it does not fit. */
int specoptim_trace_enable(int32_t enable);
int64_t specoptim_launch_count(void);
int specoptim_trace_reset(void);
int specoptim_trace_report(char *buf, int64_t len);

/* Failure-detection self-test: launches one kernel that waits on a device
 * barrier nothing ever completes, with the same bounded-spin mechanism every
 * kernel of the library uses (spin_limit probes of ~64 ns, in [1, 2^24]).
 * The wait gives up, records its code in the library's device error flag and
 * the kernel returns; the call then synchronises `stream`, reads and clears
 * the flag and returns SPECOPTIM_ERR_TIMEOUT.  The CUDA context stays usable.
 * Any other return value means the mechanism is broken. */
int specoptim_selftest_wait_timeout(uint32_t spin_limit, void *stream);

/* Synchronises `stream` and reports whether a bounded device-side wait of any
 * of the library's kernels (the asynchronous calls of this header, of
 * mask_fused.h and of dpsync.h) gave up since the last check:
 * SPECOPTIM_ERR_TIMEOUT (the flag is cleared; the results of the kernels
 * launched since the last check are not to be trusted) or SPECOPTIM_OK.
 * A library built with -DSPECOPTIM_CHECK (a test build) also verifies, in the
 * mask kernels, that every kept index is below H; a failure skips the access
 * and is reported here as SPECOPTIM_ERR_BOUNDS. */
int specoptim_check_device(void *stream);

/* Message of the last failed call on this thread ("" if none). */
const char *specoptim_last_error(void);

/* ------------------------------------------------------------------------
 * Activation mask, key design 1: h~ = h (.) m, K = round((1-p) H) kept dims
 * per token, m = g(layer, step, batch metadata, S, H) regenerated on both
 * sides; backward dL/dh = (dL/dh~) (.) m with the same indices.
 *
 * g: row r (flattened token index b*T + t of the call) keeps the dims
 * pi_r(0), ..., pi_r(K-1) of a keyed pseudo-random permutation pi_r of
 * [0, H).  Keys: seed = sm64(sm64(sm64(layer) ^ step) ^ batch_id),
 * rowkey = sm64(seed ^ r), k_i = low32(sm64(rowkey + i)), i < 4, with sm64
 * the SplitMix64 output function.  pi_r: 4 alternating Feistel rounds on
 * w = ceil(log2 H) bits (hi = w/2 bits, lo = w - w/2 bits; rounds
 * hi ^= f(lo ^ k0), lo ^= f(hi ^ k1), hi ^= f(lo ^ k2), lo ^= f(hi ^ k3),
 * f = MurmurHash3 fmix32 masked to the half width), repeated while the
 * value is >= H.  Packed order is k order.
 *
 * dense: [rows][H], packed: [rows][K], element size elem_bytes (2 = bf16 /
 * fp16, 4 = fp32); values are copied bit for bit.  0 <= K <= H <= 2^30.
 * ------------------------------------------------------------------------ */

/* K = floor((1 - p) * H + 0.5) evaluated in double; -1 if p is outside
 * [0, 1] or H < 1. */
int32_t mask_keep_count(double p, int32_t H);

/* Forward (or activation-gradient) pack: packed[r][k] = dense[r][pi_r(k)]. */
int mask_pack(const void *dense, void *packed, int64_t rows, int32_t H, int32_t K,
              int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id, void *stream);

/* Receiver unpack: dense[r][pi_r(k)] = packed[r][k]; all other entries are
 * written as +0 (all-zero bits), whatever the sign or NaN-ness of h. */
int mask_unpack(const void *packed, void *dense, int64_t rows, int32_t H, int32_t K,
                int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id,
                void *stream);

/* The kept indices themselves: idx_out[r][k] = pi_r(k), int32, device
 * (for tests and for callers that build their own fused ops). */
int mask_indices(int32_t *idx_out, int64_t rows, int32_t H, int32_t K, uint32_t layer,
                 uint64_t step, uint64_t batch_id, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECOPTIM_H */
