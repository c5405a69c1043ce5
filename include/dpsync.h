/*
 * dpsync -- GB300 (sm_103a) kernels for the data-parallel side of
 * "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"
 * (NeurIPS 2026, arXiv 2609.14339; papernotes.org notes), key design 4 (dual
 * compression): each weight matrix's outer synchronisation (Streaming DiLoCo)
 * travels PowerSGD-compressed, 64x fewer values than the matrix.
 *
 * The pages name the two methods and the ratio only.  The steps follow the
 * methods' own publications (PowerSGD, Vogels, Karimireddy and Jaggi 2019:
 * one warm-started rank-k power step with error feedback; DiLoCo, Douillard et
 * al. 2023: outer SGD with Nesterov momentum on the pseudo-gradient
 * theta - W_local).  Per matrix and worker:
 *
 *   compress_p      M = E + (X - Y);  E <- M;  P = M Q           -> sum P over workers
 *   orthogonalize   P^ = orthonormal basis of the columns of P (thin QR factor,
 *                   positive diagonal; dependent columns become zero)
 *   compress_q      Q = M^T P^                                     -> sum Q over workers
 *   decompress      D = s P^ Q^T;  E <- M - D;  out = D           (s = 1 / workers)
 *   outer_step      D as above, then  b <- mu b + D;  theta <- theta - eta (D + mu b);
 *                   W_local <- (1 - mix) theta + mix W_local
 *
 * The sums over workers are the caller's (an all-reduce of P and of Q between
 * the calls; nothing to do for one worker).  Orthogonalisation and the
 * decompressed result do not depend on whether P was summed or averaged; Q is
 * summed and scaled by s inside decompress / outer_step.
 *
 * Conventions: as in specoptim.h (device pointers of the current device,
 * fp32 row-major, 16-byte aligned; `stream` a cudaStream_t as void*; status
 * codes SPECOPTIM_*; message in specoptim_last_error()).  Weight matrices are
 * m x n with ld = n, n a multiple of 4; 1 <= k <= 64.  A handle serves one
 * weight matrix and is not thread-safe.
 */
#ifndef DPSYNC_H
#define DPSYNC_H

#include <stdint.h>

#include "specoptim.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DPSYNC_MAX_RANK 64
#define DPSYNC_MAX_BATCH 16

typedef struct dpsync dpsync_t;

typedef struct {
    int32_t m, n;           /* weight shape (n a multiple of 4)                          */
    int32_t rank;           /* k; 0 = dpsync_rank(m, n, ratio)                          */
    float ratio;            /* target compression mn / ((m + n) k), default 64           */
    int32_t error_feedback; /* 1 (default): keep what the compression left out in E     */
    float outer_lr;         /* outer step eta (default 0.7)                              */
    float outer_momentum;   /* outer Nesterov mu (default 0.9)                           */
    float mix;              /* weight of W_local in the restart (default 0: replaced)    */
} dpsync_config;

/* k = floor(mn / (ratio (m + n)) + 1/2) clamped to [1, min(m, n)], evaluated in
 * double; -1 if m, n < 1 or ratio <= 0.  (Not clamped to DPSYNC_MAX_RANK.) */
int32_t dpsync_rank(int32_t m, int32_t n, float ratio);

/* Fills *cfg with the defaults above for an m x n weight. */
int dpsync_config_default(dpsync_config *cfg, int32_t m, int32_t n);

/* Creates the synchronisation state of one weight matrix on the current
 * device: error E (m x n, zero), outer momentum b (m x n, zero), outer
 * weights theta (m x n, set by dpsync_set_outer), the orthonormal basis P^
 * (m x 64 max) and small work buffers.  P (m x k) and Q (n x k) are
 * caller-owned device buffers, fp32 row-major with ld = k, that stay valid
 * for the handle's lifetime: the caller all-reduces them between the calls.
 * Q must hold the starting Q (e.g. seeded N(0, 1) values, the same on every
 * worker) before the first compress_p; each compress_q overwrites it and the
 * next sync starts from it (warm start).  *out receives the handle; the
 * handle's rank is cfg->rank or dpsync_rank(m, n, ratio) when 0, and must be
 * <= 64 (SPECOPTIM_ERR_INVALID_ARG otherwise). */
int dpsync_create(dpsync_t **out, const dpsync_config *cfg, float *P, float *Q, void *stream);

/* The rank k of a handle. */
int32_t dpsync_handle_rank(const dpsync_t *h);

/* Frees the handle's device memory (synchronises the device first). */
int dpsync_destroy(dpsync_t *h);

/* theta <- W (device m x n, read only), b <- 0: starts the outer optimizer. */
int dpsync_set_outer(dpsync_t *h, const float *W, void *stream);

/* First half of the power step for 1 to 16 handles: M = E + X - Y (E left out
 * without error feedback), stored in E, and P = M Q.  X[i], Y[i]: device
 * m x n (host arrays of device pointers); X == NULL or X[i] == NULL takes the
 * handle's theta (outer synchronisation: the pseudo-gradient theta - W_local
 * with Y[i] = W_local); Y == NULL or Y[i] == NULL subtracts nothing. */
int dpsync_compress_p_many(dpsync_t *const *handles, int32_t count, const float *const *X,
                           const float *const *Y, void *stream);

/* P^ = orthonormal basis of the columns of the (summed) P, kept in the handle:
 * the Q factor of the thin QR of P with a positive diagonal of R; a column
 * whose residual against the earlier columns has norm^2 <= 1e-10 of its own
 * norm^2 is dependent and becomes zero.  Computed as two passes of Cholesky
 * QR (Gram matrix accumulated in two-float precision, Cholesky in fp64). */
int dpsync_orthogonalize_many(dpsync_t *const *handles, int32_t count, void *stream);

/* Second half of the power step: Q = M^T P^ into the caller's Q. */
int dpsync_compress_q_many(dpsync_t *const *handles, int32_t count, void *stream);

/* D = q_scale P^ Q^T with Q the (summed) caller Q; E <- M - D (with error
 * feedback); out[i] (device m x n, may be NULL) <- D. */
int dpsync_decompress_many(dpsync_t *const *handles, int32_t count, float *const *out,
                           float q_scale, void *stream);

/* D as in dpsync_decompress_many, then the outer Nesterov step on theta and b
 * and the restart W_local[i] <- (1 - mix) theta + mix W_local[i] (device
 * m x n, in/out).  Requires dpsync_set_outer. */
int dpsync_outer_step_many(dpsync_t *const *handles, int32_t count, float *const *W_local,
                           float q_scale, void *stream);

/* Copies state to caller device buffers (any may be NULL): E, theta, b
 * (m x n each), P^ (m x k, ld = k). */
int dpsync_get_state(const dpsync_t *h, float *E, float *theta, float *mom, float *P_hat,
                     void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DPSYNC_H */
