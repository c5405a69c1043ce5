// Element-wise kernels (elementwise.cu).
#pragma once

#include <cmath>

#include "common.cuh"

namespace spco {

// host-computed scalars of one AdamW step (bias corrections in double)
struct AdamWScalars {
    float beta1, beta2, eps;
    float decay;         // 1 - lr * weight_decay
    float step_size;     // lr / (1 - beta1^t)
    float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
};

AdamWScalars adamw_scalars(int64_t t, float lr, float beta1, float beta2, float eps, float wd);
int ema_run(float *M, const float *G, int64_t n, float beta, cudaStream_t st);
int adamw_run(float *W, const float *G, float *m1, float *m2, int64_t n, const AdamWScalars &s,
              cudaStream_t st);
// dst (cols x rows) = src (rows x cols)^T, rounded to TF32 (nearest) when
// `round`; up to 16 of them in one launch
struct TransposeJob {
    const float *src;
    float *dst;
    int rows, cols;
    bool round;
};
int transpose_many(int count, const TransposeJob *jobs, cudaStream_t st);
// out (rows x cols) = X diag(d): column j of X scaled by d[j]
int scale_cols_run(const float *X, const float *d, int64_t rows, int cols, float *out, cudaStream_t st);

}  // namespace spco
