// HBM-bound element-wise kernels: the anchor EMA (key design 2 of
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes") and
// plain AdamW for tensors outside the spectral correction.  128-bit loads and
// stores, grid sized to a multiple of the SM count, scalar tail.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "elementwise.cuh"

namespace spco {
namespace {

int stream_grid(int64_t vec_items) {
    int64_t g = (vec_items + 255) / 256;
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)num_sms() * 8));
}

// M <- beta M + (1 - beta) G
__global__ void __launch_bounds__(256)
ema_kernel(float *__restrict__ M, const float *__restrict__ G, int64_t n, float beta) {
    const float one_minus = 1.f - beta;
    const int64_t nv = n / 4;
    float4 *M4 = reinterpret_cast<float4 *>(M);
    const float4 *G4 = reinterpret_cast<const float4 *>(G);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += stride) {
        float4 m = M4[i];
        const float4 g = __ldcs(&G4[i]);
        m.x = beta * m.x + one_minus * g.x;
        m.y = beta * m.y + one_minus * g.y;
        m.z = beta * m.z + one_minus * g.z;
        m.w = beta * m.w + one_minus * g.w;
        M4[i] = m;
    }
    for (int64_t i = nv * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride)
        M[i] = beta * M[i] + one_minus * G[i];
}

__device__ __forceinline__ void adamw_one(float &w, float g, float &m, float &v, const AdamWScalars &s) {
    w *= s.decay;
    m = s.beta1 * m + (1.f - s.beta1) * g;
    v = s.beta2 * v + (1.f - s.beta2) * g * g;
    w -= s.step_size * m / (sqrtf(v) * s.inv_sqrt_bc2 + s.eps);
}

__global__ void __launch_bounds__(256)
adamw_kernel(float *__restrict__ W, const float *__restrict__ G, float *__restrict__ M1,
             float *__restrict__ M2, int64_t n, AdamWScalars s) {
    const int64_t nv = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += stride) {
        float4 w = reinterpret_cast<float4 *>(W)[i];
        const float4 g = __ldcs(reinterpret_cast<const float4 *>(G) + i);
        float4 m = reinterpret_cast<float4 *>(M1)[i];
        float4 v = reinterpret_cast<float4 *>(M2)[i];
        adamw_one(w.x, g.x, m.x, v.x, s);
        adamw_one(w.y, g.y, m.y, v.y, s);
        adamw_one(w.z, g.z, m.z, v.z, s);
        adamw_one(w.w, g.w, m.w, v.w, s);
        reinterpret_cast<float4 *>(W)[i] = w;
        reinterpret_cast<float4 *>(M1)[i] = m;
        reinterpret_cast<float4 *>(M2)[i] = v;
    }
    for (int64_t i = nv * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride)
        adamw_one(W[i], G[i], M1[i], M2[i], s);
}

// dst (cols x rows) = src (rows x cols)^T, optionally rounded to TF32 (round to
// nearest, ties away).  64 x 64 tiles through a padded shared tile; when both
// dimensions are multiples of 4 each thread moves four float4 in and four
// float4 out (16 values in flight per thread), else the scalar path runs.
__device__ __forceinline__ float maybe_round(float v, int round) {
    if (round) {
        uint32_t b;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(b) : "f"(v));
        v = __uint_as_float(b);
    }
    return v;
}

// Up to kMaxTranspose transposes in one launch (the step's G^T of every tall
// matrix): tiles numbered job by job.
constexpr int kMaxTranspose = 16;
struct TransposeBatch {
    int count;
    const float *src[kMaxTranspose];
    float *dst[kMaxTranspose];
    int rows[kMaxTranspose], cols[kMaxTranspose], round[kMaxTranspose];
    int64_t tile_off[kMaxTranspose + 1];
};

__global__ void __launch_bounds__(256)
transpose_kernel(const TransposeBatch tb) {
    __shared__ float tile[64][65];
    const int tid = threadIdx.x;
    const int64_t tiles = tb.tile_off[tb.count];
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        int j = 0;
        while (j + 1 < tb.count && t >= tb.tile_off[j + 1]) ++j;
        const float *__restrict__ src = tb.src[j];
        float *__restrict__ dst = tb.dst[j];
        const int rows = tb.rows[j], cols = tb.cols[j], round = tb.round[j];
        const int64_t tiles_c = (cols + 63) / 64, local = t - tb.tile_off[j];
        const bool vec = ((rows | cols) & 3) == 0;
        const int r0 = (int)(local / tiles_c) * 64, c0 = (int)(local % tiles_c) * 64;
        __syncthreads();
        if (vec) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // 16 threads per row, 16 rows per pass
                const int r = r0 + u * 16 + tid / 16, c = c0 + (tid % 16) * 4;
                v[u] = (r < rows && c < cols) ? __ldcs(reinterpret_cast<const float4 *>(&src[(int64_t)r * cols + c]))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = u * 16 + tid / 16, cc = (tid % 16) * 4;
                tile[rr][cc] = maybe_round(v[u].x, round);
                tile[rr][cc + 1] = maybe_round(v[u].y, round);
                tile[rr][cc + 2] = maybe_round(v[u].z, round);
                tile[rr][cc + 3] = maybe_round(v[u].w, round);
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // output row = input column
                const int cc = u * 16 + tid / 16, rr = (tid % 16) * 4;
                const int c = c0 + cc, r = r0 + rr;
                if (c < cols && r < rows)
                    *reinterpret_cast<float4 *>(&dst[(int64_t)c * rows + r]) =
                        make_float4(tile[rr][cc], tile[rr + 1][cc], tile[rr + 2][cc], tile[rr + 3][cc]);
            }
        } else {
            for (int e = tid; e < 64 * 64; e += 256) {
                const int rr = e / 64, cc = e % 64, r = r0 + rr, c = c0 + cc;
                tile[rr][cc] = (r < rows && c < cols) ? maybe_round(src[(int64_t)r * cols + c], round) : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < 64 * 64; e += 256) {
                const int cc = e / 64, rr = e % 64, r = r0 + rr, c = c0 + cc;
                if (c < cols && r < rows) dst[(int64_t)c * rows + r] = tile[rr][cc];
            }
        }
    }
}

}  // namespace

int transpose_many(int count, const TransposeJob *jobs, cudaStream_t st) {
    if (count < 1 || count > kMaxTranspose) return fail(SPECOPTIM_ERR_INVALID_ARG, "transpose: 1 to 16 jobs");
    TransposeBatch tb;
    std::memset(&tb, 0, sizeof(tb));
    for (int i = 0; i < count; ++i) {
        const TransposeJob &q = jobs[i];
        const int64_t tiles = (q.rows > 0 && q.cols > 0) ? (int64_t)((q.rows + 63) / 64) * ((q.cols + 63) / 64) : 0;
        tb.src[tb.count] = q.src;
        tb.dst[tb.count] = q.dst;
        tb.rows[tb.count] = q.rows;
        tb.cols[tb.count] = q.cols;
        tb.round[tb.count] = q.round ? 1 : 0;
        tb.tile_off[tb.count + 1] = tb.tile_off[tb.count] + tiles;
        if (tiles) ++tb.count;
    }
    if (tb.count == 0) return SPECOPTIM_OK;
    const int64_t tiles = tb.tile_off[tb.count];
    // 8 CTAs of 256 threads per SM (16.6 KB of shared memory each)
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms() * 8));
    SPCO_LAUNCH("transpose", st, transpose_kernel<<<grid, 256, 0, st>>>(tb));
    SPECOPTIM_LAUNCHED("transpose_kernel");
    return SPECOPTIM_OK;
}

int transpose_run(const float *src, float *dst, int rows, int cols, bool round, cudaStream_t st) {
    const TransposeJob j{src, dst, rows, cols, round};
    return transpose_many(1, &j, st);
}

AdamWScalars adamw_scalars(int64_t t, float lr, float beta1, float beta2, float eps, float wd) {
    AdamWScalars s;
    const double bc1 = 1.0 - std::pow((double)beta1, (double)t);
    const double bc2 = 1.0 - std::pow((double)beta2, (double)t);
    s.beta1 = beta1;
    s.beta2 = beta2;
    s.eps = eps;
    s.decay = (float)(1.0 - (double)lr * (double)wd);
    s.step_size = (float)((double)lr / bc1);
    s.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    return s;
}

int ema_run(float *M, const float *G, int64_t n, float beta, cudaStream_t st) {
    if (n <= 0) return SPECOPTIM_OK;
    SPCO_LAUNCH("anchor_ema", st, ema_kernel<<<stream_grid(n / 4 + 1), 256, 0, st>>>(M, G, n, beta));
    SPECOPTIM_LAUNCHED("ema_kernel");
    return SPECOPTIM_OK;
}

int adamw_run(float *W, const float *G, float *m1, float *m2, int64_t n, const AdamWScalars &s,
              cudaStream_t st) {
    if (n <= 0) return SPECOPTIM_OK;
    SPCO_LAUNCH("adamw", st, adamw_kernel<<<stream_grid(n / 4 + 1), 256, 0, st>>>(W, G, m1, m2, n, s));
    SPECOPTIM_LAUNCHED("adamw_kernel");
    return SPECOPTIM_OK;
}

namespace {
__global__ void __launch_bounds__(256)
scale_cols_kernel(const float *__restrict__ X, const float *__restrict__ d, int64_t total, int cols,
                  float *__restrict__ out) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x)
        out[e] = X[e] * d[e % cols];
}
}  // namespace

int scale_cols_run(const float *X, const float *d, int64_t rows, int cols, float *out, cudaStream_t st) {
    const int64_t total = rows * cols;
    if (total == 0) return SPECOPTIM_OK;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 8 * 152);
    SPCO_LAUNCH("scale_cols", st, scale_cols_kernel<<<blocks, 256, 0, st>>>(X, d, total, cols, out));
    SPECOPTIM_LAUNCHED("scale_cols_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
