// GEMM interface of the library: C (M x N) = op(A) (M x K) . op(B) (K x N),
// fp32 in / fp32 out, row-major storage, with the epilogues the spectral step
// needs.  Two implementations sit behind it: tcgen05 tensor cores
// (kind::tf32, gemm_tc.cu) and fp32 FMA on the SIMT cores (gemm_simt.cu).
#pragma once

#include "common.cuh"

namespace spco {

enum EpiMode : int {
    EPI_STORE = 0,     // C[i,j] = acc
    EPI_SCALE = 1,     // C[i,j] = acc * row_scale[i] * col_scale[j]  (either may be null)
    EPI_ADAMW = 2,     // blend + AdamW on W, m1, m2 (the last product of the step)
};

// Operand of a GEMM: element (i, k) of op(A) sits at
//   ptr[i * ld + k]  when !trans   (row-major, K contiguous)
//   ptr[k * ld + i]  when  trans   (the stored matrix is the transpose)
struct Operand {
    const float *ptr;
    int64_t ld;
    bool trans;
};

struct Epilogue {
    int mode = EPI_STORE;
    float *C = nullptr;  // output (EPI_STORE / EPI_SCALE), row-major, ldc
    int64_t ldc = 0;
    const float *row_scale = nullptr;
    const float *col_scale = nullptr;
    bool round_tf32 = false;  // round the stored result to TF32 (it feeds another TF32 GEMM)
    // EPI_ADAMW: acc is G_filt[i,j]; every array below is m x n with leading dimension ld
    const float *G = nullptr;  // masked gradient
    float *W = nullptr, *m1 = nullptr, *m2 = nullptr;
    float *Gf_out = nullptr, *Gp_out = nullptr;  // optional debug outputs
    int64_t ld = 0;
    float alpha = 0.f, beta1 = 0.f, beta2 = 0.f, eps = 0.f;
    float decay = 1.f;         // 1 - lr * weight_decay
    float step_size = 0.f;     // lr / (1 - beta1^t)
    float inv_sqrt_bc2 = 1.f;  // 1 / sqrt(1 - beta2^t)
};

// element-wise epilogue shared by both implementations
__device__ __forceinline__ float round_to_tf32(float x) {
    // round to nearest (ties away from zero) at 10 mantissa bits
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void epilogue_apply(const Epilogue &e, int64_t i, int64_t j, float acc) {
    if (e.mode == EPI_ADAMW) {
        const int64_t o = i * e.ld + j;
        const float g = e.G[o];
        const float gp = e.alpha * g + (1.f - e.alpha) * acc;
        float w = e.W[o] * e.decay;
        const float m = e.beta1 * e.m1[o] + (1.f - e.beta1) * gp;
        const float v = e.beta2 * e.m2[o] + (1.f - e.beta2) * gp * gp;
        w -= e.step_size * m / (sqrtf(v) * e.inv_sqrt_bc2 + e.eps);
        e.W[o] = w;
        e.m1[o] = m;
        e.m2[o] = v;
        if (e.Gf_out) e.Gf_out[o] = acc;
        if (e.Gp_out) e.Gp_out[o] = gp;
        return;
    }
    float c = acc;
    if (e.mode == EPI_SCALE) {
        if (e.row_scale) c *= e.row_scale[i];
        if (e.col_scale) c *= e.col_scale[j];
    }
    if (e.round_tf32) c = round_to_tf32(c);
    e.C[i * e.ldc + j] = c;
}

// One product of a grouped launch: C = op(A) op(B) with its own epilogue.
struct GemmProblem {
    int64_t M, N, K;
    Operand A, B;
    Epilogue epi;
};

// tcgen05 TF32 path (C = A B^T, both K-contiguous, 16-byte rows): one product,
// or up to 8 independent products sharing one persistent launch.
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, Operand A, Operand B);
int gemm_tc(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
            cudaStream_t stream);
int gemm_tc_group(int count, const GemmProblem *probs, cudaStream_t stream);

// fp32-accurate product on the tensor cores (3xTF32 with K-concatenated split
// operands); needs gemm3_workspace_floats(M, N, K) floats of 16-byte aligned
// workspace.  Falls back to gemm_simt when the shape does not allow it.
size_t gemm3_workspace_floats(int64_t M, int64_t N, int64_t K);
int gemm_fp32x3(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
                float *ws, cudaStream_t st);

// fp32 SIMT GEMM (any shape, any transposition, any alignment)
int gemm_simt(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
              cudaStream_t stream);

}  // namespace spco
