// fp32-accurate products on the TF32 tensor cores ("3xTF32").
//
// x = hi + lo with hi = round_tf32(x) and lo = round_tf32(x - hi) carries ~22
// mantissa bits; a.b ~= hi_a.hi_b + hi_a.lo_b + lo_a.hi_b (the lo.lo term is
// below fp32 rounding).  Each operand row is written once as the K-concatenated
// row [hi | lo | hi | hi] (4K floats); then op(A) = columns 0..3K of A's buffer
// ([hi lo hi]) and op(B) = columns K..4K of B's buffer ([lo hi hi]) give the
// three products in one TF32 GEMM with K' = 3K, fp32 accumulation in TMEM.
// Used by the SVD refresh (Gram matrix, warm start, Newton-Schulz, factor
// recovery), where fp32 accuracy matters and TF32 alone (2^-11) would not do.
#include <algorithm>

#include "gemm.cuh"

namespace spco {
namespace {

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// dst (rows x 4K, ld 4K): row i = [hi | lo | hi | hi] of row i of op(src) (rows x K),
// where op(src)(i, k) = src[i * ld + k] (trans = 0) or src[k * ld + i] (trans = 1).
// 32 x 32 tiles through shared memory, so both layouts read coalesced.
__global__ void __launch_bounds__(256)
split4_kernel(const float *__restrict__ src, int64_t ld, int trans, int rows, int K,
              float *__restrict__ dst) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    const int64_t tk = (K + 31) / 32, tiles = tk * ((rows + 31) / 32);
    const int64_t K4 = 4 * (int64_t)K;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int i0 = (int)(t / tk) * 32, k0 = (int)(t % tk) * 32;
        __syncthreads();
        for (int y = ty; y < 32; y += 8) {
            float v = 0.f;
            if (trans) {  // element (i0+tx, k0+y) sits at src[(k0+y) * ld + i0 + tx]
                if (k0 + y < K && i0 + tx < rows) v = src[(int64_t)(k0 + y) * ld + i0 + tx];
                tile[tx][y] = v;
            } else {      // element (i0+y, k0+tx) sits at src[(i0+y) * ld + k0 + tx]
                if (i0 + y < rows && k0 + tx < K) v = src[(int64_t)(i0 + y) * ld + k0 + tx];
                tile[y][tx] = v;
            }
        }
        __syncthreads();
        for (int y = ty; y < 32; y += 8) {
            const int i = i0 + y, k = k0 + tx;
            if (i >= rows || k >= K) continue;
            const float x = tile[y][tx];
            const float hi = tf32_rna(x), lo = tf32_rna(x - hi);
            float *row = dst + (int64_t)i * K4;
            row[k] = hi;
            row[K + k] = lo;
            row[2 * (int64_t)K + k] = hi;
            row[3 * (int64_t)K + k] = hi;
        }
    }
}

int split4(const Operand &op, int rows, int K, float *dst, cudaStream_t st) {
    const int64_t tiles = (int64_t)((K + 31) / 32) * ((rows + 31) / 32);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms() * 16));
    SPCO_LAUNCH("split_tf32x3", st, split4_kernel<<<grid, 256, 0, st>>>(op.ptr, op.ld, op.trans ? 1 : 0, rows, K, dst));
    SPECOPTIM_LAUNCHED("split4_kernel");
    return SPECOPTIM_OK;
}

}  // namespace

size_t gemm3_workspace_floats(int64_t M, int64_t N, int64_t K) {
    return (size_t)((M + N) * 4 * K + 64);
}

// C = op(A) (M x K) . op(B) (K x N) with fp32-level accuracy.  Operand
// conventions as in gemm_simt.  Falls back to the fp32 SIMT kernel when K is
// not a multiple of 4 (the split rows must stay 16-byte aligned for TMA).
int gemm_fp32x3(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
                float *ws, cudaStream_t st) {
    if (M <= 0 || N <= 0) return SPECOPTIM_OK;
    if ((K & 3) || K > (1 << 28) || !aligned16(ws)) return gemm_simt(M, N, K, A, B, epi, st);
    float *Asplit = ws;
    float *Bsplit = ws + (size_t)M * 4 * K;
    Bsplit = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(Bsplit) + 15) & ~uintptr_t(15));
    int rc;
    if ((rc = split4(A, (int)M, (int)K, Asplit, st))) return rc;
    // op(B)^T row j = column j of op(B): element (j, k) of op(B)^T is op(B)(k, j)
    Operand Bt{B.ptr, B.ld, !B.trans};
    if ((rc = split4(Bt, (int)N, (int)K, Bsplit, st))) return rc;
    Operand a{Asplit, 4 * K, false};      // [hi lo hi]
    Operand b{Bsplit + K, 4 * K, true};   // [lo hi hi] (B^T rows, K-contiguous)
    if (!gemm_tc_supported(M, N, 3 * K, a, b)) return gemm_simt(M, N, K, A, B, epi, st);
    return gemm_tc(M, N, 3 * K, a, b, epi, st);
}

}  // namespace spco
