// fp32 GEMM on the SIMT cores: 128 x 128 output tile per 256-thread CTA,
// 8 x 8 outputs per thread, K staged through shared memory 16 deep with a
// register prefetch of the next slab.  Exact fp32 FMA arithmetic; used for the
// Gram matrix and the factor recovery of the SVD refresh and as the
// SPECOPTIM_PREC_FP32 path of the projection.
#include "gemm.cuh"

namespace spco {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, TM = 8, TN = 8, NT = 256;

__device__ __forceinline__ float load_op(const Operand &op, int64_t i, int64_t k, int64_t rows,
                                         int64_t K) {
    if (i >= rows || k >= K) return 0.f;
    return op.trans ? op.ptr[k * op.ld + i] : op.ptr[i * op.ld + k];
}

__global__ void __launch_bounds__(NT) gemm_simt_kernel(int64_t M, int64_t N, int64_t K, Operand A,
                                                       Operand B, Epilogue epi) {
    __shared__ float As[2][BK][BM + 4];
    __shared__ float Bs[2][BK][BN + 4];
    const int tid = threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int tr = tid / (BN / TN), tc = tid % (BN / TN);  // 16 x 16 thread grid

    // each thread stages 8 elements of the A slab and 8 of the B slab
    // A slab: BM x BK = 2048 elements.  Coalesce along the contiguous index.
    float ra[8], rb[8];
    auto fetch = [&](int64_t k0) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            int e = tid + q * NT;
            int ii, kk;
            if (A.trans) { ii = e % BM; kk = e / BM; } else { kk = e % BK; ii = e / BK; }
            ra[q] = load_op(A, m0 + ii, k0 + kk, M, K);
            int jj, kb;
            if (B.trans) { jj = e % BN; kb = e / BN; } else { kb = e % BK; jj = e / BK; }
            rb[q] = load_op(B, n0 + jj, k0 + kb, N, K);
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            int e = tid + q * NT;
            int ii, kk;
            if (A.trans) { ii = e % BM; kk = e / BM; } else { kk = e % BK; ii = e / BK; }
            As[buf][kk][ii] = ra[q];
            int jj, kb;
            if (B.trans) { jj = e % BN; kb = e / BN; } else { kb = e % BK; jj = e / BK; }
            Bs[buf][kb][jj] = rb[q];
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int a = 0; a < TM; ++a)
#pragma unroll
        for (int b = 0; b < TN; ++b) acc[a][b] = 0.f;

    fetch(0);
    stash(0);
    __syncthreads();
    int buf = 0;
    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        const bool more = k0 + BK < K;
        if (more) fetch(k0 + BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int x = 0; x < TM; ++x) a[x] = As[buf][kk][tr * TM + x];
#pragma unroll
            for (int y = 0; y < TN; ++y) b[y] = Bs[buf][kk][tc * TN + y];
#pragma unroll
            for (int x = 0; x < TM; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        if (more) {
            stash(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }
#pragma unroll
    for (int x = 0; x < TM; ++x) {
        int64_t i = m0 + tr * TM + x;
        if (i >= M) continue;
#pragma unroll
        for (int y = 0; y < TN; ++y) {
            int64_t j = n0 + tc * TN + y;
            if (j < N) epilogue_apply(epi, i, j, acc[x][y]);
        }
    }
}

}  // namespace

// B is passed as "op(B) (K x N)"; internally it is read as the (j, k) operand
// of B^T, so its transposition flag is flipped here.
int gemm_simt(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
              cudaStream_t stream) {
    if (M <= 0 || N <= 0) return SPECOPTIM_OK;
    Operand Bt = B;
    Bt.trans = !B.trans;
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    SPCO_LAUNCH("gemm_simt", stream, gemm_simt_kernel<<<grid, NT, 0, stream>>>(M, N, K, A, Bt, epi));
    SPECOPTIM_LAUNCHED("gemm_simt_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
