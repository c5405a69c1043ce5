// SVD refresh of the anchor momentum, key design 3 of "Communication-Efficient
// LLM Adaptation over Decentralized GPU Meshes": M = U S V^T and the Tikhonov
// filter d_i = s_i / (s_i + tau_p).
//
// GPU formulation (fp32):
//   1. Gram matrix of the short side, A = M^T M (m >= n) or M M^T (m < n),
//      r x r, zero-padded to Np (a multiple of 32).
//   2. Block-Jacobi eigen-decomposition A = Q diag(lambda) Q^T.  The Np/16
//      blocks of 16 indices meet in round-robin order; in each round every
//      pair of blocks forms a 32 x 32 subproblem that one warp diagonalises in
//      shared memory (cyclic Jacobi, parallel order), giving a 32 x 32
//      rotation R_p per pair.  A second kernel applies all rotations at once:
//      every 32 x 32 tile (pair p1, pair p2) of A becomes R_p1^T A R_p2 and
//      every 32-row slab of Q becomes Q R_p.  Sweeps repeat until the
//      off-diagonal Frobenius norm falls below tol times the total norm.
//      Padded indices have exactly zero rows and columns, so they are never
//      rotated and stay out of the real eigenvectors.
//   3. The eigenvectors are re-orthonormalised by two Newton-Schulz steps.
//   4. P = M V (or M^T U); s_i = |P e_i| sorted descending, d_i = s_i/(s_i+tau_p),
//      and the long-side factor is P diag(1/s), zero columns where s_i = 0.
// The fp32 Gram squares the condition number; the filter makes that harmless
// (d_i ~ s_i/tau_p for the small directions, so the error of those directions
// enters G_filt multiplied by d_i).
#include <algorithm>
#include <vector>

#include "gemm.cuh"
#include "svd.cuh"

namespace spco {
namespace {

constexpr int kB = 16;      // block size of the block-Jacobi
constexpr int kP = 2 * kB;  // subproblem size (one warp)

// round-robin schedule over `players` (even): pair i of round k
__host__ __device__ __forceinline__ void rr_pair(int players, int round, int i, int &a, int &b) {
    const int n1 = players - 1;
    if (i == 0) {
        a = n1;
        b = round;
    } else {
        a = (round + i) % n1;
        b = (round - i + n1) % n1;
    }
}

// global index of local index l (0..31) of pair p in round `round` (nb blocks)
__device__ __forceinline__ int pair_index(int nb, int round, int p, int l) {
    int a, b;
    rr_pair(nb, round, p, a, b);
    return (l < kB ? a : b) * kB + (l & (kB - 1));
}

// Jacobi rotation (c, s) that zeroes the (p,q) entry of [[app, apq], [apq, aqq]]
__device__ __forceinline__ void jacobi_cs(float app, float aqq, float apq, float &c, float &s) {
    if (apq == 0.f) {
        c = 1.f;
        s = 0.f;
        return;
    }
    const float theta = (aqq - app) / (2.f * apq);
    float t;
    if (fabsf(theta) > 1e18f) {
        t = 0.5f / theta;
    } else {
        t = 1.f / (fabsf(theta) + sqrtf(1.f + theta * theta));
        if (theta < 0.f) t = -t;
    }
    c = rsqrtf(1.f + t * t);
    s = t * c;
}

constexpr int kWarpsPerBlock = 4;

// One warp per pair: load the 32x32 subproblem, run `inner_sweeps` cyclic
// Jacobi sweeps (parallel order, 16 disjoint rotations per step), write R.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
jacobi_solve_kernel(const float *__restrict__ A, int Np, int round, float *__restrict__ R,
                    int inner_sweeps) {
    __shared__ float S[kWarpsPerBlock][kP][kP + 1];
    __shared__ float Q[kWarpsPerBlock][kP][kP + 1];
    __shared__ float cs[kWarpsPerBlock][kB][2];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nb = Np / kB;
    const int pair = blockIdx.x * kWarpsPerBlock + warp;
    if (pair >= nb / 2) return;  // whole warp leaves together
    float(*s)[kP + 1] = S[warp];
    float(*q)[kP + 1] = Q[warp];
    const int gl = pair_index(nb, round, pair, lane);
    for (int i = 0; i < kP; ++i) {
        const int gi = pair_index(nb, round, pair, i);
        s[i][lane] = A[(size_t)gi * Np + gl];
        q[i][lane] = (i == lane) ? 1.f : 0.f;
    }
    __syncwarp();
    for (int sweep = 0; sweep < inner_sweeps; ++sweep) {
        float offmax = 0.f;
        for (int step = 0; step < kP - 1; ++step) {
            if (lane < kB) {
                int p, r;
                rr_pair(kP, step, lane, p, r);
                const float apq = s[p][r];
                float c, sn;
                jacobi_cs(s[p][p], s[r][r], apq, c, sn);
                cs[warp][lane][0] = c;
                cs[warp][lane][1] = sn;
                offmax = fmaxf(offmax, fabsf(apq));
            }
            __syncwarp();
            // rows: lane owns column `lane`
            for (int i = 0; i < kB; ++i) {
                int p, r;
                rr_pair(kP, step, i, p, r);
                const float c = cs[warp][i][0], sn = cs[warp][i][1];
                const float x = s[p][lane], y = s[r][lane];
                s[p][lane] = c * x - sn * y;
                s[r][lane] = sn * x + c * y;
            }
            __syncwarp();
            // columns of S and of Q: lane owns row `lane`
            for (int i = 0; i < kB; ++i) {
                int p, r;
                rr_pair(kP, step, i, p, r);
                const float c = cs[warp][i][0], sn = cs[warp][i][1];
                float x = s[lane][p], y = s[lane][r];
                s[lane][p] = c * x - sn * y;
                s[lane][r] = sn * x + c * y;
                x = q[lane][p];
                y = q[lane][r];
                q[lane][p] = c * x - sn * y;
                q[lane][r] = sn * x + c * y;
            }
            __syncwarp();
        }
        // stop early once no off-diagonal entry is above fp32 noise of the diagonal
        float dmax = fabsf(s[lane][lane]);
        for (int o = 16; o > 0; o >>= 1) {
            offmax = fmaxf(offmax, __shfl_xor_sync(0xffffffffu, offmax, o));
            dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
        }
        if (offmax <= 1e-7f * dmax) break;
    }
    float *Rp = R + (size_t)pair * kP * kP;
    for (int i = 0; i < kP; ++i) Rp[i * kP + lane] = q[i][lane];
}

// Applies the round's rotations: tiles of A (pair x pair) and 32-row slabs of Qacc.
__global__ void __launch_bounds__(256)
jacobi_apply_kernel(float *__restrict__ A, float *__restrict__ Qacc, int Np, int round,
                    const float *__restrict__ R) {
    __shared__ float X[kP][kP + 1];
    __shared__ float T[kP][kP + 1];
    __shared__ float R1[kP][kP + 1];
    __shared__ float R2[kP][kP + 1];
    const int nb = Np / kB, np = nb / 2;
    const int64_t atiles = (int64_t)np * np;
    const int tid = threadIdx.x;
    const int tx = tid % kP, ty = tid / kP;  // 32 x 8
    for (int64_t t = blockIdx.x; t < atiles + (int64_t)(Np / kP) * np; t += gridDim.x) {
        __syncthreads();
        if (t < atiles) {
            const int p1 = (int)(t / np), p2 = (int)(t % np);
            for (int i = ty; i < kP; i += 8) {
                const int gi = pair_index(nb, round, p1, i), gj = pair_index(nb, round, p2, tx);
                X[i][tx] = A[(size_t)gi * Np + gj];
                R1[i][tx] = R[(size_t)p1 * kP * kP + i * kP + tx];
                R2[i][tx] = R[(size_t)p2 * kP * kP + i * kP + tx];
            }
            __syncthreads();
            for (int i = ty; i < kP; i += 8) {  // T = R1^T X
                float acc = 0.f;
#pragma unroll 8
                for (int k = 0; k < kP; ++k) acc = fmaf(R1[k][i], X[k][tx], acc);
                T[i][tx] = acc;
            }
            __syncthreads();
            for (int i = ty; i < kP; i += 8) {  // A' = T R2
                float acc = 0.f;
#pragma unroll 8
                for (int k = 0; k < kP; ++k) acc = fmaf(T[i][k], R2[k][tx], acc);
                const int gi = pair_index(nb, round, p1, i), gj = pair_index(nb, round, p2, tx);
                A[(size_t)gi * Np + gj] = acc;
            }
        } else {
            const int64_t u = t - atiles;
            const int slab = (int)(u / np), p = (int)(u % np);
            for (int i = ty; i < kP; i += 8) {
                const int gj = pair_index(nb, round, p, tx);
                X[i][tx] = Qacc[(size_t)(slab * kP + i) * Np + gj];
                R2[i][tx] = R[(size_t)p * kP * kP + i * kP + tx];
            }
            __syncthreads();
            for (int i = ty; i < kP; i += 8) {
                float acc = 0.f;
#pragma unroll 8
                for (int k = 0; k < kP; ++k) acc = fmaf(X[i][k], R2[k][tx], acc);
                const int gj = pair_index(nb, round, p, tx);
                Qacc[(size_t)(slab * kP + i) * Np + gj] = acc;
            }
        }
    }
}

__global__ void eye_kernel(float *__restrict__ Q, int Np) {
    const int64_t total = (int64_t)Np * Np;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x)
        Q[e] = (e / Np == e % Np) ? 1.f : 0.f;
}

// sums of squares: out[0] = off-diagonal, out[1] = all (double atomics)
__global__ void offnorm_kernel(const float *__restrict__ A, int Np, double *out) {
    double off = 0.0, all = 0.0;
    const int64_t total = (int64_t)Np * Np;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const double v = A[e];
        all += v * v;
        if (e / Np != e % Np) off += v * v;
    }
    for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&out[0], off);
        atomicAdd(&out[1], all);
    }
}

// short-side factor before sorting: out[row][c] = Qacc[row][c], row, c < r
__global__ void extract_kernel(const float *__restrict__ Qacc, int Np, int r, float *__restrict__ out) {
    const int64_t total = (int64_t)r * r;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x)
        out[e] = Qacc[(e / r) * Np + e % r];
}

// Newton-Schulz orthogonalisation step: X <- 1.5 X - 0.5 T with T = X (X^T X)
__global__ void ns_update_kernel(float *__restrict__ X, const float *__restrict__ T, int64_t n) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x)
        X[e] = 1.5f * X[e] - 0.5f * T[e];
}

// column norms of P (rows x r, row-major): thread per column, coalesced across columns
__global__ void colnorm_kernel(const float *__restrict__ P, int64_t rows, int r, float *__restrict__ out) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < r; j += gridDim.x * blockDim.x) {
        double acc = 0.0;
        for (int64_t i = 0; i < rows; ++i) {
            const double v = P[i * r + j];
            acc += v * v;
        }
        out[j] = (float)sqrt(acc);
    }
}

// rank of each singular value (descending, ties by index) -> order[rank] = index
__global__ void rank_kernel(const float *__restrict__ sv, int r, int *__restrict__ order) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < r; i += gridDim.x * blockDim.x) {
        const float si = sv[i];
        int rank = 0;
        for (int j = 0; j < r; ++j) {
            const float sj = sv[j];
            rank += (sj > si) || (sj == si && j < i);
        }
        order[rank] = i;
    }
}

// sorted s, d = s / (s + tau), and 1/s
__global__ void spectrum_kernel(const float *__restrict__ sv, int r, const int *__restrict__ order,
                                float tau, float *__restrict__ s, float *__restrict__ d,
                                float *__restrict__ inv_s) {
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < r; c += gridDim.x * blockDim.x) {
        const float v = sv[order[c]];
        s[c] = v;
        d[c] = (v + tau) > 0.f ? v / (v + tau) : 0.f;
        inv_s[c] = v > 0.f ? 1.f / v : 0.f;
    }
}

// out[row][c] = in[row][order[c]] * (scale ? scale[c] : 1), rows x r row-major
__global__ void permute_cols_kernel(const float *__restrict__ in, int64_t rows, int r,
                                    const int *__restrict__ order, const float *__restrict__ scale,
                                    float *__restrict__ out) {
    const int64_t total = rows * r;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / r;
        const int c = (int)(e % r);
        const float v = in[row * r + order[c]];
        out[e] = scale ? v * scale[c] : v;
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)num_sms() * 8));
}

}  // namespace

size_t svd_workspace_floats(int m, int n) {
    const int r = m < n ? m : n, L = m < n ? n : m;
    const int64_t Np = ((r + kP - 1) / kP) * kP;
    const int64_t np = Np / kP;
    // A, Qacc, rotations, short factor + NS temp (2 r^2), long factor P (L r),
    // s_raw, inv_s, order (int), 2 doubles
    return (size_t)(2 * Np * Np + np * kP * kP + 2 * (int64_t)r * r + (int64_t)L * r + 3 * r + 8);
}

int svd_refresh_run(const SvdArgs &a, cudaStream_t st, int *sweeps_out) {
    const bool tall = a.m >= a.n;
    const int r = tall ? a.n : a.m;
    const int64_t L = tall ? a.m : a.n;  // long side
    const int Np = ((r + kP - 1) / kP) * kP;
    const int nb = Np / kB, np = nb / 2;
    float *A = a.work;
    float *Qacc = A + (size_t)Np * Np;
    float *R = Qacc + (size_t)Np * Np;
    float *Sf = R + (size_t)np * kP * kP;  // short-side factor, unsorted (r x r)
    float *Tmp = Sf + (size_t)r * r;       // r x r scratch
    float *P = Tmp + (size_t)r * r;        // long-side M V (or M^T U), unsorted (L x r)
    float *s_raw = P + (size_t)L * r;
    float *inv_s = s_raw + r;
    int *order = reinterpret_cast<int *>(inv_s + r);
    double *norms = reinterpret_cast<double *>(
        (reinterpret_cast<uintptr_t>(order + r) + 15) & ~uintptr_t(15));

    // 1. Gram matrix of the short side into the padded A
    SPECOPTIM_CUDA(cudaMemsetAsync(A, 0, sizeof(float) * (size_t)Np * Np, st));
    Epilogue e;
    e.C = A;
    e.ldc = Np;
    int rc;
    if (tall)  // A = M^T M : op(A)(i,k) = M[k][i], op(B)(k,j) = M[k][j]
        rc = gemm_simt(r, r, a.m, Operand{a.M, a.n, true}, Operand{a.M, a.n, false}, e, st);
    else       // A = M M^T
        rc = gemm_simt(r, r, a.n, Operand{a.M, a.n, false}, Operand{a.M, a.n, true}, e, st);
    if (rc) return rc;

    // 2. block Jacobi
    SPCO_LAUNCH("svd_eye", st, eye_kernel<<<grid_for((int64_t)Np * Np, 256), 256, 0, st>>>(Qacc, Np));
    SPECOPTIM_LAUNCHED("eye_kernel");
    const int solve_blocks = (np + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t apply_work = (int64_t)np * np + (int64_t)(Np / kP) * np;
    const int apply_grid = (int)std::min<int64_t>(apply_work, (int64_t)num_sms() * 8);
    int sweep = 0;
    bool converged = false;
    double host_norms[2] = {0.0, 0.0};
    for (sweep = 0; sweep < a.max_sweeps && !converged; ++sweep) {
        for (int round = 0; round < nb - 1; ++round) {
            SPCO_LAUNCH("svd_jacobi_solve", st, jacobi_solve_kernel<<<solve_blocks, 32 * kWarpsPerBlock, 0, st>>>(A, Np, round, R, 4));
            SPCO_LAUNCH("svd_jacobi_apply", st, jacobi_apply_kernel<<<apply_grid, 256, 0, st>>>(A, Qacc, Np, round, R));
        }
        SPECOPTIM_LAUNCHED("jacobi sweep");
        SPECOPTIM_CUDA(cudaMemsetAsync(norms, 0, 2 * sizeof(double), st));
        SPCO_LAUNCH("svd_offnorm", st, offnorm_kernel<<<grid_for((int64_t)Np * Np, 256), 256, 0, st>>>(A, Np, norms));
        SPECOPTIM_LAUNCHED("offnorm_kernel");
        SPECOPTIM_CUDA(cudaMemcpyAsync(host_norms, norms, 2 * sizeof(double),
                                       cudaMemcpyDeviceToHost, st));
        SPECOPTIM_CUDA(cudaStreamSynchronize(st));
        converged = host_norms[0] <= (double)a.tol * a.tol * host_norms[1];
    }
    if (sweeps_out) *sweeps_out = sweep;
    if (!converged)
        return fail(SPECOPTIM_ERR_NOT_CONVERGED,
                    "svd_refresh: Jacobi did not reach svd_tol within svd_max_sweeps; "
                    "previous factors kept");

    // 3. short-side factor, re-orthonormalised: two Newton-Schulz steps
    //    X <- X (3 I - X^T X) / 2 remove the drift that thousands of fp32
    //    rotations leave in the accumulated eigenvectors.
    const int64_t rr = (int64_t)r * r;
    SPCO_LAUNCH("svd_extract", st, extract_kernel<<<grid_for(rr, 256), 256, 0, st>>>(Qacc, Np, r, Sf));
    SPECOPTIM_LAUNCHED("extract_kernel");
    for (int it = 0; it < 2; ++it) {
        Epilogue g;
        g.C = A;  // X^T X (r x r, ld r) reuses the Gram buffer
        g.ldc = r;
        if ((rc = gemm_simt(r, r, r, Operand{Sf, r, true}, Operand{Sf, r, false}, g, st))) return rc;
        Epilogue t;
        t.C = Tmp;
        t.ldc = r;
        if ((rc = gemm_simt(r, r, r, Operand{Sf, r, false}, Operand{A, r, false}, t, st))) return rc;
        SPCO_LAUNCH("svd_ns_update", st, ns_update_kernel<<<grid_for(rr, 256), 256, 0, st>>>(Sf, Tmp, rr));
        SPECOPTIM_LAUNCHED("ns_update_kernel");
    }

    // 4. long side P = M X (tall) or M^T X (wide); s_i = |P e_i|, sorted descending;
    //    long factor = P diag(1/s), zero columns where s_i = 0
    Epilogue f;
    f.C = P;
    f.ldc = r;
    if (tall)
        rc = gemm_simt(L, r, a.n, Operand{a.M, a.n, false}, Operand{Sf, r, false}, f, st);
    else
        rc = gemm_simt(L, r, a.m, Operand{a.M, a.n, true}, Operand{Sf, r, false}, f, st);
    if (rc) return rc;
    SPCO_LAUNCH("svd_colnorm", st, colnorm_kernel<<<grid_for(r, 128), 128, 0, st>>>(P, L, r, s_raw));
    SPCO_LAUNCH("svd_rank", st, rank_kernel<<<grid_for(r, 128), 128, 0, st>>>(s_raw, r, order));
    SPCO_LAUNCH("svd_spectrum", st, spectrum_kernel<<<grid_for(r, 128), 128, 0, st>>>(s_raw, r, order, a.tau, a.s, a.d, inv_s));
    float *short_out = tall ? a.V : a.U;
    float *long_out = tall ? a.U : a.V;
    SPCO_LAUNCH("svd_permute", st, permute_cols_kernel<<<grid_for(rr, 256), 256, 0, st>>>(Sf, r, r, order, nullptr, short_out));
    SPCO_LAUNCH("svd_permute", st, permute_cols_kernel<<<grid_for(L * r, 256), 256, 0, st>>>(P, L, r, order, inv_s, long_out));
    SPECOPTIM_LAUNCHED("svd spectrum kernels");
    return SPECOPTIM_OK;
}

}  // namespace spco
