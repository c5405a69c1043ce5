// Two-sided rotation of the Gram matrix in one pass, on the tcgen05 tensor cores:
// A <- R^T A R for one Jacobi round, written in place.
//
// A is symmetric, so only its upper "super-tiles" are read.  Pairs 2s and 2s+1
// of the round form super-pair s (four 32-index blocks, 128 indices); task
// (S1, S2), S1 <= S2, takes X = A[rows(S1), cols(S2)] (128 x 128) and, with
// p, p' the pairs of S1 and c, c' those of S2:
//   stage 1   Y_c = X[:, cols(c)] R_c                 (M 128, N 64, K 64; twice)
//   stage 2   [Y_c ; Y_c'](rows of p)^T R_p = Z^T       (M 128, N 64, K 64; twice)
// where Z = R_p^T X R_c... is the rotated super-tile; each product is 3xTF32
// (hi.hi + hi.lo + lo.hi, operands split in shared memory).  Stage 2 takes its
// A operand from the stage-1 accumulators (TMEM -> registers -> shared, hi and
// lo), its rows being the transposed columns of Y.  The result leaves through
// TMA twice: the TMEM rows are rows of the mirror super-tile (S2, S1), and a
// transposed copy gives (S1, S2); a diagonal super-tile (S1 = S2) needs only the
// first.  Every block pair of A is read and written by exactly one task, so
// the update is in place.
//
// One CTA (8 warps) per SM walks its super-tiles; the phases of a task run one
// after the other (split, MMAs, TMEM -> shared, MMAs, staging, stores) inside
// 192 KB of shared memory and 256 TMEM columns, with the loads in flight
// behind other work: the next task's X (both column pairs) while this one
// writes its result, the stage-2 rotations during the TMEM -> shared copy.  Every mbarrier wait is
// bounded; a wait that gives up records a code in the library's device flag and
// the CTA stops after letting its copies land.
#include <algorithm>
#include <cstring>

#include "gemm.cuh"
#include "jacobi.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int kApThreads = 256;
constexpr uint32_t kKB = 1024;
// Shared memory (192 KB) in three 64 KB regions, the same roles in every task:
//   P0 = [0, 64) KB     X_0 (32 KB, raw then hi) + R^T hi / lo of column pair 0
//   P1 = [64, 128) KB   X_1 + R^T of column pair 1
//   LO = [128, 192) KB  X_0 lo, X_1 lo
// After stage 1: A2_r hi + lo (64 KB per row pair r) in P0 and P1, the row
// pairs' R^T hi / lo in LO.  After stage 2: P0 and P1 take the next task's
// loads while LO stages the mirror super-tile for its TMA stores; the
// transposed copy goes to global memory straight from registers (each store
// of a warp is one 128-byte line).
constexpr uint32_t kLO = 128 * kKB;
constexpr size_t kApSmem = 192 * (size_t)kKB + 1024 /*align*/ + 128;
static_assert(kApSmem <= 232448, "shared memory budget of one CTA");
constexpr uint32_t kApTmemCols = 256;  // D1_0, D1_1, D2_0, D2_1 (64 columns each)
constexpr uint32_t kApIdesc = tf32_idesc(128, kP);

struct ApBatch {
    int count;
    int total;
    ApJob job[kApMaxJobs];
    int task_off[kApMaxJobs + 1];
};

struct ApTask {
    const ApJob *job;
    int rowblk[4];  // blocks of S1: a(2 S1), b(2 S1), a(2 S1 + 1), b(2 S1 + 1)
    int colblk[4];  // blocks of S2
    int rrow[2];    // rotation-tensor rows of pairs 2 S1, 2 S1 + 1 (hi; lo is 64 rows below)
    int crow[2];    // ... of pairs 2 S2, 2 S2 + 1
    bool diag;
};

__device__ __forceinline__ ApTask ap_task(const ApBatch &ab, int t) {
    int j = 0;
    while (j + 1 < ab.count && t >= ab.task_off[j + 1]) ++j;
    ApTask k;
    k.job = &ab.job[j];
    const int nb = k.job->Np / kB, ns = k.job->Np / 128;
    int local = t - ab.task_off[j];
    int s1 = 0;  // row-major over the upper triangle: row s1 has ns - s1 super-tiles
    while (local >= ns - s1) {
        local -= ns - s1;
        ++s1;
    }
    const int s2 = s1 + local;
    k.diag = s1 == s2;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        rr_pair(nb, k.job->round, 2 * s1 + u, k.rowblk[2 * u], k.rowblk[2 * u + 1]);
        rr_pair(nb, k.job->round, 2 * s2 + u, k.colblk[2 * u], k.colblk[2 * u + 1]);
        k.rrow[u] = (2 * s1 + u) * 2 * kP;
        k.crow[u] = (2 * s2 + u) * 2 * kP;
    }
    return k;
}

__device__ __forceinline__ void split4(float4 *h4, float4 *l4, int e) {
    const float4 v = h4[e];
    float4 h, l;
    h.x = tf32_split(v.x, l.x);
    h.y = tf32_split(v.y, l.y);
    h.z = tf32_split(v.z, l.z);
    h.w = tf32_split(v.w, l.w);
    h4[e] = h;
    l4[e] = l;
}

// 24 MMAs: D = Ahi.Bhi + Ahi.Blo + Alo.Bhi, A 128 x 64 (two 16 KB atoms),
// B 64 x 64 (two 8 KB atoms)
__device__ __forceinline__ void mma_3xtf32(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi,
                                           uint32_t b_lo) {
    const uint32_t as[3] = {a_hi, a_hi, a_lo}, bs[3] = {b_hi, b_lo, b_hi};
    uint32_t acc = 0;
#pragma unroll
    for (int u = 0; u < 3; ++u)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mma_tf32(d, smem_desc_sw128(as[u] + kk * 16 * kKB + q * 32),
                         smem_desc_sw128(bs[u] + kk * 8 * kKB + q * 32), kApIdesc, acc);
                acc = 1;
            }
}

// stage-1 loads of column pair c: X_c (four row blocks x two column blocks, 32 x 32
// boxes) to x, R_c^T hi / lo to r
__device__ __forceinline__ void load_stage1(const ApTask &k, int c, unsigned char *x, unsigned char *r,
                                            uint64_t *bar) {
    mbar_arrive_expect_tx(bar, 64 * kKB);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int rb = 0; rb < 4; ++rb)
            tma_load_2d(x + kk * 16 * kKB + rb * 4 * kKB, k.job->a32, k.colblk[2 * c + kk] * kB,
                        k.rowblk[rb] * kB, bar);
    tma_load_2d(r, k.job->rot, 0, k.crow[c], bar);
    tma_load_2d(r + 8 * kKB, k.job->rot, kB, k.crow[c], bar);
    tma_load_2d(r + 16 * kKB, k.job->rot, 0, k.crow[c] + kP, bar);
    tma_load_2d(r + 24 * kKB, k.job->rot, kB, k.crow[c] + kP, bar);
}

__global__ void __launch_bounds__(kApThreads, 1)
jacobi_apply_kernel(const __grid_constant__ ApBatch ab, unsigned *flag) {
    extern __shared__ __align__(1024) unsigned char ap_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ap_smem_raw) + 1023) & ~uintptr_t(1023));
    // [0] X_0, [1] X_1, [2] stage-2 rotations, [3] stage-1 MMAs, [4] stage-2 MMAs; each
    // completes once per task, so a task's waits use parity (task index & 1)
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 192 * kKB);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 5);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int q = warp & 3, h = warp >> 2;  // TMEM lane quarter, column half
    unsigned char *LO = smem + kLO;
    // thread 0: operations issued / seen complete per barrier (a clean stop after a timeout)
    int iss[5] = {0, 0, 0, 0, 0}, seen[5] = {0, 0, 0, 0, 0};
    auto load_x = [&](const ApTask &k) {  // both column pairs of a task into P0, P1
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            unsigned char *p = smem + c * 64 * kKB;
            load_stage1(k, c, p, p + 32 * kKB, &bar[c]);
            ++iss[c];
        }
    };
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
        if ((int)blockIdx.x < ab.total) load_x(ap_task(ab, blockIdx.x));
    }
    if (warp == 0) {
        tmem_alloc(tslot, kApTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tq = (uint32_t)(32 * q) << 16;  // this warp's TMEM lanes

    // all threads wait; thread 0 counts; the result is made uniform over the CTA
    auto wait_all = [&](int b, uint32_t par, unsigned code) -> bool {
        const bool w = mbar_wait_bounded(&bar[b], par, flag, code);
        if (w && tid == 0) ++seen[b];
        return __syncthreads_and(w) != 0;
    };

    bool ok = true;
    int it = 0;
    for (int t = blockIdx.x; t < ab.total && ok; t += gridDim.x, ++it) {
        const ApTask k = ap_task(ab, t);
        const uint32_t par = (uint32_t)it & 1u;
        if (tid == 0) bulk_wait_read<0>();  // the previous task's stores have read LO
        // ---- stage 1: Y_c = X_c R_c into TMEM columns 64 c
        for (int c = 0; c < 2; ++c) {
            unsigned char *x = smem + c * 64 * kKB, *xl = LO + c * 32 * kKB, *r = x + 32 * kKB;
            if (!(ok = wait_all(c, par, 0x301u + c))) break;
            float4 *h4 = reinterpret_cast<float4 *>(x), *l4 = reinterpret_cast<float4 *>(xl);
#pragma unroll 4
            for (int e = tid; e < (int)(32 * kKB / 16); e += kApThreads) split4(h4, l4, e);
            fence_proxy_async_smem();  // the tensor core reads what these threads wrote
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                mma_3xtf32(tmem + 64u * c, smem_u32(x), smem_u32(xl), smem_u32(r), smem_u32(r) + 16 * kKB);
                if (c == 1) {
                    mma_commit(&bar[3]);
                    ++iss[3];
                }
            }
        }
        if (!ok || !(ok = wait_all(3, par, 0x303u))) break;
        tc_fence_after();
        float v[2][32];
        tmem_ld32(tmem + 32u * h + tq, v[0]);       // Y_0[rho][32 h ..], rho = 32 q + lane
        tmem_ld32(tmem + 64u + 32u * h + tq, v[1]);  // Y_1[rho][32 h ..]
        // the stage-1 buffers are free: rotations of the row pairs for stage 2 into LO
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar[2], 64 * kKB);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                unsigned char *rr = LO + r * 32 * kKB;
                tma_load_2d(rr, k.job->rot, 0, k.rrow[r], &bar[2]);
                tma_load_2d(rr + 8 * kKB, k.job->rot, kB, k.rrow[r], &bar[2]);
                tma_load_2d(rr + 16 * kKB, k.job->rot, 0, k.rrow[r] + kP, &bar[2]);
                tma_load_2d(rr + 24 * kKB, k.job->rot, kB, k.rrow[r] + kP, &bar[2]);
            }
            ++iss[2];
        }
        // A2_r[c*64 + j][k] = Y_c[r*64 + k][j]: row rho = 32 q + lane is k = 32 (q & 1) + lane of
        // row pair r = q / 2, i.e. column `lane` of K-atom (q & 1); 128-byte swizzled rows
        {
            unsigned char *a2h = smem + (q >> 1) * 64 * kKB + (q & 1) * 16 * kKB, *a2l = a2h + 32 * kKB;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int row = c * 64 + 32 * h + jj;
                    const uint32_t off = row * 128 + ((((uint32_t)lane >> 2) ^ (row & 7)) << 4) + (lane & 3) * 4;
                    float lo;
                    *reinterpret_cast<float *>(a2h + off) = tf32_split(v[c][jj], lo);
                    *reinterpret_cast<float *>(a2l + off) = lo;
                }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (!(ok = wait_all(2, par, 0x304u))) break;
        // ---- stage 2: Z^T rows of row pair r into TMEM columns 128 + 64 r
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t a = smem_u32(smem + r * 64 * kKB), b = smem_u32(LO + r * 32 * kKB);
                mma_3xtf32(tmem + 128u + 64u * r, a, a + 32 * kKB, b, b + 16 * kKB);
            }
            mma_commit(&bar[4]);
            ++iss[4];
        }
        if (!(ok = wait_all(4, par, 0x305u))) break;
        tc_fence_after();
        // P0, P1 and LO are free: the next task's loads go out now
        if (tid == 0 && t + (int)gridDim.x < ab.total) load_x(ap_task(ab, t + gridDim.x));
        tmem_ld32(tmem + 128u + 32u * h + tq, v[0]);  // D2_0[L][32 h ..], L = 32 q + lane
        tmem_ld32(tmem + 192u + 32u * h + tq, v[1]);  // D2_1[L][32 h ..]
        tc_fence_before();
        // row L = c*64 + j of D2_r is row colidx(c, j) of the mirror super-tile and
        // column colidx(c, j) of the super-tile itself
        const int L = 32 * q + lane;
        const int gcol = k.colblk[q] * kB + lane;
        float *A = k.job->A;
        const int64_t ld = k.job->Np;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            unsigned char *mir = LO + r * 32 * kKB + h * 16 * kKB + L * 128;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *reinterpret_cast<float4 *>(mir + ((c4 ^ (L & 7)) << 4)) =
                    make_float4(v[r][4 * c4], v[r][4 * c4 + 1], v[r][4 * c4 + 2], v[r][4 * c4 + 3]);
            if (!k.diag) {
                float *dst = A + (int64_t)(k.rowblk[2 * r + h] * kB) * ld + gcol;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) dst[ii * ld] = v[r][ii];
            }
        }
        fence_proxy_async_smem();  // the TMA engine reads what these threads wrote
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int qb = 0; qb < 4; ++qb)
#pragma unroll
                    for (int kap = 0; kap < 2; ++kap)
                        tma_store_2d(k.job->a32, LO + r * 32 * kKB + kap * 16 * kKB + qb * 4 * kKB,
                                     k.rowblk[2 * r + kap] * kB, k.colblk[qb] * kB);
            bulk_commit();
        }
    }
    if (tid == 0) {
        if (!ok)  // let copies and MMAs still in flight land (bounded) before the CTA exits
            for (int b = 0; b < 5; ++b)
                for (int n = seen[b]; n < iss[b]; ++n) mbar_wait_bounded(&bar[b], (uint32_t)n & 1u, flag, 0x306u);
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kApTmemCols);
    }
}

}  // namespace

int jacobi_apply(const ApJob *jobs, int count, cudaStream_t st) {
    if (count < 1 || count > kApMaxJobs) return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_apply: 1 to 16 matrices");
    ApBatch ab;
    std::memset(&ab, 0, sizeof(ab));
    for (int i = 0; i < count; ++i) {
        if (jobs[i].Np % kNpAlign != 0 || jobs[i].Np < kNpAlign)
            return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_apply: Np must be a positive multiple of 128");
        if (!jobs[i].active) continue;  // converged matrices drop out of the task list
        const int ns = jobs[i].Np / 128;
        ab.job[ab.count] = jobs[i];
        ab.task_off[ab.count + 1] = ab.task_off[ab.count] + ns * (ns + 1) / 2;
        ++ab.count;
    }
    if (ab.count == 0) return SPECOPTIM_OK;
    ab.total = ab.task_off[ab.count];
    static bool attr = false;
    if (!attr) {
        SPECOPTIM_CUDA(cudaFuncSetAttribute(jacobi_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kApSmem));
        attr = true;
    }
    const int grid = std::min(num_sms(), ab.total);
    SPCO_LAUNCH("svd_jacobi_apply", st, jacobi_apply_kernel<<<grid, kApThreads, kApSmem, st>>>(ab, device_flag_ptr()));
    SPECOPTIM_LAUNCHED("jacobi_apply_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
