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
// One CTA per SM walks its super-tiles with warp roles, so that the epilogue of
// one super-tile overlaps the loads, split and stage-1 MMAs of the next:
//   warp 0      TMA producer (X of both column pairs, then the stage-2 rotations)
//   warp 1      TMEM (256 columns: D1 of both column pairs, D2 of both row pairs)
//               and the MMA issuer
//   warps 2-5   transform: split X into hi / lo; build A2 from D1 (first column pair)
//   warps 6-9   epilogue: build A2 (second column pair); D2 -> both orientations in
//               whole 128-byte lines
//               (the transposed copy straight from registers, the mirror
//               through a 32 x 33 shared tile per warp)
// Every mbarrier wait is bounded; a wait that gives up records a code in the
// library's device flag and that role stops (the producer and the MMA issuer
// first let their last copies and MMAs land).  The kernel is launched as a
// programmatic dependent of the round's solve when the solve fits in one wave
// beside the Q rotation: its set-up (barriers, TMEM) then runs on the SMs the
// solve's CTAs leave, before the solve has finished.
#include <algorithm>
#include <cstring>
#include <string>

#include "gemm.cuh"
#include "jacobi.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int kApThreads = 320;  // producer, MMA, 4 transform and 4 epilogue warps
constexpr uint32_t kKB = 1024;
// Shared memory (192 KB) in three 64 KB regions:
//   P0 = [0, 64) KB     X_0 (32 KB, raw then hi) + R^T hi / lo of column pair 0
//   P1 = [64, 128) KB   X_1 + R^T of column pair 1
//   LO = [128, 192) KB  X_0 lo, X_1 lo
// After the stage-1 MMAs: A2_r hi + lo (64 KB per row pair r) in P0 and P1, the
// row pairs' R^T hi / lo in LO.  After the stage-2 MMAs all three regions take
// the next super-tile.
constexpr uint32_t kLO = 128 * kKB;
constexpr size_t kApSmem = 192 * (size_t)kKB + 128 /*barriers*/ + 4 * 32 * 33 * 4 /*epilogue tiles*/ + 1024 /*align*/;
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
        k.rrow[u] = (k.job->slot * (k.job->Np / kP) + 2 * s1 + u) * 2 * kP;
        k.crow[u] = (k.job->slot * (k.job->Np / kP) + 2 * s2 + u) * 2 * kP;
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

// A2_r[c*64 + j][k] = Y_c[r*64 + k][j] for one column pair c: the thread of TMEM lane
// rho = 32 q + lane holds k = 32 (q & 1) + lane of row pair r = q / 2, i.e. column
// `lane` of K-atom (q & 1) in every row c*64 + j; 128-byte swizzled rows, hi and lo
__device__ __forceinline__ void build_a2(unsigned char *smem, uint32_t tmem, int q, int lane, int c) {
    const uint32_t tq = (uint32_t)(32 * q) << 16;
    unsigned char *a2h = smem + (q >> 1) * 64 * kKB + (q & 1) * 16 * kKB, *a2l = a2h + 32 * kKB;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32(tmem + 64u * c + 32u * hh + tq, v);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int row = c * 64 + 32 * hh + jj;
            const uint32_t off = row * 128 + ((((uint32_t)lane >> 2) ^ (row & 7)) << 4) + (lane & 3) * 4;
            float lo;
            *reinterpret_cast<float *>(a2h + off) = tf32_split(v[jj], lo);
            *reinterpret_cast<float *>(a2l + off) = lo;
        }
    }
}

__global__ void __launch_bounds__(kApThreads, 1)
jacobi_apply_kernel(const __grid_constant__ ApBatch ab, unsigned *flag) {
    extern __shared__ __align__(1024) unsigned char ap_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ap_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 192 * kKB);
    uint64_t *xfull = bar;        // [2] X_c and R_c^T landed (producer, tx bytes)
    uint64_t *xsplit = bar + 2;   // [2] X_c split into hi / lo (128 transform threads)
    uint64_t *s1done = bar + 4;   // stage-1 MMAs complete (commit)
    uint64_t *r2full = bar + 5;   // stage-2 rotations landed (producer, tx bytes)
    uint64_t *a2ready = bar + 6;  // A2 built, D1 read (128 transform + 128 epilogue threads)
    uint64_t *s2done = bar + 7;   // stage-2 MMAs complete (commit)
    uint64_t *d2free = bar + 8;   // D2 read by the epilogue (128 epilogue threads)
    uint64_t *s2half = bar + 9;   // stage-2 MMAs of row pair 0 complete (P0 and LO[0, 32) free)
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 10);
    float *etile = reinterpret_cast<float *>(smem + 192 * kKB + 128);  // 4 epilogue warps x 32 x 33
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned char *LO = smem + kLO;
    // this CTA's tasks: t = blockIdx.x + i * gridDim.x, i < n
    const int n = ab.total > (int)blockIdx.x ? (ab.total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&xfull[b], 1);
            mbar_init(&xsplit[b], 128);
        }
        mbar_init(s1done, 1);
        mbar_init(r2full, 1);
        mbar_init(a2ready, 256);
        mbar_init(s2done, 1);
        mbar_init(d2free, 128);
        mbar_init(s2half, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, kApTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // Launched as a programmatic dependent of the round's solve: the set-up above
    // overlaps the solve's last CTAs; A and the rotations are read only past here.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int i = 0, iss[2] = {0, 0}, r_iss = 0;
            for (; i < n; ++i) {
                const ApTask k = ap_task(ab, blockIdx.x + i * gridDim.x);
                const uint32_t par = (uint32_t)i & 1u;
                // P_c (and LO's half c) held the previous task's A2 (and R^T) of row pair c until
                // its stage-2 MMAs of that row pair completed
                bool ok = true;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!(ok = mbar_wait_bounded(c ? s2done : s2half, par ^ 1u, flag, 0x311u))) break;
                    unsigned char *p = smem + c * 64 * kKB;
                    load_stage1(k, c, p, p + 32 * kKB, &xfull[c]);
                    ++iss[c];
                }
                if (!ok) break;
                // LO holds this task's X lo until its stage-1 MMAs completed
                if (!mbar_wait_bounded(s1done, par, flag, 0x312u)) break;
                mbar_arrive_expect_tx(r2full, 64 * kKB);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    unsigned char *rr = LO + r * 32 * kKB;
                    tma_load_2d(rr, k.job->rot, 0, k.rrow[r], r2full);
                    tma_load_2d(rr + 8 * kKB, k.job->rot, kB, k.rrow[r], r2full);
                    tma_load_2d(rr + 16 * kKB, k.job->rot, 0, k.rrow[r] + kP, r2full);
                    tma_load_2d(rr + 24 * kKB, k.job->rot, kB, k.rrow[r] + kP, r2full);
                }
                ++r_iss;
            }
            if (i < n) {  // gave up: let the last loads issued land before the CTA exits
                for (int c = 0; c < 2; ++c)
                    if (iss[c] > 0) mbar_wait_bounded(&xfull[c], (uint32_t)(iss[c] - 1) & 1u, flag, 0x313u);
                if (r_iss > 0) mbar_wait_bounded(r2full, (uint32_t)(r_iss - 1) & 1u, flag, 0x313u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int i = 0;
            bool pending = false;
            uint64_t *last = nullptr;
            uint32_t last_par = 0;
            for (; i < n; ++i) {
                const uint32_t par = (uint32_t)i & 1u;
                bool ok = true;
                for (int c = 0; c < 2 && ok; ++c) {
                    if (!(ok = mbar_wait_bounded(&xsplit[c], par, flag, 0x321u))) break;
                    tc_fence_after();
                    const uint32_t x = smem_u32(smem + c * 64 * kKB), xl = smem_u32(LO + c * 32 * kKB);
                    mma_3xtf32(tmem + 64u * c, x, xl, x + 32 * kKB, x + 48 * kKB);
                }
                if (!ok) break;
                mma_commit(s1done);
                pending = true;
                last = s1done;
                last_par = par;
                if (!mbar_wait_bounded(a2ready, par, flag, 0x322u)) break;
                if (!mbar_wait_bounded(r2full, par, flag, 0x323u)) break;
                if (!mbar_wait_bounded(d2free, par ^ 1u, flag, 0x324u)) break;  // D2 of the previous task read
                tc_fence_after();
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t a = smem_u32(smem + r * 64 * kKB), b = smem_u32(LO + r * 32 * kKB);
                    mma_3xtf32(tmem + 128u + 64u * r, a, a + 32 * kKB, b, b + 16 * kKB);
                    mma_commit(r ? s2done : s2half);
                }
                last = s2done;
            }
            if (i < n && pending) mbar_wait_bounded(last, last_par, flag, 0x325u);
        }
    } else if (warp < 6) {
        // ---------------- transform: split X, then A2 from the stage-1 accumulators
        const int tid = threadIdx.x - 64, q = warp & 3;
        for (int i = 0; i < n; ++i) {
            const uint32_t par = (uint32_t)i & 1u;
            bool ok = true;
            for (int c = 0; c < 2; ++c) {
                if (!(ok = mbar_wait_bounded(&xfull[c], par, flag, 0x331u))) break;
                float4 *h4 = reinterpret_cast<float4 *>(smem + c * 64 * kKB);
                float4 *l4 = reinterpret_cast<float4 *>(LO + c * 32 * kKB);
#pragma unroll 4
                for (int e = tid; e < (int)(32 * kKB / 16); e += 128) split4(h4, l4, e);
                fence_proxy_async_smem();  // the tensor core reads what these threads wrote
                mbar_arrive(&xsplit[c]);
            }
            if (!ok || !mbar_wait_bounded(s1done, par, flag, 0x332u)) break;
            tc_fence_after();
            build_a2(smem, tmem, q, lane, 0);  // rows c = 0 of A2; the epilogue warps build c = 1
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(a2ready);
        }
    } else {
        // ---------------- epilogue: D2 rows -> both orientations in global memory
        const int q = warp & 3;
        const uint32_t tq = (uint32_t)(32 * q) << 16;
        for (int i = 0; i < n; ++i) {
            const ApTask k = ap_task(ab, blockIdx.x + i * gridDim.x);
            const uint32_t par = (uint32_t)i & 1u;
            if (!mbar_wait_bounded(s1done, par, flag, 0x342u)) break;
            tc_fence_after();
            build_a2(smem, tmem, q, lane, 1);  // rows c = 1 of A2
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(a2ready);
            if (!mbar_wait_bounded(s2done, par, flag, 0x341u)) break;
            tc_fence_after();
            float v[2][2][32];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) tmem_ld32(tmem + 128u + 64u * r + 32u * hh + tq, v[r][hh]);
            tc_fence_before();
            mbar_arrive(d2free);
            // row L = c*64 + j of D2_r is row colidx(c, j) of the mirror super-tile
            // and column colidx(c, j) of the super-tile; i = 32 hh + ii.  The
            // transposed copy is written column by column (each store of the warp
            // is one 128-byte line); the mirror goes through a 32 x 33 tile of
            // this warp so that it, too, leaves in whole lines.
            float *A = k.job->A;
            const int64_t ld = k.job->Np;
            const int gl = k.colblk[q] * kB + lane;  // colidx(L), L = 32 q + lane
            float *tile = etile + (warp - 6) * 32 * 33;
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int rb = k.rowblk[2 * r + hh] * kB;
                    if (!k.diag) {
                        float *dst = A + (int64_t)rb * ld + gl;
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) dst[ii * ld] = v[r][hh][ii];
                    }
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) tile[lane * 33 + ii] = v[r][hh][ii];
                    __syncwarp();
                    float *mir = A + (int64_t)(k.colblk[q] * kB) * ld + rb + lane;
#pragma unroll
                    for (int row = 0; row < 32; ++row) mir[row * ld] = tile[row * 33 + lane];
                    __syncwarp();
                }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kApTmemCols);
    }
}

}  // namespace

int jacobi_apply(const ApJob *jobs, int count, cudaStream_t st, bool after_solve) {
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
    if (int rc = set_smem_limit(reinterpret_cast<const void *>(&jacobi_apply_kernel), kApSmem)) return rc;
    const int grid = std::min(num_sms(), ab.total);
    // programmatic dependent launch (after_solve): the CTAs may start on SMs the
    // solve before it leaves, and wait (griddepcontrol.wait) for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kApThreads);
    cfg.dynamicSmemBytes = kApSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_solve ? 1 : 0;
    unsigned *flag = device_flag_ptr();
    cudaError_t err = cudaSuccess;
    SPCO_LAUNCH("svd_jacobi_apply", st, err = cudaLaunchKernelEx(&cfg, jacobi_apply_kernel, ab, flag));
    if (err != cudaSuccess) return fail(SPECOPTIM_ERR_CUDA, std::string("jacobi_apply: ") + cudaGetErrorString(err));
    SPECOPTIM_LAUNCHED("jacobi_apply_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
