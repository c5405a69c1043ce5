// Rotation kernel of the block-Jacobi eigen-solver on the tcgen05 tensor cores.
//
// One CTA (4 warps) per task = (matrix, 128-row slab, pair p):
//   X (128 x 64)  = IN[slab rows, cols(p)]        two TMA boxes of 32 columns
//   R_p^T hi / lo (64 x 64 each)                  four TMA boxes
//   X is split in shared memory into hi = rna_tf32(x) and lo = rna_tf32(x - hi)
//   (element-wise, so the 128-byte swizzle of the TMA layout is kept), then one
//   thread issues 24 tcgen05.mma (M = 128, N = 64, K = 8) into a 64-column TMEM
//   accumulator:  D = Xhi.Rhi + Xhi.Rlo + Xlo.Rhi  (3xTF32, fp32-accurate, the
//   lo.lo term is below fp32 rounding).
//   The 4 warps read D back (tcgen05.ld, one row per thread), stage it in the
//   shared memory of X in the swizzled box layout (as is, or transposed), and
//   one thread stores it with TMA.
// Every mbarrier wait is bounded; a wait that gives up records a code in the
// library's device flag and the CTA skips the rest of its work (TMEM is freed).
#include <algorithm>
#include <cstring>

#include "gemm.cuh"
#include "jacobi.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int kCtRows = 128;                    // slab rows = MMA M
constexpr int kCtThreads = 128;
constexpr uint32_t kXAtom = kCtRows * 128;      // 32 columns x 128 rows of fp32: 16 KB
constexpr uint32_t kXBytes = 2 * kXAtom;        // the 64 columns of a pair
constexpr uint32_t kRAtom = kP * 128;           // 32 columns x 64 rows: 8 KB
constexpr uint32_t kRBytes = 2 * kRAtom;        // one part (hi or lo) of R_p^T
constexpr uint32_t kTmemCols = 64;
constexpr size_t kCtSmem = 2 * (size_t)kXBytes + 2 * (size_t)kRBytes + 1024 /*align*/ + 64;
constexpr uint32_t kCtIdesc = tf32_idesc(kCtRows, kP);

struct CtBatch {
    int count;
    CtJob job[kCtMaxJobs];
    int task_off[kCtMaxJobs + 1];
};

__device__ __forceinline__ float4 split_hi(float4 v, float4 &lo) {
    float4 h;
    h.x = round_to_tf32(v.x);
    h.y = round_to_tf32(v.y);
    h.z = round_to_tf32(v.z);
    h.w = round_to_tf32(v.w);
    lo.x = round_to_tf32(v.x - h.x);
    lo.y = round_to_tf32(v.y - h.y);
    lo.z = round_to_tf32(v.z - h.z);
    lo.w = round_to_tf32(v.w - h.w);
    return h;
}

__global__ void __launch_bounds__(kCtThreads)
jacobi_rotate_kernel(const __grid_constant__ CtBatch cb, unsigned *flag) {
    extern __shared__ __align__(1024) unsigned char ct_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ct_smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *xh = smem, *xl = smem + kXBytes;
    unsigned char *rh = smem + 2 * kXBytes, *rl = rh + kRBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(rl + kRBytes);  // [0] loads, [1] MMAs
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    int j = 0;
    while (j + 1 < cb.count && (int)blockIdx.x >= cb.task_off[j + 1]) ++j;
    const CtJob &job = cb.job[j];
    if (!job.active) return;  // whole CTA
    const int np = job.Np / kP, nb = job.Np / kB;
    const int local = (int)blockIdx.x - cb.task_off[j];
    const int slab = local / np, pair = local % np;
    int blk_a, blk_b;
    rr_pair(nb, job.round, pair, blk_a, blk_b);
    const int row0 = slab * kCtRows;

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], kXBytes + 2 * kRBytes);
        tma_load_2d(xh, job.in, blk_a * kB, row0, &bar[0]);
        tma_load_2d(xh + kXAtom, job.in, blk_b * kB, row0, &bar[0]);
        const int rrow = (job.slot * np + pair) * 2 * kP;
        tma_load_2d(rh, job.rot, 0, rrow, &bar[0]);
        tma_load_2d(rh + kRAtom, job.rot, kB, rrow, &bar[0]);
        tma_load_2d(rl, job.rot, 0, rrow + kP, &bar[0]);
        tma_load_2d(rl + kRAtom, job.rot, kB, rrow + kP, &bar[0]);
    }
    bool ok = mbar_wait_bounded(&bar[0], 0, flag, 0x201u);
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        float4 *h4 = reinterpret_cast<float4 *>(xh), *l4 = reinterpret_cast<float4 *>(xl);
#pragma unroll 4
        for (int e = tid; e < (int)(kXBytes / 16); e += kCtThreads) {
            float4 lo;
            h4[e] = split_hi(h4[e], lo);
            l4[e] = lo;
        }
    }
    fence_proxy_async_smem();  // the tensor core reads what these threads wrote
    __syncthreads();
    if (ok && tid == 0) {
        tc_fence_after();
        const uint32_t a_hi = smem_u32(xh), a_lo = smem_u32(xl), b_hi = smem_u32(rh), b_lo = smem_u32(rl);
        const uint32_t as[3] = {a_hi, a_hi, a_lo}, bs[3] = {b_hi, b_lo, b_hi};
        uint32_t acc = 0;
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    mma_tf32(tmem, smem_desc_sw128(as[t] + kk * kXAtom + s * 32),
                             smem_desc_sw128(bs[t] + kk * kRAtom + s * 32), kCtIdesc, acc);
                    acc = 1;
                }
        mma_commit(&bar[1]);
    }
    if (ok) ok = mbar_wait_bounded(&bar[1], 0, flag, 0x202u);
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    if (ok) {
        // this thread's accumulator row: slab row `r`, 64 columns
        const int r = warp * 32 + lane;
        float v[2][32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), v[0]);
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32, v[1]);
        // X's buffer is free (the MMAs completed): stage the result there
        if (!job.transposed) {
            // box layout of the load: atom kk, row r, 16-byte chunk c at c ^ (r % 8)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4 *>(xh + kk * kXAtom + r * 128 + ((c ^ (r & 7)) << 4)) =
                        make_float4(v[kk][4 * c], v[kk][4 * c + 1], v[kk][4 * c + 2], v[kk][4 * c + 3]);
        } else {
            // transposed: output row jj (0..63) = column jj of the pair, output
            // column r; 32-row boxes, box (warp, jj / 32) at warp * 8 KB + (jj / 32) * 4 KB
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int jj = kk * 32 + i;
                    *reinterpret_cast<float *>(xh + warp * (kP * 128) + jj * 128 +
                                               (((lane >> 2) ^ (jj & 7)) << 4) + (lane & 3) * 4) = v[kk][i];
                }
        }
    }
    fence_proxy_async_smem();  // the TMA engine reads what these threads wrote
    __syncthreads();
    if (ok && tid == 0) {
        if (!job.transposed) {
            tma_store_2d(job.out, xh, blk_a * kB, row0);
            tma_store_2d(job.out, xh + kXAtom, blk_b * kB, row0);
        } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                tma_store_2d(job.out, xh + w * (kP * 128), row0 + w * 32, blk_a * kB);
                tma_store_2d(job.out, xh + w * (kP * 128) + 32 * 128, row0 + w * 32, blk_b * kB);
            }
        }
        bulk_commit();
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int jacobi_rotate(const CtJob *jobs, int count, cudaStream_t st) {
    if (count < 1 || count > kCtMaxJobs) return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_rotate: 1 to 32 matrices");
    CtBatch cb;
    std::memset(&cb, 0, sizeof(cb));
    cb.count = count;
    for (int i = 0; i < count; ++i) {
        if (jobs[i].Np % kNpAlign != 0 || jobs[i].Np < kNpAlign)
            return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_rotate: Np must be a positive multiple of 128");
        cb.job[i] = jobs[i];
        cb.task_off[i + 1] = cb.task_off[i] + (jobs[i].Np / kCtRows) * (jobs[i].Np / kP);
    }
    static bool attr = false;
    if (!attr) {
        SPECOPTIM_CUDA(cudaFuncSetAttribute(jacobi_rotate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kCtSmem));
        attr = true;
    }
    SPCO_LAUNCH("svd_jacobi_rotate", st,
                jacobi_rotate_kernel<<<cb.task_off[count], kCtThreads, kCtSmem, st>>>(cb, device_flag_ptr()));
    SPECOPTIM_LAUNCHED("jacobi_rotate_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
