// Rotation kernel of the block-Jacobi eigen-solver on the tcgen05 tensor cores.
//
// Task = (matrix, 128-row slab, pair p):
//   X (128 x 64)  = IN[slab rows, cols(p)]        two TMA boxes of 32 columns
//   R_p^T hi / lo (64 x 64 each)                  four TMA boxes
//   X is split into hi = rna_tf32(x), kept in place in the swizzled shared
//   tile, and lo = rna_tf32(x - hi), written to TMEM (lane = row of the slab);
//   then one thread issues 24 tcgen05.mma (M = 128, N = 64, K = 8) into a
//   64-column TMEM accumulator:  D = Xhi.Rhi + Xhi.Rlo + Xlo.Rhi  (3xTF32,
//   fp32-accurate, the lo.lo term is below fp32 rounding), the last 8 with
//   their A operand read from TMEM.  D is staged in shared memory in the box
//   layout of the output (as is, or transposed) and stored with TMA.
// Keeping X lo out of shared memory leaves room for three stages of 64 KB.
// One persistent CTA per SM takes a contiguous range of tasks, with warp roles:
//   warp 0      TMA producer into a three-stage ring (X, R hi, R lo per stage)
//   warp 1      TMEM (two 64-column accumulators, X lo of each stage) and the
//               MMA issuer
//   warps 2-5   split X of the next stage: one thread per row, lo to its TMEM lane
//   warps 6-9   epilogue: tcgen05.ld of their lane quarter, staging, TMA store
// so the loads of tasks i+1 and i+2, the split of task i+1, the MMAs of task i
// and the stores of task i-1 overlap.  Every mbarrier wait is bounded; a wait
// that gives up records a code in the library's device flag and the role stops.
#include <algorithm>
#include <cstring>

#include "gemm.cuh"
#include "jacobi.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int kCtRows = 128;                    // slab rows = MMA M
constexpr int kCtThreads = 320;
constexpr uint32_t kXAtom = kCtRows * 128;      // 32 columns x 128 rows of fp32: 16 KB
constexpr uint32_t kXBytes = 2 * kXAtom;        // the 64 columns of a pair
constexpr uint32_t kRAtom = kP * 128;           // 32 columns x 64 rows: 8 KB
constexpr uint32_t kRBytes = 2 * kRAtom;        // one part (hi or lo) of R_p^T
constexpr uint32_t kLoadBytes = kXBytes + 2 * kRBytes;   // X raw + R hi + R lo
constexpr uint32_t kStageBytes = kLoadBytes;             // X lo lives in TMEM
constexpr uint32_t kTmemCols = 512;                      // two accumulators + X lo of each stage
constexpr uint32_t kLoCol = 128;                         // X lo of stage s at columns kLoCol + 64 s
// stages, output staging (one 128 x 64 tile), barriers
constexpr size_t ct_smem(int stages) { return (size_t)stages * kStageBytes + kXBytes + 1024 /*align*/ + 128; }
constexpr int kStages = 3;
static_assert(ct_smem(kStages) <= 232448, "shared memory budget of one CTA");
static_assert(kLoCol + 64 * kStages <= kTmemCols, "TMEM columns");
constexpr uint32_t kCtIdesc = tf32_idesc(kCtRows, kP);

struct CtBatch {
    int count;
    int total;
    CtJob job[kCtMaxJobs];
    int task_off[kCtMaxJobs + 1];
};

// task t of the batch: matrix j, then pair-major with the slab fastest, so a
// CTA's contiguous range reuses one R_p (L2-hot) across consecutive tasks
struct CtTask {
    const CtJob *job;
    int slab, blk_a, blk_b, rrow;
};

__device__ __forceinline__ CtTask ct_task(const CtBatch &cb, int t) {
    int j = 0;
    while (j + 1 < cb.count && t >= cb.task_off[j + 1]) ++j;
    CtTask k;
    k.job = &cb.job[j];
    const int np = k.job->Np / kP, nb = k.job->Np / kB, ns = k.job->Np / kCtRows;
    const int local = t - cb.task_off[j];
    k.slab = local % ns;
    const int pair = local / ns;
    rr_pair(nb, k.job->round, pair, k.blk_a, k.blk_b);
    k.rrow = (k.job->slot * np + pair) * 2 * kP;
    return k;
}

// loads X of task k into `stage`, and R_p^T hi / lo unless the stage already
// holds them (same rotation tensor and row)
__device__ __forceinline__ void ct_load(const CtTask &k, unsigned char *stage, uint64_t *bar, bool with_r) {
    unsigned char *x = stage, *rh = stage + kXBytes, *rl = rh + kRBytes;
    mbar_arrive_expect_tx(bar, with_r ? kLoadBytes : kXBytes);
    tma_load_2d(x, k.job->in, k.blk_a * kB, k.slab * kCtRows, bar);
    tma_load_2d(x + kXAtom, k.job->in, k.blk_b * kB, k.slab * kCtRows, bar);
    if (!with_r) return;
    tma_load_2d(rh, k.job->rot, 0, k.rrow, bar);
    tma_load_2d(rh + kRAtom, k.job->rot, kB, k.rrow, bar);
    tma_load_2d(rl, k.job->rot, 0, k.rrow + kP, bar);
    tma_load_2d(rl + kRAtom, k.job->rot, kB, k.rrow + kP, bar);
}

__device__ __forceinline__ float4 split_hi(float4 v, float4 &lo) {
    float4 h;
    h.x = tf32_split(v.x, lo.x);
    h.y = tf32_split(v.y, lo.y);
    h.z = tf32_split(v.z, lo.z);
    h.w = tf32_split(v.w, lo.w);
    return h;
}

// 64 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const float (&v)[64]) {
    uint32_t u[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) u[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
        "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, "
        "%33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, "
        "%49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};"
        :
        : "r"(taddr),
          "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
          "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]),
          "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]),
          "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31]),
          "r"(u[32]), "r"(u[33]), "r"(u[34]), "r"(u[35]), "r"(u[36]), "r"(u[37]), "r"(u[38]), "r"(u[39]),
          "r"(u[40]), "r"(u[41]), "r"(u[42]), "r"(u[43]), "r"(u[44]), "r"(u[45]), "r"(u[46]), "r"(u[47]),
          "r"(u[48]), "r"(u[49]), "r"(u[50]), "r"(u[51]), "r"(u[52]), "r"(u[53]), "r"(u[54]), "r"(u[55]),
          "r"(u[56]), "r"(u[57]), "r"(u[58]), "r"(u[59]), "r"(u[60]), "r"(u[61]), "r"(u[62]), "r"(u[63])
        : "memory");
}

// D (TMEM) += A . B^T with A (128 x 8 tf32) in TMEM (lane = row, column = k)
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <int STAGES>
__global__ void __launch_bounds__(kCtThreads, 1)
jacobi_rotate_kernel(const __grid_constant__ CtBatch cb, unsigned *flag) {
    extern __shared__ __align__(1024) unsigned char ct_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ct_smem_raw) + 1023) & ~uintptr_t(1023));
    // barriers after the output staging tile (which starts at STAGES * kStageBytes)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * kStageBytes + kXBytes);
    uint64_t *full = bars;                 // [STAGES] TMA landed
    uint64_t *split = full + STAGES;      // [STAGES] X split (128 arrivals)
    uint64_t *empty = split + STAGES;     // [STAGES] MMAs done with the stage
    uint64_t *tfull = empty + STAGES;     // [2] accumulator ready
    uint64_t *tempty = tfull + 2;          // [2] accumulator read (128 arrivals)
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tempty + 2);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // this CTA's contiguous task range
    const int per = cb.total / (int)gridDim.x, extra = cb.total % (int)gridDim.x;
    const int t0 = (int)blockIdx.x * per + min((int)blockIdx.x, extra);
    const int n = per + ((int)blockIdx.x < extra ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&split[s], 128);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int i = 0;
            const CUtensorMap *held_map[STAGES];
            int held_row[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) {
                held_map[s] = nullptr;
                held_row[s] = -1;
            }
            for (; i < n; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait_bounded(&empty[s], ((uint32_t)(i / STAGES) & 1u) ^ 1u, flag, 0x201u)) break;
                const CtTask k = ct_task(cb, t0 + i);
                const bool with_r = held_map[s] != k.job->rot || held_row[s] != k.rrow;
                held_map[s] = k.job->rot;
                held_row[s] = k.rrow;
                ct_load(k, smem + s * kStageBytes, &full[s], with_r);
            }
            if (i < n)  // gave up: let the loads already issued land before the CTA exits
                for (int q = (i > STAGES ? i - STAGES : 0); q < i; ++q)
                    mbar_wait_bounded(&full[q % STAGES], (uint32_t)(q / STAGES) & 1u, flag, 0x205u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int i = 0;
            for (; i < n; ++i) {
                const int s = i % STAGES, a = i & 1;
                if (!mbar_wait_bounded(&split[s], (uint32_t)(i / STAGES) & 1u, flag, 0x202u)) break;
                if (!mbar_wait_bounded(&tempty[a], ((uint32_t)(i >> 1) & 1u) ^ 1u, flag, 0x203u)) break;
                tc_fence_after();
                unsigned char *st = smem + s * kStageBytes;
                const uint32_t a_hi = smem_u32(st), b_hi = a_hi + kXBytes, b_lo = b_hi + kRBytes;
                const uint32_t a_lo = tmem + kLoCol + 64u * (uint32_t)s;
                const uint32_t bs[2] = {b_hi, b_lo};
                const uint32_t d = tmem + (uint32_t)(a * kP);
                uint32_t acc = 0;
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            mma_tf32(d, smem_desc_sw128(a_hi + kk * kXAtom + q * 32),
                                     smem_desc_sw128(bs[u] + kk * kRAtom + q * 32), kCtIdesc, acc);
                            acc = 1;
                        }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        mma_tf32_ta(d, a_lo + (uint32_t)(8 * (4 * kk + q)),
                                    smem_desc_sw128(b_hi + kk * kRAtom + q * 32), kCtIdesc, 1u);
                mma_commit(&empty[s]);  // stage free once these MMAs have read it
                mma_commit(&tfull[a]);  // accumulator ready once they completed
            }
            if (i < n && i > 0)  // gave up: the last MMAs issued finish before TMEM is freed
                mbar_wait_bounded(&tfull[(i - 1) & 1], (uint32_t)((i - 1) >> 1) & 1u, flag, 0x206u);
        }
    } else if (warp < 6) {
        // ---------------- split X into hi (in place) and lo
        // thread = row r of the slab = TMEM lane r (this warp's lane quarter)
        const int q = warp & 3, r = 32 * q + lane;
        for (int i = 0; i < n; ++i) {
            const int s = i % STAGES;
            if (!mbar_wait_bounded(&full[s], (uint32_t)(i / STAGES) & 1u, flag, 0x204u)) break;
            unsigned char *st = smem + s * kStageBytes;
            float lo[64];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    // 16-byte chunk c of row r of atom kk sits at chunk c ^ (r % 8) (128-byte swizzle)
                    float4 *p = reinterpret_cast<float4 *>(st + kk * kXAtom + r * 128 + ((c ^ (r & 7)) << 4));
                    float4 l;
                    *p = split_hi(*p, l);
                    lo[32 * kk + 4 * c] = l.x;
                    lo[32 * kk + 4 * c + 1] = l.y;
                    lo[32 * kk + 4 * c + 2] = l.z;
                    lo[32 * kk + 4 * c + 3] = l.w;
                }
            tmem_st64(tmem + ((uint32_t)(32 * q) << 16) + kLoCol + 64u * (uint32_t)s, lo);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            fence_proxy_async_smem();  // the tensor core reads what these threads wrote
            tc_fence_before();
            mbar_arrive(&split[s]);
        }
    } else {
        // ---------------- epilogue: TMEM lane quarter q = rows 32q .. 32q+31 of the slab,
        // staged in the box layout of the output map, stored by TMA
        const int q = warp % 4;
        const bool leader = warp == 6 && lane == 0;
        unsigned char *out = smem + STAGES * kStageBytes;
        for (int i = 0; i < n; ++i) {
            const int a = i & 1;
            if (!mbar_wait_bounded(&tfull[a], (uint32_t)(i >> 1) & 1u, flag, 0x207u)) break;
            tc_fence_after();
            float v[2][32];
            const uint32_t taddr = tmem + (uint32_t)(a * kP) + ((uint32_t)(q * 32) << 16);
            tmem_ld32(taddr, v[0]);
            tmem_ld32(taddr + 32, v[1]);
            tc_fence_before();
            mbar_arrive(&tempty[a]);
            const CtTask k = ct_task(cb, t0 + i);
            // the previous task's TMA store has finished reading the staging tile
            if (leader) bulk_wait_read<0>();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int r = q * 32 + lane;  // row within the slab
            if (!k.job->transposed) {
                // atom kk (32 columns), row r, 16-byte chunk c at c ^ (r % 8)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4 *>(out + kk * kXAtom + r * 128 + ((c ^ (r & 7)) << 4)) =
                            make_float4(v[kk][4 * c], v[kk][4 * c + 1], v[kk][4 * c + 2], v[kk][4 * c + 3]);
            } else {
                // output row jj (pair index), output column r: 32 x 32 boxes, box (q, jj / 32)
                // at q * 8 KB + (jj / 32) * 4 KB
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int jj = kk * 32 + c;
                        *reinterpret_cast<float *>(out + q * (kP * 128) + jj * 128 +
                                                   (((lane >> 2) ^ (jj & 7)) << 4) + (lane & 3) * 4) = v[kk][c];
                    }
            }
            fence_proxy_async_smem();  // the TMA engine reads what these threads wrote
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (leader) {
                const int row0 = k.slab * kCtRows;
                if (!k.job->transposed) {
                    tma_store_2d(k.job->out, out, k.blk_a * kB, row0);
                    tma_store_2d(k.job->out, out + kXAtom, k.blk_b * kB, row0);
                } else {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        tma_store_2d(k.job->out, out + w * (kP * 128), row0 + w * 32, k.blk_a * kB);
                        tma_store_2d(k.job->out, out + w * (kP * 128) + 32 * 128, row0 + w * 32, k.blk_b * kB);
                    }
                }
                bulk_commit();
            }
        }
        if (leader) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int jacobi_rotate(const CtJob *jobs, int count, cudaStream_t st, int max_ctas) {
    if (count < 1 || count > kCtMaxJobs) return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_rotate: 1 to 32 matrices");
    CtBatch cb;
    std::memset(&cb, 0, sizeof(cb));
    for (int i = 0; i < count; ++i) {
        if (jobs[i].Np % kNpAlign != 0 || jobs[i].Np < kNpAlign)
            return fail(SPECOPTIM_ERR_INVALID_ARG, "jacobi_rotate: Np must be a positive multiple of 128");
        if (!jobs[i].active) continue;  // converged matrices drop out of the task list
        cb.job[cb.count] = jobs[i];
        cb.task_off[cb.count + 1] = cb.task_off[cb.count] + (jobs[i].Np / kCtRows) * (jobs[i].Np / kP);
        ++cb.count;
    }
    if (cb.count == 0) return SPECOPTIM_OK;
    cb.total = cb.task_off[cb.count];
    if (int rc = set_smem_limit(reinterpret_cast<const void *>(&jacobi_rotate_kernel<kStages>), ct_smem(kStages)))
        return rc;
    // one CTA per SM (or per SM of the share given) with at least two tasks each
    int grid = std::max(1, std::min(max_ctas > 0 ? max_ctas : num_sms(), cb.total / 2));
    SPCO_LAUNCH("svd_jacobi_rotate", st,
                jacobi_rotate_kernel<kStages><<<grid, kCtThreads, ct_smem(kStages), st>>>(cb, device_flag_ptr()));
    SPECOPTIM_LAUNCHED("jacobi_rotate_kernel");
    return SPECOPTIM_OK;
}

}  // namespace spco
