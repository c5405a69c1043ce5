// Data-parallel outer synchronisation of one weight matrix (key design 4 of
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes": the
// Streaming DiLoCo outer step travels PowerSGD-compressed, 64x).
//
// The m x n streams are HBM-bound with O(k) fp32 work per element (k <= 64):
// persistent CTAs fed by 1D bulk copies (cp.async.bulk) into a ring of
// shared-memory stages, fp32 FMA on the SIMT cores in 8 x 8 (or 4 x 8)
// register tiles, and deterministic split reductions in a fixed order.  The
// k x k orthogonalisation never touches fp64 (slow on this part): products and
// sums are carried in two floats (hi + lo) and the triangular factors are
// applied in fp32.
//
//   dp_pad_q_kernel      Q (n x k) -> Qp (n x (kp+4)), zero padded, for bulk copies
//   dp_compress_p_kernel M = E + X - Y -> E;  P = M Q
//   dp_gram_kernel       Gram matrix of P (pass 0) or of P R1^-1 (pass 1) in two
//                        floats; the last CTA of a matrix factors it (Cholesky,
//                        two floats) and stores R with its reciprocal diagonal
//   dp_orth_apply_kernel P^ = (P R1^-1) R2^-1 by forward substitution
//   dp_compress_q_kernel partial Q = M^T P^ per row range
//   dp_q_reduce_kernel   Q = sum of the partials (range order)
//   dp_update_kernel     D = s P^ Q^T;  E <- M - D;  out = D, or the outer
//                        Nesterov step and the restart of W_local
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dpsync.h"
#include "tc.cuh"

struct dpsync {
    dpsync_config cfg;
    int m, n, k, kp;
    float *P, *Q;          // caller-owned m x k, n x k
    float *E;              // m x n: M between compress_p and decompress, then the error
    float *theta, *mom;    // m x n each, allocated by set_outer
    float *Ph;             // m x kp orthonormal basis (padded columns are zero)
    float *Qp;             // n x (kp + 4) padded copy of Q for compress_p
    float *T;              // 2 x kp x kp: R1, R2 (strict upper part) with reciprocal diagonals
    float *Gpart;          // gram tasks x blocks x 16 x 2 partial Gram matrices (hi, lo)
    float *Qpart;          // q row ranges x ncb*128 x kp partial Q
    int *counters;         // [0, 2): gram passes
    CUtensorMap *maps;     // device: X, Y, E (compress_p boxes), Qp, E (compress_q boxes), P^
    const float *map_x, *map_y;  // the X and Y the first two maps describe
    int gram_tasks, q_ranges, ncb;
    bool have_outer;
};

namespace spco {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxJobs = DPSYNC_MAX_BATCH;
constexpr int kPBC = 128;        // compress_p columns per stage
constexpr int kPMaxStages = 6;
constexpr int kGramRows = 128;   // rows per Gram task
constexpr int kQRows = 512;      // rows per compress_q task
constexpr int kQCols = 128;      // columns per compress_q task
constexpr int kURows = 256;      // rows per dp_update task
constexpr int kUTile = 32;       // rows per dp_update tile (8 warps x 4 rows)
constexpr int kUCols = 128;      // columns per dp_update task
constexpr int kApplyRows = 256;  // rows per dp_orth_apply CTA (one per thread)
constexpr float kDrop = 1e-10f;  // dependent column: residual^2 <= kDrop * norm^2

inline int pad_rank(int k) { return k <= 8 ? 8 : k <= 16 ? 16 : k <= 32 ? 32 : 64; }

__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

__device__ __forceinline__ int find_job(const int *begins, int count, int b) {
    int j = 0;
    while (j + 1 < count && b >= begins[j + 1]) ++j;
    return j;
}

// cp.async (sm_80+): 16-byte asynchronous copy global -> shared
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sum of the 64 values v over the 32 lanes of a warp; afterwards lane l holds
// the totals of entries 2l and 2l+1 in v[0], v[1].
__device__ __forceinline__ void warp_reduce64(float (&v)[64], int lane) {
#pragma unroll
    for (int o = 16, half = 32; o >= 1; o >>= 1, half >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
}

// ---------------------------------------------------------------------------
// two-float arithmetic (x = hi + lo, |lo| <= ulp(hi) / 2): error-free sum
// (Knuth) and product (fma), with every operation rounded explicitly so that
// the compiler cannot contract them.
// ---------------------------------------------------------------------------
struct df {
    float hi, lo;
};
__device__ __forceinline__ df two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ df quick_two_sum(float a, float b) {  // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df df_add(df x, df y) {
    const df s = two_sum(x.hi, y.hi);
    return quick_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ df df_neg(df x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ df df_mul(df x, df y) {
    const float p = __fmul_rn(x.hi, y.hi);
    float e = __fmaf_rn(x.hi, y.hi, -p);
    e = __fmaf_rn(x.hi, y.lo, e);
    e = __fmaf_rn(x.lo, y.hi, e);
    return quick_two_sum(p, e);
}
// 1 / sqrt(x): fp32 estimate y and one Newton step y + y (1 - x y^2) / 2 in two floats (x > 0)
__device__ __forceinline__ df df_rsqrt(df x) {
    const float y = rsqrtf(x.hi);
    const float yy = __fmul_rn(y, y);
    const df y2{yy, __fmaf_rn(y, y, -yy)};                              // y^2 exactly
    const df e = df_add(df{1.f, 0.f}, df_neg(df_mul(x, y2)));          // 1 - x y^2
    const df c = df_mul(df{y, 0.f}, e);
    return df_add(df{y, 0.f}, df{__fmul_rn(0.5f, c.hi), __fmul_rn(0.5f, c.lo)});
}
// (hi, lo) accumulation of a product of two floats: the product split exactly
// by an fma, the running sum by TwoSum; lo collects all rounding errors.
__device__ __forceinline__ void df_acc(float &hi, float &lo, float a, float b) {
    const float p = __fmul_rn(a, b);
    const float pe = __fmaf_rn(a, b, -p);
    const df s = two_sum(hi, p);
    hi = s.hi;
    lo = __fadd_rn(lo, __fadd_rn(s.lo, pe));
}

// tf32 hi (round to nearest, ties away) and lo = tf32(x - hi) of four floats
__device__ __forceinline__ float tf32_rna(float x) { return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u); }
__device__ __forceinline__ float4 split_hi4(float4 v, float4 &lo) {
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    lo = make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
    return h;
}

// ---------------------------------------------------------------------------
// dp_pad_q_kernel: Qp[j][c] = Q[j][c] for c < k, 0 for k <= c < kp + 4
// ---------------------------------------------------------------------------
struct PadJob {
    const float *Q;
    float *Qp;
    int n, k, kp;
    int64_t begin;
};
struct PadBatch {
    PadJob job[kMaxJobs];
    int count;
    int64_t total;
};

__global__ void __launch_bounds__(kThreads) dp_pad_q_kernel(const __grid_constant__ PadBatch B) {
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < B.total; e += (int64_t)gridDim.x * kThreads) {
        int j = 0;
        while (j + 1 < B.count && e >= B.job[j + 1].begin) ++j;
        const PadJob &J = B.job[j];
        const int64_t f = e - J.begin;
        const int w = J.kp + 4;
        const int64_t row = f / w;
        const int c = (int)(f % w);
        J.Qp[f] = c < J.k ? J.Q[row * J.k + c] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// compress_p:  M = E + X - Y -> E (global);  P = M Q
// Task: R rows (16; 8 for kp = 64) of one matrix over all its columns, in
// stages of 128 columns (512-byte row segments: narrower boxes cost DRAM
// efficiency, wider ones leave no room for the Q box).  Thread 0 keeps a ring
// of stages in flight: per stage one 2D TMA box (128 columns x R rows) of each
// of X, Y, E and one of Qp (the stage's 128 rows of Q, padded), all
// completing on the stage's mbarrier; the
// boxes are zero-filled outside the matrices.  The warps form M (written to
// global E from registers and in place of the E box), and the 8 warps
// accumulate P in 8 x 8 register tiles ((R/8)(kp/8) tiles, cs warps per tile
// splitting the columns); the task's last stage reduces the tiles over lanes
// and warps.  A stage is refilled as soon as it is consumed.
// ---------------------------------------------------------------------------
constexpr int kPRows = 16;
struct PJob {
    const CUtensorMap *mx, *my, *me, *mq;
    float *E, *P;
    int m, n, k, kp, hasY, ef, R, nch, task_begin;
};
struct PBatch {
    PJob job[kMaxJobs];
    int count, total_tasks, stages;
    uint32_t stage_bytes;
    unsigned *flag;
};
constexpr int kPBuf = kPRows * kPBC;  // floats of one input box (R x 128)

struct PCursor {
    int task, chunk, job;  // task < 0: past the end
};
__device__ __forceinline__ void p_first(PCursor &c, const PBatch &B, const int *begins) {
    c.task = blockIdx.x < (unsigned)B.total_tasks ? (int)blockIdx.x : -1;
    c.chunk = 0;
    c.job = c.task >= 0 ? find_job(begins, B.count, c.task) : 0;
}
__device__ __forceinline__ void p_advance(PCursor &c, const PBatch &B, const int *begins) {
    if (c.task < 0) return;
    if (++c.chunk < B.job[c.job].nch) return;
    c.chunk = 0;
    c.task += gridDim.x;
    if (c.task >= B.total_tasks) {
        c.task = -1;
        return;
    }
    c.job = find_job(begins, B.count, c.task);
}

__device__ __forceinline__ void p_issue(const PBatch &B, const PCursor &c, unsigned char *stage, uint64_t *bar) {
    const PJob &J = B.job[c.job];
    const int row0 = (c.task - J.task_begin) * J.R, col0 = c.chunk * kPBC;
    const uint32_t box = (uint32_t)J.R * kPBC * 4u, qbox = (uint32_t)kPBC * (J.kp + 4) * 4u;
    const uint32_t nin = 1u + (J.hasY ? 1u : 0u) + (J.ef ? 1u : 0u);
    float *xs = reinterpret_cast<float *>(stage), *ys = xs + kPBuf, *es = ys + kPBuf, *qs = es + kPBuf;
    mbar_arrive_expect_tx(bar, box * nin + qbox);
    tma_load_2d(xs, J.mx, col0, row0, bar);
    if (J.hasY) tma_load_2d(ys, J.my, col0, row0, bar);
    if (J.ef) tma_load_2d(es, J.me, col0, row0, bar);
    tma_load_2d(qs, J.mq, 0, col0, bar);
}

// P tile += M_stage Q_stage (zero outside the matrix) for padded rank KP
template <int KP>
__device__ __forceinline__ void p_fma(const float *es, const float *qs, float (&acc)[64], int warp, int lane) {
    constexpr int R = KP == 64 ? 8 : 16, TILES = (R / 8) * (KP / 8), CS = 8 / TILES, GS = 32 * CS;
    constexpr int QS = KP + 4, U = (kPBC + GS - 1) / GS;
    const int tile = warp % TILES, csplit = warp / TILES;
    const int rt = tile % (R / 8), kt = tile / (R / 8);
#pragma unroll
    for (int v = 0; v < U; ++v) {
        const int j = csplit * 32 + lane + GS * v;
        if (GS * (v + 1) > kPBC && j >= kPBC) break;
        float a[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) a[r] = es[(rt * 8 + r) * kPBC + j];
        const float4 b0 = *reinterpret_cast<const float4 *>(qs + j * QS + kt * 8);
        const float4 b1 = *reinterpret_cast<const float4 *>(qs + j * QS + kt * 8 + 4);
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r * 8 + q] = fmaf(a[r], b[q], acc[r * 8 + q]);
    }
}

__global__ void __launch_bounds__(kThreads, 2) dp_compress_p_kernel(const __grid_constant__ PBatch B) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int begins[kMaxJobs];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + 128);  // 8 warps x 64
    unsigned char *ring = smem + 128 + 8 * 64 * sizeof(float);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < B.count) begins[tid] = B.job[tid].task_begin;
    if (tid == 0) {
        for (int s = 0; s < B.stages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int j = 0; j < B.count; ++j) {
            prefetch_tmap(B.job[j].mx);
            prefetch_tmap(B.job[j].mq);
        }
    }
    __syncthreads();
    PCursor cur, pc;
    p_first(cur, B, begins);
    pc = cur;
    if (tid == 0)
        for (int s = 0; s < B.stages && pc.task >= 0; ++s) {
            p_issue(B, pc, ring + (size_t)s * B.stage_bytes, &bar[s]);
            p_advance(pc, B, begins);
        }
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int it = 0; cur.task >= 0; ++it) {
        const int s = it % B.stages;
        unsigned char *stage = ring + (size_t)s * B.stage_bytes;
        float *xs = reinterpret_cast<float *>(stage), *ys = xs + kPBuf, *es = ys + kPBuf, *qs = es + kPBuf;
        const PJob &J = B.job[cur.job];
        const int R = J.R, row0 = (cur.task - J.task_begin) * R, col0 = cur.chunk * kPBC;
        if (ok) ok = mbar_wait_bounded(&bar[s], (uint32_t)(it / B.stages) & 1u, B.flag, 3u);
        if (ok) {
            // M = E + X - Y over the box: to global E (inside the matrix) and in place of the E box
            for (int f = tid; f < R * (kPBC / 4); f += kThreads) {
                float4 x = reinterpret_cast<const float4 *>(xs)[f];
                if (J.hasY) {
                    const float4 y = reinterpret_cast<const float4 *>(ys)[f];
                    x.x -= y.x; x.y -= y.y; x.z -= y.z; x.w -= y.w;
                }
                if (J.ef) {
                    const float4 e = reinterpret_cast<const float4 *>(es)[f];
                    x.x = e.x + x.x; x.y = e.y + x.y; x.z = e.z + x.z; x.w = e.w + x.w;
                }
                reinterpret_cast<float4 *>(es)[f] = x;
                const int r = row0 + f / (kPBC / 4), c = col0 + 4 * (f % (kPBC / 4));
                if (r < J.m && c < J.n) __stcs(reinterpret_cast<float4 *>(J.E + (size_t)r * J.n + c), x);
            }
        }
        ok = __syncthreads_and(ok) != 0;
        if (!ok) break;
        switch (J.kp) {
            case 8: p_fma<8>(es, qs, acc, warp, lane); break;
            case 16: p_fma<16>(es, qs, acc, warp, lane); break;
            case 32: p_fma<32>(es, qs, acc, warp, lane); break;
            default: p_fma<64>(es, qs, acc, warp, lane); break;
        }
        const bool last = cur.chunk == J.nch - 1;
        __syncthreads();  // this stage is consumed: refill it
        if (tid == 0 && pc.task >= 0) {
            p_issue(B, pc, stage, &bar[s]);
            p_advance(pc, B, begins);
        }
        if (last) {
            // task done: sum the tiles over lanes (shuffles) and column-split warps (smem)
            const int tiles = (R / 8) * (J.kp / 8), cs = 8 / tiles;
            warp_reduce64(acc, lane);
            red[warp * 64 + 2 * lane] = acc[0];
            red[warp * 64 + 2 * lane + 1] = acc[1];
            __syncthreads();
            for (int e = tid; e < tiles * 64; e += kThreads) {
                const int tt = e / 64, idx = e % 64;
                float sum = 0.f;
                for (int q = 0; q < cs; ++q) sum += red[(tt + q * tiles) * 64 + idx];
                const int row = row0 + (tt % (R / 8)) * 8 + idx / 8, col = (tt / (R / 8)) * 8 + idx % 8;
                if (row < J.m && col < J.k) J.P[(size_t)row * J.k + col] = sum;
            }
            __syncthreads();  // red is free again
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.f;
        }
        p_advance(cur, B, begins);
    }
}

// ---------------------------------------------------------------------------
// orthogonalisation: two passes of Cholesky QR.  Pass p forms the Gram matrix
// of Y = P (p = 0) or Y = P R1^-1 (p = 1) with every product and sum carried in
// two floats, factors it as R^T R in two floats (a pivot <= kDrop x the
// column's own squared norm marks the column dependent: its row of R is zero
// and its reciprocal pivot 0) and stores R in fp32: strict upper part and the
// reciprocal pivots on the diagonal.
// ---------------------------------------------------------------------------

// y <- y R^-1 for one row held in registers (forward substitution), R as
// stored above.  The Gram pass and the apply kernel both go through this
// function, so the second pass factors exactly the rows the apply kernel
// produces.
template <int KP>
__device__ __forceinline__ void tri_solve_row(float (&y)[KP], const float *R) {
#pragma unroll
    for (int c = 0; c < KP; ++c) {
        float s = y[c];
#pragma unroll
        for (int a = 0; a < c; ++a) s = fmaf(-y[a], R[a * KP + c], s);
        y[c] = s * R[c * KP + c];
    }
}

struct GJob {
    const float *P, *R1;
    float *Gpart, *Rout;
    int *counter;
    int m, k, kp, tasks, task_begin;
};
struct GBatch {
    GJob job[kMaxJobs];
    int count, pass;
};

// (bi, bj) of upper-triangular 4 x 4 block b of an nb x nb block grid
__device__ __forceinline__ void block_pair(int b, int nb, int &bi, int &bj) {
    bi = 0;
    while (b >= nb - bi) {
        b -= nb - bi;
        ++bi;
    }
    bj = bi + b;
}

template <int KP>
__device__ void gram_task(const GBatch &B, const GJob &J, int task, unsigned char *smem) {
    constexpr int NB = KP / 4, NBLK = NB * (NB + 1) / 2;
    constexpr int RG = NBLK >= kThreads ? 1 : kThreads / NBLK;
    constexpr int XS = KP + 1;  // row stride of the staged rows (odd: conflict-free per-row access)
    __shared__ int is_last;
    float *xs = reinterpret_cast<float *>(smem);  // kGramRows x XS
    float *r1 = xs + kGramRows * XS;              // KP x KP
    float *red = r1 + KP * KP;                    // 32 x kThreads
    const int tid = threadIdx.x;
    const int r0 = task * kGramRows, rows = min(kGramRows, J.m - r0);
    for (int e = tid; e < kGramRows * KP; e += kThreads) {
        const int r = e / KP, c = e % KP;
        xs[r * XS + c] = (r < rows && c < J.k) ? J.P[(size_t)(r0 + r) * J.k + c] : 0.f;
    }
    if (B.pass == 1)
        for (int e = tid; e < KP * KP; e += kThreads) r1[e] = J.R1[e];
    __syncthreads();
    if (B.pass == 1) {
        if (tid < rows) {
            float y[KP];
#pragma unroll
            for (int c = 0; c < KP; ++c) y[c] = xs[tid * XS + c];
            tri_solve_row<KP>(y, r1);
#pragma unroll
            for (int c = 0; c < KP; ++c) xs[tid * XS + c] = y[c];
        }
        __syncthreads();
    }
    // 4 x 4 blocks of the upper triangle, RG row groups per block
    const int blk = tid % NBLK, rg = tid / NBLK;
    const bool active = rg < RG && tid < NBLK * RG;
    int bi, bj;
    block_pair(blk, NB, bi, bj);
    float hi[16], lo[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0.f;
    if (active)
        for (int r = rg; r < rows; r += RG) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = xs[r * XS + 4 * bi + i];
                b[i] = xs[r * XS + 4 * bj + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) df_acc(hi[i * 4 + j], lo[i * 4 + j], a[i], b[j]);
        }
    // tree over the row groups: slot = rg * NBLK + blk, element-major in red
    for (int cnt = RG; cnt > 1;) {
        const int h = (cnt + 1) / 2;
        if (active && rg >= h && rg < cnt) {
            const int slot = (rg - h) * NBLK + blk;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                red[(2 * e) * kThreads + slot] = hi[e];
                red[(2 * e + 1) * kThreads + slot] = lo[e];
            }
        }
        __syncthreads();
        if (active && rg < cnt - h) {
            const int slot = rg * NBLK + blk;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const df s = df_add(df{hi[e], lo[e]}, df{red[(2 * e) * kThreads + slot], red[(2 * e + 1) * kThreads + slot]});
                hi[e] = s.hi;
                lo[e] = s.lo;
            }
        }
        __syncthreads();
        cnt = h;
    }
    if (active && rg == 0) {
        float2 *gp = reinterpret_cast<float2 *>(J.Gpart) + ((size_t)task * NBLK + blk) * 16;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const df s = quick_two_sum(hi[e], lo[e]);
            gp[e] = make_float2(s.hi, s.lo);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(J.counter, 1) == J.tasks - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // last CTA of the matrix: G = sum of the partials in task order, then Cholesky
    float *gh = reinterpret_cast<float *>(smem);  // KP x KP (upper triangle)
    float *gl = gh + KP * KP;
    float *dg = gl + KP * KP;                      // original diagonal (hi)
    float *pinv = dg + KP;                         // reciprocal pivots (0: dependent)
    for (int e = tid; e < NBLK * 16; e += kThreads) {
        const int b = e / 16, w = e % 16;
        df s{0.f, 0.f};
        const float2 *src = reinterpret_cast<const float2 *>(J.Gpart) + (size_t)b * 16 + w;
        const size_t stride = (size_t)NBLK * 16;
        int t = 0;
        for (; t + 8 <= J.tasks; t += 8) {  // eight loads in flight, then the ordered sums
            float2 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (size_t)(t + u) * stride);
#pragma unroll
            for (int u = 0; u < 8; ++u) s = df_add(s, df{v[u].x, v[u].y});
        }
        for (; t < J.tasks; ++t) {
            const float2 v = __ldcg(src + (size_t)t * stride);
            s = df_add(s, df{v.x, v.y});
        }
        int pbi, pbj;
        block_pair(b, NB, pbi, pbj);
        const int r = 4 * pbi + w / 4, c = 4 * pbj + w % 4;
        if (r <= c) {
            gh[r * KP + c] = s.hi;
            gl[r * KP + c] = s.lo;
            if (r == c) dg[r] = s.hi;
        }
    }
    __syncthreads();
    // pivot j: 1 / sqrt(d), or 0 when the residual d is at most kDrop of the column's norm^2
    auto recip_pivot = [&](df d, int j) -> df {
        return d.hi > kDrop * dg[j] ? df_rsqrt(d) : df{0.f, 0.f};
    };
    // row 0 of R
    {
        const df inv = recip_pivot(df{gh[0], gl[0]}, 0);
        for (int c = 1 + tid; c < KP; c += kThreads) {
            const df r = df_mul(df{gh[c], gl[c]}, inv);
            gh[c] = r.hi;
            gl[c] = r.lo;
        }
        if (tid == 0) pinv[0] = inv.hi;
    }
    __syncthreads();
    // step j: trailing update with row j of R; the threads holding row j + 1
    // finish it in the same pass (each recomputes the new pivot), so one
    // barrier per step
    for (int j = 0; j + 1 < KP; ++j) {
        const int L = KP - j - 1;
        // the pairs j < a <= c, a-major: a = j + 1 + ra with ra from the triangular index
        for (int idx = tid; idx < L * (L + 1) / 2; idx += kThreads) {
            int ra = 0, rem = idx;
            while (rem >= L - ra) {
                rem -= L - ra;
                ++ra;
            }
            const int a = j + 1 + ra, c = a + rem;
            const df rja{gh[j * KP + a], gl[j * KP + a]};
            const df g = df_add(df{gh[a * KP + c], gl[a * KP + c]},
                                df_neg(df_mul(rja, df{gh[j * KP + c], gl[j * KP + c]})));
            if (a == j + 1) {
                const df d = df_add(df{gh[a * KP + a], gl[a * KP + a]}, df_neg(df_mul(rja, rja)));
                const df inv = recip_pivot(d, a);
                if (c == a) {
                    pinv[a] = inv.hi;
                } else {
                    const df r = df_mul(g, inv);
                    gh[a * KP + c] = r.hi;
                    gl[a * KP + c] = r.lo;
                }
            } else {
                gh[a * KP + c] = g.hi;
                gl[a * KP + c] = g.lo;
            }
        }
        __syncthreads();
    }
    for (int e = tid; e < KP * KP; e += kThreads) {
        const int r = e / KP, c = e % KP;
        J.Rout[e] = r < c ? gh[e] : r == c ? pinv[r] : 0.f;
    }
    if (tid == 0) *J.counter = 0;
}

__global__ void __launch_bounds__(kThreads, 1) dp_gram_kernel(const __grid_constant__ GBatch B) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int begins[kMaxJobs];
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].task_begin;
    __syncthreads();
    const GJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    const int task = blockIdx.x - J.task_begin;
    switch (J.kp) {
        case 8: gram_task<8>(B, J, task, smem); break;
        case 16: gram_task<16>(B, J, task, smem); break;
        case 32: gram_task<32>(B, J, task, smem); break;
        default: gram_task<64>(B, J, task, smem); break;
    }
}

inline size_t gram_smem_bytes(int kp) {
    const size_t p1 = sizeof(float) * ((size_t)kGramRows * (kp + 1) + (size_t)kp * kp + 32 * kThreads);
    const size_t p2 = sizeof(float) * (2 * (size_t)kp * kp + 2 * kp);
    return std::max(p1, p2);
}

// P^ = (P R1^-1) R2^-1 into the handle's m x kp basis, one row per thread.
struct AJob {
    const float *P, *R;  // R: R1 then R2, kp x kp each
    float *Ph;
    int m, k, kp, cta_begin;
};
struct ABatch {
    AJob job[kMaxJobs];
    int count;
};

template <int KP>
__device__ void orth_apply_rows(const AJob &J, unsigned char *smem_raw) {
    const int tid = threadIdx.x;
    const int r0 = (blockIdx.x - J.cta_begin) * kApplyRows, rows = min(kApplyRows, J.m - r0);
    float *r12 = reinterpret_cast<float *>(smem_raw);  // R1, R2
    for (int e = tid; e < 2 * KP * KP; e += kThreads) r12[e] = J.R[e];
    __syncthreads();
    if (tid >= rows) return;
    const int row = r0 + tid;
    float y[KP];
#pragma unroll
    for (int c = 0; c < KP; ++c) y[c] = c < J.k ? J.P[(size_t)row * J.k + c] : 0.f;
    tri_solve_row<KP>(y, r12);
    tri_solve_row<KP>(y, r12 + KP * KP);
    float4 *dst = reinterpret_cast<float4 *>(J.Ph + (size_t)row * KP);
#pragma unroll
    for (int c = 0; c < KP; c += 4) dst[c / 4] = make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]);
}

__global__ void __launch_bounds__(kThreads) dp_orth_apply_kernel(const __grid_constant__ ABatch B) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ int begins[kMaxJobs];
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].cta_begin;
    __syncthreads();
    const AJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    switch (J.kp) {
        case 8: orth_apply_rows<8>(J, smem_raw); break;
        case 16: orth_apply_rows<16>(J, smem_raw); break;
        case 32: orth_apply_rows<32>(J, smem_raw); break;
        default: orth_apply_rows<64>(J, smem_raw); break;
    }
}

// ---------------------------------------------------------------------------
// compress_q on the tcgen05 tensor cores:  partial Q = M^T P^ over one row
// range, 3xTF32 (hi.hi + hi.lo + lo.hi, fp32-accurate).
// Task (column block of 128, row range of 512) accumulates
//   D (128 x NP, TMEM) += A (128 x 32) . B (NP x 32)^T   per chunk of 32 rows,
// A[j][i] = M[r0 + i][col0 + j], B[c][i] = P^[r0 + i][c] (NP = kp, at least 16).
// The raw chunk arrives by TMA (boxes of 128 x 32 of M and kp x 32 of P^,
// zero outside the matrices) into a ring of kQtRaw stages; four split warps
// transpose it into the K-major, 128-byte-swizzled operand tiles, split into
// tf32 hi and lo, in a ring of kQtOps stages (the raw ring runs further ahead
// than the operands, which only wait for the MMAs).  Warp roles:
//   warp 0      TMA producer
//   warp 1      TMEM (two accumulators) and the MMA issuer (12 MMAs per chunk)
//   warps 2-9   transpose + split
//   warps 10-13 epilogue: the task's accumulator to its partial in Qpart
// Every mbarrier wait is bounded; a wait that gives up records a code in the
// library's device flag and that role stops.
// ---------------------------------------------------------------------------
constexpr int kQtK = 32;                       // rows of M per chunk (the MMA K of one atom)
constexpr int kQtMaxRaw = 8, kQtOps = 2;
constexpr int kQtThreads = 448;
constexpr int kQtSplitThreads = 256;  // warps 2-9
constexpr uint32_t kQtRawM = kQtK * kQCols * 4;       // 16 KB
constexpr uint32_t kQtA = kQCols * 128;               // 16 KB: 128 rows of 128 bytes
constexpr size_t kQtSmem = 232448 - 1024;             // all of shared memory but the static part
// ring layout for the largest padded rank of a launch: raw stages (M box, P^ box),
// then two operand stages (A hi, A lo, B hi, B lo); as many raw stages as fit
struct QtLayout {
    uint32_t raw_stage, op_stage, b_bytes, op_base;
    int raw;
};
__host__ __device__ inline QtLayout qt_layout(int kpmax) {
    QtLayout L;
    const int np = kpmax < 16 ? 16 : kpmax;
    L.raw_stage = (kQtRawM + (uint32_t)kQtK * kpmax * 4 + 1023) & ~1023u;
    L.b_bytes = (uint32_t)np * 128;
    L.op_stage = (2 * kQtA + 2 * L.b_bytes + 1023) & ~1023u;
    L.raw = (int)((kQtSmem - 1024 - 256 - kQtOps * (size_t)L.op_stage) / L.raw_stage);
    if (L.raw > kQtMaxRaw) L.raw = kQtMaxRaw;
    L.op_base = (uint32_t)L.raw * L.raw_stage;
    return L;
}
constexpr uint32_t kQtTmemCols = 128;                 // two accumulators of up to 64 columns

struct QJob {
    const CUtensorMap *mm, *mp;
    float *Qpart;
    int m, n, kp, ranges, ncb, task_begin;
};
struct QBatch {
    QJob job[kMaxJobs];
    int count, total_tasks, kpmax;
    unsigned *flag;
};

struct QCursor {
    int task, chunk, job, nch;
};
__device__ __forceinline__ int q_nch(const QJob &J, int task) {
    const int range = (task - J.task_begin) / J.ncb;
    const int rows = min(kQRows, J.m - range * kQRows);
    return (rows + kQtK - 1) / kQtK;
}
__device__ __forceinline__ void q_first(QCursor &c, const QBatch &B, const int *begins) {
    c.task = blockIdx.x < (unsigned)B.total_tasks ? (int)blockIdx.x : -1;
    c.chunk = 0;
    c.job = c.task >= 0 ? find_job(begins, B.count, c.task) : 0;
    c.nch = c.task >= 0 ? q_nch(B.job[c.job], c.task) : 0;
}
__device__ __forceinline__ bool q_advance(QCursor &c, const QBatch &B, const int *begins) {  // true: new task
    if (c.task < 0) return false;
    if (++c.chunk < c.nch) return false;
    c.chunk = 0;
    c.task += gridDim.x;
    if (c.task >= B.total_tasks) {
        c.task = -1;
        return true;
    }
    c.job = find_job(begins, B.count, c.task);
    c.nch = q_nch(B.job[c.job], c.task);
    return true;
}

__global__ void __launch_bounds__(kQtThreads, 1) dp_compress_q_kernel(const __grid_constant__ QBatch B) {
    extern __shared__ __align__(1024) unsigned char qt_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(qt_raw) + 1023) & ~uintptr_t(1023));
    const QtLayout L = qt_layout(B.kpmax);
    const int kQtRaw = L.raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.op_base + kQtOps * L.op_stage);
    uint64_t *full = bars;                   // [kQtMaxRaw] raw chunk landed
    uint64_t *rfree = full + kQtMaxRaw;      // [kQtMaxRaw] raw chunk consumed
    uint64_t *ready = rfree + kQtRaw;        // [kQtOps] operands written (128 arrivals)
    uint64_t *ofree = ready + kQtOps;        // [kQtOps] MMAs done with the operands
    uint64_t *tfull = ofree + kQtOps;        // [2] accumulator complete
    uint64_t *tempty = tfull + 2;            // [2] accumulator read (128 arrivals)
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tempty + 2);
    __shared__ int begins[kMaxJobs];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].task_begin;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQtRaw; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&rfree[s], kQtSplitThreads);
        }
        for (int o = 0; o < kQtOps; ++o) {
            mbar_init(&ready[o], kQtSplitThreads);
            mbar_init(&ofree[o], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, kQtTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    unsigned *flag = B.flag;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            for (int j = 0; j < B.count; ++j) {
                prefetch_tmap(B.job[j].mm);
                prefetch_tmap(B.job[j].mp);
            }
            QCursor c;
            q_first(c, B, begins);
            int i = 0;
            for (; c.task >= 0; ++i, q_advance(c, B, begins)) {
                const int s = i % kQtRaw;
                if (!mbar_wait_bounded(&rfree[s], ((uint32_t)(i / kQtRaw) & 1u) ^ 1u, flag, 0x301u)) break;
                const QJob &J = B.job[c.job];
                const int t = c.task - J.task_begin, cb = t % J.ncb, range = t / J.ncb;
                const int r0 = range * kQRows + c.chunk * kQtK;
                unsigned char *st = smem + s * L.raw_stage;
                mbar_arrive_expect_tx(&full[s], kQtRawM + (uint32_t)kQtK * J.kp * 4u);
                tma_load_2d(st, J.mm, cb * kQCols, r0, &full[s]);
                tma_load_2d(st + kQtRawM, J.mp, 0, r0, &full[s]);
            }
            if (c.task >= 0)  // gave up: let the loads already issued land before the CTA exits
                for (int q = (i > kQtRaw ? i - kQtRaw : 0); q < i; ++q)
                    mbar_wait_bounded(&full[q % kQtRaw], (uint32_t)(q / kQtRaw) & 1u, flag, 0x305u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            QCursor c;
            q_first(c, B, begins);
            int i = 0, task_i = 0;
            bool ok = true;
            for (; c.task >= 0; ++i) {
                const int o = i % kQtOps, a = task_i & 1;
                const QJob &J = B.job[c.job];
                const int np = J.kp < 16 ? 16 : J.kp;
                if (!(ok = mbar_wait_bounded(&ready[o], (uint32_t)(i / kQtOps) & 1u, flag, 0x302u))) break;
                if (c.chunk == 0 && !(ok = mbar_wait_bounded(&tempty[a], ((uint32_t)(task_i >> 1) & 1u) ^ 1u, flag, 0x303u)))
                    break;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + L.op_base + o * L.op_stage);
                const uint32_t ah = st, al = st + kQtA, bh = st + 2 * kQtA, bl = bh + L.b_bytes;
                const uint32_t as[3] = {ah, ah, al}, bs[3] = {bh, bl, bh};
                const uint32_t d = tmem + (uint32_t)(a * 64);
                const uint32_t idesc = tf32_idesc(128, np);
#pragma unroll
                for (int u = 0; u < 3; ++u)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        mma_tf32(d, smem_desc_sw128(as[u] + q * 32), smem_desc_sw128(bs[u] + q * 32), idesc,
                                 (c.chunk > 0 || u > 0 || q > 0) ? 1u : 0u);
                mma_commit(&ofree[o]);
                const bool last = c.chunk == c.nch - 1;
                if (last) mma_commit(&tfull[a]);
                if (q_advance(c, B, begins)) ++task_i;
            }
            if (!ok && i > 0)  // gave up: the MMAs issued finish before TMEM is freed
                mbar_wait_bounded(&ofree[(i - 1) % kQtOps], (uint32_t)((i - 1) / kQtOps) & 1u, flag, 0x306u);
        }
    } else if (warp < 10) {
        // ---------------- transpose + split: raw M (32 x 128) -> A[j][i], raw P^ (32 x kp) -> B[c][i]
        const int tid = threadIdx.x - 64;
        QCursor c;
        q_first(c, B, begins);
        for (int i = 0; c.task >= 0; ++i, q_advance(c, B, begins)) {
            const int s = i % kQtRaw, o = i % kQtOps;
            if (!mbar_wait_bounded(&full[s], (uint32_t)(i / kQtRaw) & 1u, flag, 0x304u)) break;
            if (!mbar_wait_bounded(&ofree[o], ((uint32_t)(i / kQtOps) & 1u) ^ 1u, flag, 0x308u)) break;
            const unsigned char *rs = smem + s * L.raw_stage;
            unsigned char *st = smem + L.op_base + o * L.op_stage;
            const float *rm = reinterpret_cast<const float *>(rs), *rp = reinterpret_cast<const float *>(rs + kQtRawM);
            const int kp = B.job[c.job].kp;
#pragma unroll 4
            for (int e = tid; e < kQCols * 8; e += kQtSplitThreads) {  // (row j of A, 16-byte chunk cc: i = 4 cc .. 4 cc + 3)
                const int j = e % kQCols, cc = e / kQCols;
                float4 lo;
                const float4 hi = split_hi4(make_float4(rm[(4 * cc) * kQCols + j], rm[(4 * cc + 1) * kQCols + j],
                                                        rm[(4 * cc + 2) * kQCols + j], rm[(4 * cc + 3) * kQCols + j]), lo);
                const uint32_t off = (uint32_t)j * 128 + ((uint32_t)(cc ^ (j & 7)) << 4);
                *reinterpret_cast<float4 *>(st + off) = hi;
                *reinterpret_cast<float4 *>(st + kQtA + off) = lo;
            }
            for (int e = tid; e < kp * 8; e += kQtSplitThreads) {  // (row r of B, chunk cc)
                const int r = e % kp, cc = e / kp;
                float4 lo;
                const float4 hi = split_hi4(make_float4(rp[(4 * cc) * kp + r], rp[(4 * cc + 1) * kp + r],
                                                        rp[(4 * cc + 2) * kp + r], rp[(4 * cc + 3) * kp + r]), lo);
                const uint32_t off = (uint32_t)r * 128 + ((uint32_t)(cc ^ (r & 7)) << 4);
                *reinterpret_cast<float4 *>(st + 2 * kQtA + off) = hi;
                *reinterpret_cast<float4 *>(st + 2 * kQtA + L.b_bytes + off) = lo;
            }
            fence_proxy_async_smem();  // the tensor core reads what these threads wrote
            mbar_arrive(&rfree[s]);
            mbar_arrive(&ready[o]);
        }
    } else {
        // ---------------- epilogue: TMEM lane quarter q = columns 32q .. 32q+31 of the block
        const int q = warp % 4;
        QCursor c;
        q_first(c, B, begins);
        for (int task_i = 0; c.task >= 0; ++task_i) {
            const int a = task_i & 1;
            const QJob &J = B.job[c.job];
            const int t = c.task - J.task_begin, cb = t % J.ncb, range = t / J.ncb;
            if (!mbar_wait_bounded(&tfull[a], (uint32_t)(task_i >> 1) & 1u, flag, 0x307u)) break;
            tc_fence_after();
            float v0[32], v1[32];
            const uint32_t taddr = tmem + (uint32_t)(a * 64) + ((uint32_t)(q * 32) << 16);
            tmem_ld32(taddr, v0);
            if (J.kp > 32) tmem_ld32(taddr + 32, v1);
            tc_fence_before();
            mbar_arrive(&tempty[a]);
            const int ldp = J.ncb * kQCols, col = cb * kQCols + q * 32 + lane;
            float4 *dst = reinterpret_cast<float4 *>(J.Qpart + ((size_t)range * ldp + col) * J.kp);
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (4 * x < J.kp) dst[x] = make_float4(v0[4 * x], v0[4 * x + 1], v0[4 * x + 2], v0[4 * x + 3]);
            if (J.kp > 32) {
#pragma unroll
                for (int x = 0; x < 8; ++x) dst[8 + x] = make_float4(v1[4 * x], v1[4 * x + 1], v1[4 * x + 2], v1[4 * x + 3]);
            }
            // next task (the cursor walks chunk by chunk)
            do {
            } while (!q_advance(c, B, begins));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kQtTmemCols);
    }
}

// Q[j][c] = sum over the row ranges (in order) of the partials
struct RJob {
    const float *Qpart;
    float *Q;
    int n, k, kp, ranges, ldp;
    int64_t begin;
};
struct RBatch {
    RJob job[kMaxJobs];
    int count;
    int64_t total;
};

__global__ void __launch_bounds__(kThreads) dp_q_reduce_kernel(const __grid_constant__ RBatch B) {
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < B.total; e += (int64_t)gridDim.x * kThreads) {
        int j = 0;
        while (j + 1 < B.count && e >= B.job[j + 1].begin) ++j;
        const RJob &J = B.job[j];
        const int64_t f = e - J.begin;
        const int64_t col = f / J.k;
        const int c = (int)(f % J.k);
        float s = 0.f;
        for (int r = 0; r < J.ranges; ++r) s += J.Qpart[((size_t)r * J.ldp + col) * J.kp + c];
        J.Q[f] = s;
    }
}

// ---------------------------------------------------------------------------
// decompress / outer step.  Task (row block of 256, column block of 128) of a
// persistent CTA (two per SM): the task's Q rows go transposed into shared
// memory once, the P^ rows of each 32-row tile arrive by cp.async one tile
// ahead, and each thread holds a 4 x 4 tile of D = s P^ Q^T (rows 4w..4w+3 of
// the tile, columns 4l..4l+3).  The thread's E (and theta, momentum) values
// are loaded before D is formed, so the FMA work covers the memory latency;
// then per element
//   E <- M - D (error feedback);  out <- D                       (mode 0)
//   b <- mu b + D;  theta <- theta - lr (D + mu b);
//   W <- (1 - mix) theta + mix W                                 (mode 1)
// ---------------------------------------------------------------------------
struct UJob {
    const float *Ph, *Q;
    float *E, *out, *theta, *mom, *W;
    int m, n, k, kp, ef, tiles_c, task_begin;
    float lr, mu, mix;
};
struct UBatch {
    UJob job[kMaxJobs];
    int count, mode, total_tasks;
    float q_scale;
};
constexpr int kQsStride = kUCols + 4;

__global__ void __launch_bounds__(kThreads, 2) dp_update_kernel(const __grid_constant__ UBatch B) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int begins[kMaxJobs];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < B.count) begins[tid] = B.job[tid].task_begin;
    __syncthreads();
    float *qs = reinterpret_cast<float *>(smem);  // kp x kQsStride (kp of the largest job)
    const float s = B.q_scale;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int task = blockIdx.x; task < B.total_tasks; task += gridDim.x) {
        const UJob &J = B.job[find_job(begins, B.count, task)];
        const int kp = J.kp, t = task - J.task_begin;
        const int rbeg = (t / J.tiles_c) * kURows, c0 = (t % J.tiles_c) * kUCols;
        const int rend = min(J.m, rbeg + kURows), ntile = (rend - rbeg + kUTile - 1) / kUTile;
        const int col = c0 + 4 * lane;
        const bool col_in = col < J.n;
        float *ps = qs + kp * kQsStride;  // 2 x kUTile x kp
        __syncthreads();                  // the previous task is done with qs and ps
        for (int e = tid; e < kUCols * kp; e += kThreads) {
            const int j = e / kp, c = e % kp;
            qs[c * kQsStride + j] = (c < J.k && c0 + j < J.n) ? J.Q[(size_t)(c0 + j) * J.k + c] : 0.f;
        }
        auto load_ph = [&](int tile) {
            const int r = rbeg + tile * kUTile, rows = min(kUTile, rend - r);
            float *dst = ps + (tile & 1) * kUTile * kp;
            const float *src = J.Ph + (size_t)r * kp;
            for (int f = tid; f < rows * kp / 4; f += kThreads) cp_async16(dst + 4 * f, src + 4 * f);
            cp_async_commit();
        };
        load_ph(0);
        for (int tl = 0; tl < ntile; ++tl) {
            const int rowb = rbeg + tl * kUTile + 4 * warp;
            // this thread's operands, loaded ahead of the FMA work
            float4 ev[4], tv[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool in = col_in && rowb + i < rend;
                const size_t idx = in ? (size_t)(rowb + i) * J.n + col : 0;
                ev[i] = (in && J.ef) ? __ldcs(reinterpret_cast<const float4 *>(J.E + idx)) : zero;
                tv[i] = (in && B.mode == 1) ? __ldcs(reinterpret_cast<const float4 *>(J.theta + idx)) : zero;
                bv[i] = (in && B.mode == 1) ? __ldcs(reinterpret_cast<const float4 *>(J.mom + idx)) : zero;
            }
            if (tl + 1 < ntile) {
                load_ph(tl + 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();  // P^ rows of this tile (and qs) are visible
            const float *pr = ps + (tl & 1) * kUTile * kp + 4 * warp * kp;
            float acc[16];  // [4 rows][4 columns]
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
            for (int c4 = 0; c4 < kp; c4 += 4) {
                float4 p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = *reinterpret_cast<const float4 *>(pr + i * kp + c4);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const float4 q = *reinterpret_cast<const float4 *>(qs + (c4 + cc) * kQsStride + 4 * lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float pv = cc == 0 ? p[i].x : cc == 1 ? p[i].y : cc == 2 ? p[i].z : p[i].w;
                        acc[i * 4 + 0] = fmaf(pv, q.x, acc[i * 4 + 0]);
                        acc[i * 4 + 1] = fmaf(pv, q.y, acc[i * 4 + 1]);
                        acc[i * 4 + 2] = fmaf(pv, q.z, acc[i * 4 + 2]);
                        acc[i * 4 + 3] = fmaf(pv, q.w, acc[i * 4 + 3]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = rowb + i;
                if (!col_in || row >= rend) continue;
                const size_t idx = (size_t)row * J.n + col;
                const float4 D = make_float4(s * acc[i * 4], s * acc[i * 4 + 1], s * acc[i * 4 + 2], s * acc[i * 4 + 3]);
                if (J.ef) {
                    const float4 M = ev[i];
                    __stcs(reinterpret_cast<float4 *>(J.E + idx), make_float4(M.x - D.x, M.y - D.y, M.z - D.z, M.w - D.w));
                }
                if (B.mode == 0) {
                    if (J.out) __stcs(reinterpret_cast<float4 *>(J.out + idx), D);
                    continue;
                }
                const float mu = J.mu, lr = J.lr;
                float4 b = bv[i], th = tv[i];
                b.x = fmaf(mu, b.x, D.x); b.y = fmaf(mu, b.y, D.y);
                b.z = fmaf(mu, b.z, D.z); b.w = fmaf(mu, b.w, D.w);
                th.x = fmaf(-lr, fmaf(mu, b.x, D.x), th.x); th.y = fmaf(-lr, fmaf(mu, b.y, D.y), th.y);
                th.z = fmaf(-lr, fmaf(mu, b.z, D.z), th.z); th.w = fmaf(-lr, fmaf(mu, b.w, D.w), th.w);
                __stcs(reinterpret_cast<float4 *>(J.mom + idx), b);
                __stcs(reinterpret_cast<float4 *>(J.theta + idx), th);
                float4 w = th;
                if (J.mix != 0.f) {
                    const float4 wl = *reinterpret_cast<const float4 *>(J.W + idx);
                    const float keep = 1.f - J.mix;
                    w.x = fmaf(J.mix, wl.x, keep * th.x); w.y = fmaf(J.mix, wl.y, keep * th.y);
                    w.z = fmaf(J.mix, wl.z, keep * th.z); w.w = fmaf(J.mix, wl.w, keep * th.w);
                }
                __stcs(reinterpret_cast<float4 *>(J.W + idx), w);
            }
            __syncthreads();  // this tile's P^ buffer may be refilled
        }
    }
}

}  // namespace
}  // namespace spco

// ---------------------------------------------------------------------------
// host API (include/dpsync.h)
// ---------------------------------------------------------------------------
using namespace spco;

namespace {

constexpr size_t kSmemBudget = 232448;  // 227 KB: one CTA per SM

int validate_batch(dpsync_t *const *hs, int32_t count, const char *what) {
    if (!hs || count < 1 || count > DPSYNC_MAX_BATCH)
        return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": 1 to 16 handles");
    for (int i = 0; i < count; ++i) {
        if (!hs[i]) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": null handle");
        for (int j = 0; j < i; ++j)
            if (hs[j] == hs[i]) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": repeated handle");
    }
    return SPECOPTIM_OK;
}

int set_smem(const void *fn, size_t bytes) {
    return set_smem_limit(fn, bytes);
}

int gram_blocks(int kp) { return (kp / 4) * (kp / 4 + 1) / 2; }
int p_rows(int kp) { return kp == 64 ? 8 : 16; }

// launch order of a batch: largest work first, so the tail of the grid is short
std::vector<int> by_size(dpsync_t *const *hs, int count) {
    std::vector<int> order(count);
    for (int i = 0; i < count; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        return (int64_t)hs[a]->m * hs[a]->n > (int64_t)hs[b]->m * hs[b]->n;
    });
    return order;
}

void free_all(dpsync *h) {
    for (void *p : {(void *)h->E, (void *)h->theta, (void *)h->mom, (void *)h->Ph, (void *)h->Qp, (void *)h->T,
                    (void *)h->Gpart, (void *)h->Qpart, (void *)h->counters, (void *)h->maps})
        if (p) cudaFree(p);
}

}  // namespace

extern "C" int32_t dpsync_rank(int32_t m, int32_t n, float ratio) {
    if (m < 1 || n < 1 || !(ratio > 0.f)) return -1;
    double k = std::floor((double)m * (double)n / ((double)ratio * ((double)m + (double)n)) + 0.5);
    k = std::max(1.0, std::min((double)std::min(m, n), k));
    return (int32_t)k;
}

extern "C" int dpsync_config_default(dpsync_config *cfg, int32_t m, int32_t n) {
    clear_error();
    if (!cfg) return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_config_default: null cfg");
    cfg->m = m;
    cfg->n = n;
    cfg->rank = 0;
    cfg->ratio = 64.f;
    cfg->error_feedback = 1;
    cfg->outer_lr = 0.7f;
    cfg->outer_momentum = 0.9f;
    cfg->mix = 0.f;
    return SPECOPTIM_OK;
}

extern "C" int dpsync_create(dpsync_t **out, const dpsync_config *cfg, float *P, float *Q, void *stream) {
    clear_error();
    if (!out || !cfg || !P || !Q) return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_create: null argument");
    *out = nullptr;
    if (cfg->m < 1 || cfg->n < 1 || cfg->n % 4 != 0)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_create: need m, n >= 1 and n a multiple of 4");
    if (cfg->rank < 0 || (cfg->rank == 0 && !(cfg->ratio > 0.f)) || !(cfg->mix >= 0.f && cfg->mix <= 1.f))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_create: bad rank, ratio or mix");
    const int k = cfg->rank > 0 ? cfg->rank : dpsync_rank(cfg->m, cfg->n, cfg->ratio);
    if (k > DPSYNC_MAX_RANK || k > std::min(cfg->m, cfg->n))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_create: rank above 64 or min(m, n)");
    if ((reinterpret_cast<uintptr_t>(P) | reinterpret_cast<uintptr_t>(Q)) & 3u)
        return fail(SPECOPTIM_ERR_MISALIGNED, "dpsync_create: P and Q must be 4-byte aligned");
    if (int rc = bind_device()) return rc;
    dpsync *h = new dpsync();
    h->cfg = *cfg;
    h->m = cfg->m;
    h->n = cfg->n;
    h->k = k;
    h->kp = pad_rank(k);
    h->P = P;
    h->Q = Q;
    h->gram_tasks = (h->m + kGramRows - 1) / kGramRows;
    h->q_ranges = (h->m + kQRows - 1) / kQRows;
    h->ncb = (h->n + kQCols - 1) / kQCols;
    const size_t mn = (size_t)h->m * h->n, kp = h->kp;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMalloc(&h->E, sizeof(float) * mn);
    if (e == cudaSuccess) e = cudaMalloc(&h->Ph, sizeof(float) * (size_t)h->m * kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->Qp, sizeof(float) * (size_t)h->n * (kp + 4));
    if (e == cudaSuccess) e = cudaMalloc(&h->T, sizeof(float) * 2 * kp * kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->Gpart, sizeof(float) * 32 * (size_t)gram_blocks(h->kp) * h->gram_tasks);
    if (e == cudaSuccess) e = cudaMalloc(&h->Qpart, sizeof(float) * (size_t)h->q_ranges * h->ncb * kQCols * kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->counters, sizeof(int) * 2);
    if (e == cudaSuccess) e = cudaMalloc(&h->maps, sizeof(CUtensorMap) * 6);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->E, 0, sizeof(float) * mn, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->Ph, 0, sizeof(float) * (size_t)h->m * kp, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->T, 0, sizeof(float) * 2 * kp * kp, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->counters, 0, sizeof(int) * 2, st);
    if (e != cudaSuccess) {
        free_all(h);
        delete h;
        return cuda_status(e, "dpsync_create");
    }
    // tensor maps of the handle's own buffers (those of X and Y follow each call)
    CUtensorMap hm[4];
    const uint32_t R = (uint32_t)p_rows(h->kp);
    int rc = make_tmap_2d_ex(&hm[0], h->E, h->m, h->n, h->n, kPBC, R, false);
    if (!rc) rc = make_tmap_2d_ex(&hm[1], h->Qp, h->n, h->kp + 4, h->kp + 4, h->kp + 4, kPBC, false);
    if (!rc) rc = make_tmap_2d_ex(&hm[2], h->E, h->m, h->n, h->n, kQCols, kQtK, false);
    if (!rc) rc = make_tmap_2d_ex(&hm[3], h->Ph, h->m, h->kp, h->kp, h->kp, kQtK, false);
    if (!rc) rc = cuda_status(cudaMemcpyAsync(h->maps + 2, hm, sizeof(hm), cudaMemcpyHostToDevice, st),
                              "dpsync_create: tensor maps");
    if (!rc) rc = cuda_status(cudaStreamSynchronize(st), "dpsync_create");
    if (rc) {
        free_all(h);
        delete h;
        return rc;
    }
    *out = h;
    return SPECOPTIM_OK;
}

extern "C" int32_t dpsync_handle_rank(const dpsync_t *h) { return h ? h->k : -1; }

extern "C" int dpsync_destroy(dpsync_t *h) {
    clear_error();
    if (!h) return SPECOPTIM_OK;
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
    return SPECOPTIM_OK;
}

extern "C" int dpsync_set_outer(dpsync_t *h, const float *W, void *stream) {
    clear_error();
    if (!h || !W) return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_set_outer: null argument");
    const size_t bytes = sizeof(float) * (size_t)h->m * h->n;
    if (!h->theta) {
        SPECOPTIM_CUDA(cudaMalloc(&h->theta, bytes));
        SPECOPTIM_CUDA(cudaMalloc(&h->mom, bytes));
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPECOPTIM_CUDA(cudaMemcpyAsync(h->theta, W, bytes, cudaMemcpyDeviceToDevice, st));
    SPECOPTIM_CUDA(cudaMemsetAsync(h->mom, 0, bytes, st));
    h->have_outer = true;
    return SPECOPTIM_OK;
}

extern "C" int dpsync_compress_p_many(dpsync_t *const *hs, int32_t count, const float *const *X,
                                      const float *const *Y, void *stream) {
    clear_error();
    int rc;
    if ((rc = validate_batch(hs, count, "dpsync_compress_p_many"))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PadBatch pad{};
    PBatch b{};
    pad.count = b.count = count;
    int64_t pad_total = 0;
    int tasks = 0, kpmax = 8;
    const std::vector<int> order = by_size(hs, count);
    for (int slot = 0; slot < count; ++slot) {
        const int i = order[slot];
        dpsync *h = hs[i];
        const float *x = X ? X[i] : nullptr;
        if (!x) {
            if (!h->have_outer)
                return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_compress_p_many: X is NULL and set_outer was not called");
            x = h->theta;
        }
        const float *y = Y ? Y[i] : nullptr;
        if (!aligned16(x) || (y && !aligned16(y)))
            return fail(SPECOPTIM_ERR_MISALIGNED, "dpsync_compress_p_many: X and Y must be 16-byte aligned");
        PadJob &pj = pad.job[slot];
        pj.Q = h->Q;
        pj.Qp = h->Qp;
        pj.n = h->n;
        pj.k = h->k;
        pj.kp = h->kp;
        pj.begin = pad_total;
        pad_total += (int64_t)h->n * (h->kp + 4);
        if (x != h->map_x || (y && y != h->map_y)) {
            CUtensorMap xm[2];
            const uint32_t R = (uint32_t)p_rows(h->kp);
            int r2 = make_tmap_2d_ex(&xm[0], x, h->m, h->n, h->n, kPBC, R, false);
            if (!r2) r2 = make_tmap_2d_ex(&xm[1], y ? y : x, h->m, h->n, h->n, kPBC, R, false);
            if (r2) return r2;
            SPECOPTIM_CUDA(cudaMemcpyAsync(h->maps, xm, sizeof(xm), cudaMemcpyHostToDevice, st));
            h->map_x = x;
            h->map_y = y ? y : x;
        }
        PJob &j = b.job[slot];
        j.mx = h->maps;
        j.my = h->maps + 1;
        j.me = h->maps + 2;
        j.mq = h->maps + 3;
        j.hasY = y ? 1 : 0;
        j.E = h->E;
        j.P = h->P;
        j.m = h->m;
        j.n = h->n;
        j.k = h->k;
        j.kp = h->kp;
        j.ef = h->cfg.error_feedback ? 1 : 0;
        j.R = p_rows(h->kp);
        j.nch = (h->n + kPBC - 1) / kPBC;
        j.task_begin = tasks;
        tasks += (h->m + j.R - 1) / j.R;
        kpmax = std::max(kpmax, h->kp);
    }
    pad.total = pad_total;
    b.total_tasks = tasks;
    b.stage_bytes = (uint32_t)align128(sizeof(float) * (3 * (size_t)kPBuf + (size_t)kPBC * (kpmax + 4)));
    // two CTAs per SM when two stages each fit in half of shared memory, else one with more stages
    const size_t fixed = 128 + 8 * 64 * sizeof(float);
    const int per_sm = fixed + 2 * (size_t)b.stage_bytes <= kSmemBudget / 2 ? 2 : 1;
    b.stages = (int)std::min<size_t>(kPMaxStages, (kSmemBudget / per_sm - fixed) / b.stage_bytes);
    b.flag = device_flag_ptr();
    const size_t smem = fixed + (size_t)b.stages * b.stage_bytes;
    if ((rc = set_smem((const void *)dp_compress_p_kernel, smem))) return rc;
    const int pad_grid = (int)std::min<int64_t>((pad_total + kThreads - 1) / kThreads, 4 * num_sms());
    SPCO_LAUNCH("dp_pad_q", st, dp_pad_q_kernel<<<pad_grid, kThreads, 0, st>>>(pad));
    SPECOPTIM_LAUNCHED("dp_pad_q_kernel");
    const int grid = std::min(tasks, per_sm * num_sms());
    SPCO_LAUNCH("dp_compress_p", st, dp_compress_p_kernel<<<grid, kThreads, smem, st>>>(b));
    SPECOPTIM_LAUNCHED("dp_compress_p_kernel");
    return SPECOPTIM_OK;
}

extern "C" int dpsync_orthogonalize_many(dpsync_t *const *hs, int32_t count, void *stream) {
    clear_error();
    int rc;
    if ((rc = validate_batch(hs, count, "dpsync_orthogonalize_many"))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int kpmax = 8;
    for (int i = 0; i < count; ++i) kpmax = std::max(kpmax, hs[i]->kp);
    const std::vector<int> order = by_size(hs, count);
    const size_t gsmem = gram_smem_bytes(kpmax);
    if ((rc = set_smem((const void *)dp_gram_kernel, gsmem))) return rc;
    for (int pass = 0; pass < 2; ++pass) {
        GBatch g{};
        g.count = count;
        g.pass = pass;
        int total = 0;
        for (int slot = 0; slot < count; ++slot) {
            dpsync *h = hs[order[slot]];
            GJob &j = g.job[slot];
            j.P = h->P;
            j.R1 = h->T;
            j.Gpart = h->Gpart;
            j.Rout = h->T + (size_t)pass * h->kp * h->kp;
            j.counter = h->counters + pass;
            j.m = h->m;
            j.k = h->k;
            j.kp = h->kp;
            j.tasks = h->gram_tasks;
            j.task_begin = total;
            total += h->gram_tasks;
        }
        SPCO_LAUNCH("dp_gram", st, dp_gram_kernel<<<total, kThreads, gsmem, st>>>(g));
        SPECOPTIM_LAUNCHED("dp_gram_kernel");
    }
    ABatch a{};
    a.count = count;
    int total = 0;
    for (int slot = 0; slot < count; ++slot) {
        dpsync *h = hs[order[slot]];
        AJob &j = a.job[slot];
        j.P = h->P;
        j.R = h->T;
        j.Ph = h->Ph;
        j.m = h->m;
        j.k = h->k;
        j.kp = h->kp;
        j.cta_begin = total;
        total += (h->m + kApplyRows - 1) / kApplyRows;
    }
    const size_t asmem = sizeof(float) * 2 * (size_t)kpmax * kpmax;
    if ((rc = set_smem((const void *)dp_orth_apply_kernel, asmem))) return rc;
    SPCO_LAUNCH("dp_orth_apply", st, dp_orth_apply_kernel<<<total, kThreads, asmem, st>>>(a));
    SPECOPTIM_LAUNCHED("dp_orth_apply_kernel");
    return SPECOPTIM_OK;
}

extern "C" int dpsync_compress_q_many(dpsync_t *const *hs, int32_t count, void *stream) {
    clear_error();
    int rc;
    if ((rc = validate_batch(hs, count, "dpsync_compress_q_many"))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    QBatch b{};
    RBatch r{};
    b.count = r.count = count;
    int tasks = 0, kpmax = 8;
    int64_t rtotal = 0;
    const std::vector<int> order = by_size(hs, count);
    for (int slot = 0; slot < count; ++slot) {
        dpsync *h = hs[order[slot]];
        QJob &j = b.job[slot];
        j.mm = h->maps + 4;
        j.mp = h->maps + 5;
        j.Qpart = h->Qpart;
        j.m = h->m;
        j.n = h->n;
        j.kp = h->kp;
        j.ranges = h->q_ranges;
        j.ncb = h->ncb;
        j.task_begin = tasks;
        tasks += h->q_ranges * h->ncb;
        kpmax = std::max(kpmax, h->kp);
        RJob &rj = r.job[slot];
        rj.Qpart = h->Qpart;
        rj.Q = h->Q;
        rj.n = h->n;
        rj.k = h->k;
        rj.kp = h->kp;
        rj.ranges = h->q_ranges;
        rj.ldp = h->ncb * kQCols;
        rj.begin = rtotal;
        rtotal += (int64_t)h->n * h->k;
    }
    b.total_tasks = tasks;
    r.total = rtotal;
    b.flag = device_flag_ptr();
    b.kpmax = kpmax;
    if ((rc = set_smem((const void *)dp_compress_q_kernel, kQtSmem))) return rc;
    const int grid = std::min(tasks, num_sms());
    SPCO_LAUNCH("dp_compress_q", st, dp_compress_q_kernel<<<grid, kQtThreads, kQtSmem, st>>>(b));
    SPECOPTIM_LAUNCHED("dp_compress_q_kernel");
    const int rgrid = (int)std::min<int64_t>((rtotal + kThreads - 1) / kThreads, 4 * num_sms());
    SPCO_LAUNCH("dp_q_reduce", st, dp_q_reduce_kernel<<<rgrid, kThreads, 0, st>>>(r));
    SPECOPTIM_LAUNCHED("dp_q_reduce_kernel");
    return SPECOPTIM_OK;
}

namespace {
int launch_update(dpsync_t *const *hs, int32_t count, float *const *ptrs, float q_scale, int mode,
                  void *stream, const char *what) {
    int rc;
    if ((rc = validate_batch(hs, count, what))) return rc;
    if (!std::isfinite(q_scale)) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": q_scale");
    UBatch b{};
    b.count = count;
    b.mode = mode;
    b.q_scale = q_scale;
    int total = 0, kpmax = 8;
    const std::vector<int> order = by_size(hs, count);
    for (int slot = 0; slot < count; ++slot) {
        const int i = order[slot];
        dpsync *h = hs[i];
        float *p = ptrs ? ptrs[i] : nullptr;
        if (mode == 1 && (!p || !h->have_outer))
            return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": needs W_local and set_outer");
        if (p && !aligned16(p)) return fail(SPECOPTIM_ERR_MISALIGNED, std::string(what) + ": 16-byte alignment");
        UJob &j = b.job[slot];
        j.Ph = h->Ph;
        j.Q = h->Q;
        j.E = h->E;
        j.out = mode == 0 ? p : nullptr;
        j.theta = h->theta;
        j.mom = h->mom;
        j.W = mode == 1 ? p : nullptr;
        j.m = h->m;
        j.n = h->n;
        j.k = h->k;
        j.kp = h->kp;
        j.ef = h->cfg.error_feedback ? 1 : 0;
        j.tiles_c = (h->n + kUCols - 1) / kUCols;
        j.task_begin = total;
        j.lr = h->cfg.outer_lr;
        j.mu = h->cfg.outer_momentum;
        j.mix = h->cfg.mix;
        total += ((h->m + kURows - 1) / kURows) * j.tiles_c;
        kpmax = std::max(kpmax, h->kp);
    }
    b.total_tasks = total;
    const size_t smem = sizeof(float) * (size_t)kpmax * (kQsStride + 2 * kUTile);
    if ((rc = set_smem((const void *)dp_update_kernel, smem))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int per_sm = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dp_update_kernel, kThreads, smem);
    const int grid = std::min(total, std::max(1, per_sm) * num_sms());
    SPCO_LAUNCH(mode == 0 ? "dp_decompress" : "dp_outer_step", st,
                dp_update_kernel<<<grid, kThreads, smem, st>>>(b));
    SPECOPTIM_LAUNCHED("dp_update_kernel");
    return SPECOPTIM_OK;
}
}  // namespace

extern "C" int dpsync_decompress_many(dpsync_t *const *hs, int32_t count, float *const *out,
                                      float q_scale, void *stream) {
    clear_error();
    return launch_update(hs, count, out, q_scale, 0, stream, "dpsync_decompress_many");
}

extern "C" int dpsync_outer_step_many(dpsync_t *const *hs, int32_t count, float *const *W_local,
                                      float q_scale, void *stream) {
    clear_error();
    return launch_update(hs, count, W_local, q_scale, 1, stream, "dpsync_outer_step_many");
}

extern "C" int dpsync_get_state(const dpsync_t *h, float *E, float *theta, float *mom, float *P_hat,
                                void *stream) {
    clear_error();
    if (!h) return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_get_state: null handle");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = sizeof(float) * (size_t)h->m * h->n;
    if ((theta || mom) && !h->have_outer)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_get_state: set_outer was not called");
    if (E) SPECOPTIM_CUDA(cudaMemcpyAsync(E, h->E, bytes, cudaMemcpyDeviceToDevice, st));
    if (theta) SPECOPTIM_CUDA(cudaMemcpyAsync(theta, h->theta, bytes, cudaMemcpyDeviceToDevice, st));
    if (mom) SPECOPTIM_CUDA(cudaMemcpyAsync(mom, h->mom, bytes, cudaMemcpyDeviceToDevice, st));
    if (P_hat)
        SPECOPTIM_CUDA(cudaMemcpy2DAsync(P_hat, sizeof(float) * h->k, h->Ph, sizeof(float) * h->kp,
                                         sizeof(float) * h->k, h->m, cudaMemcpyDeviceToDevice, st));
    return SPECOPTIM_OK;
}
