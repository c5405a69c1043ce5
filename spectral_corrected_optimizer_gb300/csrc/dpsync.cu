// Data-parallel outer synchronisation of one weight matrix (key design 4 of
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes": the
// Streaming DiLoCo outer step travels PowerSGD-compressed, 64x).
//
// Every kernel here streams the m x n matrices once and does O(k) fp32 work
// per element (k <= 64), so they are HBM-bound: fp32 FMA on the SIMT cores
// from operands staged in shared memory with cp.async, 8 x 8 register tiles
// (one shared-memory load per four FMAs), grids sized by rows / tiles, and
// deterministic split reductions (partials + last-arriving CTA, fixed order).
//
//   dp_compress_p_kernel   M = E + X - Y -> E;  P = M Q
//   dp_gram_kernel         Gram matrix of P (or of P T1) in two-float precision,
//                          then (last CTA) Cholesky in fp64 and T = R^-1
//   dp_orth_apply_kernel   P^ = (P T1) T2      (two passes of Cholesky QR)
//   dp_compress_q_kernel   Q = M^T P^
//   dp_update_kernel       D = s P^ Q^T;  E <- M - D;  out = D  or the outer
//                          Nesterov step and the restart of W_local
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dpsync.h"
#include "common.cuh"

struct dpsync {
    dpsync_config cfg;
    int m, n, k, kp;
    float *P, *Q;          // caller-owned m x k, n x k
    float *E;              // m x n: M between compress_p and decompress, then the error
    float *theta, *mom;    // m x n each, allocated by set_outer
    float *Ph;             // m x kp orthonormal basis (padded columns are zero)
    float *T;              // 2 x kp x kp: R1^-1, R2^-1 of the two Cholesky QR passes
    double *Gpart;         // gram tasks x kp(kp+1)/2 partial Gram matrices
    float *Qpart;          // q row ranges x ncb*128 x kp partial Q
    int *counters;         // [0, 2): gram passes; [2, 2 + ncb): Q column blocks
    int gram_tasks, q_ranges, ncb;
    bool have_outer;
};

namespace spco {
namespace {

constexpr int kThreads = 256;
constexpr int kGramRows = 128;   // rows per Gram task
constexpr int kQRows = 512;      // rows per compress_q task
constexpr int kQCols = 128;      // columns per compress_q task
constexpr int kQChunk = 16;      // rows per compress_q stage
constexpr int kQStages = 4;
constexpr int kPStages = 2;
constexpr int kTileRows = 64;    // dp_update tile
constexpr int kTileCols = 256;
constexpr double kDrop = 1e-10;  // dependent column: residual^2 <= kDrop * norm^2

inline int pad_rank(int k) { return k <= 8 ? 8 : k <= 16 ? 16 : k <= 32 ? 32 : 64; }

// compress_p tiling per padded rank: R rows per CTA streamed in BC-column chunks.
struct PCfg {
    int R, BC, tiles, cs;
};
__host__ __device__ inline PCfg p_cfg(int kp) {
    // 8 x 8 register tiles: (R/8)(kp/8) tiles over 8 warps, cs warps per tile
    // split the columns
    PCfg c;
    c.R = kp == 64 ? 8 : 16;
    c.BC = 128;
    c.tiles = (c.R / 8) * (kp / 8);
    c.cs = 8 / c.tiles;
    return c;
}
inline int p_stage_floats(int kp) { return 3 * 2048 + 128 * (kp + 4); }

// ---------------------------------------------------------------------------
// cp.async (sm_80+): 16-byte and 4-byte asynchronous copies global -> shared;
// a source size of 0 fills the destination with zeros.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(valid ? 4 : 0)
                 : "memory");
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
// compress_p:  M = E + X - Y -> E (global);  P = M Q
// ---------------------------------------------------------------------------
struct PJob {
    const float *X, *Y;
    float *E;
    const float *Q;
    float *P;
    int m, n, k, kp, ef, cta_begin;
};
struct PBatch {
    PJob job[DPSYNC_MAX_BATCH];
    int count, stage_floats;
};

__device__ __forceinline__ int find_job(const int *begins, int count, int b) {
    int j = 0;
    while (j + 1 < count && b >= begins[j + 1]) ++j;
    return j;
}

__global__ void __launch_bounds__(kThreads, 2) dp_compress_p_kernel(const __grid_constant__ PBatch B) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int begins[DPSYNC_MAX_BATCH];
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].cta_begin;
    __syncthreads();
    const int ji = find_job(begins, B.count, blockIdx.x);
    const PJob &J = B.job[ji];
    const PCfg C = p_cfg(J.kp);
    const int row0 = (blockIdx.x - J.cta_begin) * C.R;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qs = J.kp + 4;  // Q row stride in shared memory
    float *red = smem + kPStages * B.stage_floats;  // 8 warps x 64

    // zero the Q buffers once: cp.async writes only columns < k
    for (int i = tid; i < kPStages * B.stage_floats; i += kThreads) smem[i] = 0.f;
    __syncthreads();

    const bool hasY = J.Y != nullptr, ef = J.ef != 0;
    const int nch = (J.n + C.BC - 1) / C.BC;
    const int f4_per_row = C.BC / 4, nf4 = C.R * f4_per_row;

    auto issue = [&](int c) {
        float *st = smem + (c % kPStages) * B.stage_floats;
        float *xs = st, *ys = st + 2048, *es = st + 4096, *qsm = st + 6144;
        const int col0 = c * C.BC;
        for (int f = tid; f < nf4; f += kThreads) {
            const int r = f / f4_per_row, c4 = f % f4_per_row;
            const int gr = row0 + r, gc = col0 + 4 * c4;
            const bool ok = gr < J.m && gc < J.n;
            const size_t off = ok ? (size_t)gr * J.n + gc : 0;
            cp_async16(xs + 4 * f, J.X + off, ok);
            if (hasY) cp_async16(ys + 4 * f, J.Y + off, ok);
            if (ef) cp_async16(es + 4 * f, J.E + off, ok);
        }
        const int nq = C.BC * J.k;
        for (int e = tid; e < nq; e += kThreads) {
            const int j = e / J.k, cc = e % J.k;
            const bool ok = col0 + j < J.n;
            cp_async4(qsm + j * qs + cc, J.Q + (ok ? (size_t)(col0 + j) * J.k + cc : 0), ok);
        }
    };

    const int tile = warp % C.tiles, csplit = warp / C.tiles;
    const int rt = tile % (C.R / 8), kt = tile / (C.R / 8);
    const int g = csplit * 32 + lane, gstride = 32 * C.cs, u = C.BC / gstride;
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;

    issue(0);
    cp_async_commit();
    for (int c = 0; c < nch; ++c) {
        if (c + 1 < nch) issue(c + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        float *st = smem + (c % kPStages) * B.stage_floats;
        float *xs = st, *ys = st + 2048, *es = st + 4096, *qsm = st + 6144;
        const int col0 = c * C.BC;
        // M = E + X - Y into es and global E
        for (int f = tid; f < nf4; f += kThreads) {
            float4 x = reinterpret_cast<float4 *>(xs)[f];
            if (hasY) {
                const float4 y = reinterpret_cast<float4 *>(ys)[f];
                x.x -= y.x; x.y -= y.y; x.z -= y.z; x.w -= y.w;
            }
            if (ef) {
                const float4 e = reinterpret_cast<float4 *>(es)[f];
                x.x = e.x + x.x; x.y = e.y + x.y; x.z = e.z + x.z; x.w = e.w + x.w;
            }
            reinterpret_cast<float4 *>(es)[f] = x;
            const int r = f / f4_per_row, c4 = f % f4_per_row;
            const int gr = row0 + r, gc = col0 + 4 * c4;
            if (gr < J.m && gc < J.n) *reinterpret_cast<float4 *>(J.E + (size_t)gr * J.n + gc) = x;
        }
        __syncthreads();
        // P_tile += M_chunk Q_chunk over this thread's columns
        for (int v = 0; v < u; ++v) {
            const int j = g + gstride * v;
            float a[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) a[r] = es[(rt * 8 + r) * C.BC + j];
            const float4 b0 = *reinterpret_cast<const float4 *>(qsm + j * qs + kt * 8);
            const float4 b1 = *reinterpret_cast<const float4 *>(qsm + j * qs + kt * 8 + 4);
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[r * 8 + q] = fmaf(a[r], b[q], acc[r * 8 + q]);
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    warp_reduce64(acc, lane);
    red[warp * 64 + 2 * lane] = acc[0];
    red[warp * 64 + 2 * lane + 1] = acc[1];
    __syncthreads();
    for (int e = tid; e < C.tiles * 64; e += kThreads) {
        const int t = e / 64, idx = e % 64;
        float s = 0.f;
        for (int q = 0; q < C.cs; ++q) s += red[(t + q * C.tiles) * 64 + idx];
        const int trt = t % (C.R / 8), tkt = t / (C.R / 8);
        const int row = row0 + trt * 8 + idx / 8, col = tkt * 8 + idx % 8;
        if (row < J.m && col < J.k) J.P[(size_t)row * J.k + col] = s;
    }
}

// ---------------------------------------------------------------------------
// compress_q:  Q = M^T P^.  Task (column block of 128, row range of 512): the
// partial of its rows into Qpart; the last task of a column block to finish
// sums the partials in row-range order into the caller's Q.
// ---------------------------------------------------------------------------
struct QJob {
    const float *M, *Ph;
    float *Qpart, *Q;
    int *counter;
    int m, n, k, kp, ranges, ncb, task_begin;
};
struct QBatch {
    QJob job[DPSYNC_MAX_BATCH];
    int count, stage_floats;
};

__global__ void __launch_bounds__(kThreads, 2) dp_compress_q_kernel(const __grid_constant__ QBatch B) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int begins[DPSYNC_MAX_BATCH];
    __shared__ int is_last;
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].task_begin;
    __syncthreads();
    const QJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    const int task = blockIdx.x - J.task_begin;
    const int cb = task % J.ncb, range = task / J.ncb;
    const int col0 = cb * kQCols, rbeg = range * kQRows, rend = min(J.m, rbeg + kQRows);
    const int nch = (rend - rbeg + kQChunk - 1) / kQChunk;
    const int tid = threadIdx.x;
    const int kp = J.kp;

    auto issue = [&](int c) {
        float *st = smem + (c % kQStages) * B.stage_floats;
        float *ms = st, *ps = st + kQChunk * kQCols;
        const int r0 = rbeg + c * kQChunk;
        for (int f = tid; f < kQChunk * kQCols / 4; f += kThreads) {
            const int r = f / (kQCols / 4), c4 = f % (kQCols / 4);
            const int gr = r0 + r, gc = col0 + 4 * c4;
            const bool ok = gr < rend && gc < J.n;
            cp_async16(ms + 4 * f, J.M + (ok ? (size_t)gr * J.n + gc : 0), ok);
        }
        for (int f = tid; f < kQChunk * kp / 4; f += kThreads) {
            const int r = f / (kp / 4), c4 = f % (kp / 4);
            const bool ok = r0 + r < rend;
            cp_async16(ps + 4 * f, J.Ph + (ok ? (size_t)(r0 + r) * kp + 4 * c4 : 0), ok);
        }
    };

    const int tiles = 2 * kp, rg_count = kThreads / tiles;
    const int tile = tid % tiles, rg = tid / tiles;
    const int ct = tile % 16, kt = tile / 16;
    float acc[64];  // [8 columns][8 ranks]
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;

#pragma unroll
    for (int s = 0; s < kQStages - 1; ++s) {
        if (s < nch) issue(s);
        cp_async_commit();
    }
    for (int c = 0; c < nch; ++c) {
        cp_async_wait<kQStages - 2>();
        __syncthreads();
        const float *st = smem + (c % kQStages) * B.stage_floats;
        const float *ms = st, *ps = st + kQChunk * kQCols;
        for (int i = rg; i < kQChunk; i += rg_count) {
            const float4 a0 = *reinterpret_cast<const float4 *>(ms + i * kQCols + 4 * ct);
            const float4 a1 = *reinterpret_cast<const float4 *>(ms + i * kQCols + 64 + 4 * ct);
            const float4 b0 = *reinterpret_cast<const float4 *>(ps + i * kp + kt * 8);
            const float4 b1 = *reinterpret_cast<const float4 *>(ps + i * kp + kt * 8 + 4);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int x = 0; x < 8; ++x)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[x * 8 + q] = fmaf(a[x], b[q], acc[x * 8 + q]);
        }
        if (c + kQStages - 1 < nch) issue(c + kQStages - 1);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    // sum the row groups in the (now idle) stage ring: halving steps
    for (int half = rg_count / 2; half >= 1; half /= 2) {
        const int nt = half * tiles;
        if (rg >= half && rg < 2 * half) {
            const int idx = (rg - half) * tiles + tile;
#pragma unroll
            for (int v = 0; v < 64; ++v) smem[v * nt + idx] = acc[v];
        }
        __syncthreads();
        if (rg < half) {
            const int idx = rg * tiles + tile;
#pragma unroll
            for (int v = 0; v < 64; ++v) acc[v] += smem[v * nt + idx];
        }
        __syncthreads();
    }
    const int ldp = J.ncb * kQCols;  // Qpart: [ranges][ldp][kp]
    if (rg == 0) {
        float *dst = J.Qpart + ((size_t)range * ldp + col0) * kp + kt * 8;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int col = x < 4 ? 4 * ct + x : 64 + 4 * ct + (x - 4);
            float4 *d = reinterpret_cast<float4 *>(dst + (size_t)col * kp);
            d[0] = make_float4(acc[x * 8 + 0], acc[x * 8 + 1], acc[x * 8 + 2], acc[x * 8 + 3]);
            d[1] = make_float4(acc[x * 8 + 4], acc[x * 8 + 5], acc[x * 8 + 6], acc[x * 8 + 7]);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(J.counter + cb, 1) == J.ranges - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int ncols = min(kQCols, J.n - col0);
    for (int e = tid; e < ncols * J.k; e += kThreads) {
        const int j = e / J.k, q = e % J.k;
        float s = 0.f;
        for (int r = 0; r < J.ranges; ++r) s += __ldcg(J.Qpart + ((size_t)r * ldp + col0 + j) * kp + q);
        J.Q[(size_t)(col0 + j) * J.k + q] = s;
    }
    if (tid == 0) J.counter[cb] = 0;
}

// ---------------------------------------------------------------------------
// orthogonalisation: two passes of Cholesky QR.  Pass p forms the Gram matrix
// of Y = P (p = 0) or Y = P T1 (p = 1) with every product and sum carried in
// two floats (hi + lo, error-free product and sum), factors it in fp64 as
// R^T R (a pivot <= kDrop x the column's own squared norm marks the column
// dependent: its row of R and column of R^-1 are zero) and stores T = R^-1.
// ---------------------------------------------------------------------------

// y_c = sum_{a <= c} x_a T[a][c] in a fixed order: the gram pass and the apply
// kernel evaluate P T1 through this one function, so the second pass sees
// exactly the rows the apply kernel produces.
__device__ __forceinline__ float upper_times(const float *x, const float *T, int kp, int c) {
    float s = 0.f;
    for (int a = 0; a <= c; ++a) s = fmaf(x[a], T[a * kp + c], s);
    return s;
}

// (hi, lo) += a * b with the product split exactly (fma) and the sum by TwoSum
__device__ __forceinline__ void df_acc(float &hi, float &lo, float a, float b) {
    const float p = __fmul_rn(a, b);
    const float pe = fmaf(a, b, -p);
    const float s = __fadd_rn(hi, p);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(p, bb));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, pe));
}

struct GJob {
    const float *P, *T1;
    double *Gpart;
    float *Tout;
    int *counter;
    int m, k, kp, tasks, task_begin;
};
struct GBatch {
    GJob job[DPSYNC_MAX_BATCH];
    int count, pass;
};
constexpr int kMaxEntries = (64 * 65 / 2 + kThreads - 1) / kThreads;  // 9

__global__ void __launch_bounds__(kThreads, 1) dp_gram_kernel(const __grid_constant__ GBatch B) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int begins[DPSYNC_MAX_BATCH];
    __shared__ int is_last;
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].task_begin;
    __syncthreads();
    const GJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    const int task = blockIdx.x - J.task_begin;
    const int kp = J.kp, tid = threadIdx.x;
    const int r0 = task * kGramRows, rows = min(kGramRows, J.m - r0);
    float *xs = smem;                       // kGramRows x kp
    float *ys = xs + kGramRows * kp;        // kGramRows x kp
    float *t1 = ys + kGramRows * kp;        // kp x kp

    for (int e = tid; e < kGramRows * kp; e += kThreads) {
        const int r = e / kp, c = e % kp;
        xs[e] = (r < rows && c < J.k) ? J.P[(size_t)(r0 + r) * J.k + c] : 0.f;
    }
    if (B.pass == 1)
        for (int e = tid; e < kp * kp; e += kThreads) t1[e] = J.T1[e];
    __syncthreads();
    const float *y = xs;
    if (B.pass == 1) {
        for (int e = tid; e < kGramRows * kp; e += kThreads) {
            const int r = e / kp, c = e % kp;
            ys[e] = upper_times(xs + r * kp, t1, kp, c);
        }
        __syncthreads();
        y = ys;
    }
    // this thread's entries (a <= b) of the upper triangle, row-major order
    const int E = kp * (kp + 1) / 2;
    int ea[kMaxEntries], eb[kMaxEntries];
    float hi[kMaxEntries], lo[kMaxEntries];
#pragma unroll
    for (int v = 0; v < kMaxEntries; ++v) {
        int e = tid + v * kThreads, a = 0;
        if (e >= E) e = -1;
        if (e >= 0)
            while (e >= kp - a) { e -= kp - a; ++a; }
        ea[v] = e >= 0 ? a : -1;
        eb[v] = e >= 0 ? a + e : 0;
        hi[v] = lo[v] = 0.f;
    }
    for (int r = 0; r < rows; ++r) {
#pragma unroll
        for (int v = 0; v < kMaxEntries; ++v)
            if (ea[v] >= 0) df_acc(hi[v], lo[v], y[r * kp + ea[v]], y[r * kp + eb[v]]);
    }
    double *gp = J.Gpart + (size_t)task * E;
#pragma unroll
    for (int v = 0; v < kMaxEntries; ++v)
        if (ea[v] >= 0) gp[tid + v * kThreads] = (double)hi[v] + (double)lo[v];
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(J.counter, 1) == J.tasks - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // last CTA: G = sum of the partials (task order), Cholesky, T = R^-1
    double *G = reinterpret_cast<double *>(smem);  // kp x kp (upper triangle used)
    double *Ti = G + kp * kp;                       // kp x kp
    double *piv = Ti + kp * kp;                     // kp
    double *dg = piv + kp;                          // kp: original diagonal
    for (int e = tid; e < E; e += kThreads) {
        double s = 0.0;
        for (int t = 0; t < J.tasks; ++t) s += __ldcg(J.Gpart + (size_t)t * E + e);
        int a = 0, f = e;
        while (f >= kp - a) { f -= kp - a; ++a; }
        G[a * kp + a + f] = s;
        if (f == 0) dg[a] = s;
    }
    __syncthreads();
    for (int j = 0; j < kp; ++j) {
        const double d = G[j * kp + j];
        const bool dep = !(d > kDrop * dg[j]);
        const double pj = dep ? 0.0 : sqrt(d);
        for (int c = j + 1 + tid; c < kp; c += kThreads) G[j * kp + c] = dep ? 0.0 : G[j * kp + c] / pj;
        if (tid == 0) piv[j] = pj;
        __syncthreads();
        if (!dep) {
            const int L = kp - j - 1;
            for (int idx = tid; idx < L * L; idx += kThreads) {
                const int a = j + 1 + idx / L, b = j + 1 + idx % L;
                if (a <= b) G[a * kp + b] -= G[j * kp + a] * G[j * kp + b];
            }
        }
        __syncthreads();
    }
    // columns of R^-1 by back substitution, one thread per column
    if (tid < kp) {
        const int c = tid;
        for (int i = c; i >= 0; --i) {
            double t;
            if (piv[i] == 0.0) {
                t = 0.0;
            } else if (i == c) {
                t = 1.0 / piv[i];
            } else {
                double s = 0.0;
                for (int p = i + 1; p <= c; ++p) s += G[i * kp + p] * Ti[p * kp + c];
                t = -s / piv[i];
            }
            Ti[i * kp + c] = t;
        }
    }
    __syncthreads();
    for (int e = tid; e < kp * kp; e += kThreads) {
        const int i = e / kp, c = e % kp;
        J.Tout[e] = i <= c ? (float)Ti[e] : 0.f;
    }
    if (tid == 0) *J.counter = 0;
}

// P^ = (P T1) T2 into the handle's m x kp basis.
struct AJob {
    const float *P, *T;  // T: T1 then T2, kp x kp each
    float *Ph;
    int m, k, kp, cta_begin;
};
struct ABatch {
    AJob job[DPSYNC_MAX_BATCH];
    int count;
};
constexpr int kApplyRows = 64;

__global__ void __launch_bounds__(kThreads) dp_orth_apply_kernel(const __grid_constant__ ABatch B) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int begins[DPSYNC_MAX_BATCH];
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].cta_begin;
    __syncthreads();
    const AJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    const int kp = J.kp, tid = threadIdx.x;
    const int r0 = (blockIdx.x - J.cta_begin) * kApplyRows, rows = min(kApplyRows, J.m - r0);
    float *xs = smem, *ys = xs + kApplyRows * kp, *t1 = ys + kApplyRows * kp, *t2 = t1 + kp * kp;
    for (int e = tid; e < kApplyRows * kp; e += kThreads) {
        const int r = e / kp, c = e % kp;
        xs[e] = (r < rows && c < J.k) ? J.P[(size_t)(r0 + r) * J.k + c] : 0.f;
    }
    for (int e = tid; e < 2 * kp * kp; e += kThreads) t1[e] = J.T[e];
    __syncthreads();
    for (int e = tid; e < kApplyRows * kp; e += kThreads) {
        const int r = e / kp, c = e % kp;
        ys[e] = upper_times(xs + r * kp, t1, kp, c);
    }
    __syncthreads();
    for (int e = tid; e < rows * kp; e += kThreads) {
        const int r = e / kp, c = e % kp;
        J.Ph[(size_t)(r0 + r) * kp + c] = upper_times(ys + r * kp, t2, kp, c);
    }
}

// ---------------------------------------------------------------------------
// decompress / outer step over 64 x 256 tiles:  D = s P^ Q^T (8 x 8 per thread,
// P^ and Q staged transposed in shared memory), then per element
//   E <- M - D (error feedback);  out <- D                       (mode 0)
//   b <- mu b + D;  theta <- theta - lr (D + mu b);
//   W <- (1 - mix) theta + mix W                                 (mode 1)
// ---------------------------------------------------------------------------
struct UJob {
    const float *Ph, *Q;
    float *E, *out, *theta, *mom, *W;
    int m, n, k, kp, ef, tiles_n, cta_begin;
    float lr, mu, mix;
};
struct UBatch {
    UJob job[DPSYNC_MAX_BATCH];
    int count, mode;
    float q_scale;
};
constexpr int kPsStride = kTileRows + 4;
constexpr int kQsStride = kTileCols + 4;

__global__ void __launch_bounds__(kThreads, 2) dp_update_kernel(const __grid_constant__ UBatch B) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int begins[DPSYNC_MAX_BATCH];
    if (threadIdx.x < B.count) begins[threadIdx.x] = B.job[threadIdx.x].cta_begin;
    __syncthreads();
    const UJob &J = B.job[find_job(begins, B.count, blockIdx.x)];
    const int t = blockIdx.x - J.cta_begin;
    const int r0 = (t / J.tiles_n) * kTileRows, c0 = (t % J.tiles_n) * kTileCols;
    const int kp = J.kp, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *ps = smem;                   // kp x kPsStride: P^ rows of the tile, transposed
    float *qs = ps + kp * kPsStride;    // kp x kQsStride: Q rows of the tile, transposed
    for (int e = tid; e < kTileRows * kp; e += kThreads) {
        const int r = e / kp, c = e % kp;
        ps[c * kPsStride + r] = r0 + r < J.m ? J.Ph[(size_t)(r0 + r) * kp + c] : 0.f;
    }
    for (int e = tid; e < kTileCols * kp; e += kThreads) {
        const int j = e / kp, c = e % kp;
        qs[c * kQsStride + j] = (c < J.k && c0 + j < J.n) ? J.Q[(size_t)(c0 + j) * J.k + c] : 0.f;
    }
    __syncthreads();
    float acc[64];  // [8 rows][8 columns]
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    for (int c = 0; c < kp; ++c) {
        const float4 p0 = *reinterpret_cast<const float4 *>(ps + c * kPsStride + 8 * warp);
        const float4 p1 = *reinterpret_cast<const float4 *>(ps + c * kPsStride + 8 * warp + 4);
        const float4 q0 = *reinterpret_cast<const float4 *>(qs + c * kQsStride + 4 * lane);
        const float4 q1 = *reinterpret_cast<const float4 *>(qs + c * kQsStride + 128 + 4 * lane);
        const float a[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        const float b[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int x = 0; x < 8; ++x) acc[r * 8 + x] = fmaf(a[r], b[x], acc[r * 8 + x]);
    }
    const float s = B.q_scale;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int row = r0 + 8 * warp + r;
        if (row >= J.m) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = c0 + 128 * h + 4 * lane;
            if (col >= J.n) continue;
            const size_t idx = (size_t)row * J.n + col;
            const float4 D = make_float4(s * acc[r * 8 + 4 * h], s * acc[r * 8 + 4 * h + 1],
                                         s * acc[r * 8 + 4 * h + 2], s * acc[r * 8 + 4 * h + 3]);
            if (J.ef) {
                float4 M = *reinterpret_cast<const float4 *>(J.E + idx);
                M.x -= D.x; M.y -= D.y; M.z -= D.z; M.w -= D.w;
                *reinterpret_cast<float4 *>(J.E + idx) = M;
            }
            if (B.mode == 0) {
                if (J.out) *reinterpret_cast<float4 *>(J.out + idx) = D;
            } else {
                float4 th = *reinterpret_cast<const float4 *>(J.theta + idx);
                float4 b = *reinterpret_cast<const float4 *>(J.mom + idx);
                const float mu = J.mu, lr = J.lr;
                b.x = fmaf(mu, b.x, D.x); b.y = fmaf(mu, b.y, D.y);
                b.z = fmaf(mu, b.z, D.z); b.w = fmaf(mu, b.w, D.w);
                th.x = fmaf(-lr, fmaf(mu, b.x, D.x), th.x); th.y = fmaf(-lr, fmaf(mu, b.y, D.y), th.y);
                th.z = fmaf(-lr, fmaf(mu, b.z, D.z), th.z); th.w = fmaf(-lr, fmaf(mu, b.w, D.w), th.w);
                *reinterpret_cast<float4 *>(J.mom + idx) = b;
                *reinterpret_cast<float4 *>(J.theta + idx) = th;
                float4 w = th;
                if (J.mix != 0.f) {
                    const float4 wl = *reinterpret_cast<const float4 *>(J.W + idx);
                    const float keep = 1.f - J.mix;
                    w.x = fmaf(J.mix, wl.x, keep * th.x); w.y = fmaf(J.mix, wl.y, keep * th.y);
                    w.z = fmaf(J.mix, wl.z, keep * th.z); w.w = fmaf(J.mix, wl.w, keep * th.w);
                }
                *reinterpret_cast<float4 *>(J.W + idx) = w;
            }
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
    return cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes),
                       "cudaFuncSetAttribute");
}

int gram_smem_bytes(int kp) {
    const size_t p1 = sizeof(float) * (2 * (size_t)kGramRows * kp + (size_t)kp * kp);
    const size_t p2 = sizeof(double) * (2 * (size_t)kp * kp + 2 * (size_t)kp);
    return (int)std::max(p1, p2);
}

void free_all(dpsync *h) {
    for (void *p : {(void *)h->E, (void *)h->theta, (void *)h->mom, (void *)h->Ph, (void *)h->T,
                    (void *)h->Gpart, (void *)h->Qpart, (void *)h->counters})
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
    const size_t mn = (size_t)h->m * h->n, E = (size_t)h->kp * (h->kp + 1) / 2;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMalloc(&h->E, sizeof(float) * mn);
    if (e == cudaSuccess) e = cudaMalloc(&h->Ph, sizeof(float) * (size_t)h->m * h->kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->T, sizeof(float) * 2 * (size_t)h->kp * h->kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->Gpart, sizeof(double) * E * h->gram_tasks);
    if (e == cudaSuccess)
        e = cudaMalloc(&h->Qpart, sizeof(float) * (size_t)h->q_ranges * h->ncb * kQCols * h->kp);
    if (e == cudaSuccess) e = cudaMalloc(&h->counters, sizeof(int) * (2 + h->ncb));
    if (e == cudaSuccess) e = cudaMemsetAsync(h->E, 0, sizeof(float) * mn, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->Ph, 0, sizeof(float) * (size_t)h->m * h->kp, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->T, 0, sizeof(float) * 2 * (size_t)h->kp * h->kp, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->counters, 0, sizeof(int) * (2 + h->ncb), st);
    if (e != cudaSuccess) {
        free_all(h);
        delete h;
        return cuda_status(e, "dpsync_create");
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
    PBatch b{};
    b.count = count;
    int total = 0, kpmax = 8;
    for (int i = 0; i < count; ++i) {
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
        PJob &j = b.job[i];
        j.X = x;
        j.Y = y;
        j.E = h->E;
        j.Q = h->Q;
        j.P = h->P;
        j.m = h->m;
        j.n = h->n;
        j.k = h->k;
        j.kp = h->kp;
        j.ef = h->cfg.error_feedback ? 1 : 0;
        j.cta_begin = total;
        total += (h->m + p_cfg(h->kp).R - 1) / p_cfg(h->kp).R;
        kpmax = std::max(kpmax, h->kp);
    }
    b.stage_floats = p_stage_floats(kpmax);
    const size_t smem = sizeof(float) * ((size_t)kPStages * b.stage_floats + 8 * 64);
    if ((rc = set_smem((const void *)dp_compress_p_kernel, smem))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("dp_compress_p", st, dp_compress_p_kernel<<<total, kThreads, smem, st>>>(b));
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
    const size_t gsmem = gram_smem_bytes(kpmax);
    if ((rc = set_smem((const void *)dp_gram_kernel, gsmem))) return rc;
    for (int pass = 0; pass < 2; ++pass) {
        GBatch g{};
        g.count = count;
        g.pass = pass;
        int total = 0;
        for (int i = 0; i < count; ++i) {
            dpsync *h = hs[i];
            GJob &j = g.job[i];
            j.P = h->P;
            j.T1 = h->T;
            j.Gpart = h->Gpart;
            j.Tout = h->T + (size_t)pass * h->kp * h->kp;
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
    for (int i = 0; i < count; ++i) {
        dpsync *h = hs[i];
        AJob &j = a.job[i];
        j.P = h->P;
        j.T = h->T;
        j.Ph = h->Ph;
        j.m = h->m;
        j.k = h->k;
        j.kp = h->kp;
        j.cta_begin = total;
        total += (h->m + kApplyRows - 1) / kApplyRows;
    }
    const size_t asmem = sizeof(float) * (2 * (size_t)kApplyRows * kpmax + 2 * (size_t)kpmax * kpmax);
    if ((rc = set_smem((const void *)dp_orth_apply_kernel, asmem))) return rc;
    SPCO_LAUNCH("dp_orth_apply", st, dp_orth_apply_kernel<<<total, kThreads, asmem, st>>>(a));
    SPECOPTIM_LAUNCHED("dp_orth_apply_kernel");
    return SPECOPTIM_OK;
}

extern "C" int dpsync_compress_q_many(dpsync_t *const *hs, int32_t count, void *stream) {
    clear_error();
    int rc;
    if ((rc = validate_batch(hs, count, "dpsync_compress_q_many"))) return rc;
    QBatch b{};
    b.count = count;
    int total = 0, kpmax = 8;
    for (int i = 0; i < count; ++i) {
        dpsync *h = hs[i];
        QJob &j = b.job[i];
        j.M = h->E;
        j.Ph = h->Ph;
        j.Qpart = h->Qpart;
        j.Q = h->Q;
        j.counter = h->counters + 2;
        j.m = h->m;
        j.n = h->n;
        j.k = h->k;
        j.kp = h->kp;
        j.ranges = h->q_ranges;
        j.ncb = h->ncb;
        j.task_begin = total;
        total += h->q_ranges * h->ncb;
        kpmax = std::max(kpmax, h->kp);
    }
    b.stage_floats = kQChunk * kQCols + kQChunk * kpmax;
    const size_t smem = sizeof(float) * (size_t)kQStages * b.stage_floats;
    if ((rc = set_smem((const void *)dp_compress_q_kernel, smem))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("dp_compress_q", st, dp_compress_q_kernel<<<total, kThreads, smem, st>>>(b));
    SPECOPTIM_LAUNCHED("dp_compress_q_kernel");
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
    for (int i = 0; i < count; ++i) {
        dpsync *h = hs[i];
        float *p = ptrs ? ptrs[i] : nullptr;
        if (mode == 1 && (!p || !h->have_outer))
            return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": needs W_local and set_outer");
        if (p && !aligned16(p)) return fail(SPECOPTIM_ERR_MISALIGNED, std::string(what) + ": 16-byte alignment");
        UJob &j = b.job[i];
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
        j.tiles_n = (h->n + kTileCols - 1) / kTileCols;
        j.cta_begin = total;
        j.lr = h->cfg.outer_lr;
        j.mu = h->cfg.outer_momentum;
        j.mix = h->cfg.mix;
        total += ((h->m + kTileRows - 1) / kTileRows) * j.tiles_n;
        kpmax = std::max(kpmax, h->kp);
    }
    const size_t smem = sizeof(float) * (size_t)kpmax * (kPsStride + kQsStride);
    if ((rc = set_smem((const void *)dp_update_kernel, smem))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH(mode == 0 ? "dp_decompress" : "dp_outer_step", st,
                dp_update_kernel<<<total, kThreads, smem, st>>>(b));
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
    if (E) SPECOPTIM_CUDA(cudaMemcpyAsync(E, h->E, bytes, cudaMemcpyDeviceToDevice, st));
    if ((theta || mom) && !h->have_outer)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "dpsync_get_state: set_outer was not called");
    if (theta) SPECOPTIM_CUDA(cudaMemcpyAsync(theta, h->theta, bytes, cudaMemcpyDeviceToDevice, st));
    if (mom) SPECOPTIM_CUDA(cudaMemcpyAsync(mom, h->mom, bytes, cudaMemcpyDeviceToDevice, st));
    if (P_hat)
        SPECOPTIM_CUDA(cudaMemcpy2DAsync(P_hat, sizeof(float) * h->k, h->Ph, sizeof(float) * h->kp,
                                         sizeof(float) * h->k, h->m, cudaMemcpyDeviceToDevice, st));
    return SPECOPTIM_OK;
}
