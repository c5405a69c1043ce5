// SVD refresh of the anchor momentum, key design 3 of "Communication-Efficient
// LLM Adaptation over Decentralized GPU Meshes": M = U S V^T and the Tikhonov
// filter d_i = s_i / (s_i + tau_p).
//
// GPU formulation (fp32):
//   1. Gram matrix of the short side, A = M^T M (m >= n) or M M^T (m < n),
//      r x r, zero-padded to Np (a multiple of 128), in fp32-accurate 3xTF32
//      tensor-core products; with a previous factor W the start is W^T A W.
//   2. Block-Jacobi eigen-decomposition A = Q diag(lambda) Q^T.  The Np/32
//      blocks of 32 indices meet in round-robin order; in each round every
//      pair of blocks forms a 64 x 64 subproblem that 256 threads sweep in
//      shared memory (cyclic Jacobi, parallel order; two pairs per CTA),
//      giving a 64 x 64 rotation R_p
//      per pair (R = the block-diagonal of all R_p in the round's order).  The
//      rotations are applied on the tensor cores (3xTF32): A <- R^T A R in one
//      pass over its upper 128 x 128 super-tiles (jacobi_apply_tc.cu), and
//      Q <- Q R (jacobi_tc.cu) on a second stream beside the next solves.
//      Sweeps repeat until the off-diagonal Frobenius norm falls below tol
//      times the total norm.  Padded indices have exactly zero rows and
//      columns, so they are never rotated and stay out of the real eigenvectors.
//   3. The eigenvectors are re-orthonormalised by two Newton-Schulz steps.
//   4. P = M V (or M^T U); s_i = |P e_i| sorted descending, d_i = s_i/(s_i+tau_p),
//      and the long-side factor is P diag(1/s), zero columns where s_i = 0.
// The fp32 Gram squares the condition number; the filter makes that harmless
// (d_i ~ s_i/tau_p for the small directions, so the error of those directions
// enters G_filt multiplied by d_i).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "gemm.cuh"
#include "jacobi.cuh"
#include "svd.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int kMaxBatch = 16;

// All matrices of one batched refresh.  Each matrix i has Np[i] (a multiple of
// 128) padded indices in nb = Np/32 blocks; in its round `round[i]` the blocks
// meet in Np/64 pairs.  The solve kernel takes 256 threads per pair (two pairs
// per CTA), the pairs numbered over the whole batch through pair_off.  R[i] points at the rotation slot of the
// round: per pair, R_p^T split for 3xTF32 (hi block, then lo block, 64 x 64 each).
struct JacBatch {
    int count;
    float *A[kMaxBatch];
    float *R[kMaxBatch];
    int Np[kMaxBatch];
    int round[kMaxBatch];
    int active[kMaxBatch];
    int pair_off[kMaxBatch + 1];
};

__device__ __forceinline__ int find_job(const int *off, int count, int item) {
    int i = 0;
    while (i + 1 < count && item >= off[i + 1]) ++i;
    return i;
}

constexpr int kSolveThreads = 256;  // threads per pair subproblem
// Two pairs per CTA, each 256-thread half with a named barrier of its own: the
// round's solves then hold half as many SMs (88 for the 1B layer's 176 pairs),
// so the Q rotation launched beside them on 3/8 of the SMs finds its SMs free
// (measured: two 256-thread CTAs on one SM run the solve as fast as one).
constexpr int kSolvePairsPerCta = 2;

// barrier of this thread's pair (id 0 is the CTA-wide __syncthreads)
__device__ __forceinline__ void pair_sync() {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + (int)(threadIdx.x / kSolveThreads)), "n"(kSolveThreads) : "memory");
}

// Rotation (c, s) of one pair from approximate reciprocal / square-root
// intrinsics (a few ulp each): c^2 + s^2 = 1 to a few ulp, the same order as
// with correctly rounded operations; the rotation only has to be orthogonal to
// fp32 accuracy and close to the exact Jacobi angle.
__device__ __forceinline__ void jacobi_cs_fast(float app, float aqq, float apq, float &c, float &s) {
    const float theta = __fdividef(aqq - app, 2.f * apq);
    const float at = fabsf(theta);
    const float x = fmaf(theta, theta, 1.f);
    // t = 1 / (|theta| + sqrt(1 + theta^2)); beyond |theta| = 1e18 the square
    // would overflow and t = 1 / (2 |theta|) to fp32 accuracy
    float t = at > 1e18f ? __fdividef(0.5f, at) : __fdividef(1.f, at + x * rsqrtf(x));
    t = copysignf(t, theta);
    c = rsqrtf(fmaf(t, t, 1.f));
    s = t * c;
    if (apq == 0.f) {
        c = 1.f;
        s = 0.f;
    }
}

// The subproblem is kept in "position" order (the circle method of the
// round-robin, with the data moving instead of the indices): positions k (top)
// and 32 + k (bottom) form pair k in every step, and after a step the element
// at position p moves to cat_next(p): top 0 stays, top k -> k + 1, top 31 ->
// bottom 31, bottom k -> k - 1, bottom 0 -> top 1.  The other 63 positions form
// one cycle, so any two indices meet exactly once in the 63 steps of a sweep
// and a sweep ends in the order it started from.
__host__ __device__ __forceinline__ int cat_next(int p) {
    if (p == 0) return 0;
    if (p < kB - 1) return p + 1;
    if (p == kB - 1) return kP - 1;
    if (p == kB) return 1;
    return p - 1;
}

// Physical column of position c in a row of S: bottom positions are rotated by
// two banks, so that for a fixed row the 32 lanes of a warp reading columns l
// or 32 + l, or writing the moved columns cat_next(l) or cat_next(32 + l),
// each touch 32 distinct banks (and so do the reads of the pair entries).
__device__ __forceinline__ int sphys(int c) { return c < kB ? c : kB + ((c - kB + 2) & (kB - 1)); }

constexpr int kSP = kP;  // row pitch of S (every row starts at bank 0)
constexpr int kSBuf = kP * kSP;  // floats per copy of S

// Rotation table of a step: (c, s) of pair k at float2 index cs_index(k).  The
// thread that owns pairs 8m .. 8m+7 reads them as four 16-byte loads; group m
// starts at 64 m + 16 (m / 2) bytes, so the four groups read in one phase of a
// 16-byte load fall in four different bank quads.
constexpr int kCsSlot = 36;  // float2 per slot (4 x 8 entries + skew, 16-byte multiple)
__device__ __forceinline__ int cs_index(int k) { return (k >> 3) * 8 + (k & 7) + ((k >> 4) << 1); }

// 8 warps per pair (half a CTA): load the 64 x 64 subproblem S, run up to
// `inner_sweeps` cyclic Jacobi sweeps (32 disjoint rotations per step) and
// write the accumulated rotation R (64 x 64), split for 3xTF32.
//  * Every warp computes all 32 rotations of a step itself (lane l owns pair
//    l), so the block updates need no barrier and no shared rotation table.
//  * S is double buffered: a step reads one copy and writes the moved blocks
//    into the other, so one barrier per step separates the steps.  Thread
//    (warp w, lane l) updates the 2 x 2 blocks (pair w + 8u rows, pair l
//    columns), u = 0..3, at loop-invariant addresses (the copy a step reads is
//    a template argument, so every access is register + immediate).
//  * R lives in registers: thread (w, l) holds row 8w + l/4 of R, positions of
//    pairs 8m .. 8m+7 (m = l % 4).  After the barrier of a step it applies the
//    step's rotations (from a two-slot table that warp 0 fills) and moves its
//    values to the next positions, exchanging one value with each
//    neighbouring quarter by shuffles.
constexpr size_t kSolveSmem = (2 * (size_t)kSBuf + 2 * 2 * (size_t)kCsSlot) * 4 + 16;
static_assert(kSolveSmem % 16 == 0, "each pair's shared memory starts 16-byte aligned");

struct SolveState {
    float rt[8], rb[8];       // this thread's part of R (top / bottom positions of 8 pairs)
    int rd_t[4], rd_b[4];     // row offsets of the blocks read (pair rows ka, 32 + ka)
    int wr_t[4], wr_b[4];     // row offsets after the move
    int a_pp, a_qq, a_pq;     // pair `lane`'s entries
    int cbot, wct, wcb;       // columns: bottom of `lane`, and both after the move
    int m;
    float offmax, dmax;
};

// One Jacobi step reading copy FROM of S and writing copy 1 - FROM; its
// rotations go to table slot FROM (consecutive steps alternate).
template <int FROM>
__device__ __forceinline__ void solve_step(float *S0, float2 *csb, SolveState &st, int lane, int warp,
                                           bool track) {
    const float *S = S0 + FROM * kSBuf;
    float *Sn = S0 + (1 - FROM) * kSBuf;
    float c, sn;
    {
        const float app = S[st.a_pp], aqq = S[st.a_qq], apq = S[st.a_pq];
        jacobi_cs_fast(app, aqq, apq, c, sn);
        if (track) {
            st.offmax = fmaxf(st.offmax, fabsf(apq));
            st.dmax = fmaxf(st.dmax, fmaxf(fabsf(app), fabsf(aqq)));
        }
    }
    if (warp == 0) csb[FROM * kCsSlot + cs_index(lane)] = make_float2(c, sn);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int ka = warp + 8 * u;
        const float ca = __shfl_sync(0xffffffffu, c, ka), sa = __shfl_sync(0xffffffffu, sn, ka);
        const float x11 = S[st.rd_t[u] + lane], x12 = S[st.rd_t[u] + st.cbot];
        const float x21 = S[st.rd_b[u] + lane], x22 = S[st.rd_b[u] + st.cbot];
        // rows: J_a^T X, then columns: (J_a^T X) J_b
        const float y11 = ca * x11 - sa * x21, y21 = sa * x11 + ca * x21;
        const float y12 = ca * x12 - sa * x22, y22 = sa * x12 + ca * x22;
        float z12 = sn * y11 + c * y12, z21 = c * y21 - sn * y22;
        if (ka == lane) z12 = z21 = 0.f;  // the rotated pair is now decoupled
        Sn[st.wr_t[u] + st.wct] = c * y11 - sn * y12;
        Sn[st.wr_t[u] + st.wcb] = z12;
        Sn[st.wr_b[u] + st.wct] = z21;
        Sn[st.wr_b[u] + st.wcb] = sn * y21 + c * y22;
    }
    pair_sync();
    // R <- R J_step on this thread's pairs, then the positions move on
    const float4 *cs4 = reinterpret_cast<const float4 *>(csb + FROM * kCsSlot + 8 * st.m + 2 * (st.m >> 1));
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float4 w = cs4[h];
        float x = st.rt[2 * h], y = st.rb[2 * h];
        st.rt[2 * h] = w.x * x - w.y * y;
        st.rb[2 * h] = w.y * x + w.x * y;
        x = st.rt[2 * h + 1];
        y = st.rb[2 * h + 1];
        st.rt[2 * h + 1] = w.z * x - w.w * y;
        st.rb[2 * h + 1] = w.w * x + w.z * y;
    }
    const float top_last = st.rt[7], bot_first = st.rb[0];
    const float top_in = __shfl_up_sync(0xffffffffu, top_last, 1);     // quarter m-1, same row
    const float bot_in = __shfl_down_sync(0xffffffffu, bot_first, 1);  // quarter m+1, same row
#pragma unroll
    for (int q = 7; q >= 1; --q) st.rt[q] = st.rt[q - 1];
    if (st.m == 0) {
        st.rt[1] = bot_first;  // bottom 0 -> top 1; top 0 stays (rt[0] unchanged)
    } else {
        st.rt[0] = top_in;
    }
#pragma unroll
    for (int q = 0; q < 7; ++q) st.rb[q] = st.rb[q + 1];
    st.rb[7] = st.m == 3 ? top_last : bot_in;  // top 31 -> bottom 31
}

__device__ void solve_pair(const JacBatch &jb, int item, int inner_sweeps, unsigned char *smem) {
    float *S0 = reinterpret_cast<float *>(smem);
    float2 *csb = reinterpret_cast<float2 *>(S0 + 2 * kSBuf);  // [2][kCsSlot] (c, s) of a step
    float *red = reinterpret_cast<float *>(csb + 2 * kCsSlot);
    const int job = find_job(jb.pair_off, jb.count, item);
    if (!jb.active[job]) return;
    const int Np = jb.Np[job], nb = Np / kB, round = jb.round[job];
    const int pair = item - jb.pair_off[job];
    const float *A = jb.A[job];
    const int tid = threadIdx.x % kSolveThreads, lane = tid & 31, warp = tid >> 5;
    // the subproblem in its start order (position = local index), copy 0
    for (int e = tid; e < kP * (kP / 4); e += kSolveThreads) {
        const int i = e / (kP / 4), j4 = (e % (kP / 4)) * 4;
        const float4 v = *reinterpret_cast<const float4 *>(
            &A[(size_t)pair_index(nb, round, pair, i) * Np + pair_index(nb, round, pair, j4)]);
        S0[i * kSP + sphys(j4)] = v.x;
        S0[i * kSP + sphys(j4 + 1)] = v.y;
        S0[i * kSP + sphys(j4 + 2)] = v.z;
        S0[i * kSP + sphys(j4 + 3)] = v.w;
    }
    SolveState st;
    const int ri = warp * 8 + (lane >> 2);
    st.m = lane & 3;
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // R = I
        st.rt[q] = ri == 8 * st.m + q ? 1.f : 0.f;
        st.rb[q] = ri == kB + 8 * st.m + q ? 1.f : 0.f;
    }
    st.cbot = sphys(kB + lane);
    st.a_pp = lane * kSP + lane;
    st.a_qq = (kB + lane) * kSP + st.cbot;
    st.a_pq = lane * kSP + st.cbot;
    st.wct = sphys(cat_next(lane));
    st.wcb = sphys(cat_next(kB + lane));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int ka = warp + 8 * u;
        st.rd_t[u] = ka * kSP;
        st.rd_b[u] = (kB + ka) * kSP;
        st.wr_t[u] = cat_next(ka) * kSP;
        st.wr_b[u] = cat_next(kB + ka) * kSP;
    }
    pair_sync();
    // A sweep has an odd number of steps (63): the copy holding S alternates
    // between sweeps.  The convergence test only matters with more than one sweep.
    const bool track = inner_sweeps > 1;
    int from = 0;
    for (int sweep = 0; sweep < inner_sweeps; ++sweep) {
        st.offmax = 0.f;
        st.dmax = 0.f;
        if (from == 0) {
            for (int step = 0; step + 1 < kP - 1; step += 2) {
                solve_step<0>(S0, csb, st, lane, warp, track);
                solve_step<1>(S0, csb, st, lane, warp, track);
            }
            solve_step<0>(S0, csb, st, lane, warp, track);
        } else {
            for (int step = 0; step + 1 < kP - 1; step += 2) {
                solve_step<1>(S0, csb, st, lane, warp, track);
                solve_step<0>(S0, csb, st, lane, warp, track);
            }
            solve_step<1>(S0, csb, st, lane, warp, track);
        }
        from ^= 1;
        if (!track) break;
        // stop once no off-diagonal entry rotated in this sweep was above fp32 noise
        if (warp == 0) {
            for (int o = 16; o > 0; o >>= 1) {
                st.offmax = fmaxf(st.offmax, __shfl_xor_sync(0xffffffffu, st.offmax, o));
                st.dmax = fmaxf(st.dmax, __shfl_xor_sync(0xffffffffu, st.dmax, o));
            }
            if (lane == 0) {
                red[0] = st.offmax;
                red[1] = st.dmax;
            }
        }
        pair_sync();
        // red is rewritten only after the next sweep's barriers
        if (red[0] <= 1e-7f * red[1]) break;
    }
    // R_p^T = hi + lo for the tensor-core rotation: R^T[j][k] = R[k][j].  R goes
    // through shared memory (pitch 65, S is no longer read) so that both the
    // staging and the row-wise writes of R^T are coalesced.
    constexpr int kTP = kP + 1;
    float *Rs = S0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        Rs[ri * kTP + 8 * st.m + q] = st.rt[q];
        Rs[ri * kTP + kB + 8 * st.m + q] = st.rb[q];
    }
    pair_sync();
    float *Rp = jb.R[job] + (size_t)pair * 2 * kP * kP;
    for (int e = tid; e < kP * kP / 2; e += kSolveThreads) {
        const int jj = e / (kP / 2), k2 = (e % (kP / 2)) * 2;
        const float x0 = Rs[k2 * kTP + jj], x1 = Rs[(k2 + 1) * kTP + jj];
        float l0, l1;
        const float h0 = tf32_split(x0, l0), h1 = tf32_split(x1, l1);
        *reinterpret_cast<float2 *>(&Rp[jj * kP + k2]) = make_float2(h0, h1);
        *reinterpret_cast<float2 *>(&Rp[kP * kP + jj * kP + k2]) = make_float2(l0, l1);
    }
}

// Subproblem solves of one round: kSolvePairsPerCta pairs per CTA, each on its
// own 256 threads and its own part of shared memory.
__global__ void __launch_bounds__(kSolveThreads * kSolvePairsPerCta)
jacobi_solve_kernel(const JacBatch js, int inner_sweeps, int pairs) {
    extern __shared__ __align__(16) unsigned char solve_smem[];
    // the apply that follows (a programmatic dependent) may set up on SMs this grid leaves
    asm volatile("griddepcontrol.launch_dependents;");
    const int half = threadIdx.x / kSolveThreads, item = blockIdx.x * kSolvePairsPerCta + half;
    if (item >= pairs) return;  // a whole half: it takes part in no barrier
    solve_pair(js, item, inner_sweeps, solve_smem + half * kSolveSmem);
}

__global__ void eye_kernel(float *__restrict__ Q, int Np) {
    const int64_t total = (int64_t)Np * Np;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x)
        Q[e] = (e / Np == e % Np) ? 1.f : 0.f;
}

// Qacc = [W 0; 0 I] with W the previous short-side factor (r x r, row-major)
__global__ void init_q_kernel(float *__restrict__ Q, int Np, int r, const float *__restrict__ W) {
    const int64_t total = (int64_t)Np * Np;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(e / Np), j = (int)(e % Np);
        Q[e] = (i < r && j < r) ? W[(size_t)i * r + j] : (i == j ? 1.f : 0.f);
    }
}

// Sums of squares of A (Np x Np, Np a multiple of 4): out[0] += off-diagonal,
// out[1] += all.  A is a Gram matrix rotated by orthogonal similarities, so no
// entry exceeds its largest diagonal entry in magnitude: each block scales by
// the power of two just above that entry (exact, no overflow, underflow only
// below 2^-75 of it) and sums the scaled squares in fp32 per thread (a few
// hundred terms each); the per-thread sums are combined in double, one pair of
// atomics per block.  fp64 arithmetic, slow on this part, is kept out of the
// per-element loop.  One launch covers the batch: blockIdx.y picks the matrix.
struct OffBatch {
    const float *A[kMaxBatch];
    double *out[kMaxBatch];
    int Np[kMaxBatch];
};

__global__ void __launch_bounds__(256) offnorm_kernel(const OffBatch ob) {
    __shared__ float smax[8];
    __shared__ double sred[2][8];
    const float *__restrict__ A = ob.A[blockIdx.y];
    double *out = ob.out[blockIdx.y];
    const int Np = ob.Np[blockIdx.y];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float dm = 0.f;
    for (int i = tid; i < Np; i += blockDim.x) dm = fmaxf(dm, fabsf(A[(size_t)i * Np + i]));
    for (int o = 16; o > 0; o >>= 1) dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, o));
    if (lane == 0) smax[warp] = dm;
    __syncthreads();
    dm = smax[0];
    for (int w = 1; w < 8; ++w) dm = fmaxf(dm, smax[w]);
    int e = 0;
    frexpf(dm, &e);  // dm = f 2^e, f in [0.5, 1)
    const float sc = (dm > 0.f && isfinite(dm)) ? ldexpf(1.f, -e) : 1.f;
    float off = 0.f, all = 0.f;
    // this block's rows are i = blockIdx.x + r gridDim.x; its float4s are walked
    // flat, four loads in flight per thread
    const int n4 = Np >> 2;
    const int nrows = Np > (int)blockIdx.x ? (Np - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = nrows * n4;
    for (int e0 = tid; e0 < total; e0 += 4 * (int)blockDim.x) {
        float4 v[4];
        int d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * (int)blockDim.x;
            if (e < total) {
                const int r = e / n4, c = e - r * n4;
                const int i = (int)blockIdx.x + r * (int)gridDim.x;
                v[u] = reinterpret_cast<const float4 *>(A + (size_t)i * Np)[c];
                d[u] = i - 4 * c;  // position of the diagonal entry in this float4, if any
            } else {
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                d[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float x = v[u].x * sc, y = v[u].y * sc, z = v[u].z * sc, w = v[u].w * sc;
            const float sx = x * x, sy = y * y, sz = z * z, sw = w * w;
            all += (sx + sy) + (sz + sw);
            off += ((d[u] == 0 ? 0.f : sx) + (d[u] == 1 ? 0.f : sy)) + ((d[u] == 2 ? 0.f : sz) + (d[u] == 3 ? 0.f : sw));
        }
    }
    double doff = off, dall = all;
    for (int o = 16; o > 0; o >>= 1) {
        doff += __shfl_xor_sync(0xffffffffu, doff, o);
        dall += __shfl_xor_sync(0xffffffffu, dall, o);
    }
    if (lane == 0) {
        sred[0][warp] = doff;
        sred[1][warp] = dall;
    }
    __syncthreads();
    if (tid == 0) {
        double so = 0.0, sa = 0.0;
        for (int w = 0; w < 8; ++w) {
            so += sred[0][w];
            sa += sred[1][w];
        }
        atomicAdd(&out[0], so);
        atomicAdd(&out[1], sa);
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

// squared column norms of P (rows x r, row-major) accumulated in double:
// block (x, y) covers 32 columns and a 1/gridDim.y share of the rows
__global__ void __launch_bounds__(256)
colnorm_kernel(const float *__restrict__ P, int64_t rows, int r, double *__restrict__ out2) {
    __shared__ double part[8][33];
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    const int j = blockIdx.x * 32 + tx;
    double acc = 0.0;
    if (j < r)
        for (int64_t i = blockIdx.y * 8 + ty; i < rows; i += (int64_t)gridDim.y * 8) {
            const double v = P[i * r + j];
            acc += v * v;
        }
    part[ty][tx] = acc;
    __syncthreads();
    if (ty == 0 && j < r) {
        double t = 0.0;
        for (int y = 0; y < 8; ++y) t += part[y][tx];
        atomicAdd(&out2[j], t);
    }
}

__global__ void sqrt_kernel(const double *__restrict__ in2, int r, float *__restrict__ out) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < r; j += gridDim.x * blockDim.x)
        out[j] = (float)sqrt(in2[j]);
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

namespace {

int64_t padded_order(int r) { return ((int64_t)(r + kNpAlign - 1) / kNpAlign) * kNpAlign; }

constexpr int kMaps = 3;                         // A (32 x 32 boxes), Q (32 x 128), rotations (32 x 64)
constexpr int64_t kMapFloats = kMaps * 32 + 32;  // 128-byte maps + 128-byte alignment slack

}  // namespace

size_t svd_workspace_floats(int m, int n) {
    const int r = m < n ? m : n, L = m < n ? n : m;
    const int64_t Np = padded_order(r);
    // A, Qacc (Np^2 each), two rotation slots (Np/64 pairs x R^T hi/lo, 64 x 64 each),
    // TMA maps, short factor + scratch (2 r^2), long factor P (L r), s_raw, inv_s,
    // order (int), 2 doubles
    return (size_t)(2 * Np * Np + 2 * (Np / kP) * 2 * kP * kP + kMapFloats + 2 * (int64_t)r * r +
                    (int64_t)L * r + 3 * r + 8);
}

namespace {

struct JobBufs {
    int r, Np, nb;
    int64_t L;
    bool tall;
    float *A, *Qacc, *Rt, *Sf, *Tmp, *P, *s_raw, *inv_s;
    CUtensorMap *maps;  // device: A (32 x 32 boxes), Q (32 x 128), R^T (32 x 64)
    int *order;
    double *norms;
};

JobBufs carve(const SvdJob &a) {
    JobBufs b;
    b.tall = a.m >= a.n;
    b.r = b.tall ? a.n : a.m;
    b.L = b.tall ? a.m : a.n;
    b.Np = (int)padded_order(b.r);
    b.nb = b.Np / kB;
    const size_t NN = (size_t)b.Np * b.Np;
    b.A = a.work;
    b.Qacc = b.A + NN;
    b.Rt = b.Qacc + NN;
    float *mp = b.Rt + (size_t)2 * (b.Np / kP) * 2 * kP * kP;
    b.maps = reinterpret_cast<CUtensorMap *>((reinterpret_cast<uintptr_t>(mp) + 127) & ~uintptr_t(127));
    b.Sf = mp + kMapFloats;
    b.Tmp = b.Sf + (size_t)b.r * b.r;
    b.P = b.Tmp + (size_t)b.r * b.r;
    b.s_raw = b.P + (size_t)b.L * b.r;
    b.inv_s = b.s_raw + b.r;
    b.order = reinterpret_cast<int *>(b.inv_s + b.r);
    b.norms = reinterpret_cast<double *>((reinterpret_cast<uintptr_t>(b.order + b.r) + 15) & ~uintptr_t(15));
    return b;
}

// TMA maps of one matrix's Jacobi tensors, encoded on the host and copied to
// the workspace (the rotation kernel reads them from device memory)
int upload_maps(const JobBufs &b, cudaStream_t st) {
    CUtensorMap h[kMaps];
    int rc;
    const int64_t rot_rows = (int64_t)2 * (b.Np / kP) * 2 * kP;
    if ((rc = make_tmap_2d(&h[0], b.A, b.Np, b.Np, b.Np, kB, kB))) return rc;
    if ((rc = make_tmap_2d(&h[1], b.Qacc, b.Np, b.Np, b.Np, kB, 128))) return rc;
    if ((rc = make_tmap_2d(&h[2], b.Rt, rot_rows, kP, kP, kB, kP))) return rc;
    SPECOPTIM_CUDA(cudaMemcpyAsync(b.maps, h, sizeof(h), cudaMemcpyHostToDevice, st));
    return SPECOPTIM_OK;
}

// Gram matrix of the short side into the padded A, and the starting basis:
// identity, or the previous short-side factor W with A <- W^T A W.
int prepare(const SvdJob &a, const JobBufs &b, cudaStream_t st) {
    SPECOPTIM_CUDA(cudaMemsetAsync(b.A, 0, sizeof(float) * (size_t)b.Np * b.Np, st));
    Epilogue e;
    e.C = b.A;
    e.ldc = b.Np;
    int rc;
    float *ws = nullptr;
    if ((rc = scratch_floats(gemm3_workspace_floats(b.r, b.r, b.L), &ws))) return rc;
    if (b.tall)  // A = M^T M : op(A)(i,k) = M[k][i], op(B)(k,j) = M[k][j]
        rc = gemm_fp32x3(b.r, b.r, a.m, Operand{a.M, a.n, true}, Operand{a.M, a.n, false}, e, ws, st);
    else         // A = M M^T
        rc = gemm_fp32x3(b.r, b.r, a.n, Operand{a.M, a.n, false}, Operand{a.M, a.n, true}, e, ws, st);
    if (rc) return rc;
    const int64_t NN = (int64_t)b.Np * b.Np;
    if (!a.warm) {
        SPCO_LAUNCH("svd_eye", st, eye_kernel<<<grid_for(NN, 256), 256, 0, st>>>(b.Qacc, b.Np));
        SPECOPTIM_LAUNCHED("eye_kernel");
        return SPECOPTIM_OK;
    }
    SPCO_LAUNCH("svd_init_q", st, init_q_kernel<<<grid_for(NN, 256), 256, 0, st>>>(b.Qacc, b.Np, b.r, a.warm));
    SPECOPTIM_LAUNCHED("init_q_kernel");
    Epilogue t;
    t.C = b.Tmp;
    t.ldc = b.r;
    if ((rc = gemm_fp32x3(b.r, b.r, b.r, Operand{b.A, b.Np, false}, Operand{a.warm, b.r, false}, t, ws, st)))
        return rc;  // T = A W
    Epilogue w;
    w.C = b.A;
    w.ldc = b.Np;
    return gemm_fp32x3(b.r, b.r, b.r, Operand{a.warm, b.r, true}, Operand{b.Tmp, b.r, false}, w, ws, st);  // W^T T
}

// re-orthonormalised short factor, s_i = |M v_i| sorted descending, d, long factor
int finish(const SvdJob &a, const JobBufs &b, cudaStream_t st) {
    const int r = b.r;
    const int64_t rr = (int64_t)r * r, L = b.L;
    int rc;
    float *ws = nullptr;
    if ((rc = scratch_floats(std::max(gemm3_workspace_floats(r, r, r), gemm3_workspace_floats(L, r, b.tall ? a.n : a.m)), &ws)))
        return rc;
    SPCO_LAUNCH("svd_extract", st, extract_kernel<<<grid_for(rr, 256), 256, 0, st>>>(b.Qacc, b.Np, r, b.Sf));
    SPECOPTIM_LAUNCHED("extract_kernel");
    // two Newton-Schulz steps X <- X (3 I - X^T X) / 2 remove the drift that the
    // fp32 rotations leave in the accumulated eigenvectors
    for (int it = 0; it < 2; ++it) {
        Epilogue g;
        g.C = b.A;  // X^T X (r x r, ld r) reuses the Gram buffer
        g.ldc = r;
        if ((rc = gemm_fp32x3(r, r, r, Operand{b.Sf, r, true}, Operand{b.Sf, r, false}, g, ws, st))) return rc;
        Epilogue t;
        t.C = b.Tmp;
        t.ldc = r;
        if ((rc = gemm_fp32x3(r, r, r, Operand{b.Sf, r, false}, Operand{b.A, r, false}, t, ws, st))) return rc;
        SPCO_LAUNCH("svd_ns_update", st, ns_update_kernel<<<grid_for(rr, 256), 256, 0, st>>>(b.Sf, b.Tmp, rr));
        SPECOPTIM_LAUNCHED("ns_update_kernel");
    }
    Epilogue f;
    f.C = b.P;
    f.ldc = r;
    if (b.tall)
        rc = gemm_fp32x3(L, r, a.n, Operand{a.M, a.n, false}, Operand{b.Sf, r, false}, f, ws, st);
    else
        rc = gemm_fp32x3(L, r, a.m, Operand{a.M, a.n, true}, Operand{b.Sf, r, false}, f, ws, st);
    if (rc) return rc;
    // squared norms in double, in the (now free) Gram buffer
    double *norm2 = reinterpret_cast<double *>(b.A);
    SPECOPTIM_CUDA(cudaMemsetAsync(norm2, 0, sizeof(double) * (size_t)r, st));
    {
        const dim3 grid((unsigned)((r + 31) / 32), (unsigned)std::max<int64_t>(1, std::min<int64_t>(L / 64, 64)));
        SPCO_LAUNCH("svd_colnorm", st, colnorm_kernel<<<grid, 256, 0, st>>>(b.P, L, r, norm2));
        SPCO_LAUNCH("svd_colnorm", st, sqrt_kernel<<<grid_for(r, 128), 128, 0, st>>>(norm2, r, b.s_raw));
    }
    SPCO_LAUNCH("svd_rank", st, rank_kernel<<<grid_for(r, 128), 128, 0, st>>>(b.s_raw, r, b.order));
    SPCO_LAUNCH("svd_spectrum", st, spectrum_kernel<<<grid_for(r, 128), 128, 0, st>>>(b.s_raw, r, b.order, a.tau, a.s, a.d, b.inv_s));
    float *short_out = b.tall ? a.V : a.U;
    float *long_out = b.tall ? a.U : a.V;
    SPCO_LAUNCH("svd_permute", st, permute_cols_kernel<<<grid_for(rr, 256), 256, 0, st>>>(b.Sf, r, r, b.order, nullptr, short_out));
    SPCO_LAUNCH("svd_permute", st, permute_cols_kernel<<<grid_for(L * r, 256), 256, 0, st>>>(b.P, L, r, b.order, b.inv_s, long_out));
    SPECOPTIM_LAUNCHED("svd spectrum kernels");
    return SPECOPTIM_OK;
}

}  // namespace

int set_solve_attributes() {
    return set_smem_limit(reinterpret_cast<const void *>(&jacobi_solve_kernel), kSolvePairsPerCta * kSolveSmem);
}

// Streams and events of one refresh call's Jacobi loop (created per call: a few
// tens of microseconds against a refresh of many milliseconds, and concurrent
// refreshes on different streams stay independent; released when the call
// returns, which the driver defers until their work completed).
struct JacStreams {
    cudaStream_t hi = nullptr, lo = nullptr;
    cudaEvent_t a_done[2] = {}, q_done[2] = {}, ev = nullptr, norms = nullptr;
    ~JacStreams() {
        for (int k = 0; k < 2; ++k) {
            if (a_done[k]) cudaEventDestroy(a_done[k]);
            if (q_done[k]) cudaEventDestroy(q_done[k]);
        }
        if (ev) cudaEventDestroy(ev);
        if (norms) cudaEventDestroy(norms);
        if (hi) cudaStreamDestroy(hi);
        if (lo) cudaStreamDestroy(lo);
    }
    // both chains start after the caller's stream's earlier work
    int create(cudaStream_t st) {
        int least = 0, greatest = 0;
        SPECOPTIM_CUDA(cudaDeviceGetStreamPriorityRange(&least, &greatest));
        for (int k = 0; k < 2; ++k) {
            SPECOPTIM_CUDA(cudaEventCreateWithFlags(&a_done[k], cudaEventDisableTiming));
            SPECOPTIM_CUDA(cudaEventCreateWithFlags(&q_done[k], cudaEventDisableTiming));
        }
        SPECOPTIM_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
        SPECOPTIM_CUDA(cudaEventCreateWithFlags(&norms, cudaEventDisableTiming));
        SPECOPTIM_CUDA(cudaStreamCreateWithPriority(&hi, cudaStreamNonBlocking, greatest));
        SPECOPTIM_CUDA(cudaStreamCreateWithPriority(&lo, cudaStreamNonBlocking, least));
        SPECOPTIM_CUDA(cudaEventRecord(ev, st));
        SPECOPTIM_CUDA(cudaStreamWaitEvent(hi, ev, 0));
        SPECOPTIM_CUDA(cudaStreamWaitEvent(lo, ev, 0));
        for (int k = 0; k < 2; ++k) SPECOPTIM_CUDA(cudaEventRecord(q_done[k], lo));
        return SPECOPTIM_OK;
    }
    // the caller's stream resumes once both chains are done
    int join(cudaStream_t st) {
        SPECOPTIM_CUDA(cudaEventRecord(ev, lo));
        SPECOPTIM_CUDA(cudaStreamWaitEvent(st, ev, 0));
        SPECOPTIM_CUDA(cudaEventRecord(ev, hi));
        SPECOPTIM_CUDA(cudaStreamWaitEvent(st, ev, 0));
        return SPECOPTIM_OK;
    }
};

// One batched refresh in flight: its jobs, buffers and streams, and (for the
// asynchronous form) the library thread that runs its sweep loop.
struct SvdRun {
    int count = 0;
    SvdJob jobs[kMaxBatch];
    JobBufs b[kMaxBatch];
    JacStreams js;
    cudaEvent_t done = nullptr;  // recorded on `hi` once both chains' last kernels are queued
    std::thread worker;
    int device = 0;
    int rc = SPECOPTIM_OK;
    std::string err;
    ~SvdRun() {
        if (done) cudaEventDestroy(done);
    }
};

namespace {

std::atomic<bool> g_run_active{false};

// pinned host slots for the convergence test's sums (one run at a time)
double *host_sums() {
    static double *p = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        if (cudaMallocHost(reinterpret_cast<void **>(&p), 2 * kMaxBatch * sizeof(double)) != cudaSuccess)
            p = nullptr;
    });
    return p;
}

// Gram matrices and the Jacobi sweeps of every job, on the run's two streams.
int sweep_loop(SvdRun &R) {
    const int count = R.count;
    SvdJob *jobs = R.jobs;
    JobBufs *b = R.b;
    cudaStream_t hi = R.js.hi, lo = R.js.lo;
    int rc;
    for (int i = 0; i < count; ++i)
        if ((rc = prepare(jobs[i], b[i], hi))) return rc;
    JacBatch jb;
    std::memset(&jb, 0, sizeof(jb));
    jb.count = count;
    int max_sweeps = 1, rounds = 1;
    ApJob ajob[kMaxBatch];
    CtJob qjob[kMaxBatch];
    for (int i = 0; i < count; ++i) {
        if ((rc = upload_maps(b[i], hi))) return rc;
        jb.A[i] = b[i].A;
        jb.Np[i] = b[i].Np;
        jb.active[i] = 1;
        jb.pair_off[i + 1] = jb.pair_off[i] + b[i].Np / kP;
        max_sweeps = std::max(max_sweeps, jobs[i].max_sweeps);
        rounds = std::max(rounds, b[i].nb - 1);
        const CUtensorMap *m = b[i].maps;
        // A <- R^T A R (two-sided, upper super-tiles) and Q <- Q R
        ajob[i] = ApJob{&m[0], &m[2], b[i].A, b[i].Np, 0, 0, 1};
        qjob[i] = CtJob{&m[1], &m[1], &m[2], b[i].Np, 0, 0, 0, 1};
    }
    const int solve_grid = jb.pair_off[count];
    // the apply starts as a programmatic dependent of the solve only while the
    // solve's CTAs fit one per SM beside the Q rotation (measured: with more,
    // e.g. a 14-matrix or a 7B-shaped batch, the early apply CTAs cost more
    // than the launch they hide)
    const int q_ctas = num_sms() * 3 / 8;
    const bool apply_after_solve = (solve_grid + kSolvePairsPerCta - 1) / kSolvePairsPerCta <= num_sms() - q_ctas;
    int inner = 1;
    for (int i = 0; i < count; ++i) inner = std::max(inner, jobs[i].inner_sweeps);
    if ((rc = set_solve_attributes())) return rc;
    auto set_round = [&](long g) {
        for (int i = 0; i < count; ++i) {
            const int round = (int)(g % (b[i].nb - 1));
            jb.round[i] = round;
            const int slot = (int)(g & 1);
            jb.R[i] = b[i].Rt + (size_t)slot * (b[i].Np / kP) * 2 * kP * kP;
            ajob[i].slot = qjob[i].slot = slot;
            ajob[i].round = qjob[i].round = round;
            ajob[i].active = qjob[i].active = jb.active[i];
        }
    };
    // Two chains.  `hi` (highest priority): solve(g) -> A <- R^T A R -> solve(g+1)
    // ...; `lo`: Q <- Q R for round g, released with solve(g+1) (which does not
    // need it) so that the two share the SMs.  Rotations of round g live in
    // slot g % 2; solve(g+1) rewrites the slot of round g-1 once Q(g-1) read it.
    JacStreams &js_ = R.js;
    auto solve = [&](long gg) -> int {
        set_round(gg);
        SPECOPTIM_CUDA(cudaStreamWaitEvent(hi, js_.q_done[gg & 1], 0));
        SPCO_LAUNCH("svd_jacobi_solve", hi,
                    jacobi_solve_kernel<<<(solve_grid + kSolvePairsPerCta - 1) / kSolvePairsPerCta,
                                          kSolveThreads * kSolvePairsPerCta, kSolvePairsPerCta * kSolveSmem, hi>>>(
                        jb, inner, solve_grid));
        SPECOPTIM_LAUNCHED("jacobi_solve_kernel");
        return SPECOPTIM_OK;
    };
    // the convergence test's sums land in pinned host memory, so the copies stay
    // asynchronous and the host waits on an event, not on the stream
    double *host = host_sums();
    if (!host) return fail(SPECOPTIM_ERR_CUDA, "svd_refresh: pinned host memory for the convergence test");
    int active = count;
    long g = 0;
    if ((rc = solve(0))) return rc;
    for (int sweep = 0; sweep < max_sweeps && active > 0; ++sweep) {
        for (int k = 0; k < rounds; ++k, ++g) {
            set_round(g);
            if ((rc = jacobi_apply(ajob, count, hi, apply_after_solve))) return rc;
            SPECOPTIM_CUDA(cudaEventRecord(js_.a_done[g & 1], hi));
            SPECOPTIM_CUDA(cudaStreamWaitEvent(lo, js_.a_done[g & 1], 0));
            // on 3/8 of the SMs: the solves take the rest, and the next round's
            // rotation of A finds SMs free sooner (measured best among 1/4 .. all)
            if ((rc = jacobi_rotate(qjob, count, lo, q_ctas))) return rc;
            SPECOPTIM_CUDA(cudaEventRecord(js_.q_done[g & 1], lo));
            // the sweep's last solve (the next sweep's first) goes after the convergence test
            if (k + 1 < rounds && (rc = solve(g + 1))) return rc;
        }
        SPECOPTIM_LAUNCHED("jacobi sweep");
        // convergence test of the active matrices: one launch, then the next
        // sweep's first solve runs while the host waits for the sums
        OffBatch ob;
        int nt = 0, max_np = 0;
        for (int i = 0; i < count; ++i) {
            if (!jb.active[i]) continue;
            jobs[i].sweeps = sweep + 1;
            SPECOPTIM_CUDA(cudaMemsetAsync(b[i].norms, 0, 2 * sizeof(double), hi));
            ob.A[nt] = b[i].A;
            ob.out[nt] = b[i].norms;
            ob.Np[nt] = b[i].Np;
            max_np = std::max(max_np, b[i].Np);
            ++nt;
        }
        if (nt == 0) break;  // unreachable: the loop runs only while a matrix is active
        const dim3 ogrid((unsigned)std::max(1, std::min(max_np, (2 * num_sms() + nt - 1) / nt)), (unsigned)nt);
        SPCO_LAUNCH("svd_offnorm", hi, offnorm_kernel<<<ogrid, 256, 0, hi>>>(ob));
        SPECOPTIM_LAUNCHED("offnorm_kernel");
        for (int i = 0; i < count; ++i)
            if (jb.active[i])
                SPECOPTIM_CUDA(cudaMemcpyAsync(&host[2 * i], b[i].norms, 2 * sizeof(double),
                                               cudaMemcpyDeviceToHost, hi));
        SPECOPTIM_CUDA(cudaEventRecord(js_.norms, hi));
        if ((rc = solve(g))) return rc;
        SPECOPTIM_CUDA(cudaEventSynchronize(js_.norms));
        for (int i = 0; i < count; ++i) {
            if (!jb.active[i]) continue;
            const double tol = jobs[i].tol;
            int now_active = 1;
            if (host[2 * i] <= tol * tol * host[2 * i + 1]) {
                now_active = 0;
            } else if (jobs[i].sweeps >= jobs[i].max_sweeps) {
                now_active = 0;
                jobs[i].status = SPECOPTIM_ERR_NOT_CONVERGED;
            }
            if (!now_active) {
                jb.active[i] = 0;
                --active;
            }
        }
    }
    for (int i = 0; i < count; ++i)
        if (jb.active[i]) jobs[i].status = SPECOPTIM_ERR_NOT_CONVERGED;
    return SPECOPTIM_OK;
}

// the run's loop, then `done` after both chains (also after a failure, so that
// the caller can still order its stream after whatever was queued)
void run_loop(SvdRun *R) {
    R->rc = sweep_loop(*R);
    if (R->rc) R->err = specoptim_last_error();
    if (cudaEventRecord(R->js.ev, R->js.lo) != cudaSuccess ||
        cudaStreamWaitEvent(R->js.hi, R->js.ev, 0) != cudaSuccess ||
        cudaEventRecord(R->done, R->js.hi) != cudaSuccess) {
        if (!R->rc) {
            R->rc = SPECOPTIM_ERR_CUDA;
            R->err = "svd_refresh: recording the end of the sweeps failed";
        }
    }
}

}  // namespace

int svd_refresh_start(const SvdJob *jobs, int count, cudaStream_t st, bool async, SvdRun **out) {
    *out = nullptr;
    if (count < 1 || count > kMaxBatch)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_refresh: 1 to 16 matrices per batch");
    bool expected = false;
    if (!g_run_active.compare_exchange_strong(expected, true))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_refresh: another refresh is in progress in this process "
                                               "(finish it with specoptim_svd_refresh_end first)");
    SvdRun *R = new SvdRun();
    R->count = count;
    int rc = SPECOPTIM_OK;
    size_t need = 0;
    for (int i = 0; i < count; ++i) {
        R->jobs[i] = jobs[i];
        R->jobs[i].sweeps = 0;
        R->jobs[i].status = SPECOPTIM_OK;
        R->b[i] = carve(R->jobs[i]);
        need = std::max(need, gemm3_workspace_floats(R->b[i].r, R->b[i].r, R->b[i].L));
    }
    float *ws = nullptr;
    // the Gram products' scratch is grown here, on the calling thread, so that the
    // sweep thread never reallocates it
    if (!rc) rc = scratch_floats(need, &ws);
    if (!rc) rc = cudaGetDevice(&R->device) == cudaSuccess ? R->js.create(st) : fail(SPECOPTIM_ERR_CUDA, "cudaGetDevice");
    if (!rc && cudaEventCreateWithFlags(&R->done, cudaEventDisableTiming) != cudaSuccess)
        rc = fail(SPECOPTIM_ERR_CUDA, "svd_refresh: cudaEventCreate");
    if (rc) {
        delete R;
        g_run_active.store(false);
        return rc;
    }
    if (async) {
        try {
            R->worker = std::thread([R] {
                if (cudaSetDevice(R->device) != cudaSuccess) {
                    R->rc = SPECOPTIM_ERR_CUDA;
                    R->err = "svd_refresh: cudaSetDevice on the sweep thread failed";
                    cudaEventRecord(R->done, R->js.hi);
                    return;
                }
                run_loop(R);
            });
        } catch (...) {
            run_loop(R);  // no thread could be started: run the loop here
        }
    } else {
        run_loop(R);
    }
    *out = R;
    return SPECOPTIM_OK;
}

int svd_refresh_complete(SvdRun *R, SvdJob *jobs, cudaStream_t st) {
    if (R->worker.joinable()) R->worker.join();
    int rc = R->rc;
    std::string err = R->err;
    if (cudaStreamWaitEvent(st, R->done, 0) != cudaSuccess && !rc) {
        rc = SPECOPTIM_ERR_CUDA;
        err = "svd_refresh: ordering the stream after the sweeps failed";
    }
    const int count = R->count;
    int first_bad = SPECOPTIM_OK;
    for (int i = 0; i < count && !rc; ++i) {
        jobs[i].sweeps = R->jobs[i].sweeps;
        jobs[i].status = R->jobs[i].status;
        if (jobs[i].status != SPECOPTIM_OK) {
            if (!first_bad) first_bad = jobs[i].status;
            continue;
        }
        if ((rc = finish(R->jobs[i], R->b[i], st))) err = specoptim_last_error();
    }
    delete R;  // the streams go once their queued work is done
    g_run_active.store(false);
    if (rc) return fail(rc, err);
    if (first_bad)
        return fail(first_bad, "svd_refresh: Jacobi did not reach svd_tol within svd_max_sweeps; "
                               "previous factors kept for the matrices concerned");
    return SPECOPTIM_OK;
}

int svd_refresh_batch(SvdJob *jobs, int count, cudaStream_t st) {
    SvdRun *R = nullptr;
    int rc = svd_refresh_start(jobs, count, st, false, &R);
    if (rc) return rc;
    return svd_refresh_complete(R, jobs, st);
}

}  // namespace spco
