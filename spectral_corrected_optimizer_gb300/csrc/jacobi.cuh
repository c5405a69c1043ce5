// Block-Jacobi eigen-solver of the SVD refresh: the round-robin schedule and
// the tensor-core rotation kernel shared by svd.cu and jacobi_tc.cu.
//
// The padded order Np (a multiple of 128) is cut into nb = Np/32 blocks of 32
// indices.  In round k the blocks meet in Np/64 pairs (round-robin over nb
// players); pair p of round k owns the 64 indices of its two blocks.  Each
// round rotates every pair's 64 x 64 subproblem by an orthogonal R_p.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace spco {

constexpr int kB = 32;      // block size of the block-Jacobi
constexpr int kP = 2 * kB;  // subproblem size (one pair of blocks)
constexpr int kNpAlign = 128;  // Np granularity: whole 128-row slabs for the rotation kernel

// 3xTF32 operand split x = hi + lo: hi is x rounded to the 10 explicit mantissa
// bits of TF32, to nearest with ties away from zero (half a unit of the 13
// dropped bits is added to the magnitude, then they are cleared; for finite x
// below the largest float), and lo = x - hi (exact) rounded the same way.  The
// tensor core reads the top 19 bits of each.  Integer operations only.
__device__ __forceinline__ float tf32_round(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}
__device__ __forceinline__ float tf32_split(float x, float &lo) {
    const float hi = tf32_round(x);
    lo = tf32_round(x - hi);
    return hi;
}

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

// global index of local index l (0..63) of pair p of the given round (nb blocks)
__host__ __device__ __forceinline__ int pair_index(int nb, int round, int p, int l) {
    int a, b;
    rr_pair(nb, round, p, a, b);
    return (l < kB ? a : b) * kB + (l & (kB - 1));
}

// One matrix of a rotation launch:  OUT[rows, cols(p)] = IN[rows, cols(p)] . R_p
// for every 128-row slab and every pair p of round `round` (cols(p) = the 64
// indices of pair p), or, with `transposed`, OUT[cols(p), rows] = that product
// transposed.  R_p comes pre-split for 3xTF32 as R_p^T = hi + lo (two 64 x 64
// row-major fp32 blocks, hi then lo) at row ((slot * Np/64 + p) * 2) * 64 of
// the rotation tensor.  All three tensors are reached through TMA maps that
// live in device memory: `in` and `out` with boxes of 32 columns x 128 rows
// (transposed output: 32 x 32), `rot` with 32 x 64.  OUT may be IN itself
// (every task reads and writes only its own slab and pair).
struct CtJob {
    const CUtensorMap *in, *out, *rot;
    int Np, round, slot, transposed, active;
};

constexpr int kCtMaxJobs = 32;

// One matrix of a two-sided rotation launch (jacobi_apply_tc.cu): A <- R^T A R
// in place for round `round`, A symmetric Np x Np (row-major, leading
// dimension Np).  `a32` is a TMA map of A with 32 x 32 boxes, `rot` the
// rotation tensor's map (rotations of the round in slot `slot`, as for CtJob).
struct ApJob {
    const CUtensorMap *a32, *rot;
    float *A;
    int Np, round, slot, active;
};

constexpr int kApMaxJobs = 16;

// Launches the two-sided rotation of `count` (<= 16) matrices in one kernel;
// `after_solve`: as a programmatic dependent of the solve launched just before
// it on `st` (the kernel waits for that solve's results before reading A).
int jacobi_apply(const ApJob *jobs, int count, cudaStream_t st, bool after_solve = false);

// Launches the rotation of `count` (<= 32) matrices in one kernel on at most
// `max_ctas` SMs (0: all of them).
int jacobi_rotate(const CtJob *jobs, int count, cudaStream_t st, int max_ctas = 0);

}  // namespace spco
