// The activation mask's index function g, shared by the mask kernels and the
// mask ops fused with the layer boundary.
//
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
// key design 1: row r keeps pi_r(0..K-1) of a keyed permutation pi_r of
// [0, H), built from four alternating Feistel rounds over ceil(log2 H) bits
// with MurmurHash3's fmix32 as round function and SplitMix64-derived round
// keys; values >= H are walked on through the permutation's cycle.
#pragma once

#include <stdint.h>

namespace spco {

// ---- g: keyed permutation ---------------------------------------------------

__host__ __device__ __forceinline__ uint64_t splitmix_out(uint64_t state) {
    uint64_t z = state + 0x9e3779b97f4a7c15ULL;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t murmur_fmix(uint32_t x) {
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}

struct RowKeys {
    uint32_t k[4];
};

__device__ __forceinline__ RowKeys row_keys(uint64_t seed, uint64_t row) {
    uint64_t rk = splitmix_out(seed ^ row);
    RowKeys out;
#pragma unroll
    for (int i = 0; i < 4; ++i) out.k[i] = static_cast<uint32_t>(splitmix_out(rk + (uint64_t)i));
    return out;
}

// permutation geometry for a given H
struct PermShape {
    uint32_t H;
    int lo_bits;
    uint32_t hi_mask, lo_mask;
    uint32_t walk_limit;
};

__host__ __device__ inline PermShape perm_shape(uint32_t H) {
    int w = 0;
    while ((1ull << w) < (unsigned long long)H) ++w;
    PermShape s;
    s.H = H;
    s.lo_bits = w - w / 2;
    s.hi_mask = (1u << (w / 2)) - 1u;
    s.lo_mask = (1u << s.lo_bits) - 1u;
    s.walk_limit = 1u << w;
    return s;
}

__device__ __forceinline__ uint32_t feistel4(const RowKeys &key, const PermShape &ps, uint32_t x) {
    uint32_t lo = x & ps.lo_mask;
    uint32_t hi = x >> ps.lo_bits;
    hi ^= murmur_fmix(lo ^ key.k[0]) & ps.hi_mask;
    lo ^= murmur_fmix(hi ^ key.k[1]) & ps.lo_mask;
    hi ^= murmur_fmix(lo ^ key.k[2]) & ps.hi_mask;
    lo ^= murmur_fmix(hi ^ key.k[3]) & ps.lo_mask;
    return (hi << ps.lo_bits) | lo;
}

// pi_r(k): the k-th kept dim of the row (cycle walking bounded by the domain size)
__device__ __forceinline__ uint32_t kept_dim(const RowKeys &key, const PermShape &ps, uint32_t k) {
    uint32_t x = feistel4(key, ps, k);
    for (uint32_t g = 0; x >= ps.H && g < ps.walk_limit; ++g) x = feistel4(key, ps, x);
    return x;
}

// Flag value of a failed index check in the checked build (bit 31 set, the
// check's site number in the low bits).
constexpr unsigned kBoundsFlag = 0x80000000u;

// kept_dim as an index into a row of H values.  The checked build
// (-DSPECOPTIM_CHECK, for tests) verifies j < H -- the permutation's output
// after cycle walking -- records a failure in *flag with its site number and
// returns 0 instead, so the access it feeds stays inside the row; the normal
// build returns kept_dim unchanged.
__device__ __forceinline__ uint32_t kept_index(const RowKeys &key, const PermShape &ps, uint32_t k,
                                               unsigned *flag, unsigned site) {
    const uint32_t j = kept_dim(key, ps, k);
#ifdef SPECOPTIM_CHECK
    if (j >= ps.H) {
        if (flag) atomicCAS(flag, 0u, kBoundsFlag | site);
        return 0u;
    }
#else
    (void)flag;
    (void)site;
#endif
    return j;
}

// seed of one (layer, step, batch) boundary
__host__ __device__ inline uint64_t mask_seed(uint32_t layer, uint64_t step, uint64_t batch_id) {
    return splitmix_out(splitmix_out(splitmix_out((uint64_t)layer) ^ step) ^ batch_id);
}


}  // namespace spco
