// The activation mask fused with the ops at a pipeline-stage boundary
// (include/mask_fused.h): pack of the residual sum on the sender, unpack +
// RMSNorm on the receiver, RMSNorm backward + pack on the receiver, unpack-add
// into the residual gradient on the sender.
//
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
// key design 1: only the K kept dims of each token travel, chosen by the
// shared function g (mask_g.cuh) in both directions.
//
// One warp per row.  The ops that read dense tensors only at the kept dims
// (pack_add, rmsnorm_backward_pack, unpack_add) gather those elements straight
// from global memory: at K/H = 0.05 a row touches about 56 % of its 32-byte
// sectors, which is all the DRAM traffic they cost.  unpack_rmsnorm writes two
// dense rows: each warp builds them in shared memory (zero-fill + scatter) and
// stores them with 16-byte coalesced stores.
#include <algorithm>
#include <string>

#include "../../include/mask_fused.h"
#include "common.cuh"
#include "mask_g.cuh"

namespace spco {
namespace {

constexpr int kWarps = 8;
constexpr int kThreadsF = kWarps * 32;

__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// float -> bf16 bits, nearest with ties to even; NaN -> 0x7FC0
__device__ __forceinline__ uint16_t bf16_rne(float x) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7FC0;
    return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Gathers at the kept dims take them in batches of kBatch per lane: all the
// batch's indices are hashed first, then all its loads are issued, so each lane
// keeps kBatch independent loads in flight per tensor.
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kThreadsF) pack_add_kernel(const uint16_t *__restrict__ a, const uint16_t *__restrict__ b,
                                                           uint16_t *__restrict__ packed, int64_t rows, int H,
                                                           int K, uint64_t seed, unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    const int lane = threadIdx.x & 31;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < rows; r += (int64_t)gridDim.x * kWarps) {
        const RowKeys key = row_keys(seed, (uint64_t)r);
        const uint16_t *ar = a + r * H, *br = b + r * H;
        for (int k0 = 0; k0 < K; k0 += 32 * kBatch) {
            uint32_t j[kBatch];
            uint16_t va[kBatch], vb[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                j[u] = k < K ? kept_index(key, ps, (uint32_t)k, flag, 6u) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const bool in = k0 + 32 * u + lane < K;
                va[u] = in ? __ldg(ar + j[u]) : (uint16_t)0;
                vb[u] = in ? __ldg(br + j[u]) : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                if (k < K) packed[r * K + k] = bf16_rne(bf16_val(va[u]) + bf16_val(vb[u]));
            }
        }
    }
}

__global__ void __launch_bounds__(kThreadsF) unpack_rmsnorm_kernel(const uint16_t *__restrict__ packed,
                                                                 const uint16_t *__restrict__ gamma, float eps,
                                                                 uint16_t *__restrict__ h_out,
                                                                 uint16_t *__restrict__ x_out, int64_t rows,
                                                                 int H, int K, uint64_t seed, int warps,
                                                                 unsigned *flag) {
    extern __shared__ __align__(16) uint16_t rowbuf[];  // per warp: h row, x row (H + pad each)
    const PermShape ps = perm_shape((uint32_t)H);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w >= warps) return;
    const int stride = (H + 7) & ~7;  // 16-byte multiple
    uint16_t *hb = rowbuf + (size_t)w * 2 * stride, *xb = hb + stride;
    const float inv_h = 1.f / (float)H;
    for (int64_t r = (int64_t)blockIdx.x * warps + w; r < rows; r += (int64_t)gridDim.x * warps) {
        const uint16_t *pr = packed + r * K;
        float ss = 0.f;
        for (int k = lane; k < K; k += 32) {
            const float v = bf16_val(__ldg(pr + k));
            ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        const float rinv = 1.f / sqrtf(fmaf(ss, inv_h, eps));
        // zero both rows (16 bytes per lane-step), then scatter the kept dims
        uint4 *h4 = reinterpret_cast<uint4 *>(hb), *x4 = reinterpret_cast<uint4 *>(xb);
        for (int i = lane; i < stride / 8; i += 32) h4[i] = x4[i] = make_uint4(0, 0, 0, 0);
        __syncwarp();
        const RowKeys key = row_keys(seed, (uint64_t)r);
        for (int k = lane; k < K; k += 32) {
            const uint32_t j = kept_index(key, ps, (uint32_t)k, flag, 7u);
            const uint16_t p = __ldg(pr + k);
            hb[j] = p;
            xb[j] = bf16_rne(bf16_val(p) * rinv * bf16_val(__ldg(gamma + j)));
        }
        __syncwarp();
        uint16_t *ho = h_out + r * H, *xo = x_out + r * H;
        if ((H & 7) == 0 && ((reinterpret_cast<uintptr_t>(h_out) | reinterpret_cast<uintptr_t>(x_out)) & 15) == 0) {
            uint4 *ho4 = reinterpret_cast<uint4 *>(ho), *xo4 = reinterpret_cast<uint4 *>(xo);
            for (int i = lane; i < H / 8; i += 32) {
                __stcs(ho4 + i, h4[i]);
                __stcs(xo4 + i, x4[i]);
            }
        } else {
            for (int i = lane; i < H; i += 32) {
                ho[i] = hb[i];
                xo[i] = xb[i];
            }
        }
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kThreadsF) rmsnorm_bwd_pack_kernel(const uint16_t *__restrict__ packed_h,
                                                                   const uint16_t *__restrict__ gamma, float eps,
                                                                   const uint16_t *__restrict__ dx,
                                                                   const uint16_t *__restrict__ g_res,
                                                                   uint16_t *__restrict__ out, int64_t rows, int H,
                                                                   int K, uint64_t seed, unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    const int lane = threadIdx.x & 31;
    const float inv_h = 1.f / (float)H;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < rows; r += (int64_t)gridDim.x * kWarps) {
        const RowKeys key = row_keys(seed, (uint64_t)r);
        const uint16_t *pr = packed_h + r * K, *dr = dx + r * H;
        const uint16_t *gr = g_res ? g_res + r * H : nullptr;
        if (K <= 32 * kBatch) {
            // one batch: the kept dims' operands stay in registers between the two passes
            uint32_t j[kBatch];
            float hv[kBatch], gd[kBatch], rv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = 32 * u + lane;
                j[u] = k < K ? kept_index(key, ps, (uint32_t)k, flag, 8u) : 0u;
            }
            float ss = 0.f, s = 0.f;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = 32 * u + lane;
                const bool in = k < K;
                hv[u] = in ? bf16_val(__ldg(pr + k)) : 0.f;
                gd[u] = in ? bf16_val(__ldg(gamma + j[u])) * bf16_val(__ldg(dr + j[u])) : 0.f;
                rv[u] = (in && gr) ? bf16_val(__ldg(gr + j[u])) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                ss = fmaf(hv[u], hv[u], ss);
                s = fmaf(gd[u], hv[u], s);
            }
            ss = warp_sum(ss);
            s = warp_sum(s);
            const float rr = sqrtf(fmaf(ss, inv_h, eps)), rinv = 1.f / rr;
            const float c = s * inv_h * rinv * rinv * rinv;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = 32 * u + lane;
                if (k < K) out[r * K + k] = bf16_rne(gd[u] * rinv - hv[u] * c + rv[u]);
            }
            continue;
        }
        // pass 1: mean of squares of h~ and sum_i gamma_i dx_i h~_i over the kept dims
        float ss = 0.f, s = 0.f;
        for (int k0 = 0; k0 < K; k0 += 32 * kBatch) {
            uint32_t j[kBatch];
            uint16_t hv[kBatch], gv[kBatch], dv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                j[u] = k < K ? kept_index(key, ps, (uint32_t)k, flag, 8u) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                const bool in = k < K;
                hv[u] = in ? __ldg(pr + k) : (uint16_t)0;
                gv[u] = in ? __ldg(gamma + j[u]) : (uint16_t)0;
                dv[u] = in ? __ldg(dr + j[u]) : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const float h = bf16_val(hv[u]);
                ss = fmaf(h, h, ss);
                s = fmaf(bf16_val(gv[u]) * bf16_val(dv[u]), h, s);
            }
        }
        ss = warp_sum(ss);
        s = warp_sum(s);
        const float rr = sqrtf(fmaf(ss, inv_h, eps)), rinv = 1.f / rr;
        const float c = s * inv_h * rinv * rinv * rinv;
        // pass 2: the kept dims' gradient (the operands come back from L1 / L2)
        for (int k0 = 0; k0 < K; k0 += 32 * kBatch) {
            uint32_t j[kBatch];
            uint16_t hv[kBatch], gv[kBatch], dv[kBatch], rv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                j[u] = k < K ? kept_index(key, ps, (uint32_t)k, flag, 8u) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                const bool in = k < K;
                hv[u] = in ? __ldg(pr + k) : (uint16_t)0;
                gv[u] = in ? __ldg(gamma + j[u]) : (uint16_t)0;
                dv[u] = in ? __ldg(dr + j[u]) : (uint16_t)0;
                rv[u] = (in && gr) ? __ldg(gr + j[u]) : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                if (k < K) {
                    const float v = bf16_val(gv[u]) * bf16_val(dv[u]) * rinv - bf16_val(hv[u]) * c + bf16_val(rv[u]);
                    out[r * K + k] = bf16_rne(v);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreadsF) unpack_add_kernel(const uint16_t *__restrict__ packed, uint16_t *__restrict__ g,
                                                             int64_t rows, int H, int K, uint64_t seed, unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    const int lane = threadIdx.x & 31;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < rows; r += (int64_t)gridDim.x * kWarps) {
        const RowKeys key = row_keys(seed, (uint64_t)r);
        uint16_t *gr = g + r * H;
        const uint16_t *pr = packed + r * K;
        for (int k0 = 0; k0 < K; k0 += 32 * kBatch) {
            uint32_t j[kBatch];
            uint16_t gv[kBatch], pv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                j[u] = k < K ? kept_index(key, ps, (uint32_t)k, flag, 9u) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                const bool in = k < K;
                gv[u] = in ? gr[j[u]] : (uint16_t)0;
                pv[u] = in ? __ldg(pr + k) : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int k = k0 + 32 * u + lane;
                if (k < K) gr[j[u]] = bf16_rne(bf16_val(gv[u]) + bf16_val(pv[u]));
            }
        }
    }
}

int check(int64_t rows, int32_t H, int32_t K, const char *what) {
    if (rows < 0) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": rows < 0");
    if (H < 1 || H > (1 << 30)) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": H outside [1, 2^30]");
    if (K < 0 || K > H) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": K outside [0, H]");
    return SPECOPTIM_OK;
}

bool aligned2(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1) == 0; }

int grid_rows(int64_t rows, int warps) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((rows + warps - 1) / warps, (int64_t)num_sms() * 32));
}

}  // namespace
}  // namespace spco

using namespace spco;

extern "C" int mask_pack_add(const void *a, const void *b, void *packed, int64_t rows, int32_t H, int32_t K,
                             uint32_t layer, uint64_t step, uint64_t batch_id, void *stream) {
    clear_error();
    int rc = check(rows, H, K, "mask_pack_add");
    if (rc) return rc;
    if (rows == 0 || K == 0) return SPECOPTIM_OK;
    if (!a || !b || !packed) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_pack_add: null pointer");
    if (!aligned2(a) || !aligned2(b) || !aligned2(packed))
        return fail(SPECOPTIM_ERR_MISALIGNED, "mask_pack_add: bf16 pointers must be 2-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("mask_pack_add", st,
                pack_add_kernel<<<grid_rows(rows, kWarps), kThreadsF, 0, st>>>(
                    static_cast<const uint16_t *>(a), static_cast<const uint16_t *>(b),
                    static_cast<uint16_t *>(packed), rows, H, K, mask_seed(layer, step, batch_id),
                    device_flag_ptr()));
    SPECOPTIM_LAUNCHED("pack_add_kernel");
    return SPECOPTIM_OK;
}

extern "C" int mask_unpack_rmsnorm(const void *packed, const void *gamma, float eps, void *h_out, void *x_out,
                                   int64_t rows, int32_t H, int32_t K, uint32_t layer, uint64_t step,
                                   uint64_t batch_id, void *stream) {
    clear_error();
    int rc = check(rows, H, K, "mask_unpack_rmsnorm");
    if (rc) return rc;
    if (!(eps >= 0.f)) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_unpack_rmsnorm: eps must be >= 0");
    if (rows == 0) return SPECOPTIM_OK;
    if ((K > 0 && !packed) || !gamma || !h_out || !x_out)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_unpack_rmsnorm: null pointer");
    if (!aligned2(packed) || !aligned2(gamma) || !aligned2(h_out) || !aligned2(x_out))
        return fail(SPECOPTIM_ERR_MISALIGNED, "mask_unpack_rmsnorm: bf16 pointers must be 2-byte aligned");
    const size_t row_bytes = 2 * sizeof(uint16_t) * (size_t)((H + 7) & ~7);
    const int warps = (int)std::min<size_t>(kWarps, 200 * 1024 / row_bytes);
    if (warps < 1) return fail(SPECOPTIM_ERR_NOT_IMPLEMENTED, "mask_unpack_rmsnorm: H too large for the row buffers");
    const size_t smem = row_bytes * warps;
    if (int rc = set_smem_limit(reinterpret_cast<const void *>(&unpack_rmsnorm_kernel), smem)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("mask_unpack_rmsnorm", st,
                unpack_rmsnorm_kernel<<<grid_rows(rows, warps), kThreadsF, smem, st>>>(
                    static_cast<const uint16_t *>(packed), static_cast<const uint16_t *>(gamma), eps,
                    static_cast<uint16_t *>(h_out), static_cast<uint16_t *>(x_out), rows, H, K,
                    mask_seed(layer, step, batch_id), warps, device_flag_ptr()));
    SPECOPTIM_LAUNCHED("unpack_rmsnorm_kernel");
    return SPECOPTIM_OK;
}

extern "C" int mask_rmsnorm_backward_pack(const void *packed_h, const void *gamma, float eps, const void *dx,
                                          const void *g_res, void *packed_grad, int64_t rows, int32_t H, int32_t K,
                                          uint32_t layer, uint64_t step, uint64_t batch_id, void *stream) {
    clear_error();
    int rc = check(rows, H, K, "mask_rmsnorm_backward_pack");
    if (rc) return rc;
    if (!(eps >= 0.f)) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_rmsnorm_backward_pack: eps must be >= 0");
    if (rows == 0 || K == 0) return SPECOPTIM_OK;
    if (!packed_h || !gamma || !dx || !packed_grad)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_rmsnorm_backward_pack: null pointer");
    if (!aligned2(packed_h) || !aligned2(gamma) || !aligned2(dx) || !aligned2(packed_grad) || (g_res && !aligned2(g_res)))
        return fail(SPECOPTIM_ERR_MISALIGNED, "mask_rmsnorm_backward_pack: bf16 pointers must be 2-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("mask_rmsnorm_bwd_pack", st,
                rmsnorm_bwd_pack_kernel<<<grid_rows(rows, kWarps), kThreadsF, 0, st>>>(
                    static_cast<const uint16_t *>(packed_h), static_cast<const uint16_t *>(gamma), eps,
                    static_cast<const uint16_t *>(dx), static_cast<const uint16_t *>(g_res),
                    static_cast<uint16_t *>(packed_grad), rows, H, K, mask_seed(layer, step, batch_id),
                    device_flag_ptr()));
    SPECOPTIM_LAUNCHED("rmsnorm_bwd_pack_kernel");
    return SPECOPTIM_OK;
}

extern "C" int mask_unpack_add(const void *packed, void *g, int64_t rows, int32_t H, int32_t K, uint32_t layer,
                               uint64_t step, uint64_t batch_id, void *stream) {
    clear_error();
    int rc = check(rows, H, K, "mask_unpack_add");
    if (rc) return rc;
    if (rows == 0 || K == 0) return SPECOPTIM_OK;
    if (!packed || !g) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_unpack_add: null pointer");
    if (!aligned2(packed) || !aligned2(g))
        return fail(SPECOPTIM_ERR_MISALIGNED, "mask_unpack_add: bf16 pointers must be 2-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("mask_unpack_add", st,
                unpack_add_kernel<<<grid_rows(rows, kWarps), kThreadsF, 0, st>>>(
                    static_cast<const uint16_t *>(packed), static_cast<uint16_t *>(g), rows, H, K,
                    mask_seed(layer, step, batch_id), device_flag_ptr()));
    SPECOPTIM_LAUNCHED("unpack_add_kernel");
    return SPECOPTIM_OK;
}
