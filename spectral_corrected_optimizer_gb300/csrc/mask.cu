// In-graph activation mask: pack / unpack / indices.
//
// "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
// key design 1: h~ = h (.) m keeps K = round((1-p)H) dims of every token; the
// mask m = g(layer, step, batch metadata, S, H) is regenerated locally by
// sender and receiver, only the K kept values are sent, and the backward pass
// dL/dh = (dL/dh~) (.) m uses the same index set.
//
// g (this library's definition; the pages fix only its properties): row r
// keeps pi_r(0..K-1) of a keyed permutation pi_r of [0, H), built from four
// alternating Feistel rounds over ceil(log2 H) bits with MurmurHash3's fmix32
// as round function and SplitMix64-derived round keys; values >= H are walked
// on through the permutation's cycle.  Costs K permutation evaluations per row
// (no sort, no per-dim hash of all H dims), and for H a power of two no cycle
// walking at all.
//
// Data path (HBM-bound streaming): a persistent CTA takes chunks of CH rows
// (see the pipelined kernels below).  Dense chunks move between HBM and shared memory
// with 1D bulk copies (cp.async.bulk) in a multi-stage pipeline; the gather
// (pack) or the zero-fill + scatter (unpack) happens in shared memory; the
// result leaves with one bulk store per chunk.  Rows that do not fill a chunk,
// unaligned pointers and very long rows take a plain per-row kernel.
#include <algorithm>

#include "common.cuh"
#include "mask_g.cuh"

namespace spco {
namespace {

// ---- pipelined bulk-copy kernels --------------------------------------------
//
// A CTA of CH = 8 warps takes chunks of 8 rows (8 * elem_bytes * X is a
// multiple of 16 bytes for any X, so every chunk of dense and of packed rows
// starts and ends 16-byte aligned).  Warp w owns row w of the chunk: it derives
// the row's keys in registers and gathers / scatters that row, so no block
// barrier is needed inside a row.  Dense (pack) or packed (unpack) input chunks
// arrive by 1D bulk copies into a ring of `stages` buffers, each with its own
// mbarrier; outputs leave by bulk stores from a ring of kOutBufs buffers.
// Thread 0 lets at most one store group stay in flight after issuing a store,
// so by the next block barrier the buffer two iterations ahead is free: one
// __syncthreads per chunk.

constexpr int CH = 8;                   // rows per chunk = warps per CTA
constexpr int kThreads = CH * 32;
constexpr int kMaxStages = 4;
constexpr int kOutBufs = 3;
constexpr size_t kSmemBudget = 232448;  // 227 KB, one CTA per SM

__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

// shared memory carve-up (identical on host and device): barriers, input ring, output ring
struct RingLayout {
    size_t in, out, in_stride, out_stride, total;
};

__host__ __device__ inline RingLayout ring_layout(size_t in_bytes, size_t out_bytes, int stages) {
    RingLayout L;
    L.in = 128;  // mbarriers live in the first 128 bytes
    L.in_stride = align128(in_bytes);
    L.out = L.in + (size_t)stages * L.in_stride;
    L.out_stride = align128(out_bytes);
    L.total = L.out + (size_t)kOutBufs * L.out_stride;
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 3)
pack_bulk_kernel(const T *__restrict__ dense, T *__restrict__ packed, int64_t nchunks, int H,
                 int K, uint64_t seed, int stages, unsigned *flag) {
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t in_bytes = (uint32_t)((size_t)CH * H * sizeof(T));
    const uint32_t out_bytes = (uint32_t)((size_t)CH * K * sizeof(T));
    const RingLayout L = ring_layout(in_bytes, out_bytes, stages);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    const PermShape ps = perm_shape((uint32_t)H);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int64_t grid = gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            int64_t c = blockIdx.x + s * grid;
            if (c < nchunks) {
                mbar_arrive_expect_tx(&bar[s], in_bytes);
                bulk_load(smem + L.in + s * L.in_stride, dense + c * CH * (int64_t)H, in_bytes, &bar[s]);
            }
        }
    }
    bool ok = true;
    int it = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += grid, ++it) {
        const int stage = it % stages;
        const uint32_t parity = (uint32_t)(it / stages) & 1u;
        const RowKeys key = row_keys(seed, (uint64_t)(c * CH + warp));
        const T *src = reinterpret_cast<const T *>(smem + L.in + stage * L.in_stride) + (size_t)warp * H;
        T *out = reinterpret_cast<T *>(smem + L.out + (it % kOutBufs) * L.out_stride);
        if (ok) ok = mbar_wait_bounded(&bar[stage], parity, flag, 1u);
        if (ok)
            for (int k = lane; k < K; k += 32) out[warp * K + k] = src[kept_index(key, ps, (uint32_t)k, flag, 1u)];
        fence_proxy_async_smem();
        ok = __syncthreads_and(ok) != 0;  // row gathers done; block control flow stays uniform
        if (!ok) break;
        if (tid == 0) {
            bulk_store(packed + c * CH * (int64_t)K, out, out_bytes);
            bulk_commit();
            bulk_wait_read<1>();  // the buffer of iteration it-1 is free again
            int64_t nxt = c + stages * grid;
            if (nxt < nchunks) {
                mbar_arrive_expect_tx(&bar[stage], in_bytes);
                bulk_load(smem + L.in + stage * L.in_stride, dense + nxt * CH * (int64_t)H, in_bytes,
                          &bar[stage]);
            }
        }
    }
    if (tid == 0) bulk_wait_all();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
unpack_bulk_kernel(const T *__restrict__ packed, T *__restrict__ dense, int64_t nchunks, int H,
                   int K, uint64_t seed, int stages, unsigned *flag) {
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t in_bytes = (uint32_t)((size_t)CH * K * sizeof(T));
    const uint32_t out_bytes = (uint32_t)((size_t)CH * H * sizeof(T));
    const RingLayout L = ring_layout(in_bytes, out_bytes, stages);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    const PermShape ps = perm_shape((uint32_t)H);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int64_t grid = gridDim.x;
    const uint32_t row_bytes = (uint32_t)(H * sizeof(T));

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            int64_t c = blockIdx.x + s * grid;
            if (c < nchunks) {
                mbar_arrive_expect_tx(&bar[s], in_bytes);
                bulk_load(smem + L.in + s * L.in_stride, packed + c * CH * (int64_t)K, in_bytes, &bar[s]);
            }
        }
    }
    bool ok = true;
    int it = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += grid, ++it) {
        const int stage = it % stages;
        const uint32_t parity = (uint32_t)(it / stages) & 1u;
        const RowKeys key = row_keys(seed, (uint64_t)(c * CH + warp));
        unsigned char *row = smem + L.out + (it % kOutBufs) * L.out_stride + (size_t)warp * row_bytes;
        // exact +0 off the mask: zero the row (16-byte stores when the row allows it)
        if ((row_bytes & 15u) == 0) {
            uint4 *z = reinterpret_cast<uint4 *>(row);
            for (uint32_t j = lane; j < row_bytes / 16; j += 32) z[j] = make_uint4(0, 0, 0, 0);
        } else {
            for (uint32_t j = lane; j < row_bytes; j += 32) row[j] = 0;
        }
        __syncwarp();
        if (ok) ok = mbar_wait_bounded(&bar[stage], parity, flag, 2u);
        if (ok) {
            const T *src = reinterpret_cast<const T *>(smem + L.in + stage * L.in_stride) + (size_t)warp * K;
            T *dst = reinterpret_cast<T *>(row);
            for (int k = lane; k < K; k += 32) dst[kept_index(key, ps, (uint32_t)k, flag, 2u)] = src[k];
        }
        fence_proxy_async_smem();
        ok = __syncthreads_and(ok) != 0;
        if (!ok) break;
        if (tid == 0) {
            bulk_store(dense + c * CH * (int64_t)H, smem + L.out + (it % kOutBufs) * L.out_stride, out_bytes);
            bulk_commit();
            bulk_wait_read<1>();
            int64_t nxt = c + stages * grid;
            if (nxt < nchunks) {
                mbar_arrive_expect_tx(&bar[stage], in_bytes);
                bulk_load(smem + L.in + stage * L.in_stride, packed + nxt * CH * (int64_t)K, in_bytes,
                          &bar[stage]);
            }
        }
    }
    if (tid == 0) bulk_wait_all();
}

// ---- plain per-row kernels (ragged tails, unaligned pointers, long rows) ----

template <typename T>
__global__ void pack_rows_kernel(const T *__restrict__ dense, T *__restrict__ packed, int64_t row0,
                                 int64_t rows, int H, int K, uint64_t seed, unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    for (int64_t r = row0 + blockIdx.x; r < rows; r += gridDim.x) {
        RowKeys key = row_keys(seed, (uint64_t)r);
        for (int k = threadIdx.x; k < K; k += blockDim.x)
            packed[r * K + k] = dense[r * H + kept_index(key, ps, (uint32_t)k, flag, 3u)];
    }
}

template <typename T>
__global__ void unpack_rows_kernel(const T *__restrict__ packed, T *__restrict__ dense,
                                   int64_t row0, int64_t rows, int H, int K, uint64_t seed,
                                   unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    for (int64_t r = row0 + blockIdx.x; r < rows; r += gridDim.x) {
        for (int j = threadIdx.x; j < H; j += blockDim.x) dense[r * H + j] = T(0);
        __syncthreads();
        RowKeys key = row_keys(seed, (uint64_t)r);
        for (int k = threadIdx.x; k < K; k += blockDim.x)
            dense[r * H + kept_index(key, ps, (uint32_t)k, flag, 4u)] = packed[r * K + k];
        __syncthreads();
    }
}

__global__ void indices_kernel(int32_t *__restrict__ idx, int64_t rows, int H, int K,
                               uint64_t seed, unsigned *flag) {
    const PermShape ps = perm_shape((uint32_t)H);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        RowKeys key = row_keys(seed, (uint64_t)r);
        for (int k = threadIdx.x; k < K; k += blockDim.x)
            idx[r * K + k] = (int32_t)kept_index(key, ps, (uint32_t)k, flag, 5u);
    }
}

int check_args(int64_t rows, int32_t H, int32_t K, int32_t elem_bytes) {
    if (rows < 0) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask: rows < 0");
    if (H < 1 || H > (1 << 30)) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask: H outside [1, 2^30]");
    if (K < 0 || K > H) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask: K outside [0, H]");
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "mask: elem_bytes must be 2 or 4");
    return SPECOPTIM_OK;
}

int row_grid(int64_t rows) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(rows, (int64_t)num_sms() * 16));
}

// Ring configuration: two CTAs per SM (16 warps to hide the hash latency) when
// a ring of at least 3 input stages fits in half the shared memory, else one
// CTA per SM with as many stages as fit; stages = 0 means the bulk path does
// not fit at all.
struct RingPlan {
    int stages, ctas_per_sm;
};

RingPlan pick_ring(size_t in_bytes, size_t out_bytes, int max_ctas) {
    if (max_ctas >= 3 && ring_layout(in_bytes, out_bytes, 2).total <= kSmemBudget / 3 - 1024) return {2, 3};
    for (int st = kMaxStages; st >= 3; --st)
        if (ring_layout(in_bytes, out_bytes, st).total <= kSmemBudget / 2 - 1024) return {st, 2};
    for (int st = kMaxStages; st >= 1; --st)
        if (ring_layout(in_bytes, out_bytes, st).total <= kSmemBudget) return {st, 1};
    return {0, 1};
}

template <typename T>
int run_pack(const void *dense, void *packed, int64_t rows, int H, int K, uint64_t seed,
             cudaStream_t st) {
    const T *d = static_cast<const T *>(dense);
    T *p = static_cast<T *>(packed);
    const size_t in_b = (size_t)CH * H * sizeof(T), out_b = (size_t)CH * K * sizeof(T);
    const RingPlan plan = pick_ring(in_b, out_b, 3);
    const int stages = plan.stages;
    int64_t nfull = (aligned16(dense) && aligned16(packed) && stages > 0) ? rows / CH : 0;
    if (nfull > 0) {
        size_t smem = ring_layout(in_b, out_b, stages).total;
        if (int rc = set_smem_limit(reinterpret_cast<const void *>(&pack_bulk_kernel<T>), kSmemBudget)) return rc;
        int grid = (int)std::min<int64_t>(nfull, (int64_t)num_sms() * plan.ctas_per_sm);
        SPCO_LAUNCH("mask_pack_bulk", st, pack_bulk_kernel<T><<<grid, kThreads, smem, st>>>(d, p, nfull, H, K, seed, stages,
                                                          device_flag_ptr()));
        SPECOPTIM_LAUNCHED("mask_pack bulk kernel");
    }
    int64_t row0 = nfull * CH;
    if (row0 < rows) {
        SPCO_LAUNCH("mask_pack_rows", st, pack_rows_kernel<T><<<row_grid(rows - row0), 128, 0, st>>>(d, p, row0, rows, H, K, seed,
                                                                             device_flag_ptr()));
        SPECOPTIM_LAUNCHED("mask_pack row kernel");
    }
    return SPECOPTIM_OK;
}

template <typename T>
int run_unpack(const void *packed, void *dense, int64_t rows, int H, int K, uint64_t seed,
               cudaStream_t st) {
    const T *p = static_cast<const T *>(packed);
    T *d = static_cast<T *>(dense);
    const size_t in_b = (size_t)CH * K * sizeof(T), out_b = (size_t)CH * H * sizeof(T);
    const RingPlan plan = pick_ring(in_b, out_b, 2);
    const int stages = plan.stages;
    int64_t nfull = (aligned16(dense) && aligned16(packed) && stages > 0) ? rows / CH : 0;
    if (nfull > 0) {
        size_t smem = ring_layout(in_b, out_b, stages).total;
        if (int rc = set_smem_limit(reinterpret_cast<const void *>(&unpack_bulk_kernel<T>), kSmemBudget)) return rc;
        int grid = (int)std::min<int64_t>(nfull, (int64_t)num_sms() * plan.ctas_per_sm);
        SPCO_LAUNCH("mask_unpack_bulk", st, unpack_bulk_kernel<T><<<grid, kThreads, smem, st>>>(p, d, nfull, H, K, seed, stages,
                                                            device_flag_ptr()));
        SPECOPTIM_LAUNCHED("mask_unpack bulk kernel");
    }
    int64_t row0 = nfull * CH;
    if (row0 < rows) {
        SPCO_LAUNCH("mask_unpack_rows", st, unpack_rows_kernel<T><<<row_grid(rows - row0), 256, 0, st>>>(p, d, row0, rows, H, K, seed,
                                                                                 device_flag_ptr()));
        SPECOPTIM_LAUNCHED("mask_unpack row kernel");
    }
    return SPECOPTIM_OK;
}

}  // namespace
}  // namespace spco

using namespace spco;

extern "C" int32_t mask_keep_count(double p, int32_t H) {
    if (!(p >= 0.0 && p <= 1.0) || H < 1) return -1;
    double x = (1.0 - p) * (double)H + 0.5;
    int32_t K = (int32_t)x;  // x >= 0.5, truncation = floor
    return K > H ? H : K;
}

extern "C" int mask_pack(const void *dense, void *packed, int64_t rows, int32_t H, int32_t K,
                         int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id,
                         void *stream) {
    clear_error();
    int rc = check_args(rows, H, K, elem_bytes);
    if (rc) return rc;
    if (rows == 0 || K == 0) return SPECOPTIM_OK;
    if (!dense || !packed) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_pack: null pointer");
    uint64_t seed = mask_seed(layer, step, batch_id);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return elem_bytes == 2 ? run_pack<uint16_t>(dense, packed, rows, H, K, seed, st)
                           : run_pack<uint32_t>(dense, packed, rows, H, K, seed, st);
}

extern "C" int mask_unpack(const void *packed, void *dense, int64_t rows, int32_t H, int32_t K,
                           int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id,
                           void *stream) {
    clear_error();
    int rc = check_args(rows, H, K, elem_bytes);
    if (rc) return rc;
    if (rows == 0) return SPECOPTIM_OK;
    if (!dense || (K > 0 && !packed))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_unpack: null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        SPECOPTIM_CUDA(cudaMemsetAsync(dense, 0, (size_t)rows * H * elem_bytes, st));
        return SPECOPTIM_OK;
    }
    uint64_t seed = mask_seed(layer, step, batch_id);
    return elem_bytes == 2 ? run_unpack<uint16_t>(packed, dense, rows, H, K, seed, st)
                           : run_unpack<uint32_t>(packed, dense, rows, H, K, seed, st);
}

extern "C" int mask_indices(int32_t *idx_out, int64_t rows, int32_t H, int32_t K, uint32_t layer,
                            uint64_t step, uint64_t batch_id, void *stream) {
    clear_error();
    int rc = check_args(rows, H, K, 4);
    if (rc) return rc;
    if (rows == 0 || K == 0) return SPECOPTIM_OK;
    if (!idx_out) return fail(SPECOPTIM_ERR_INVALID_ARG, "mask_indices: null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("mask_indices", st, indices_kernel<<<row_grid(rows), 128, 0, st>>>(idx_out, rows, H, K,
                                                   mask_seed(layer, step, batch_id), device_flag_ptr()));
    SPECOPTIM_LAUNCHED("mask_indices kernel");
    return SPECOPTIM_OK;
}
