// tcgen05 tensor-core GEMM, kind::tf32 with fp32 accumulation in TMEM.
//
//   C (M x N) = A (M x K) . B (N x K)^T      A, B fp32 row-major, K contiguous
//
// It runs the products of the two-sided projection of key design 3
// ("Communication-Efficient LLM Adaptation over Decentralized GPU Meshes":
// G_filt = U diag(d) U^T G V diag(d) V^T, evaluated through the projectors
// U diag(d) U^T and V diag(d) V^T), with the diagonal scaling, the convex
// blend and the AdamW update as epilogues, and the 3xTF32 products of the SVD
// refresh (gemm3.cu).
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: 2D tiled loads (128B swizzle) of a 128 x 32 slab
//               of A and a 256 x 32 slab of B per stage, 4 stages, completion
//               counted on the stage's "full" mbarrier.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators);
//               one lane issues tcgen05.mma (M=128, N=256, K=8) four times per
//               stage and frees the stage with tcgen05.commit; after the last
//               stage of a tile it commits to the accumulator's "full" barrier.
//   warps 2-9   epilogue: tcgen05.ld of their TMEM lane quarter and column
//               half, element-wise epilogue, global stores; then release the
//               accumulator, so tile i's epilogue overlaps tile i+1's MMAs.
// Every wait on an mbarrier is bounded; a wait that gives up records a code in
// the library's device flag and the CTA winds down (TMEM freed) instead of
// hanging.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "tc.cuh"

namespace spco {
namespace {

constexpr int BM = 128, BN = 256, BK = 32;  // BK fp32 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (2 + EPI_WARPS) * 32;
constexpr uint32_t A_BYTES = BM * BK * 4;
constexpr uint32_t B_BYTES = BN * BK * 4;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int kMaxGroup = 8;
constexpr int TPITCH = 33;  // padded row of an epilogue transpose tile (conflict-free both ways)
constexpr size_t TILE_BYTES = (size_t)EPI_WARPS * 32 * TPITCH * 4;
constexpr size_t SMEM_BYTES =
    (size_t)STAGES * STAGE_BYTES + TILE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");

constexpr uint32_t kIdesc = tf32_idesc(BM, BN);

// ---- epilogue of one row segment (32 accumulator columns) ---------------------

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// Coalesced epilogue of a 32 x 32 accumulator block.  The block arrives from
// tcgen05.ld as "thread = row, registers = 32 columns"; it is transposed
// through a padded shared tile so that each warp instruction then touches four
// rows x 32 consecutive columns (four full 128-byte lines per array).
__device__ __forceinline__ void epilogue_block(const Epilogue &e, float *tile, int lane,
                                               int64_t row0, int64_t col0, int64_t M, int64_t N,
                                               const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) tile[lane * TPITCH + j] = v[j];
    __syncwarp();
    const int sub = lane >> 3;        // row within a group of 4
    const int cq = (lane & 7) * 4;    // first of this thread's 4 columns
    const int64_t col = col0 + cq;
    const bool vec = (col + 4 <= N) &&
                     (((e.mode == EPI_ADAMW) ? e.ld : e.ldc) & 3) == 0;
    if (e.mode == EPI_ADAMW) {
        if (vec) {
            // four row groups at a time: every load is issued before any store, so
            // 16 independent 16-byte loads per thread are in flight
#pragma unroll
            for (int gb = 0; gb < 8; gb += 4) {
                float4 g4[4], w4[4], m4[4], v4[4];
                int64_t off[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t row = row0 + (gb + u) * 4 + sub;
                    off[u] = row < M ? row * e.ld + col : -1;
                    if (off[u] >= 0) {
                        g4[u] = ld4_stream(e.G + off[u]);
                        w4[u] = ld4(e.W + off[u]);
                        m4[u] = ld4(e.m1 + off[u]);
                        v4[u] = ld4(e.m2 + off[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (off[u] < 0) continue;
                    const int i = (gb + u) * 4 + sub;
                    const float a[4] = {tile[i * TPITCH + cq], tile[i * TPITCH + cq + 1],
                                        tile[i * TPITCH + cq + 2], tile[i * TPITCH + cq + 3]};
                    const float gv[4] = {g4[u].x, g4[u].y, g4[u].z, g4[u].w};
                    float wv[4] = {w4[u].x, w4[u].y, w4[u].z, w4[u].w};
                    float mv[4] = {m4[u].x, m4[u].y, m4[u].z, m4[u].w};
                    float vv[4] = {v4[u].x, v4[u].y, v4[u].z, v4[u].w}, pv[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        pv[t] = e.alpha * gv[t] + (1.f - e.alpha) * a[t];
                        mv[t] = e.beta1 * mv[t] + (1.f - e.beta1) * pv[t];
                        vv[t] = e.beta2 * vv[t] + (1.f - e.beta2) * pv[t] * pv[t];
                        wv[t] = wv[t] * e.decay - e.step_size * mv[t] / (sqrtf(vv[t]) * e.inv_sqrt_bc2 + e.eps);
                    }
                    const int64_t o = off[u];
                    st4(e.W + o, make_float4(wv[0], wv[1], wv[2], wv[3]));
                    st4(e.m1 + o, make_float4(mv[0], mv[1], mv[2], mv[3]));
                    st4(e.m2 + o, make_float4(vv[0], vv[1], vv[2], vv[3]));
                    if (e.Gf_out) st4(e.Gf_out + o, make_float4(a[0], a[1], a[2], a[3]));
                    if (e.Gp_out) st4(e.Gp_out + o, make_float4(pv[0], pv[1], pv[2], pv[3]));
                }
            }
        } else {
            for (int g = 0; g < 8; ++g) {
                const int i = g * 4 + sub;
                const int64_t row = row0 + i;
                if (row >= M) continue;
                for (int t = 0; t < 4; ++t)
                    if (col + t < N) epilogue_apply(e, row, col + t, tile[i * TPITCH + cq + t]);
            }
        }
    } else {
        float cs[4] = {1.f, 1.f, 1.f, 1.f};
        if (e.mode == EPI_SCALE && e.col_scale)
            for (int t = 0; t < 4; ++t) cs[t] = (col + t < N) ? e.col_scale[col + t] : 0.f;
#pragma unroll 4
        for (int g = 0; g < 8; ++g) {
            const int i = g * 4 + sub;
            const int64_t row = row0 + i;
            if (row >= M) continue;
            const float rs = (e.mode == EPI_SCALE && e.row_scale) ? e.row_scale[row] : 1.f;
            float c[4];
            for (int t = 0; t < 4; ++t) {
                c[t] = tile[i * TPITCH + cq + t] * rs * cs[t];
                if (e.round_tf32) c[t] = round_to_tf32(c[t]);
            }
            if (vec) {
                st4(e.C + row * e.ldc + col, make_float4(c[0], c[1], c[2], c[3]));
            } else {
                for (int t = 0; t < 4; ++t)
                    if (col + t < N) e.C[row * e.ldc + col + t] = c[t];
            }
        }
    }
    __syncwarp();
}

// ---- the kernel ----------------------------------------------------------------

// Up to kMaxGroup independent products in one persistent launch.  Tiles are
// numbered problem by problem (N fastest inside a problem); every role walks
// the same sequence, so each CTA knows which problem a tile belongs to.
struct GemmGroup {
    CUtensorMap tmA[kMaxGroup];
    CUtensorMap tmB[kMaxGroup];
    Epilogue epi[kMaxGroup];
    int M[kMaxGroup], N[kMaxGroup], K[kMaxGroup];
    int tiles_n[kMaxGroup];
    int tile_off[kMaxGroup + 1];
    int count;
};

__device__ __forceinline__ void tile_coords(const GemmGroup &g, int tile, int &p, int &m0, int &n0) {
    p = 0;
    while (p + 1 < g.count && tile >= g.tile_off[p + 1]) ++p;
    const int local = tile - g.tile_off[p];
    n0 = (local % g.tiles_n[p]) * BN;  // N fastest: the A slab stays hot in L2
    m0 = (local / g.tiles_n[p]) * BM;
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_tf32_kernel(const __grid_constant__ GemmGroup grp, unsigned *flag) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *tbuf = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + TILE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int num_tiles = grp.tile_off[grp.count];

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], EPI_WARPS * 32);
        }
        fence_mbar_init();
        for (int p = 0; p < grp.count; ++p) {
            prefetch_tmap(&grp.tmA[p]);
            prefetch_tmap(&grp.tmB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            int p, m0, n0;
            tile_coords(grp, tile, p, m0, n0);
            const int num_kb = (grp.K[p] + BK - 1) / BK;
            for (int kb = 0; kb < num_kb; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, flag, 0x101u)) { ok = false; break; }
                unsigned char *sa = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                tma_load_2d(sa, &grp.tmA[p], kb * BK, m0, &full[s]);
                tma_load_2d(sa + A_BYTES, &grp.tmB[p], kb * BK, n0, &full[s]);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        uint32_t it = 0, local = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1u;
            const uint32_t aph = (local >> 1) & 1u;
            if (!mbar_wait_bounded(&tempty[acc], aph ^ 1u, flag, 0x102u)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            int p, m0, n0;
            tile_coords(grp, tile, p, m0, n0);
            const int num_kb = (grp.K[p] + BK - 1) / BK;
            for (int kb = 0; kb < num_kb; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait_bounded(&full[s], ph, flag, 0x103u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
                const uint32_t sb = sa + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 8; ++k)
                    mma_tf32(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32),
                             kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
                mma_commit(&empty[s]);  // stage free once these MMAs have read it
            }
            mma_commit(&tfull[acc]);    // accumulator ready once all MMAs completed
        }
    } else if (warp >= 2) {
        // ---------------- epilogue
        const int q = warp % 4;          // TMEM lane quarter this warp may access
        const int half = (warp - 2) / 4; // column half of the 256-wide tile
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            int p, m0, n0;
            tile_coords(grp, tile, p, m0, n0);
            const uint32_t acc = local & 1u;
            const uint32_t aph = (local >> 1) & 1u;
            if (!mbar_wait_bounded(&tfull[acc], aph, flag, 0x104u)) break;
            tc_fence_after();
            float *tbuf_w = tbuf + (warp - 2) * 32 * TPITCH;
            for (int c = 0; c < BN / 2 / 32; ++c) {
                const int col = half * (BN / 2) + c * 32;
                float v[32];
                tmem_ld32(tmem_base + acc * BN + col + ((uint32_t)(q * 32) << 16), v);
                epilogue_block(grp.epi[p], tbuf_w, lane, (int64_t)m0 + q * 32, (int64_t)n0 + col, grp.M[p],
                               grp.N[p], v);
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- host side -------------------------------------------------------------------

// rows x K fp32 matrix (K contiguous, leading dimension ld), box 32 (K) x box_rows
int make_tmap(CUtensorMap *map, const float *ptr, int64_t rows, int64_t K, int64_t ld,
              uint32_t box_rows) {
    return make_tmap_2d(map, ptr, rows, K, ld, BK, box_rows);
}

}  // namespace

// The tensor-core path takes C = A . B^T with A and B both K-contiguous, row
// pitches that are multiples of 16 bytes and 16-byte aligned bases (TMA rules).
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, Operand A, Operand B) {
    if (M < 1 || N < 1 || K < 1) return false;
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return false;
    if (A.trans || !B.trans) return false;
    if ((A.ld & 3) || (B.ld & 3) || !aligned16(A.ptr) || !aligned16(B.ptr)) return false;
    return tmap_encoder_available();
}

int gemm_tc_group(int count, const GemmProblem *probs, cudaStream_t stream) {
    if (count < 1 || count > kMaxGroup) return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_tc: 1 to 8 problems");
    GemmGroup g;
    std::memset(&g, 0, sizeof(g));
    g.count = count;
    int mode_mask = 0;
    for (int p = 0; p < count; ++p) {
        const GemmProblem &q = probs[p];
        if (!gemm_tc_supported(q.M, q.N, q.K, q.A, q.B))
            return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_tc: operand layout not supported");
        int rc = make_tmap(&g.tmA[p], q.A.ptr, q.M, q.K, q.A.ld, BM);
        if (rc) return rc;
        if ((rc = make_tmap(&g.tmB[p], q.B.ptr, q.N, q.K, q.B.ld, BN))) return rc;
        g.epi[p] = q.epi;
        g.M[p] = (int)q.M;
        g.N[p] = (int)q.N;
        g.K[p] = (int)q.K;
        g.tiles_n[p] = (int)((q.N + BN - 1) / BN);
        g.tile_off[p + 1] = g.tile_off[p] + g.tiles_n[p] * (int)((q.M + BM - 1) / BM);
        mode_mask |= 1 << q.epi.mode;
    }
    if (int rc = set_smem_limit(reinterpret_cast<const void *>(&gemm_tf32_kernel), SMEM_BYTES)) return rc;
    const int grid = std::min(g.tile_off[count], num_sms());
    const char *name = (mode_mask & (1 << EPI_ADAMW)) ? "gemm_tf32_adamw"
                       : (mode_mask & (1 << EPI_SCALE)) ? "gemm_tf32_scale"
                                                        : "gemm_tf32";
    SPCO_LAUNCH(name, stream, gemm_tf32_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(g, device_flag_ptr()));
    SPECOPTIM_LAUNCHED("gemm_tf32_kernel");
    return SPECOPTIM_OK;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}
}  // namespace

bool tmap_encoder_available() { return encode_fn() != nullptr; }

int make_tmap_2d(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld,
                 uint32_t box_cols, uint32_t box_rows) {
    return make_tmap_2d_ex(map, ptr, rows, cols, ld, box_cols, box_rows, true);
}

int make_tmap_2d_ex(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(SPECOPTIM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SPECOPTIM_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SPECOPTIM_OK;
}

int gemm_tc(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
            cudaStream_t stream) {
    GemmProblem q{M, N, K, A, B, epi};
    return gemm_tc_group(1, &q, stream);
}

}  // namespace spco
