// specoptim_filter_noalloc: the filtered gradient G_filt = U diag(d) U^T G V
// diag(d) V^T computed without allocating any device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a framework which
// owns all device memory through its own pool (a raw allocation bypasses the
// pool's accounting and can fail once the pool has reserved the GPU), and code
// on a latency-critical path where the implicit device synchronisation of
// cudaMalloc / cudaFree is not acceptable.  This entry point keeps its
// intermediates in one file-scope device array instead, so the caller passes
// only inputs and outputs.
//
// The array, kScratchBytes = 16 MiB, is part of the library's device image:
// every GPU that loads the library holds it until the process exits.  All
// calls share it and it keeps the last call's contents; nothing in it needs to
// start at zero (every intermediate is fully written before it is read).  Two
// calls whose kernels overlap on the GPU (different streams without ordering,
// or different host threads) race on it and give wrong results.
//
// Host code cannot use the array's name as a device address, so the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it; that first call should therefore come before
// any stream capture.  The cached address belongs to the device's primary
// context: after cudaDeviceReset (or any other teardown of that context) it
// is stale, and this entry point must not be called again in that process.
//
// The products follow the projection equation's literal order (U^T G first,
// then V, then U and V^T again), not the projector association that
// specoptim_step runs; with SPECOPTIM_PREC_TF32 every operand is rounded to
// TF32 (nearest) before it reaches the tensor cores, U and V included, as in
// the step.
#include <mutex>
#include <string>

#include "gemm.cuh"

namespace spco {

int transpose_run(const float *src, float *dst, int rows, int cols, bool round, cudaStream_t st);
int gemm_tc(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
            cudaStream_t stream);
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, Operand A, Operand B);

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices] = {nullptr};

// device address of the scratch array on the current device (looked up once per device)
int scratch_address(float **out) {
    int dev = 0;
    SPECOPTIM_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "filter_noalloc: device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e, "filter_noalloc: cudaGetSymbolAddress");
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return SPECOPTIM_OK;
}

size_t round_up64(size_t n) { return (n + 63) & ~size_t(63); }  // 256-byte regions

int gemm_dispatch(int prec, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                  const float *B, int64_t ldb, const Epilogue &e, cudaStream_t st) {
    Operand a{A, lda, false}, b{B, ldb, true};
    if (prec == SPECOPTIM_PREC_TF32 && gemm_tc_supported(M, N, K, a, b))
        return gemm_tc(M, N, K, a, b, e, st);
    return gemm_simt(M, N, K, a, b, e, st);
}

}  // namespace
}  // namespace spco

using namespace spco;

extern "C" int specoptim_filter_noalloc(const float *U, const float *V, const float *d,
                                        const float *G, float *G_filt, int32_t m, int32_t n,
                                        int32_t precision, void *stream) {
    clear_error();
    if (!U || !V || !d || !G || !G_filt)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "filter_noalloc: null pointer");
    if (m < 1 || n < 1) return fail(SPECOPTIM_ERR_INVALID_ARG, "filter_noalloc: m and n must be >= 1");
    if (precision != SPECOPTIM_PREC_TF32 && precision != SPECOPTIM_PREC_FP32)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "filter_noalloc: unknown precision");
    if (!aligned16(U) || !aligned16(V) || !aligned16(G) || !aligned16(G_filt))
        return fail(SPECOPTIM_ERR_MISALIGNED, "filter_noalloc: U, V, G, G_filt must be 16-byte aligned");
    const bool tall = m > n;
    const size_t r = (size_t)(tall ? n : m);
    // tall: G^T, U^T, U, V^T, V, T1, Xf; otherwise U^T, U, V^T, V, T^T, Xf^T
    const size_t need = tall ? round_up64((size_t)n * m) + 2 * round_up64(r * m) + 2 * round_up64(r * n) +
                                   round_up64(r * n) + round_up64(r * r)
                             : 2 * round_up64(r * m) + 2 * round_up64(r * n) + round_up64(r * m) +
                                   round_up64(r * r);
    if (need > kScratchFloats)
        return fail(SPECOPTIM_ERR_INVALID_ARG,
                    "filter_noalloc: a " + std::to_string(m) + " x " + std::to_string(n) +
                        " matrix needs " + std::to_string(need * sizeof(float)) +
                        " bytes of scratch; the static scratch holds " +
                        std::to_string(kScratchBytes) + " bytes");
    float *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool round = precision == SPECOPTIM_PREC_TF32;
    Epilogue plain;
    plain.round_tf32 = round;
    Epilogue scaled = plain;
    scaled.mode = EPI_SCALE;
    scaled.row_scale = d;
    scaled.col_scale = d;
    Epilogue out;
    out.C = G_filt;
    out.ldc = n;
    float *p = scratch;
    auto take = [&](size_t count) {
        float *q = p;
        p += round_up64(count);
        return q;
    };
    // U^T and V^T (rounded on the way), and U, V back from them: the operands of
    // the last two products then carry the same rounding as the first two
    float *UT = take(r * m), *Ur = take(r * m), *VT = take(r * n), *Vr = take(r * n);
    if ((rc = transpose_run(U, UT, m, (int)r, round, st))) return rc;
    if ((rc = transpose_run(V, VT, n, (int)r, round, st))) return rc;
    if ((rc = transpose_run(UT, Ur, (int)r, m, false, st))) return rc;
    if ((rc = transpose_run(VT, Vr, (int)r, n, false, st))) return rc;
    U = Ur;
    V = Vr;
    if (tall) {  // T1 = U^T G, Xf = (T1 V) o dd^T, Z^T = V Xf^T, G_filt = U Z
        float *GT = take((size_t)n * m);
        float *T1 = take(r * n), *Xf = take(r * r), *ZT = T1;
        if ((rc = transpose_run(G, GT, m, n, round, st))) return rc;
        plain.C = T1;
        plain.ldc = n;
        if ((rc = gemm_dispatch(precision, r, n, m, UT, m, GT, m, plain, st))) return rc;
        scaled.C = Xf;
        scaled.ldc = r;
        if ((rc = gemm_dispatch(precision, r, r, n, T1, n, VT, n, scaled, st))) return rc;
        plain.C = ZT;
        plain.ldc = r;
        if ((rc = gemm_dispatch(precision, n, r, r, V, r, Xf, r, plain, st))) return rc;
        return gemm_dispatch(precision, m, n, r, U, r, ZT, r, out, st);
    }
    // T^T = V^T G^T, Xf^T = (T^T U) o dd^T, Y = U Xf, G_filt = Y V^T
    float *TT = take(r * m), *XfT = take(r * r), *Y = TT;
    plain.C = TT;
    plain.ldc = m;
    if ((rc = gemm_dispatch(precision, r, m, n, VT, n, G, n, plain, st))) return rc;
    scaled.C = XfT;
    scaled.ldc = r;
    if ((rc = gemm_dispatch(precision, r, r, m, TT, m, UT, m, scaled, st))) return rc;
    plain.C = Y;
    plain.ldc = r;
    if ((rc = gemm_dispatch(precision, m, r, r, U, r, XfT, r, plain, st))) return rc;
    return gemm_dispatch(precision, m, n, r, Y, r, V, r, out, st);
}
