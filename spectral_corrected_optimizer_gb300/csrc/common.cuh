// Shared helpers of the specoptim CUDA library: status handling, error text,
// device error flags for bounded waits, and the inline-PTX wrappers for
// mbarriers and bulk (TMA) copies used by several kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/specoptim.h"

namespace spco {

// per-thread message of the last failure (specoptim_last_error)
void set_error(const std::string &msg);
void clear_error();

inline int fail(int code, const std::string &msg) {
    set_error(msg);
    return code;
}

inline int cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return SPECOPTIM_OK;
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return SPECOPTIM_ERR_CUDA;
}

#define SPECOPTIM_CUDA(call)                                                  \
    do {                                                                      \
        int _rc = ::spco::cuda_status((call), #call);                   \
        if (_rc != SPECOPTIM_OK) return _rc;                                 \
    } while (0)

#define SPECOPTIM_LAUNCHED(what)                                              \
    do {                                                                      \
        int _rc = ::spco::cuda_status(cudaGetLastError(), what);        \
        if (_rc != SPECOPTIM_OK) return _rc;                                 \
    } while (0)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the device (the library serves one device per process; read once)
inline int num_sms() {
    static const int sms = [] {
        int dev = 0, n = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }();
    return sms;
}

// Device-side error flag shared by all kernels of the library: a bounded wait
// that gives up writes its code here instead of spinning forever; the host
// reads it with check_device_flag().
int check_device_flag(cudaStream_t stream);
unsigned *device_flag_ptr();

// Tracing: every kernel launch of the library goes through SPCO_LAUNCH, which
// counts it and, while tracing is enabled, brackets it with CUDA events on the
// launching stream so that per-kernel device time can be reported.
int trace_begin(const char *name, cudaStream_t st);
void trace_end(int token, cudaStream_t st);

#define SPCO_LAUNCH(name, st, ...)                                            \
    do {                                                                      \
        int _tk = ::spco::trace_begin(name, st);                             \
        __VA_ARGS__;                                                          \
        ::spco::trace_end(_tk, st);                                          \
    } while (0)

// The library serves one device per process: its shared state (kernel
// shared-memory limits, the scratch buffer below, the device-side error flag)
// belongs to the device that is current at its first use.  bind_device()
// records that device and fails with SPECOPTIM_ERR_INVALID_ARG when another
// one is current.
int bind_device();

// Raises `fn`'s dynamic shared-memory limit to at least `bytes` (once per
// kernel and size; thread-safe).
int set_smem_limit(const void *fn, size_t bytes);

// Library-wide scratch for transient operands (the split copies of 3xTF32
// products in the SVD refresh): grown on demand with cudaMalloc on the current
// device, never shrunk, shared by all handles.  Callers use it only between
// stream syncs of the same host thread (the refresh synchronises every sweep).
int scratch_floats(size_t n, float **out);

// iteration limit of every spin on an mbarrier (each probe also sleeps a little)
constexpr uint32_t kSpinLimit = 1u << 22;

// ---------------------------------------------------------------------------
// inline PTX: mbarrier and bulk copies (sm_90+ instructions, used on sm_103a)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// kSpinLimit probes: sets *flag (if not null) to `code` and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned *flag,
                                                  unsigned code) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(32);
    }
    if (flag) atomicExch(flag, code);
    return false;
}

// Same wait with an explicit probe limit (used by the timeout self-test).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned *flag,
                                                unsigned code, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        __nanosleep(64);
    }
    if (flag) atomicExch(flag, code);
    return false;
}

// 1D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1D bulk copy shared -> global in the current bulk group
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// wait until at most N committed bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// wait until all committed bulk groups have completed (writes visible)
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace spco
