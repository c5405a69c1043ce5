// Launch counting and per-kernel CUDA-event timing of the library's kernels
// (specoptim_trace_* in the C-ABI).
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace spco {
namespace {

struct Rec {
    const char *name;
    cudaEvent_t start, stop;
};

std::atomic<int64_t> g_launches{0};
std::atomic<bool> g_enabled{false};
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void recycle_all() {
    for (auto &r : g_recs) {
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
    }
    g_recs.clear();
}

}  // namespace

int trace_begin(const char *name, cudaStream_t st) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_enabled.load(std::memory_order_relaxed)) return -1;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r{name, take_event(), take_event()};
    cudaEventRecord(r.start, st);
    g_recs.push_back(r);
    return (int)g_recs.size() - 1;
}

void trace_end(int token, cudaStream_t st) {
    if (token < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (token < (int)g_recs.size()) cudaEventRecord(g_recs[token].stop, st);
}

namespace {
std::mutex g_scratch_mu;
float *g_scratch = nullptr;
size_t g_scratch_n = 0;
std::mutex g_dev_mu;
int g_device = -1;
std::mutex g_smem_mu;
std::map<const void *, size_t> g_smem;
}  // namespace

int bind_device() {
    int dev = 0;
    SPECOPTIM_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_device < 0) g_device = dev;
    if (dev != g_device)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "the library serves one device per process (device " +
                                                   std::to_string(g_device) + " at first use, device " +
                                                   std::to_string(dev) + " current now)");
    return SPECOPTIM_OK;
}

int set_smem_limit(const void *fn, size_t bytes) {
    int rc = bind_device();
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_smem_mu);
    size_t &have = g_smem[fn];
    if (bytes > have) {
        SPECOPTIM_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
        have = bytes;
    }
    return SPECOPTIM_OK;
}

int scratch_floats(size_t n, float **out) {
    int rc = bind_device();
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (n > g_scratch_n) {
        if (g_scratch) {
            SPECOPTIM_CUDA(cudaDeviceSynchronize());
            cudaFree(g_scratch);
            g_scratch = nullptr;
            g_scratch_n = 0;
        }
        SPECOPTIM_CUDA(cudaMalloc(reinterpret_cast<void **>(&g_scratch), n * sizeof(float)));
        g_scratch_n = n;
    }
    *out = g_scratch;
    return SPECOPTIM_OK;
}

namespace {
// waits on an mbarrier phase that nothing completes, with a bounded spin
__global__ void wait_timeout_kernel(unsigned *flag, uint32_t limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait_limit(&bar, 0, flag, 0x1FFu, limit);
    }
}
}  // namespace

}  // namespace spco

using namespace spco;

extern "C" int specoptim_selftest_wait_timeout(uint32_t spin_limit, void *stream) {
    clear_error();
    if (spin_limit < 1 || spin_limit > (1u << 24))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "selftest: spin_limit must be in [1, 2^24]");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SPCO_LAUNCH("selftest_wait", st, wait_timeout_kernel<<<1, 32, 0, st>>>(device_flag_ptr(), spin_limit));
    SPECOPTIM_LAUNCHED("wait_timeout_kernel");
    return check_device_flag(st);
}

extern "C" int specoptim_check_device(void *stream) {
    clear_error();
    return check_device_flag(static_cast<cudaStream_t>(stream));
}

extern "C" int specoptim_trace_enable(int32_t enable) {
    clear_error();
    std::lock_guard<std::mutex> lk(g_mu);
    if (enable) {
        cudaDeviceSynchronize();
        recycle_all();
        g_launches.store(0);
    }
    g_enabled.store(enable != 0);
    return SPECOPTIM_OK;
}

extern "C" int64_t specoptim_launch_count(void) { return g_launches.load(); }

extern "C" int specoptim_trace_reset(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    cudaDeviceSynchronize();
    recycle_all();
    g_launches.store(0);
    return SPECOPTIM_OK;
}

extern "C" int specoptim_trace_report(char *buf, int64_t len) {
    clear_error();
    if (!buf || len < 1) return fail(SPECOPTIM_ERR_INVALID_ARG, "trace_report: no buffer");
    std::lock_guard<std::mutex> lk(g_mu);
    SPECOPTIM_CUDA(cudaDeviceSynchronize());
    std::map<std::string, std::pair<int64_t, double>> agg;
    for (auto &r : g_recs) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) ms = 0.f;
        auto &a = agg[r.name];
        a.first += 1;
        a.second += ms;
    }
    std::string out;
    for (auto &kv : agg) {
        char line[256];
        std::snprintf(line, sizeof(line), "%s %lld %.6f\n", kv.first.c_str(),
                      (long long)kv.second.first, kv.second.second);
        out += line;
    }
    if ((int64_t)out.size() + 1 > len) return fail(SPECOPTIM_ERR_INVALID_ARG, "trace_report: buffer too small");
    std::memcpy(buf, out.c_str(), out.size() + 1);
    return SPECOPTIM_OK;
}
