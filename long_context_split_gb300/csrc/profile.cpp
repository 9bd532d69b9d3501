// Launch profiler: while enabled, every kernel launch of the library is
// bracketed by CUDA events recorded on the launching stream; the totals per
// kernel are read back (after synchronising on the events) when it is
// disabled.  A measurement aid for benchmarks and the planner's calibration.
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "splitkv.h"
#include "internal.h"

namespace skv {
namespace {

struct Rec {
    int kernel;
    cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;

void release(std::vector<Rec>& recs) {
    for (Rec& r : recs) {
        if (r.start) cudaEventDestroy(r.start);
        if (r.stop) cudaEventDestroy(r.stop);
    }
    recs.clear();
}

}  // namespace

ProfileScope::ProfileScope(int kernel, cudaStream_t s) : kernel_(kernel), stream_(s), start_(nullptr), stop_(nullptr) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_on) return;
    }
    if (cudaEventCreate(&start_) != cudaSuccess || cudaEventCreate(&stop_) != cudaSuccess ||
        cudaEventRecord(start_, s) != cudaSuccess) {
        cudaGetLastError();
        if (start_) cudaEventDestroy(start_);
        if (stop_) cudaEventDestroy(stop_);
        start_ = stop_ = nullptr;
    }
}

ProfileScope::~ProfileScope() {
    if (!start_) return;
    if (cudaEventRecord(stop_, stream_) != cudaSuccess) {
        cudaGetLastError();
        cudaEventDestroy(start_);
        cudaEventDestroy(stop_);
        return;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    g_recs.push_back(Rec{kernel_, start_, stop_});
}

}  // namespace skv

extern "C" {

splitkv_status splitkv_profile_begin(void) {
    std::lock_guard<std::mutex> lock(skv::g_mu);
    skv::release(skv::g_recs);
    skv::g_on = true;
    return SPLITKV_OK;
}

splitkv_status splitkv_profile_end(splitkv_kernel_time* out) {
    std::vector<skv::Rec> recs;
    {
        std::lock_guard<std::mutex> lock(skv::g_mu);
        skv::g_on = false;
        recs.swap(skv::g_recs);
    }
    splitkv_status st = SPLITKV_OK;
    if (out)
        for (int k = 0; k < SPLITKV_KERNEL_COUNT; ++k) out[k] = splitkv_kernel_time{0, 0, 0.0};
    for (skv::Rec& r : recs) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) {
            cudaGetLastError();
            skv::set_last_error_message("splitkv_profile_end: reading a launch's events failed");
            st = SPLITKV_ERR_CUDA;
            continue;
        }
        if (out && r.kernel >= 0 && r.kernel < SPLITKV_KERNEL_COUNT) {
            out[r.kernel].launches += 1;
            out[r.kernel].total_ms += (double)ms;
        }
    }
    skv::release(recs);
    return st;
}

}  // extern "C"
