// splitkv_decode_static: the fused decode for callers that cannot allocate
// device memory.  The workspace that splitkv_decode takes from the caller
// lives here instead, in a fixed file-scope device array; the call uploads
// its plan into that array and runs the same engine.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "splitkv.h"
#include "internal.h"

namespace {

// Shared by every call on a device and kept for the life of the process on
// each GPU where the library is loaded.
static __device__ __align__(256) unsigned char g_static_scratch[SPLITKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

splitkv_status fail(splitkv_status s, const char* msg) {
    skv::set_last_error_message(msg);
    return s;
}

// Device address of the array on the current device; looked up once per device.
splitkv_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        char buf[256];
        snprintf(buf, sizeof buf, "splitkv_decode_static: cudaGetDevice: %s", cudaGetErrorString(e));
        return fail(SPLITKV_ERR_CUDA, buf);
    }
    if (dev < 0 || dev >= kMaxDevices) return fail(SPLITKV_ERR_UNSUPPORTED, "splitkv_decode_static: device index too large");
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            char buf[256];
            snprintf(buf, sizeof buf, "splitkv_decode_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return fail(SPLITKV_ERR_CUDA, buf);
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SPLITKV_OK;
}

}  // namespace

extern "C" splitkv_status splitkv_decode_static(const splitkv_problem* prob, const splitkv_plan_t* plan, void* out,
                                                float* lse_out, int32_t* dev_error_word, splitkv_stream stream) {
    if (!plan) return fail(SPLITKV_ERR_INVALID_ARG, "splitkv_decode_static: plan is NULL");
    const size_t need = splitkv_workspace_bytes(plan);
    if (need > SPLITKV_STATIC_SCRATCH_BYTES) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "splitkv_decode_static: the plan needs %zu bytes of scratch, more than the %zu-byte static array; "
                 "call splitkv_decode with a workspace instead",
                 need, (size_t)SPLITKV_STATIC_SCRATCH_BYTES);
        return fail(SPLITKV_ERR_WORKSPACE, buf);
    }
    // every argument is checked before the upload below writes the shared array
    splitkv_status s = skv::check_decode_args(prob, plan, out, lse_out, dev_error_word);
    if (s != SPLITKV_OK) return s;
    void* scratch = nullptr;
    if ((s = scratch_address(&scratch)) != SPLITKV_OK) return s;
    // the plan image carries zeroed counters, queue head and error word
    s = splitkv_plan_upload(plan, scratch, SPLITKV_STATIC_SCRATCH_BYTES, stream);
    if (s != SPLITKV_OK) return s;
    return splitkv_decode(prob, plan, scratch, SPLITKV_STATIC_SCRATCH_BYTES, out, lse_out, dev_error_word, stream);
}

extern "C" splitkv_status splitkv_read_static_device_error(int32_t clear, int32_t* raw, splitkv_stream stream) {
    void* scratch = nullptr;
    splitkv_status s = scratch_address(&scratch);
    if (s != SPLITKV_OK) return s;
    return splitkv_read_device_error(nullptr, scratch, clear, raw, stream);
}
