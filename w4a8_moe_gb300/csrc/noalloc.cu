// MoE forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs where
// allocating is not permitted or not available (a plugin or embedding host
// that owns the device memory budget and offers no allocator, code paths that
// must not call cudaMalloc because it can synchronize the device or fail at an
// arbitrary point of a latency-critical loop). For them this file provides
// moe_w4a8_forward_static: the same computation as moe_w4a8_forward, with its
// scratch space in a fixed array that the library owns. Nothing here allocates:
// the array is part of the library's device image, reserved on every GPU that
// loads the library until the process exits.
#include <mutex>

#include "w4a8_moe.h"
#include "internal.h"

namespace w4a8 {

namespace {

// Largest scratch the static variant supports: enough for decode-sized layers
// (e.g. 32 tokens of a Grok-1-shaped layer, hidden 6144 / intermediate 32768,
// top-2 of 8, needs about 28 MiB).
constexpr size_t kStaticScratchBytes = W4A8_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// The address of the array on the current device, looked up once per device.
// In host code `g_static_scratch` names a host-side stand-in, not device
// memory, so the kernels get the device address from cudaGetSymbolAddress.
void* scratch_for_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

}  // namespace w4a8

extern "C" int moe_w4a8_forward_static(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I,
                                       int E, int k, const int32_t* w_gu, const float* s_gu,
                                       const int32_t* w_d, const float* s_d, const float* a2_scale, int act,
                                       const int32_t* topk_ids, const float* topk_w, const int32_t* counts,
                                       const int32_t* offsets, const int32_t* sorted_ids,
                                       const int32_t* inv_perm, uint16_t* out_bf16, void* stream)
{
    // Reject problems whose scratch does not fit before touching the device.
    if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1 ||
        moe_w4a8_workspace_size(T, H, I, E, k) > w4a8::kStaticScratchBytes)
        return W4A8_ERR_WORKSPACE;
    void* scratch = w4a8::scratch_for_current_device();
    if (!scratch)
        return W4A8_ERR_DEVICE;
    // The regular entry point does the rest; the per-call state that must start
    // at zero (the int64 row sums of the intermediate activation) is cleared by
    // its first kernel, so the previous call's leftovers do no harm.
    return moe_w4a8_forward(x_e4m3, a1_scale, T, H, I, E, k, w_gu, s_gu, w_d, s_d, a2_scale, act, topk_ids,
                            topk_w, counts, offsets, sorted_ids, inv_perm, out_bf16, scratch,
                            w4a8::kStaticScratchBytes, stream);
}
