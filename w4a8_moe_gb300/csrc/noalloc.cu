// MoE forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs where
// allocating is not permitted or not available (a plugin or embedding host
// that owns the device memory budget and offers no allocator, code paths that
// must not call cudaMalloc because it can synchronize the device or fail at an
// arbitrary point of a latency-critical loop). For them this file provides
// moe_w4a8_forward_static: the same computation as moe_w4a8_forward, with its
// scratch space in a fixed array that the library owns. Nothing here allocates:
// the array is part of the library's device image, reserved in every CUDA
// context that loads the library until the process exits.
#include <cudaTypedefs.h>

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

// Every CUDA context that loads the library holds its own copy of the array
// (the primary context of each device, or a context a host application created
// and made current), so its device address is looked up once per context and
// cached under the context handle.
constexpr int kMaxContexts = 64;
struct ContextScratch {
    CUcontext ctx;
    void* ptr;
};
ContextScratch g_cache[kMaxContexts];
int g_cached = 0;
std::mutex g_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
bool g_ctx_tried = false;

CUcontext current_context()
{
    CUcontext c = nullptr;
    if (g_ctx_current && g_ctx_current(&c) != CUDA_SUCCESS)
        c = nullptr;
    return c;
}

// The address of the array in the current context. In host code
// `g_static_scratch` names a host-side stand-in, not device memory, so the
// kernels get the device address from cudaGetSymbolAddress.
void* scratch_for_current_context()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ctx_tried) {
        g_ctx_tried = true;
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        cudaGetLastError();
    }
    CUcontext ctx = current_context();
    if (ctx)
        for (int i = 0; i < g_cached; ++i)
            if (g_cache[i].ctx == ctx)
                return g_cache[i].ptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (!ctx)   // the lookup has made the device's primary context current
        ctx = current_context();
    if (ctx && g_cached < kMaxContexts)
        g_cache[g_cached++] = {ctx, p};
    return p;
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
    // The regular entry point's checks, in its order, then the size limit,
    // all before touching the device.
    const void* ptrs[] = {x_e4m3, a1_scale, w_gu, s_gu, w_d, s_d, a2_scale, topk_ids, topk_w,
                          counts, offsets, sorted_ids, inv_perm, out_bf16};
    if (int st = w4a8::moe_forward_check(ptrs, 14, T, H, I, E, k, act))
        return st;
    if (moe_w4a8_workspace_size(T, H, I, E, k) > w4a8::kStaticScratchBytes)
        return W4A8_ERR_WORKSPACE;
    void* scratch = w4a8::scratch_for_current_context();
    if (!scratch)
        return W4A8_ERR_DEVICE;
    // The regular entry point does the rest; the per-call state that must start
    // at zero (the int64 row sums of the intermediate activation, the per-expert
    // progress counters) is cleared by its first kernel, so the previous call's
    // leftovers do no harm.
    return moe_w4a8_forward(x_e4m3, a1_scale, T, H, I, E, k, w_gu, s_gu, w_d, s_d, a2_scale, act, topk_ids,
                            topk_w, counts, offsets, sorted_ids, inv_perm, out_bf16, scratch,
                            w4a8::kStaticScratchBytes, stream);
}

extern "C" int moe_w4a8_forward_static_error(int* code_out, void* stream)
{
    if (!code_out)
        return W4A8_ERR_NULL;
    void* scratch = w4a8::scratch_for_current_context();
    if (!scratch)
        return W4A8_ERR_DEVICE;
    return w4a8_device_error(scratch, code_out, stream);
}
