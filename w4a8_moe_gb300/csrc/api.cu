// C ABI of the library: argument validation, workspace carving, tensor-map
// encoding and kernel launches. Declarations and contracts: include/w4a8_moe.h.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/w4a8_moe.h"
#include "internal.h"

namespace w4a8 {

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;  // device error word + reserved

struct DeviceInfo {
    int checked = 0;  // 0 unknown, 1 usable, -1 not usable
    int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Returns kOK with the SM count when the current device is compute capability
// 10.3 and the kernel image loads.
int current_device(int* num_sms)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return kErrDevice;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
        ok = ok && major == 10 && minor == 3 && sms > 0;
        d.checked = ok ? 1 : -1;
        d.num_sms = sms;
        cudaGetLastError();
    }
    if (d.checked != 1)
        return kErrDevice;
    if (!g_encode_tried) {
        g_encode_tried = true;
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    }
    if (!g_encode)
        return kErrDevice;
    *num_sms = d.num_sms;
    return kOK;
}

thread_local void* g_profile_events[4] = {nullptr, nullptr, nullptr, nullptr};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Carver {
    uint8_t* base;
    size_t off = kHeader;
    explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
    template <class T>
    T* take(size_t bytes)
    {
        T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
        off = align_up(off + bytes);
        return p;
    }
};

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swz)
{
    if (!g_encode)
        return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- workspace layouts ------------------------------------------------------
// Router with the gate: the header holds the grid-wide completion counter of
// the one-launch path (byte 128); then logits (when the caller wants none),
// the per-slice partial logits and the multi-kernel path's histograms.
struct RouteGateWs {
    int* done;
    float* logits;
    float* partial;
    int32_t* hist;
    int32_t* base;
};
static size_t route_gate_ws(int T, int H, int E, int k, RouteGateWs* w, void* ws)
{
    Carver c(ws);
    w->done = ws ? reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + 128) : nullptr;
    w->logits = c.take<float>(static_cast<size_t>(T) * E * 4);
    const int hs = route_gate_slice(T, H, E, k);
    w->partial = c.take<float>(hs ? static_cast<size_t>(H / hs) * T * E * 4 : 0);
    const int64_t A = static_cast<int64_t>(T) * k;
    const int64_t nb = (A + kRouteChunk - 1) / kRouteChunk;
    w->hist = c.take<int32_t>(static_cast<size_t>(nb) * E * 4);
    w->base = c.take<int32_t>(static_cast<size_t>(nb) * E * 4);
    return c.off;
}

static size_t route_ws(int T, int E, int k, int32_t** hist, int32_t** base, void* ws)
{
    Carver c(ws);
    const int64_t A = static_cast<int64_t>(T) * k;
    const int64_t nb = (A + kRouteChunk - 1) / kRouteChunk;
    *hist = c.take<int32_t>(static_cast<size_t>(nb) * E * 4);
    *base = c.take<int32_t>(static_cast<size_t>(nb) * E * 4);
    return c.off;
}

struct MoeWs {
    uint8_t* xp;
    long long* s0x;
    uint8_t* hq;
    unsigned long long* s0h;
    float* ypart;
    float* hf;             // dynamic intermediate scale only
    unsigned int* hmax;    // header word at byte 64 (dynamic only)
    int* done;             // [256] per-expert progress counters (one-launch forward)
    uint8_t* wq8;          // prefill: the weights unpacked once per call
    int* sync;             // prefill: the down GEMM's pacing counters
};
static size_t moe_ws(int T, int H, int I, int E, int k, MoeWs* w, void* ws, bool dynamic = false)
{
    Carver c(ws);
    const size_t A = static_cast<size_t>(T) * k;
    w->xp = c.take<uint8_t>(A * H);
    w->s0x = c.take<long long>(A * 8);
    w->hq = c.take<uint8_t>(A * I);
    w->s0h = c.take<unsigned long long>(A * 8);
    w->ypart = c.take<float>(static_cast<size_t>(moe_ksplit_max(T, k)) * A * H * 4);
    w->hf = c.take<float>(dynamic ? A * I * 4 : 0);
    w->done = c.take<int>(256 * 4);
    w->wq8 = c.take<uint8_t>(moe_unpack_once(T) ? static_cast<size_t>(E) * 3 * I * H : 0);
    w->sync = c.take<int>(moe_unpack_once(T) ? static_cast<size_t>(kMoeSyncInts) * 4 : 0);
    w->hmax = ws ? reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + 64) : nullptr;
    return c.off;
}

// Shapes the MoE forward accepts (see the header).
static bool moe_shape_ok(int T, int H, int I, int E, int k)
{
    return T >= 1 && H >= 128 && H % 128 == 0 && I >= 128 && I % 128 == 0 && E >= 1 && E <= 256 && k >= 1 &&
           k <= E && static_cast<int64_t>(T) * k < (static_cast<int64_t>(1) << 30) &&
           static_cast<int64_t>(E) * 2 * I < (static_cast<int64_t>(1) << 31);
}

struct BlkWs {
    uint8_t* xq;
    float* xs_t;
    int ld_t;
    float* ypart;
    int* tile_cnt;   // split-K counters, one per (128-row weight tile, token tile)
    int n_cnt;
};
static size_t blk_ws(int M, int N, int K, BlkWs* w, void* ws)
{
    Carver c(ws);
    w->ld_t = (M + 3) / 4 * 4;
    w->xq = c.take<uint8_t>(static_cast<size_t>(M) * K);
    w->xs_t = c.take<float>(static_cast<size_t>(K / 128) * w->ld_t * 4);
    const int ks = blk_ksplit_max(M, K);
    w->ypart = c.take<float>(ks > 1 ? static_cast<size_t>(ks) * M * N * 4 : 0);
    // token tiles are at least 16 wide
    w->n_cnt = (N / 128) * ((M + 15) / 16);
    w->tile_cnt = c.take<int>(static_cast<size_t>(w->n_cnt) * 4);
    return c.off;
}

// Per-tensor FP8 linear: split-K partials, then one counter per
// (128-row weight tile, token tile) -- token tiles are at least 16 wide.
struct FpWs {
    float* ypart;
    int* tile_cnt;
};
static size_t fp_ws(int M, int N, int K, FpWs* w, void* ws)
{
    Carver c(ws);
    const int ks = fp8_ksplit_max(M, K);
    w->ypart = c.take<float>(ks > 1 ? static_cast<size_t>(ks) * M * N * 4 : 0);
    w->tile_cnt = c.take<int>(static_cast<size_t>(N / 128) * ((M + 15) / 16) * 4);
    return c.off;
}

}  // namespace w4a8

using namespace w4a8;

extern "C" {

const char* w4a8_status_string(int status)
{
    switch (status) {
    case W4A8_OK: return "W4A8_OK";
    case W4A8_ERR_NULL: return "W4A8_ERR_NULL: a required pointer is NULL";
    case W4A8_ERR_SHAPE: return "W4A8_ERR_SHAPE: unsupported size";
    case W4A8_ERR_ALIGN: return "W4A8_ERR_ALIGN: pointer not 16-byte aligned";
    case W4A8_ERR_WORKSPACE: return "W4A8_ERR_WORKSPACE: workspace missing or too small";
    case W4A8_ERR_DEVICE: return "W4A8_ERR_DEVICE: needs a compute capability 10.3 GPU";
    case W4A8_ERR_LAUNCH: return "W4A8_ERR_LAUNCH: CUDA launch or driver call failed";
    case W4A8_ERR_TIMEOUT: return "W4A8_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "W4A8: unknown status";
    }
}

int w4a8_version(void) { return 100; }

int w4a8_quantize_experts(const uint16_t* w_bf16, int E, int N, int K, int32_t* packed, float* scale,
                          void* stream)
{
    if (!w_bf16 || !packed || !scale)
        return W4A8_ERR_NULL;
    if (E < 1 || N < 1 || K < 8 || K % 8 != 0)
        return W4A8_ERR_SHAPE;
    if (!aligned16(w_bf16) || !aligned16(packed) || !aligned16(scale))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    return launch_quantize_experts(w_bf16, E, N, K, packed, scale, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_LAUNCH;
}

size_t w4a8_quantize_act_workspace_size(int64_t numel)
{
    (void)numel;
    return kHeader + align_up(1024 * sizeof(float));
}

int w4a8_quantize_act(const uint16_t* x_bf16, int64_t numel, float* scale, int compute_scale,
                      uint8_t* x_e4m3, void* ws, size_t ws_bytes, void* stream)
{
    if (!x_bf16 || !scale || !x_e4m3)
        return W4A8_ERR_NULL;
    if (numel < 16 || numel % 16 != 0)
        return W4A8_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(x_e4m3) || ((reinterpret_cast<uintptr_t>(scale) & 3u) != 0))
        return W4A8_ERR_ALIGN;
    if (compute_scale && (!ws || ws_bytes < w4a8_quantize_act_workspace_size(numel)))
        return W4A8_ERR_WORKSPACE;
    if (compute_scale && !aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* partial = compute_scale ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kHeader) : nullptr;
    const int nb = act_amax_blocks(numel);
    if (compute_scale && launch_act_amax(x_bf16, numel, partial, nb, s) != cudaSuccess)
        return W4A8_ERR_LAUNCH;
    return launch_act_encode(x_bf16, numel, scale, compute_scale, partial, nb, x_e4m3, s) == cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_LAUNCH;
}

size_t moe_route_workspace_size(int T, int E, int k)
{
    int32_t *h, *b;
    return route_ws(T, E, k, &h, &b, nullptr);
}

size_t moe_route_gate_workspace_size(int T, int H, int E, int k)
{
    RouteGateWs w;
    return route_gate_ws(T, H, E, k, &w, nullptr);
}

int moe_route_gate(const uint16_t* hidden_bf16, const uint16_t* gate_bf16, int T, int H, int E, int k,
                   int renormalize, float* logits_out, int32_t* topk_ids, float* topk_w, int32_t* counts,
                   int32_t* offsets, int32_t* sorted_ids, int32_t* inv_perm, void* ws, size_t ws_bytes,
                   void* stream)
{
    if (!hidden_bf16 || !gate_bf16 || !topk_ids || !topk_w || !counts || !offsets || !sorted_ids || !inv_perm)
        return W4A8_ERR_NULL;
    if (T < 1 || H < 128 || H % 128 != 0 || E < 1 || E > 256 || k < 1 || k > E ||
        static_cast<int64_t>(T) * k >= (static_cast<int64_t>(1) << 31))
        return W4A8_ERR_SHAPE;
    const void* ptrs[] = {hidden_bf16, gate_bf16, topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return W4A8_ERR_ALIGN;
    if (logits_out && !aligned16(logits_out))
        return W4A8_ERR_ALIGN;
    if (!ws || ws_bytes < moe_route_gate_workspace_size(T, H, E, k))
        return W4A8_ERR_WORKSPACE;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    RouteGateWs w;
    route_gate_ws(T, H, E, k, &w, ws);
    float* logits = logits_out ? logits_out : w.logits;
    return launch_route_gate(hidden_bf16, gate_bf16, T, H, E, k, renormalize ? 1 : 0, logits, logits_out ? 1 : 0,
                             topk_ids, topk_w,
                             counts, offsets, sorted_ids, inv_perm, w.partial, w.done, w.hist, w.base,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_LAUNCH;
}

int moe_route(const float* logits, int T, int E, int k, int renormalize, int32_t* topk_ids,
              float* topk_w, int32_t* counts, int32_t* offsets, int32_t* sorted_ids, int32_t* inv_perm,
              void* ws, size_t ws_bytes, void* stream)
{
    if (!logits || !topk_ids || !topk_w || !counts || !offsets || !sorted_ids || !inv_perm)
        return W4A8_ERR_NULL;
    if (T < 1 || E < 1 || E > 256 || k < 1 || k > E ||
        static_cast<int64_t>(T) * k >= (static_cast<int64_t>(1) << 31))
        return W4A8_ERR_SHAPE;
    const void* ptrs[] = {logits, topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return W4A8_ERR_ALIGN;
    if (!ws || ws_bytes < moe_route_workspace_size(T, E, k))
        return W4A8_ERR_WORKSPACE;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    int32_t *hist, *base;
    route_ws(T, E, k, &hist, &base, ws);
    return launch_route(logits, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w, counts, offsets,
                        sorted_ids, inv_perm, hist, base, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_LAUNCH;
}

size_t moe_w4a8_workspace_size(int T, int H, int I, int E, int k)
{
    MoeWs w;
    return moe_ws(T, H, I, E, k, &w, nullptr);
}

int moe_w4a8_workspace_layout(int T, int H, int I, int E, int k, int64_t* offsets)
{
    if (!offsets)
        return W4A8_ERR_NULL;
    if (!moe_shape_ok(T, H, I, E, k))
        return W4A8_ERR_SHAPE;
    MoeWs w;
    moe_ws(T, H, I, E, k, &w, reinterpret_cast<void*>(static_cast<uintptr_t>(kAlign)));
    // moe_ws carves from a non-null base; offsets are relative to it
    offsets[0] = static_cast<int64_t>(reinterpret_cast<uintptr_t>(w.hq) - kAlign);
    offsets[1] = static_cast<int64_t>(reinterpret_cast<uintptr_t>(w.xp) - kAlign);
    return W4A8_OK;
}

int moe_w4a8_plan(int T, int H, int I, int E, int k, int dynamic, int num_sms, int32_t* plan)
{
    if (!plan)
        return W4A8_ERR_NULL;
    if (!moe_shape_ok(T, H, I, E, k) || num_sms < 1)
        return W4A8_ERR_SHAPE;
    const MoeConfig c = moe_pick_config(T, H, I, E, k, num_sms, dynamic == 0);
    const bool one = c.fused && dynamic == 0;
    plan[0] = c.bn;
    plan[1] = c.kc;
    plan[2] = c.ksplit;
    plan[3] = one ? 0 : c.streamk;
    plan[4] = one ? 0 : c.nslots;
    plan[5] = one ? 1 : 0;
    // the prefill unpack, the gather, the GEMM launch(es), the dynamic scale's
    // quantizer, the combine
    plan[6] = (c.a8 ? 1 : 0) + 1 + (one ? 1 : 2) + (dynamic ? 1 : 0) + 1;
    plan[7] = (one || !c.streamk) ? c.ksplit : c.nslots;
    return W4A8_OK;
}

}  // extern "C"

// Checks of moe_w4a8_forward that need no workspace: pointers, shape, alignment.
int w4a8::moe_forward_check(const void* const* ptrs, int nptrs, int T, int H, int I, int E, int k, int act)
{
    for (int i = 0; i < nptrs; ++i)
        if (!ptrs[i])
            return W4A8_ERR_NULL;
    if (!moe_shape_ok(T, H, I, E, k) || (act != 0 && act != 1))
        return W4A8_ERR_SHAPE;
    for (int i = 0; i < nptrs; ++i)
        if (!aligned16(ptrs[i]))
            return W4A8_ERR_ALIGN;
    return W4A8_OK;
}

// The MoE forward with a static (a2_scale read) or dynamic (computed from the
// call's h and written to a2_out) intermediate scale.
static int moe_forward_common(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I, int E, int k,
                              const int32_t* w_gu, const float* s_gu, const int32_t* w_d, const float* s_d,
                              const float* a2_scale, float* a2_out, bool dynamic, int act,
                              const int32_t* topk_ids, const float* topk_w, const int32_t* counts,
                              const int32_t* offsets, const int32_t* sorted_ids, const int32_t* inv_perm,
                              uint16_t* out_bf16, void* ws, size_t ws_bytes, void* stream)
{
    const void* ptrs[] = {x_e4m3, a1_scale, w_gu, s_gu, w_d, s_d, a2_scale, topk_ids, topk_w,
                          counts, offsets, sorted_ids, inv_perm, out_bf16};
    if (int st = moe_forward_check(ptrs, 14, T, H, I, E, k, act))
        return st;
    if (!ws || ws_bytes < (dynamic ? moe_w4a8_dynamic_workspace_size(T, H, I, E, k)
                                  : moe_w4a8_workspace_size(T, H, I, E, k)))
        return W4A8_ERR_WORKSPACE;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    MoeWs w;
    moe_ws(T, H, I, E, k, &w, ws, dynamic);
    MoeLaunch L{};
    L.xq = x_e4m3;
    L.a1 = a1_scale;
    L.T = T;
    L.H = H;
    L.I = I;
    L.E = E;
    L.k = k;
    L.w_gu = w_gu;
    L.s_gu = s_gu;
    L.w_d = w_d;
    L.s_d = s_d;
    L.a2 = a2_scale;
    L.act = act;
    L.ids = topk_ids;
    L.topk_w = topk_w;
    L.counts = counts;
    L.offsets = offsets;
    L.sorted_ids = sorted_ids;
    L.inv = inv_perm;
    L.out = out_bf16;
    L.xp = w.xp;
    L.s0x = w.s0x;
    L.hq = w.hq;
    L.s0h = w.s0h;
    L.ypart = w.ypart;
    L.done = w.done;
    L.wq8 = w.wq8;
    L.sync = w.sync;
    // header words 48 and 49: the one-launch forward's claim counters, zero
    // when the workspace is allocated and left zero by every call
    L.claim = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + 192);
    L.dynamic = dynamic ? 1 : 0;
    L.hf = w.hf;
    L.hmax = w.hmax;
    L.a2_out = a2_out;
    L.err = static_cast<uint32_t*>(ws);
    for (int i = 0; i < 4; ++i)
        L.events[i] = g_profile_events[i];
    const MoeConfig cfg = moe_pick_config(T, H, I, E, k, sms, !dynamic);
    return launch_moe_forward(L, cfg, sms, static_cast<cudaStream_t>(stream));
}

extern "C" {

int moe_w4a8_forward(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I, int E, int k,
                     const int32_t* w_gu, const float* s_gu, const int32_t* w_d, const float* s_d,
                     const float* a2_scale, int act, const int32_t* topk_ids, const float* topk_w,
                     const int32_t* counts, const int32_t* offsets, const int32_t* sorted_ids,
                     const int32_t* inv_perm, uint16_t* out_bf16, void* ws, size_t ws_bytes, void* stream)
{
    return moe_forward_common(x_e4m3, a1_scale, T, H, I, E, k, w_gu, s_gu, w_d, s_d, a2_scale, nullptr, false,
                              act, topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm, out_bf16, ws, ws_bytes,
                              stream);
}

size_t moe_w4a8_dynamic_workspace_size(int T, int H, int I, int E, int k)
{
    MoeWs w;
    return moe_ws(T, H, I, E, k, &w, nullptr, true);
}

int moe_w4a8_forward_dynamic(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I, int E, int k,
                             const int32_t* w_gu, const float* s_gu, const int32_t* w_d, const float* s_d,
                             float* a2_out, int act, const int32_t* topk_ids, const float* topk_w,
                             const int32_t* counts, const int32_t* offsets, const int32_t* sorted_ids,
                             const int32_t* inv_perm, uint16_t* out_bf16, void* ws, size_t ws_bytes, void* stream)
{
    return moe_forward_common(x_e4m3, a1_scale, T, H, I, E, k, w_gu, s_gu, w_d, s_d, a2_out, a2_out, true, act,
                              topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm, out_bf16, ws, ws_bytes,
                              stream);
}

size_t fp8_block_linear_workspace_size(int M, int N, int K)
{
    BlkWs w;
    return blk_ws(M, N, K, &w, nullptr);
}

size_t fp8_linear_workspace_size(int M, int N, int K)
{
    FpWs w;
    return fp_ws(M, N, K, &w, nullptr);
}

int fp8_linear(const uint8_t* x_e4m3, const float* x_scale, int M, int N, int K, const uint8_t* w_e4m3,
               const float* w_scale, uint16_t* y_bf16, void* ws, size_t ws_bytes, void* stream)
{
    if (!x_e4m3 || !x_scale || !w_e4m3 || !w_scale || !y_bf16)
        return W4A8_ERR_NULL;
    if (M < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0)
        return W4A8_ERR_SHAPE;
    const void* ptrs[] = {x_e4m3, w_e4m3, y_bf16};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return W4A8_ERR_ALIGN;
    if (!ws || ws_bytes < fp8_linear_workspace_size(M, N, K))
        return W4A8_ERR_WORKSPACE;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    FpWs w;
    fp_ws(M, N, K, &w, ws);
    FpLaunch L;
    L.M = M;
    L.N = N;
    L.K = K;
    L.x = x_e4m3;
    L.sx = x_scale;
    L.w = w_e4m3;
    L.sw = w_scale;
    L.y = y_bf16;
    L.ypart = w.ypart;
    L.tile_cnt = w.tile_cnt;
    L.err = static_cast<uint32_t*>(ws);
    const FpConfig cfg = fp8_pick_config(M, N, K, sms);
    return launch_fp8_linear(L, cfg, sms, static_cast<cudaStream_t>(stream)) == kOK ? W4A8_OK : W4A8_ERR_LAUNCH;
}

int fp8_block_linear(const uint16_t* x_bf16, int M, int N, int K, const uint8_t* w_e4m3,
                     const float* w_scale_inv, uint16_t* y_bf16, uint8_t* xq_out, float* xs_out, void* ws,
                     size_t ws_bytes, void* stream)
{
    if (!x_bf16 || !w_e4m3 || !w_scale_inv || !y_bf16)
        return W4A8_ERR_NULL;
    if (M < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0)
        return W4A8_ERR_SHAPE;
    const void* ptrs[] = {x_bf16, w_e4m3, w_scale_inv, y_bf16};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return W4A8_ERR_ALIGN;
    if ((xq_out && !aligned16(xq_out)) || (xs_out && !aligned16(xs_out)))
        return W4A8_ERR_ALIGN;
    if (!ws || ws_bytes < fp8_block_linear_workspace_size(M, N, K))
        return W4A8_ERR_WORKSPACE;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    BlkWs w;
    blk_ws(M, N, K, &w, ws);
    uint8_t* xq = xq_out ? xq_out : w.xq;
    if (launch_block_act_quant(x_bf16, M, K, xq, xs_out, w.xs_t, w.ld_t, w.tile_cnt, w.n_cnt, s) != cudaSuccess)
        return W4A8_ERR_LAUNCH;
    BlkLaunch L{};
    L.M = M;
    L.N = N;
    L.K = K;
    L.w = w_e4m3;
    L.wsi = w_scale_inv;
    L.y = y_bf16;
    L.xq = xq;
    L.xs_t = w.xs_t;
    L.ld_t = w.ld_t;
    L.ypart = w.ypart;
    L.tile_cnt = w.tile_cnt;
    L.err = static_cast<uint32_t*>(ws);
    const BlkConfig cfg = blk_pick_config(M, N, K, sms);
    return launch_block_gemm(L, cfg, sms, s);
}

int w4a8_set_profile_events(void* const* events, int count)
{
    if (count < 0 || count > 4)
        return W4A8_ERR_SHAPE;
    for (int i = 0; i < 4; ++i)
        g_profile_events[i] = (events && i < count) ? events[i] : nullptr;
    return W4A8_OK;
}

int w4a8_selftest_wait_timeout(void* ws, void* stream)
{
    if (!ws)
        return W4A8_ERR_NULL;
    if (!aligned16(ws))
        return W4A8_ERR_ALIGN;
    int sms;
    if (int st = current_device(&sms))
        return st;
    return launch_selftest_wait_timeout(static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_LAUNCH;
}

int w4a8_device_error(void* ws, int* code_out, void* stream)
{
    if (!ws || !code_out)
        return W4A8_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return W4A8_ERR_LAUNCH;
    *code_out = (word & 1u) ? W4A8_ERR_TIMEOUT : W4A8_OK;
    return W4A8_OK;
}

}  // extern "C"
