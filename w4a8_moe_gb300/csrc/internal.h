// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units. Every launcher only enqueues work on `s` and returns the
// launch status.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace w4a8 {

// Launch `kern` as a programmatic dependent of the previous kernel in the
// stream: it may start (and run its prologue) while that kernel finishes; it
// executes griddepcontrol.wait before touching the predecessor's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- quant.cu
cudaError_t launch_quantize_experts(const uint16_t* w, int E, int N, int K, int32_t* packed,
                                    float* scale, cudaStream_t s);
int act_amax_blocks(int64_t numel);
cudaError_t launch_act_amax(const uint16_t* x, int64_t numel, float* partial, int nblocks,
                            cudaStream_t s);
cudaError_t launch_act_encode(const uint16_t* x, int64_t numel, float* scale, int compute_scale,
                              const float* partial, int nblocks, uint8_t* out, cudaStream_t s);
cudaError_t launch_block_act_quant(const uint16_t* x, int M, int K, uint8_t* xq, float* xs_rowmajor,
                                   float* xs_t, int ld_t, int* zero, int nzero, cudaStream_t s);

// ---- route.cu
constexpr int kRouteChunk = 2048;         // assignments per histogram/scatter block
constexpr int kRouteFusedMax = 4096;      // T*k up to which one block does everything
constexpr int kRouteGatePartials = 16384; // fp32 partial logits the one-launch gate path reduces
cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                         float* w, int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                         int32_t* inv, int32_t* block_hist, int32_t* block_base, cudaStream_t s);
int route_gate_slice(int T, int H, int E, int k);
cudaError_t launch_route_gate(const uint16_t* x, const uint16_t* gate, int T, int H, int E, int k,
                              int renorm, float* logits, int write_logits, int32_t* ids, float* w, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_ids, int32_t* inv, float* partial,
                              int* done, int32_t* block_hist, int32_t* block_base, cudaStream_t s);

// ---- moe.cu
constexpr int kMaxKsplit = 16;   // largest split of the down projection's K
// Prefill down GEMM pacing: a CTA's weight stream passes checkpoint c (every
// kMoeSyncEvery stages) only after every CTA passed checkpoint c - kMoeSyncSlack
// (or finished), so the CTAs sharing L2-resident panels stay within a few
// dozen K-stages of each other. kMoeSyncInts counters: checkpoints, then the
// count of CTAs done.
constexpr int kMoeSyncInts = 1024;
constexpr int kMoeSyncEvery = 32;
constexpr int kMoeSyncSlack = 2;

struct MoeConfig {
    int bn;        // token tile (MMA N upper bound)
    int kc;        // K elements per pipeline stage
    int ksplit;    // split of the down projection's K (round-robin tiles)
    int streamk;   // 1: the down GEMM takes equal K-block ranges per CTA
    int nslots;    // stream-K partial slots per output
    int fused;     // 1: gate_up and down run in one launch (K split ksplit ways)
    int a8;        // 1: the weights are unpacked once per call (moe_upcast_kernel) and
                   //    the GEMMs load them by TMA (prefill-sized calls)
};
// Whether calls of T tokens unpack the weights once per call (and need room
// for the unpacked weights in the workspace).
bool moe_unpack_once(int T);
// one_launch: whether the caller's path allows both projections in one
// launch (not with the dynamic intermediate scale, which needs max|h| first)
MoeConfig moe_pick_config(int T, int H, int I, int E, int k, int num_sms, bool one_launch);
int moe_ksplit_max(int T, int k);
struct MoeLaunch {
    const uint8_t* xq; const float* a1; int T, H, I, E, k;
    const int32_t* w_gu; const float* s_gu; const int32_t* w_d; const float* s_d;
    const float* a2; int act;
    const int32_t* ids; const float* topk_w; const int32_t* counts; const int32_t* offsets;
    const int32_t* sorted_ids; const int32_t* inv;
    uint16_t* out;
    // workspace pieces
    uint8_t* xp; long long* s0x; uint8_t* hq; unsigned long long* s0h; float* ypart;
    uint8_t* wq8;  // unpacked weights [E, 2I, H] (gate_up, tile row order) then [E, H, I]
    int* done;  // [E] per-expert gate_up progress of the one-launch forward
    int* sync;  // prefill: [kMoeSyncInts] the down GEMM's pacing counters (zeroed by the gather)
    int* claim; // [2] its tile-claim counters (zero between calls)
    // dynamic intermediate scale (moe_w4a8_forward_dynamic): h in fp32, its
    // max as float bits, the scale written to a2_out
    int dynamic; float* hf; unsigned int* hmax; float* a2_out;
    uint32_t* err;
    void* events[4];  // optional cudaEvent_t recorded around the GEMMs
};
int launch_moe_forward(const MoeLaunch& L, const MoeConfig& cfg, int num_sms, cudaStream_t s);
// The checks moe_w4a8_forward makes before it looks at the workspace, in the
// same order (null pointers, shape, alignment); returns a public status code.
int moe_forward_check(const void* const* ptrs, int nptrs, int T, int H, int I, int E, int k, int act);

// ---- block_fp8.cu
struct BlkConfig {
    int bn;
    int ksplit;
};
BlkConfig blk_pick_config(int M, int N, int K, int num_sms);
int blk_ksplit_max(int M, int K);
struct BlkLaunch {
    int M, N, K;
    const uint8_t* w; const float* wsi; uint16_t* y;
    const uint8_t* xq; const float* xs_t; int ld_t;
    float* ypart; int* tile_cnt; uint32_t* err;
};
int launch_block_gemm(const BlkLaunch& L, const BlkConfig& cfg, int num_sms, cudaStream_t s);

// ---- fp8_linear.cu
struct FpConfig {
    int bn;
    int ksplit;
};
FpConfig fp8_pick_config(int M, int N, int K, int num_sms);
int fp8_ksplit_max(int M, int K);
struct FpLaunch {
    int M, N, K;
    const uint8_t* x; const float* sx; const uint8_t* w; const float* sw; uint16_t* y;
    float* ypart; int* tile_cnt; uint32_t* err;
};
int launch_fp8_linear(const FpLaunch& L, const FpConfig& cfg, int num_sms, cudaStream_t s);

// ---- selftest.cu
cudaError_t launch_selftest_wait_timeout(uint32_t* err, cudaStream_t s);

// ---- api.cu (tensor-map encoding through the driver entry point)
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swz);

// Status codes mirrored from the public header for use inside the library.
enum {
    kOK = 0, kErrNull = 1, kErrShape = 2, kErrAlign = 3, kErrWorkspace = 4, kErrDevice = 5,
    kErrLaunch = 6, kErrTimeout = 7
};

}  // namespace w4a8
