/*
 * w4a8_moe.h -- C ABI of the GB300 (sm_103a) W4A8 mixture-of-experts library.
 *
 * The library computes the W4A8 MoE FFN of the pages
 *   "ROCm: enable trillion-parameter MoE models with INT4-FP8 single node"
 *       (sglang PR #4152; Motivation and config.json quantization_config), and
 *   "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm"
 *       (sglang PR #7392; description and review summary),
 * and the block-FP8 dense projection of
 *   "qwen4_exp: serve the block-FP8 dense projections natively (+25% decode)"
 *       (FreeToken PR #392; description and "What").
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers to caller-owned memory unless stated. The
 *    library never allocates, frees or synchronizes; every call only enqueues
 *    kernels on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *    default stream) and returns.
 *  - Arrays are row-major and contiguous; every pointer must be 16-byte
 *    aligned (W4A8_ERR_ALIGN otherwise).
 *  - bf16 is passed as uint16_t bit patterns; fp8 is OCP E4M3 ("fn": max 448,
 *    no infinity) as uint8_t codes.
 *  - Arguments are validated on the host before anything is enqueued; on an
 *    error nothing is launched and the status says why. No C++ exception
 *    crosses the ABI.
 *  - The library needs a GB300-class GPU (compute capability 10.3); on any
 *    other device, or without a device, calls return W4A8_ERR_DEVICE. There is
 *    no CPU fallback.
 *  - Workspace: calls that take `ws` need ws_bytes >= the matching
 *    *_workspace_size(). The first 256 bytes of every workspace are a header:
 *    the caller zero-fills them once when it allocates the workspace. Byte 0
 *    holds a device error word that kernels only OR bits into (a bounded wait
 *    that ran out sets bit 0); w4a8_device_error() reads and clears it. Calls
 *    may keep other counters in the header; every call leaves them zero.
 *  - Stateless and thread-safe; concurrent calls must use distinct workspaces.
 */
#ifndef W4A8_MOE_H
#define W4A8_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A8_OK = 0,
    W4A8_ERR_NULL = 1,      /* a required pointer is NULL                      */
    W4A8_ERR_SHAPE = 2,     /* a size is out of the supported range            */
    W4A8_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned                */
    W4A8_ERR_WORKSPACE = 4, /* ws is NULL or ws_bytes is too small             */
    W4A8_ERR_DEVICE = 5,    /* no sm_103 device, or the kernel image is absent */
    W4A8_ERR_LAUNCH = 6,    /* a CUDA launch or driver call failed             */
    W4A8_ERR_TIMEOUT = 7    /* reported by w4a8_device_error: a bounded wait ran out */
} w4a8_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* w4a8_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int w4a8_version(void);

/*
 * w4a8_quantize_experts -- column-wise symmetric INT4 quantization of expert
 * weights, 8 codes packed per int32 (PR #7392 review summary, "Core
 * Quantization Utilities": column-wise INT4 quantization and INT4 -> INT32
 * packing; PR #4152 config.json int4_experts {bits 4, sym true, group column}).
 *
 *   w_bf16 [E, N, K] bf16  : weights, output channel n, reduction index k.
 *   packed [E, N, K/8] i32 : out. Code k = 8j+i sits in bits 4i..4i+3 of word j
 *                            as a two's-complement nibble.
 *   scale  [E, N] fp32     : out. s = max_k |w| / 7 (1 for an all-zero row).
 *   Codes: q = clamp(rint(w / s), -8, 7), fp32 division, ties to even.
 *   Requires E >= 1, N >= 1, K a positive multiple of 8. Offline step (no ws).
 */
int w4a8_quantize_experts(const uint16_t* w_bf16, int E, int N, int K, int32_t* packed,
                          float* scale, void* stream);

/*
 * w4a8_quantize_act -- per-tensor ("tensor-wise", PR #7392 review summary)
 * FP8 quantization of activations with a static scale (PR #4152
 * quantization_config, activation_scheme "static").
 *
 *   x_bf16 [numel] bf16, numel a positive multiple of 16.
 *   scale  [1] fp32 (device). compute_scale = 1: calibrate, writes
 *          scale = max|x| / 448 (1 if x is all zero) and uses it;
 *          compute_scale = 0: reads the static scale.
 *   x_e4m3 [numel] u8: out, E4M3(x / scale) with fp32 division, RNE, +-448.
 *   ws: w4a8_quantize_act_workspace_size(numel) bytes (needed when
 *       compute_scale = 1; may be NULL with ws_bytes = 0 otherwise).
 */
int w4a8_quantize_act(const uint16_t* x_bf16, int64_t numel, float* scale, int compute_scale,
                      uint8_t* x_e4m3, void* ws, size_t ws_bytes, void* stream);
size_t w4a8_quantize_act_workspace_size(int64_t numel);

/*
 * moe_route -- softmax top-k routing with renormalized weights, expert
 * histogram and stable token permutation (the MoE gate of PR #4152 stays
 * unquantized: ignored_layers; num_experts_per_tok = k).
 *
 *   logits [T, E] fp32 : router logits (any bias already added).
 *   topk_ids [T, k] i32 : out. The k largest logits, descending; equal logits
 *                         are ranked by lower expert index.
 *   topk_w [T, k] fp32  : out. softmax(logits)[ids]; with renormalize = 1
 *                         divided by their sum (so each row sums to 1).
 *   counts [E] i32      : out. Assignments per expert.
 *   offsets [E+1] i32   : out. Exclusive prefix sum of counts; offsets[E] = T*k.
 *   sorted_ids [T*k] i32: out. Assignment a = t*k + j placed at
 *                         offsets[e] + (number of earlier assignments to e).
 *   inv_perm [T*k] i32  : out. inv_perm[sorted_ids[p]] = p.
 *   Requires T >= 1, 1 <= k <= E <= 256, T*k < 2^31.
 *   ws: moe_route_workspace_size(T, E, k) bytes.
 */
int moe_route(const float* logits, int T, int E, int k, int renormalize, int32_t* topk_ids,
              float* topk_w, int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
              int32_t* inv_perm, void* ws, size_t ws_bytes, void* stream);
size_t moe_route_workspace_size(int T, int E, int k);

/*
 * moe_route_gate -- the router gate and moe_route in one call: the MoE gate of
 * PR #4152 stays unquantized (config.json ignored_layers), so its logits are
 * computed here from the bf16 hidden states, then routed exactly as
 * moe_route does.
 *
 *   hidden_bf16 [T, H] bf16 : the MoE layer's input.
 *   gate_bf16   [E, H] bf16 : the gate weight (one row per expert).
 *   logits_out  [T, E] fp32 : optional out (NULL allowed).
 *                 logits[t, e] = sum_h hidden[t, h] * gate[e, h], products
 *                 exact in fp32, accumulated in fp32 in a fixed order (the
 *                 same inputs give the same bits).
 *   topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm: as moe_route,
 *                 computed from those fp32 logits.
 *   Requires T >= 1, H a positive multiple of 128, 1 <= k <= E <= 256,
 *   T*k < 2^31. For T*k <= 4096 the whole call is one kernel.
 *   ws: moe_route_gate_workspace_size(T, H, E, k) bytes; its first 256 bytes
 *       must be zero before the first call on that workspace (every call
 *       leaves them zero). Calls that share a workspace must not overlap on
 *       the GPU.
 */
int moe_route_gate(const uint16_t* hidden_bf16, const uint16_t* gate_bf16, int T, int H, int E, int k,
                   int renormalize, float* logits_out, int32_t* topk_ids, float* topk_w, int32_t* counts,
                   int32_t* offsets, int32_t* sorted_ids, int32_t* inv_perm, void* ws, size_t ws_bytes,
                   void* stream);
size_t moe_route_gate_workspace_size(int T, int H, int E, int k);

/*
 * moe_w4a8_forward -- the W4A8 MoE FFN (PR #7392 description: INT4 expert
 * weights upcast to FP8 so that FP8 math is used; PR #4152 Motivation: FP8
 * tensor cores, INT4 weights for lower memory bandwidth).
 *
 * For every assignment a = (t, j) with expert e = topk_ids[t, j]:
 *   gate_i = a1 * S_gu[e, i]     * sum_h x[t,h] q_gu[e, i, h]         (i < I)
 *   up_i   = a1 * S_gu[e, I + i] * sum_h x[t,h] q_gu[e, I + i, h]
 *   h_i    = act(gate_i) * up_i,  act = SiLU (act = 0) or GELU-tanh (act = 1)
 *   hq_i   = E4M3(h_i / a2)     (static scale a2; IEEE fp32 division, one RNE rounding)
 *   y_n    = a2 * S_d[e, n] * sum_i hq_i q_d[e, n, i]
 *   out[t, n] = bf16( sum_j topk_w[t, j] * y_n(t, j) )
 * with x = dec(x_e4m3) and fp32 tensor-core accumulation.
 *
 *   x_e4m3 [T, H] u8; a1_scale [1] fp32; a2_scale [1] fp32 (device pointers).
 *   w_gu [E, 2I, H/8] i32 and s_gu [E, 2I] fp32 from w4a8_quantize_experts of
 *        a [E, 2I, H] weight whose rows [0, I) are the gate, [I, 2I) the up.
 *   w_d  [E, H, I/8] i32 and s_d [E, H] fp32.
 *   topk_ids, topk_w, counts, offsets, sorted_ids, inv_perm: from moe_route.
 *   out_bf16 [T, H] bf16: out.
 *   Requires H and I positive multiples of 128, 1 <= k <= E <= 256, T >= 1.
 *   ws: moe_w4a8_workspace_size(T, H, I, E, k) bytes. Above 128 tokens this
 *       includes E * 3 * I * H bytes where the call unpacks the INT4 weights of
 *       the experts with tokens once (to E4M3 operand bytes) before the GEMMs,
 *       and 4 KB of pacing counters for the down GEMM.
 * Up to 128 tokens both projections run in one persistent launch (one CTA per
 * SM; see moe_w4a8_plan) whose down tiles wait for the gate_up tiles of the
 * same expert in other CTAs; above 128 tokens the CTAs of the down launch pace
 * their weight streams against each other (grid-wide checkpoints). Those waits
 * assume every CTA of the launch gets an SM within the bounded-wait budget
 * (about 2 s): kernels on other streams that hold SMs for longer make the call
 * report W4A8_ERR_TIMEOUT through w4a8_device_error instead of hanging.
 */
int moe_w4a8_forward(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I, int E,
                     int k, const int32_t* w_gu, const float* s_gu, const int32_t* w_d,
                     const float* s_d, const float* a2_scale, int act, const int32_t* topk_ids,
                     const float* topk_w, const int32_t* counts, const int32_t* offsets,
                     const int32_t* sorted_ids, const int32_t* inv_perm, uint16_t* out_bf16,
                     void* ws, size_t ws_bytes, void* stream);
size_t moe_w4a8_workspace_size(int T, int H, int I, int E, int k);

/*
 * moe_w4a8_plan -- the launch plan moe_w4a8_forward (dynamic = 0) or
 * moe_w4a8_forward_dynamic (dynamic = 1) uses for a shape on a GPU with
 * num_sms SMs. Host only: no device is touched, so it also runs without a
 * GPU. The plan does not change the result beyond the order in which fp32
 * partial sums of the down projection are added.
 *
 *   plan [8] int32 (host), out:
 *     [0] token tile (MMA N bound: 32, 64, 128 or 256)
 *     [1] K elements per pipeline stage
 *     [2] K split of the down projection
 *     [3] 1 when the down projection runs stream-K (equal K ranges per CTA)
 *     [4] stream-K partial slots per output (0 otherwise)
 *     [5] 1 when both projections run in one launch (static scale, token tile
 *         up to 128), 0 when gate_up and down are separate launches
 *     [6] kernel launches of one forward call
 *     [7] partial sums per output that the combine adds
 *   Returns W4A8_ERR_SHAPE for shapes moe_w4a8_forward rejects or
 *   num_sms < 1, W4A8_ERR_NULL for a null plan.
 */
int moe_w4a8_plan(int T, int H, int I, int E, int k, int dynamic, int num_sms, int32_t* plan);

/*
 * moe_w4a8_workspace_layout -- inspection hook (the pages have no
 * counterpart): where, inside the workspace of moe_w4a8_forward or
 * moe_w4a8_forward_dynamic for this shape, a call leaves its intermediate
 * tensors, so that tests can compare them with a reference. Host only.
 *
 *   offsets [2] int64 (host), out: byte offsets from the workspace start of
 *     [0] hq [T*k, I] u8: the E4M3 codes of h / a2. Row p holds assignment
 *         a = sorted_ids[p] (token a / k, slot a % k); inside every group of
 *         8 columns the codes of i = 8g + {0, 2, 4, 6, 1, 3, 5, 7}, the K
 *         order the down projection consumes.
 *     [1] xp [T*k, H] u8: the gathered E4M3 activations, same row and
 *         column orders.
 *   Returns W4A8_ERR_SHAPE for shapes moe_w4a8_forward rejects,
 *   W4A8_ERR_NULL for a null offsets.
 */
int moe_w4a8_workspace_layout(int T, int H, int I, int E, int k, int64_t* offsets);

/*
 * moe_w4a8_forward_dynamic -- moe_w4a8_forward with the intermediate
 * activation's scale calibrated on the device for every call instead of read:
 *   a2 = max |h_i| / 448 over every assignment and i of the call (1 when all
 *        h are zero), written to a2_out [1] fp32 (device), then used exactly
 *        as the static a2 of moe_w4a8_forward.
 * PR #4152 quantization_config fixes "static" activation scales; this variant
 * is for callers without a calibrated a2 (the same per-tensor scheme, taken
 * over the current batch).
 *   All other arguments as moe_w4a8_forward.
 *   ws: moe_w4a8_dynamic_workspace_size(T, H, I, E, k) bytes (it adds the
 *       fp32 intermediate [T*k, I]).
 */
int moe_w4a8_forward_dynamic(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I, int E, int k,
                             const int32_t* w_gu, const float* s_gu, const int32_t* w_d, const float* s_d,
                             float* a2_out, int act, const int32_t* topk_ids, const float* topk_w,
                             const int32_t* counts, const int32_t* offsets, const int32_t* sorted_ids,
                             const int32_t* inv_perm, uint16_t* out_bf16, void* ws, size_t ws_bytes, void* stream);
size_t moe_w4a8_dynamic_workspace_size(int T, int H, int I, int E, int k);

/*
 * moe_w4a8_forward_static -- moe_w4a8_forward for callers that cannot
 * allocate device memory. The pages have no counterpart: this is a deployment
 * variant of the same computation.
 *
 * Some callers have no allocator to give the library a workspace: a host
 * application that owns the whole device-memory budget and hands plugins only
 * their inputs and outputs, or a latency-critical loop that must never call
 * cudaMalloc (which can synchronize the device or fail at an unpredictable
 * moment). This entry point takes the same inputs and outputs as
 * moe_w4a8_forward, minus ws/ws_bytes, and uses instead a scratch array of
 * W4A8_STATIC_SCRATCH_BYTES that lives in the library's own device image: every
 * CUDA context that loads the library reserves it until the process exits. It
 * calls no allocating function.
 *
 *   - Arguments are checked as moe_w4a8_forward checks them (W4A8_ERR_NULL,
 *     W4A8_ERR_SHAPE, W4A8_ERR_ALIGN, in that order); then problems whose
 *     moe_w4a8_workspace_size(T, H, I, E, k) exceeds W4A8_STATIC_SCRATCH_BYTES
 *     return W4A8_ERR_WORKSPACE (use moe_w4a8_forward with a caller workspace
 *     for those); the limit covers decode-sized layers (e.g. 32 tokens of a
 *     Grok-1-shaped layer, or 128 tokens of a Mixtral-shaped one).
 *   - The first call in a CUDA context (the device's primary context, or a
 *     context the application made current) looks up the array's device
 *     address in that context (cudaGetSymbolAddress) and caches it under the
 *     context handle; make that first call before any stream capture. A
 *     context that is destroyed must not be followed by a new context at the
 *     same handle in the same process.
 *   - All calls in a context share the one array and it keeps the last call's
 *     contents; the state each call needs cleared is cleared by the call's
 *     first kernel. Calls whose kernels overlap on the GPU (concurrent streams,
 *     or host threads using the same device) race on the array: serialize
 *     them, e.g. on one stream.
 *   - A bounded device wait that runs out sets the array's error word (as it
 *     would a workspace's); moe_w4a8_forward_static_error reads and clears it.
 */
#define W4A8_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
int moe_w4a8_forward_static(const uint8_t* x_e4m3, const float* a1_scale, int T, int H, int I,
                            int E, int k, const int32_t* w_gu, const float* s_gu,
                            const int32_t* w_d, const float* s_d, const float* a2_scale, int act,
                            const int32_t* topk_ids, const float* topk_w, const int32_t* counts,
                            const int32_t* offsets, const int32_t* sorted_ids,
                            const int32_t* inv_perm, uint16_t* out_bf16, void* stream);

/*
 * moe_w4a8_forward_static_error -- w4a8_device_error for the built-in scratch
 * array of moe_w4a8_forward_static in the current context: *code_out receives
 * W4A8_OK, or W4A8_ERR_TIMEOUT when one of its kernels gave up on a bounded
 * wait since the last read; the word is cleared. Synchronizes `stream`.
 * Allocates nothing. Returns W4A8_OK, W4A8_ERR_NULL, W4A8_ERR_DEVICE or
 * W4A8_ERR_LAUNCH.
 */
int moe_w4a8_forward_static_error(int* code_out, void* stream);

/*
 * fp8_linear -- per-tensor FP8 dense projection ("[AMD][Quantization] Add
 * int4fp8_moe online quantization on ROCm", description: the attention
 * projections are quantized online to float8; review summary:
 * QuarkInt4Fp8LinearMethod, tensor-wise FP8 quantization).
 *
 *   y[m, n] = bf16( x_scale * w_scale * sum_k dec(x_e4m3[m, k]) * dec(w_e4m3[n, k]) )
 * with fp32 tensor-core accumulation.
 *
 *   x_e4m3 [M, K] u8, x_scale [1] fp32 (device): e.g. from w4a8_quantize_act.
 *   w_e4m3 [N, K] u8, w_scale [1] fp32 (device): the weight quantized with
 *          w4a8_quantize_act (compute_scale = 1) once, at load.
 *   y_bf16 [M, N]: out.
 *   Requires M >= 1, N and K positive multiples of 128.
 *   ws: fp8_linear_workspace_size(M, N, K) bytes, zero-filled before its first
 *       use with this function (calls leave the split-K counters at zero; after
 *       a W4A8_ERR_TIMEOUT report, zero it again). Calls that share a workspace
 *       must not overlap on the GPU.
 */
int fp8_linear(const uint8_t* x_e4m3, const float* x_scale, int M, int N, int K, const uint8_t* w_e4m3,
               const float* w_scale, uint16_t* y_bf16, void* ws, size_t ws_bytes, void* stream);
size_t fp8_linear_workspace_size(int M, int N, int K);

/*
 * fp8_block_linear -- block-FP8 dense projection y = x W^T (PR #392
 * description: FP8_PB_WO weights consumed with their weight_scale_inv, one
 * fp32 scale per 128-row x 128-col block).
 *
 *   x_bf16 [M, K] bf16: activations, quantized inside the call per token and
 *          128-column group g: xs[m, g] = max|x| / 448 (1 if zero),
 *          xq = E4M3(x / xs).
 *   w_e4m3 [N, K] u8; w_scale_inv [N/128, K/128] fp32: w ~ dec(w_e4m3) * Wsi.
 *   y_bf16 [M, N] bf16: out, y[m, n] = sum_g xs[m,g] Wsi[n/128,g]
 *          sum_{k in g} dec(xq[m,k]) dec(w[n,k]), fp32 accumulation.
 *   xq_out [M, K] u8 and xs_out [M, K/128] fp32: optional outputs (may be NULL).
 *   Requires M >= 1, N and K positive multiples of 128.
 *   ws: fp8_block_linear_workspace_size(M, N, K) bytes.
 */
int fp8_block_linear(const uint16_t* x_bf16, int M, int N, int K, const uint8_t* w_e4m3,
                     const float* w_scale_inv, uint16_t* y_bf16, uint8_t* xq_out, float* xs_out,
                     void* ws, size_t ws_bytes, void* stream);
size_t fp8_block_linear_workspace_size(int M, int N, int K);

/*
 * w4a8_set_profile_events -- measurement hook (not part of the method). Sets,
 * for the calling host thread, up to four cudaEvent_t handles that
 * moe_w4a8_forward records on its stream: [0] before the gate_up GEMM,
 * [1] after it, [2] after the down GEMM, [3] after the final combine.
 * count = 0 (or events = NULL) switches recording off. Returns W4A8_OK, or
 * W4A8_ERR_SHAPE for count outside 0..4.
 */
int w4a8_set_profile_events(void* const* events, int count);

/*
 * w4a8_selftest_wait_timeout -- test hook for the error path of the pipelined
 * kernels (the pages have no counterpart). Every mbarrier wait of those kernels
 * gives up after a cycle budget and sets the workspace error word, which
 * w4a8_device_error reports as W4A8_ERR_TIMEOUT. This call runs one small
 * kernel that waits on a barrier nothing completes, with a budget of about
 * 10 ms, so that error is recorded in ws (at least 256 bytes, 16-byte aligned)
 * without any other effect; the context stays usable.
 */
int w4a8_selftest_wait_timeout(void* ws, void* stream);

/*
 * w4a8_device_error -- read and clear the device error word of a workspace.
 * Synchronizes `stream` (the only call that does). *code_out receives
 * W4A8_OK, or W4A8_ERR_TIMEOUT when a kernel gave up on a bounded wait since
 * the last read. Returns W4A8_OK or W4A8_ERR_NULL / W4A8_ERR_LAUNCH.
 */
int w4a8_device_error(void* ws, int* code_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* W4A8_MOE_H */
