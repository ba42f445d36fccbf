// Router: softmax top-k with renormalized weights, per-expert histogram and a
// stable permutation of the T*k assignments grouped by expert.
//
// "ROCm: enable trillion-parameter MoE models with INT4-FP8 single node",
// config.json: num_local_experts, num_experts_per_tok, and ignored_layers (the
// block_sparse_moe.gate stays unquantized, so routing runs on fp32 logits).
//
// Selection ranks the fp32 logits (softmax is monotone), descending, equal
// logits by lower expert index. Weights: with renormalization
// w_j = exp(l_j - m) / sum_{j' selected} exp(l_j' - m), which equals the
// renormalized softmax probabilities; without it, the softmax over all E.
// Permutation: counting sort that keeps assignment order a = t*k + j within
// each expert, so the result is unique and compared bit-exactly.
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

constexpr int kMaxE = 256;

// Logits are read through the read-only path when they come from an earlier
// kernel, with plain loads when the same kernel has just written them.
template <bool kPlain>
__device__ __forceinline__ float load_logit(const float* p)
{
    return kPlain ? *p : __ldg(p);
}

// One warp per token; lane l holds logits l, l+32, ... (E <= 256).
template <bool kPlain = false>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int k,
                                            int renorm, int32_t* __restrict__ ids,
                                            float* __restrict__ w, int32_t* s_ids)
{
    const int lane = threadIdx.x & 31;
    float v[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? load_logit<kPlain>(logits + static_cast<int64_t>(t) * E + e) : -INFINITY;
    }
    uint32_t taken = 0;  // bit i: entry lane + 32 i already selected
    float mx = -INFINITY;
    float sel_sum = 0.0f;
    float sel_val[8];
    for (int j = 0; j < k; ++j) {
        // best among this lane's untaken entries: larger value, then lower index
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (be == 0x7FFFFFFF || v[i] > bv)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (j == 0)
            mx = bv;
        if (j < 8)
            sel_val[j] = bv;
        const float p = expf(bv - mx);
        sel_sum += p;
        if (lane == 0) {
            ids[static_cast<int64_t>(t) * k + j] = be;
            if (s_ids)
                s_ids[t * k + j] = be;
        }
    }
    float denom = sel_sum;
    if (!renorm) {
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i)
            if (lane + 32 * i < E)
                sum += expf(v[i] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        denom = sum;
    }
    if (lane == 0) {
        for (int j = 0; j < k; ++j) {
            float lv;
            if (j < 8) {
                lv = sel_val[j];
            } else {
                lv = load_logit<kPlain>(logits + static_cast<int64_t>(t) * E + ids[static_cast<int64_t>(t) * k + j]);
            }
            w[static_cast<int64_t>(t) * k + j] = __fdiv_rn(expf(lv - mx), denom);
        }
    }
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int renorm,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ w)
{
    grid_dep_wait();
    grid_dep_launch();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t < T)
        route_token(logits, t, E, k, renorm, ids, w, nullptr);
}

// Per-chunk expert histogram: block b counts assignments [b*C, (b+1)*C).
__global__ void __launch_bounds__(256) route_hist_kernel(const int32_t* __restrict__ ids, int A,
                                                         int E, int32_t* __restrict__ block_hist)
{
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int cnt[kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt[e] = 0;
    __syncthreads();
    const int a0 = blockIdx.x * kRouteChunk;
    const int a1 = min(A, a0 + kRouteChunk);
    for (int a = a0 + threadIdx.x; a < a1; a += blockDim.x)
        atomicAdd(&cnt[__ldg(ids + a)], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        block_hist[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

// Exclusive scan in (expert, block) order: base[b][e] = offsets[e] + sum of
// block_hist[b'][e] for b' < b. One block.
__global__ void __launch_bounds__(256) route_scan_kernel(const int32_t* __restrict__ block_hist,
                                                         int nb, int E, int A,
                                                         int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ block_base)
{
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int tot[kMaxE];
    __shared__ int off[kMaxE + 1];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int s = 0;
        for (int b = 0; b < nb; ++b)
            s += block_hist[static_cast<int64_t>(b) * E + e];
        tot[e] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            off[e] = run;
            run += tot[e];
        }
        off[E] = run;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        counts[e] = tot[e];
        offsets[e] = off[e];
        int run = off[e];
        for (int b = 0; b < nb; ++b) {
            block_base[static_cast<int64_t>(b) * E + e] = run;
            run += block_hist[static_cast<int64_t>(b) * E + e];
        }
    }
    if (threadIdx.x == 0)
        offsets[E] = A;
}

// Stable scatter of one chunk of assignments. Rounds of blockDim.x
// assignments in order; inside a round a warp ranks equal experts with
// match.any, warps are ordered through per-warp counts in shared memory, and
// `run` carries the per-expert count of earlier rounds.
template <int NW>
__device__ __forceinline__ void scatter_chunk(const int32_t* ids, int a0, int a1, int E,
                                              const int32_t* base, int* run, int (*wcnt)[kMaxE],
                                              int32_t* __restrict__ sorted_ids,
                                              int32_t* __restrict__ inv)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int r0 = a0; r0 < a1; r0 += NW * 32) {
        for (int e = lane; e < E; e += 32)
            wcnt[wid][e] = 0;
        __syncwarp();
        const int a = r0 + threadIdx.x;
        const bool valid = a < a1;
        const int e = valid ? ids[a] : -1;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (valid && rank == 0)
            wcnt[wid][e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int before = 0;
            for (int w2 = 0; w2 < wid; ++w2)
                before += wcnt[w2][e];
            const int pos = base[e] + run[e] + before + rank;
            sorted_ids[pos] = a;
            inv[a] = pos;
        }
        __syncthreads();
        for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
            int s = 0;
            for (int w2 = 0; w2 < NW; ++w2)
                s += wcnt[w2][e2];
            run[e2] += s;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) route_scatter_kernel(const int32_t* __restrict__ ids, int A,
                                                            int E,
                                                            const int32_t* __restrict__ block_base,
                                                            int32_t* __restrict__ sorted_ids,
                                                            int32_t* __restrict__ inv)
{
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int run[kMaxE];
    __shared__ int base[kMaxE];
    __shared__ int wcnt[8][kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        run[e] = 0;
        base[e] = block_base[static_cast<int64_t>(blockIdx.x) * E + e];
    }
    __syncthreads();
    const int a0 = blockIdx.x * kRouteChunk;
    const int a1 = min(A, a0 + kRouteChunk);
    scatter_chunk<8>(ids, a0, a1, E, base, run, wcnt, sorted_ids, inv);
}

// Small problems (T*k <= kRouteFusedMax): one block of 512 threads does
// top-k, histogram, scan and scatter.
// Histogram, scan and stable scatter of A <= kRouteFusedMax assignments whose
// experts are in s_ids (shared memory), by one block of 512 threads. Starts
// with a block barrier (s_ids written by other warps).
__device__ __forceinline__ void route_block_tail(const int32_t* s_ids, int A, int E,
                                                 int32_t* __restrict__ counts,
                                                 int32_t* __restrict__ offsets,
                                                 int32_t* __restrict__ sorted_ids,
                                                 int32_t* __restrict__ inv, int* cnt, int* base,
                                                 int (*wcnt)[kMaxE])
{
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt[e] = 0;
    __syncthreads();
    for (int a = threadIdx.x; a < A; a += blockDim.x)
        atomicAdd(&cnt[s_ids[a]], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            base[e] = run;
            offsets[e] = run;
            counts[e] = cnt[e];
            run += cnt[e];
        }
        offsets[E] = run;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt[e] = 0;  // reused as the running count
    __syncthreads();
    scatter_chunk<16>(s_ids, 0, A, E, base, cnt, wcnt, sorted_ids, inv);
}

__global__ void __launch_bounds__(512) route_fused_kernel(const float* __restrict__ logits, int T,
                                                           int E, int k, int renorm,
                                                           int32_t* __restrict__ ids,
                                                           float* __restrict__ w,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ sorted_ids,
                                                           int32_t* __restrict__ inv)
{
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int32_t s_ids[kRouteFusedMax];
    __shared__ int cnt[kMaxE];
    __shared__ int base[kMaxE];
    __shared__ int wcnt[16][kMaxE];
    const int A = T * k;
    const int wid = threadIdx.x >> 5;
    for (int t = wid; t < T; t += 16)
        route_token(logits, t, E, k, renorm, ids, w, s_ids);
    route_block_tail(s_ids, A, E, counts, offsets, sorted_ids, inv, cnt, base, wcnt);
}

// ---------------------------------------------------------------------------
// Router gate fused with routing: logits[t, e] = sum_h x[t, h] * G[e, h] in
// fp32 (bf16 operands, exact products), then the same top-k, histogram and
// permutation as above.
//
// "ROCm: enable trillion-parameter MoE models with INT4-FP8 single node",
// config.json: ignored_layers keeps the MoE gate unquantized, so it runs on the
// bf16 hidden states.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Small problems, one launch: block s computes the partial logits of H slice
// [s*HS, (s+1)*HS) for every token (one warp per token, 8 elements per lane for
// HS = 256, a fixed butterfly per expert) into partial[s, t, e]; the block that
// completes the grid-wide count sums the slices in order, routes every token
// and builds the permutation. `done` is zero at entry and left zero.
__global__ void __launch_bounds__(512) route_gate_fused_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gate, int T, int H, int E, int k,
    int renorm, int HS, float* __restrict__ partial, float* __restrict__ logits, int write_logits,
    int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ inv, int* __restrict__ done)
{
    grid_dep_wait();
    grid_dep_launch();
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ int32_t s_ids[kRouteFusedMax];
    __shared__ int cnt[kMaxE];
    __shared__ int base[kMaxE];
    __shared__ int wcnt[16][kMaxE];
    __shared__ int s_last;
    const int S = gridDim.x;
    const int s = blockIdx.x;
    const int h0 = s * HS;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int per_lane = HS / 32;   // 4, 8 or 16 elements, consecutive
    // the gate slice [E, HS] in shared memory (bf16)
    uint16_t* g_s = reinterpret_cast<uint16_t*>(dyn);
    const int chunks = E * (HS / 8);
    for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
        const int e = i / (HS / 8), c = i % (HS / 8);
        reinterpret_cast<uint4*>(g_s)[i] =
            __ldg(reinterpret_cast<const uint4*>(gate + static_cast<int64_t>(e) * H + h0) + c);
    }
    __syncthreads();
    for (int t = wid; t < T; t += 16) {
        float xv[16];
        const uint16_t* xr = x + static_cast<int64_t>(t) * H + h0 + lane * per_lane;
#pragma unroll
        for (int q = 0; q < 16; q += 8) {
            if (q + 8 <= per_lane) {   // 16-byte loads only for 8 or 16 elements per lane
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr + q));
                xv[q + 0] = bf16_lo(u.x); xv[q + 1] = bf16_hi(u.x);
                xv[q + 2] = bf16_lo(u.y); xv[q + 3] = bf16_hi(u.y);
                xv[q + 4] = bf16_lo(u.z); xv[q + 5] = bf16_hi(u.z);
                xv[q + 6] = bf16_lo(u.w); xv[q + 7] = bf16_hi(u.w);
            }
        }
        if (per_lane == 4) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(xr));
            xv[0] = bf16_lo(u.x); xv[1] = bf16_hi(u.x); xv[2] = bf16_lo(u.y); xv[3] = bf16_hi(u.y);
        }
        for (int e = 0; e < E; ++e) {
            const uint16_t* gr = g_s + e * HS + lane * per_lane;
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < 16; q += 2) {
                if (q < per_lane) {
                    const uint32_t gp = *reinterpret_cast<const uint32_t*>(gr + q);
                    acc = fmaf(xv[q], bf16_lo(gp), acc);
                    acc = fmaf(xv[q + 1], bf16_hi(gp), acc);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
            if (lane == 0)
                partial[(static_cast<int64_t>(s) * T + t) * E + e] = acc;
        }
    }
    // the last block to finish routes
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int old = atomicAdd(done, 1);
        const int last = (old == S - 1);
        if (last)
            __threadfence();
        s_last = last;
    }
    __syncthreads();
    if (!s_last)
        return;
    const int TE = T * E;
    float* red = reinterpret_cast<float*>(dyn);   // S*T*E partials (the gate slice is no longer needed)
#pragma unroll 8
    for (int i = threadIdx.x; i < S * TE; i += blockDim.x)
        red[i] = __ldcg(partial + i);
    __syncthreads();
    // the logits stay in shared memory for the routing (and go to global
    // memory only when the caller asked for them)
    float* lg = red + kRouteGatePartials;
    for (int i = threadIdx.x; i < TE; i += blockDim.x) {
        float acc = 0.0f;
        for (int q = 0; q < S; ++q)
            acc += red[q * TE + i];
        lg[i] = acc;
        if (write_logits)
            logits[i] = acc;
    }
    __syncthreads();
    for (int t = wid; t < T; t += 16)
        route_token<true>(lg, t, E, k, renorm, ids, w, s_ids);
    route_block_tail(s_ids, T * k, E, counts, offsets, sorted_ids, inv, cnt, base, wcnt);
    if (threadIdx.x == 0)
        *done = 0;
}

// Larger problems: one warp per token computes its E logits over the whole H
// (gate rows read through L2), writes them and routes the token.
__global__ void __launch_bounds__(256) route_gate_topk_kernel(const uint16_t* __restrict__ x,
                                                              const uint16_t* __restrict__ gate, int T,
                                                              int H, int E, int k, int renorm,
                                                              float* __restrict__ logits,
                                                              int32_t* __restrict__ ids,
                                                              float* __restrict__ w)
{
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T)
        return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
    for (int e = 0; e < E; ++e) {
        const uint4* gr = reinterpret_cast<const uint4*>(gate + static_cast<int64_t>(e) * H);
        float acc = 0.0f;
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 a = __ldg(xr + c), b = __ldg(gr + c);
            acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
            acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
            acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
            acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
            acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
            acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
            acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
            acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0)
            logits[static_cast<int64_t>(t) * E + e] = acc;
    }
    __syncwarp();
    route_token<true>(logits, t, E, k, renorm, ids, w, nullptr);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                         float* w, int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                         int32_t* inv, int32_t* block_hist, int32_t* block_base, cudaStream_t s)
{
    const int A = T * k;
    if (A <= kRouteFusedMax)
        return launch_dependent(route_fused_kernel, dim3(1), dim3(512), 0, s, logits, T, E, k, renorm, ids, w,
                                counts, offsets, sorted_ids, inv);
    const int nb = (A + kRouteChunk - 1) / kRouteChunk;
    cudaError_t e = launch_dependent(route_topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, logits, T, E, k,
                                     renorm, ids, w);
    if (e == cudaSuccess)
        e = launch_dependent(route_hist_kernel, dim3(nb), dim3(256), 0, s,
                             static_cast<const int32_t*>(ids), A, E, block_hist);
    if (e == cudaSuccess)
        e = launch_dependent(route_scan_kernel, dim3(1), dim3(256), 0, s, static_cast<const int32_t*>(block_hist),
                             nb, E, A, counts, offsets, block_base);
    if (e == cudaSuccess)
        e = launch_dependent(route_scatter_kernel, dim3(nb), dim3(256), 0, s, static_cast<const int32_t*>(ids), A,
                             E, static_cast<const int32_t*>(block_base), sorted_ids, inv);
    return e;
}

// Slice width of the one-launch gate path: the smallest of 128/256/512 whose
// S x T x E partials fit the reduction buffer, or 0 when none does (or when
// the problem is too large for one block to route).
int route_gate_slice(int T, int H, int E, int k)
{
    if (static_cast<int64_t>(T) * k > kRouteFusedMax)
        return 0;
    for (int hs = 128; hs <= 512; hs *= 2) {
        if (H % hs != 0)
            continue;
        const int64_t s = H / hs;
        if (s * T * E <= kRouteGatePartials && static_cast<int64_t>(E) * hs * 2 <= kRouteGatePartials * 4)
            return hs;
    }
    return 0;
}

cudaError_t launch_route_gate(const uint16_t* x, const uint16_t* gate, int T, int H, int E, int k,
                              int renorm, float* logits, int write_logits, int32_t* ids, float* w, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_ids, int32_t* inv, float* partial,
                              int* done, int32_t* block_hist, int32_t* block_base, cudaStream_t s)
{
    const int A = T * k;
    const int hs = route_gate_slice(T, H, E, k);
    if (hs) {
        // partial logits, then the summed logits [T, E] (T*E <= the partials' count)
        const size_t dyn = static_cast<size_t>(kRouteGatePartials) * 4 * 2;
        cudaError_t e = cudaFuncSetAttribute(route_gate_fused_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn));
        if (e != cudaSuccess)
            return e;
        return launch_dependent(route_gate_fused_kernel, dim3(H / hs), dim3(512), dyn, s, x, gate, T, H, E, k,
                                renorm, hs, partial, logits, write_logits, ids, w, counts, offsets, sorted_ids,
                                inv, done);
    }
    const int nb = (A + kRouteChunk - 1) / kRouteChunk;
    cudaError_t e = launch_dependent(route_gate_topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, x, gate, T, H,
                                     E, k, renorm, logits, ids, w);
    if (e == cudaSuccess)
        e = launch_dependent(route_hist_kernel, dim3(nb), dim3(256), 0, s,
                             static_cast<const int32_t*>(ids), A, E, block_hist);
    if (e == cudaSuccess)
        e = launch_dependent(route_scan_kernel, dim3(1), dim3(256), 0, s, static_cast<const int32_t*>(block_hist),
                             nb, E, A, counts, offsets, block_base);
    if (e == cudaSuccess)
        e = launch_dependent(route_scatter_kernel, dim3(nb), dim3(256), 0, s, static_cast<const int32_t*>(ids), A,
                             E, static_cast<const int32_t*>(block_base), sorted_ids, inv);
    return e;
}

}  // namespace w4a8
