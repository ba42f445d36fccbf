// Quantizers: column-wise INT4 expert weights packed 8 per int32, per-tensor
// static-scale E4M3 activations, and per-token x 128-column E4M3 activations
// for the block-FP8 projection.
//
// "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm", review
// summary ("Core Quantization Utilities": tensor-wise FP8, column-wise INT4,
// INT4 packed into INT32); "ROCm: enable trillion-parameter MoE models with
// INT4-FP8 single node", config.json quantization_config (int4_experts: bits 4,
// sym, group column; activation_scheme static); "qwen4_exp: serve the
// block-FP8 dense projections natively", description (128x128 weight blocks).
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

// ---------------------------------------------------------------------------
// INT4 experts: one warp per output channel (row of K weights). Pass 1 finds
// max|w|, s = max/7 (IEEE division; 1 for an all-zero row); pass 2 writes
// q = clamp(rint(w/s), -8, 7) as nibbles, code 8j+i in bits 4i..4i+3 of word j.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quantize_experts_kernel(const uint16_t* __restrict__ w,
                                                               int64_t rows, int K,
                                                               int32_t* __restrict__ packed,
                                                               float* __restrict__ scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    const uint4* src = reinterpret_cast<const uint4*>(w + row * K);
    const int nchunk = K / 8;  // 8 bf16 = 16 bytes = one packed word
    float amax = 0.0f;
    for (int c = lane; c < nchunk; c += 32) {
        const uint4 v = __ldg(src + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            amax = fmaxf(amax, fabsf(__uint_as_float(u[i] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(u[i] & 0xFFFF0000u)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 7.0f);
    if (lane == 0)
        scale[row] = s;
    int32_t* dst = packed + row * nchunk;
    for (int c = lane; c < nchunk; c += 32) {
        const uint4 v = __ldg(src + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(u[i] << 16);
            const float hi = __uint_as_float(u[i] & 0xFFFF0000u);
            int q0 = __float2int_rn(__fdiv_rn(lo, s));
            int q1 = __float2int_rn(__fdiv_rn(hi, s));
            q0 = min(7, max(-8, q0));
            q1 = min(7, max(-8, q1));
            word |= (static_cast<uint32_t>(q0) & 0xFu) << (8 * i);
            word |= (static_cast<uint32_t>(q1) & 0xFu) << (8 * i + 4);
        }
        dst[c] = static_cast<int32_t>(word);
    }
}

cudaError_t launch_quantize_experts(const uint16_t* w, int E, int N, int K, int32_t* packed,
                                    float* scale, cudaStream_t s)
{
    const int64_t rows = static_cast<int64_t>(E) * N;
    const int64_t blocks = (rows + 7) / 8;
    quantize_experts_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(w, rows, K, packed, scale);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-tensor activation quantization. amax: per-block maxima (deterministic,
// no atomics); encode: every block reduces the maxima itself, derives
// s = amax/448 (1 if zero), block 0 publishes it; then xq = E4M3(x / s).
// ---------------------------------------------------------------------------
int act_amax_blocks(int64_t numel)
{
    const int64_t per_block = 256 * 16;
    int64_t b = (numel + per_block - 1) / per_block;
    if (b > 1024)
        b = 1024;
    if (b < 1)
        b = 1;
    return static_cast<int>(b);
}

__device__ __forceinline__ float block_max(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (threadIdx.x == 0)
            red[0] = v;
    }
    __syncthreads();
    return red[0];
}

__global__ void __launch_bounds__(256) act_amax_kernel(const uint16_t* __restrict__ x, int64_t nvec,
                                                       float* __restrict__ partial)
{
    __shared__ float red[8];
    float m = 0.0f;
    const uint4* v = reinterpret_cast<const uint4*>(x);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 q = __ldg(v + i);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(__uint_as_float(u[j] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(u[j] & 0xFFFF0000u)));
        }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0)
        partial[blockIdx.x] = m;
}

__device__ __forceinline__ uint32_t enc4(uint32_t a, uint32_t b, float s)
{
    // a, b: 4 bf16; returns 4 E4M3 codes of x / s (IEEE division).
    const float x0 = __uint_as_float(a << 16), x1 = __uint_as_float(a & 0xFFFF0000u);
    const float x2 = __uint_as_float(b << 16), x3 = __uint_as_float(b & 0xFFFF0000u);
    const uint32_t lo = cvt_e4m3x2(__fdiv_rn(x1, s), __fdiv_rn(x0, s));
    const uint32_t hi = cvt_e4m3x2(__fdiv_rn(x3, s), __fdiv_rn(x2, s));
    return lo | (hi << 16);
}

__global__ void __launch_bounds__(256) act_encode_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                         float* __restrict__ scale, int compute,
                                                         const float* __restrict__ partial,
                                                         int nblocks, uint8_t* __restrict__ out)
{
    __shared__ float red[8];
    float s;
    if (compute) {
        float m = 0.0f;
        for (int i = threadIdx.x; i < nblocks; i += blockDim.x)
            m = fmaxf(m, partial[i]);
        m = block_max(m, red);
        s = (m == 0.0f) ? 1.0f : __fdiv_rn(m, 448.0f);
        if (blockIdx.x == 0 && threadIdx.x == 0)
            scale[0] = s;
    } else {
        s = __ldg(scale);
    }
    const uint4* v = reinterpret_cast<const uint4*>(x);
    uint4* o = reinterpret_cast<uint4*>(out);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 p = __ldg(v + 2 * i);
        const uint4 q = __ldg(v + 2 * i + 1);
        uint4 r;
        r.x = enc4(p.x, p.y, s);
        r.y = enc4(p.z, p.w, s);
        r.z = enc4(q.x, q.y, s);
        r.w = enc4(q.z, q.w, s);
        o[i] = r;
    }
}

cudaError_t launch_act_amax(const uint16_t* x, int64_t numel, float* partial, int nblocks,
                            cudaStream_t s)
{
    act_amax_kernel<<<nblocks, 256, 0, s>>>(x, numel / 8, partial);
    return cudaGetLastError();
}

cudaError_t launch_act_encode(const uint16_t* x, int64_t numel, float* scale, int compute_scale,
                              const float* partial, int nblocks, uint8_t* out, cudaStream_t s)
{
    const int64_t n16 = numel / 16;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    if (blocks < 1)
        blocks = 1;
    act_encode_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, n16, scale, compute_scale,
                                                                   partial, nblocks, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Block-FP8 activation side: one warp per (token m, 128-column group g).
// s = amax/448 (1 if zero); xq = E4M3(x / s). Writes the [M, K/128] scales
// (optional) and a transposed copy [K/128, ld_t] that the GEMM stages by TMA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) block_act_quant_kernel(const uint16_t* __restrict__ x, int M,
                                                              int K, uint8_t* __restrict__ xq,
                                                              float* __restrict__ xs,
                                                              float* __restrict__ xs_t, int ld_t,
                                                              int* __restrict__ zero, int nzero)
{
    // The one dependent of this kernel is the block-FP8 GEMM of the same call,
    // which before its own wait only streams the weights (written by no kernel
    // of this library), so it may launch at once: its weight stream then
    // overlaps this kernel and the previous call's tail. This kernel itself
    // waits before touching the workspace, which the previous call's GEMM may
    // still be using.
    grid_dep_launch();
    grid_dep_wait();
    // clear the GEMM's split-K tile counters of this call
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nzero;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        zero[i] = 0;
    const int lane = threadIdx.x & 31;
    const int G = K / 128;
    const int64_t grp = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (grp >= static_cast<int64_t>(M) * G)
        return;
    const int m = static_cast<int>(grp / G), g = static_cast<int>(grp % G);
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + static_cast<int64_t>(m) * K + g * 128) + lane);
    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
    float a = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
    const uint32_t lo = cvt_e4m3x2(__fdiv_rn(x1, s), __fdiv_rn(x0, s));
    const uint32_t hi = cvt_e4m3x2(__fdiv_rn(x3, s), __fdiv_rn(x2, s));
    reinterpret_cast<uint32_t*>(xq + static_cast<int64_t>(m) * K + g * 128)[lane] = lo | (hi << 16);
    if (lane == 0) {
        if (xs)
            xs[static_cast<int64_t>(m) * G + g] = s;
        xs_t[static_cast<int64_t>(g) * ld_t + m] = s;
    }
}

cudaError_t launch_block_act_quant(const uint16_t* x, int M, int K, uint8_t* xq, float* xs_rowmajor,
                                   float* xs_t, int ld_t, int* zero, int nzero, cudaStream_t s)
{
    const int64_t groups = static_cast<int64_t>(M) * (K / 128);
    const int64_t blocks = (groups + 7) / 8;
    return launch_dependent(block_act_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, x, M, K,
                            xq, xs_rowmajor, xs_t, ld_t, zero, nzero);
}

}  // namespace w4a8
