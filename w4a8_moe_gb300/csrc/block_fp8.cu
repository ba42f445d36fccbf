// Block-FP8 dense projection y = x W^T on sm_103a.
//
// "qwen4_exp: serve the block-FP8 dense projections natively (+25% decode)",
// description and "What": FP8_PB_WO weights e4m3 [N, K] are consumed together
// with weight_scale_inv [N/128, K/128], one fp32 scale per 128-row x 128-col
// block, instead of being dequantized to bf16 at load.
//
// Activations carry one scale per token and 128-column group, so every K-block
// of 128 has its own pair of scales: the tensor cores produce the block's fp32
// partial product in TMEM (4 MMAs of K = 32), and the epilogue warps fold it
// into register accumulators as  acc += partial * xs[m, g] * Wsi[n/128, g].
// Two TMEM partial buffers let the MMA of block g+1 overlap that fold.
//
// Roles (12 warps): warp 0 TMA (weight tile 128x128, activation tile BNx128,
// the BN activation scales of the block), warp 1 TMEM + MMA issuer, warps
// 4-11 epilogue (two warps per 32-lane TMEM quadrant, each half of the BN
// token columns). Swapped operands: M = 128 weight rows, N = BN tokens.
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

struct BlkParams {
    int M, N, K, KB;
    int kb_per_split, ksplit, mt_count, nb_count;
    const float* wsi;   // [N/128, K/128]
    float* ypart;       // [ksplit, M, N] when ksplit > 1
    uint16_t* y;        // [M, N]
    uint32_t* err;
};

template <int BN, int PST>
struct BlkTraits {
    static constexpr int kA = 128 * 128;
    static constexpr int kB = BN * 128;
    static constexpr int kS = ((BN * 4 + 1023) / 1024) * 1024;
    static constexpr int kStage = kA + kB + kS;
    static constexpr int kData = PST * kStage;
    static constexpr int kBars = 2 * PST + 4 + 1;
    static constexpr int kSmem = 1024 + kData + kBars * 8 + 16;
    static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
    static constexpr int kHalf = BN / 2;
    static constexpr int kChunk = kHalf < 32 ? kHalf : 32;
    static_assert(kB % 1024 == 0, "stage alignment");
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r);

template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t* r)
{
    uint32_t (&v)[32] = *reinterpret_cast<uint32_t(*)[32]>(r);
    tmem_ld32(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

template <int BN, int PST>
__global__ void __launch_bounds__(384, 1)
    blk_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_s, const BlkParams p)
{
    using Tr = BlkTraits<BN, PST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kData);
    uint64_t* full = bars;
    uint64_t* empty = full + PST;
    uint64_t* dfull = empty + PST;
    uint64_t* dempty = dfull + 2;
    uint64_t* drain = dempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < PST; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1 + 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&dfull[i]), 1);
            mbar_init(smem_u32(&dempty[i]), 8);
        }
        mbar_init(smem_u32(drain), 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_s);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), Tr::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int per_nb = p.mt_count * p.ksplit;
    const int total = p.nb_count * per_nb;

    auto fail = [&]() {
        *s_abort = 1;
        set_error(p.err, kErrBitTimeout);
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int ps = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
                for (int kb = 0; kb < p.kb_per_split; ++kb) {
                    if (*s_abort || !mbar_wait(smem_u32(&empty[ps]), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const int g = ks * p.kb_per_split + kb;
                    const uint32_t fb = smem_u32(&full[ps]);
                    uint8_t* st = smem + ps * Tr::kStage;
                    mbar_arrive_expect_tx(fb, Tr::kA + Tr::kB + BN * 4);
                    tma_load_2d_hint(smem_u32(st), &tm_w, g * 128, nb * 128, fb, pol_w);
                    tma_load_2d_hint(smem_u32(st + Tr::kA), &tm_x, g * 128, mt * BN, fb, pol_x);
                    tma_load_2d(smem_u32(st + Tr::kA + Tr::kB), &tm_s, mt * BN, g, fb);
                    issued |= 1u << ps;
                    last_par = (last_par & ~(1u << ps)) | (ph << ps);
                    if (++ps == PST) {
                        ps = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                fail();
                for (int s = 0; s < PST; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait(smem_u32(&full[s]), (last_par >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3_f32(128, BN);
            int ps = 0;
            uint32_t ph = 0, kc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.kb_per_split; ++kb, ++kc) {
                    const int d = kc & 1;
                    const uint32_t use = kc >> 1;
                    if (*s_abort || !mbar_wait(smem_u32(&dempty[d]), (use & 1u) ^ 1u) ||
                        !mbar_wait(smem_u32(&full[ps]), ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + ps * Tr::kStage);
                    const uint32_t b0 = a0 + Tr::kA;
                    const uint32_t dt = tmem + static_cast<uint32_t>(d * BN);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f8(dt, desc_kmajor_sw128(a0 + kk * 32), desc_kmajor_sw128(b0 + kk * 32),
                                idesc, kk ? 1u : 0u);
                    umma_commit(smem_u32(&dfull[d]));
                    umma_commit(smem_u32(&empty[ps]));
                    if (++ps == PST) {
                        ps = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                fail();
                umma_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0);
            }
        }
    } else if (warp >= 4) {
        const int q = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int c0 = hh * Tr::kHalf;
        int ps = 0;
        uint32_t ph = 0, kc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
            float acc[Tr::kHalf];
#pragma unroll
            for (int c = 0; c < Tr::kHalf; ++c)
                acc[c] = 0.0f;
            for (int kb = 0; kb < p.kb_per_split; ++kb, ++kc) {
                const int d = kc & 1;
                const uint32_t use = kc >> 1;
                // the stage's scales were written by TMA: observe its barrier too
                if (*s_abort || !mbar_wait(smem_u32(&dfull[d]), use & 1u) ||
                    !mbar_wait(smem_u32(&full[ps]), ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int g = ks * p.kb_per_split + kb;
                const float ws = __ldg(p.wsi + static_cast<int64_t>(nb) * p.KB + g);
                const float* xs = reinterpret_cast<const float*>(smem + ps * Tr::kStage + Tr::kA + Tr::kB);
                const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(d * BN + c0);
#pragma unroll
                for (int ch = 0; ch < Tr::kHalf / Tr::kChunk; ++ch) {
                    uint32_t v[Tr::kChunk];
                    tmem_ld_cols<Tr::kChunk>(tb + ch * Tr::kChunk, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < Tr::kChunk; ++c)
                        acc[ch * Tr::kChunk + c] =
                            fmaf(__uint_as_float(v[c]), xs[c0 + ch * Tr::kChunk + c] * ws,
                                 acc[ch * Tr::kChunk + c]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&dempty[d]));
                    mbar_arrive(smem_u32(&empty[ps]));
                }
                if (++ps == PST) {
                    ps = 0;
                    ph ^= 1u;
                }
            }
            if (!ok)
                break;
            const int n = nb * 128 + q * 32 + lane;
#pragma unroll
            for (int c = 0; c < Tr::kHalf; ++c) {
                const int m = mt * BN + c0 + c;
                if (m < p.M) {
                    if (p.ksplit == 1)
                        p.y[static_cast<int64_t>(m) * p.N + n] = float_to_bf16_bits(acc[c]);
                    else
                        p.ypart[(static_cast<int64_t>(ks) * p.M + m) * p.N + n] = acc[c];
                }
            }
        }
        if (!ok)
            fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Tr::kTmemCols);
    }
}

// y[m, n] = bf16( sum_s ypart[s, m, n] ), splits in order.
__global__ void __launch_bounds__(256) blk_reduce_kernel(const float* __restrict__ ypart, int ksplit,
                                                         int64_t MN, uint16_t* __restrict__ y)
{
    const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i >= MN)
        return;
    float4 a = __ldg(reinterpret_cast<const float4*>(ypart + i));
    for (int s = 1; s < ksplit; ++s) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(ypart + s * MN + i));
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
    }
    uint2 o;
    o.x = float_to_bf16_bits(a.x) | (static_cast<uint32_t>(float_to_bf16_bits(a.y)) << 16);
    o.y = float_to_bf16_bits(a.z) | (static_cast<uint32_t>(float_to_bf16_bits(a.w)) << 16);
    *reinterpret_cast<uint2*>(y + i) = o;
}

static int blk_pick_bn(int M)
{
    if (M <= 16)
        return 16;
    if (M <= 32)
        return 32;
    if (M <= 64)
        return 64;
    return 128;
}

int blk_ksplit_max(int M, int K)
{
    // split K only while the fp32 partials stay small next to the weights
    int s = K / (16 * (M < 1 ? 1 : M));
    if (s > 16)
        s = 16;
    if (s < 1)
        s = 1;
    return s;
}

BlkConfig blk_pick_config(int M, int N, int K, int num_sms)
{
    BlkConfig c;
    c.bn = blk_pick_bn(M);
    const int KB = K / 128;
    const int base = (N / 128) * ((M + c.bn - 1) / c.bn);
    const int kmax = blk_ksplit_max(M, K);
    int best = 1;
    double best_eff = 0.0;
    for (int d = 1; d <= kmax; ++d) {
        if (KB % d != 0 || KB / d < 2)
            continue;
        const int64_t tiles = static_cast<int64_t>(base) * d;
        const int64_t waves = (tiles + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(tiles) / static_cast<double>(waves * num_sms);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = d;
        }
    }
    c.ksplit = best;
    return c;
}

template <int BN, int PST>
static int launch_blk(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts,
                      const BlkParams& prm, int grid, cudaStream_t s)
{
    using Tr = BlkTraits<BN, PST>;
    auto kern = blk_gemm_kernel<BN, PST>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmem) != cudaSuccess)
        return kErrLaunch;
    kern<<<grid, 384, Tr::kSmem, s>>>(tw, tx, ts, prm);
    return cudaGetLastError() == cudaSuccess ? kOK : kErrLaunch;
}

int launch_block_gemm(const BlkLaunch& L, const BlkConfig& cfg, int num_sms, cudaStream_t s)
{
    const int BN = cfg.bn;
    const int KB = L.K / 128;
    CUtensorMap tw, tx, ts;
    if (!encode_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.w, L.K, L.N, L.K, 128, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.xq, L.K, L.M, L.K, 128, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, L.xs_t, L.ld_t, KB,
                       static_cast<uint64_t>(L.ld_t) * 4, BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return kErrLaunch;
    BlkParams p{};
    p.M = L.M;
    p.N = L.N;
    p.K = L.K;
    p.KB = KB;
    p.ksplit = cfg.ksplit;
    p.kb_per_split = KB / cfg.ksplit;
    p.mt_count = (L.M + BN - 1) / BN;
    p.nb_count = L.N / 128;
    p.wsi = L.wsi;
    p.ypart = L.ypart;
    p.y = L.y;
    p.err = L.err;
    const int64_t tiles = static_cast<int64_t>(p.nb_count) * p.mt_count * p.ksplit;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    int st;
    switch (BN) {
    case 16: st = launch_blk<16, 8>(tw, tx, ts, p, grid, s); break;
    case 32: st = launch_blk<32, 8>(tw, tx, ts, p, grid, s); break;
    case 64: st = launch_blk<64, 8>(tw, tx, ts, p, grid, s); break;
    default: st = launch_blk<128, 6>(tw, tx, ts, p, grid, s); break;
    }
    if (st != kOK || cfg.ksplit == 1)
        return st;
    const int64_t MN = static_cast<int64_t>(L.M) * L.N;
    blk_reduce_kernel<<<static_cast<unsigned>((MN / 4 + 255) / 256), 256, 0, s>>>(L.ypart, cfg.ksplit,
                                                                                 MN, L.y);
    return cudaGetLastError() == cudaSuccess ? kOK : kErrLaunch;
}

}  // namespace w4a8
