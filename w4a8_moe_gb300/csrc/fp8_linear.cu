// Per-tensor FP8 dense projection y = sx * sw * x W^T on sm_103a.
//
// "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm",
// description: the attention projections are quantized online to float8;
// review summary: QuarkInt4Fp8LinearMethod for linear layers, tensor-wise FP8
// quantization. With one scale per tensor the whole K reduction stays in the
// tensor cores: every tile accumulates in TMEM and the epilogue scales once.
//
// Roles (12 warps), operands swapped (M = 128 weight rows, N = BN tokens):
// warp 0 streams the weight tiles [128 x 128] (before the dependency wait: no
// kernel of the call writes the weights), warp 2 the activation tiles
// [BN x 128], warp 1 owns TMEM and issues the MMAs (the commit of a stage frees
// its slot; the commit of a tile hands its accumulator to the epilogue), warps
// 4-11 read the accumulator (two warps per 32-lane TMEM quadrant, each half of
// the BN columns), scale and store. Two accumulators let the epilogue of a
// tile overlap the next tile's MMAs.
//
// Small M splits K: each split writes its fp32 partial and bumps a per-tile
// counter; the CTA that completes the count sums the partials in split order,
// writes the bf16 tile and resets the counter to zero.
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

constexpr int kFpMaxKsplit = 16;

struct FpParams {
    int M, N, K, KB;
    int kb_per_split, ksplit, mt_count, nb_count;
    const float* sx;    // [1]
    const float* sw;    // [1]
    float* ypart;       // [ksplit, M, N] when ksplit > 1
    int* tile_cnt;      // [nb_count * mt_count], zero between calls
    uint16_t* y;        // [M, N]
    uint32_t* err;
};

template <int BN, int PST>
struct FpTraits {
    static constexpr int kA = 128 * 128;
    static constexpr int kB = BN * 128;
    static constexpr int kStage = kA + kB;
    static constexpr int kData = PST * kStage;
    static constexpr int kBars = 3 * PST + 4 + 1;
    static constexpr int kSmem = 1024 + kData + kBars * 8 + 32;
    static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
    static constexpr int kHalf = BN / 2;
    static constexpr int kChunk = kHalf < 32 ? kHalf : 32;
    static_assert(kB % 1024 == 0 && kStage % 1024 == 0, "stage alignment");
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(2 * BN <= 512, "tensor memory budget");
};

__device__ __forceinline__ bool fp_bar_any(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int NC>
__device__ __forceinline__ void fp_ld_cols(uint32_t taddr, uint32_t* r)
{
    if constexpr (NC == 32) {
        uint32_t (&v)[32] = *reinterpret_cast<uint32_t(*)[32]>(r);
        tmem_ld32(taddr, v);
    } else if constexpr (NC == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
              "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    } else {
        static_assert(NC == 8, "column chunk");
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                       "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    }
}

template <int BN, int PST>
__global__ void __launch_bounds__(384, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const FpParams p)
{
    using Tr = FpTraits<BN, PST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kData);
    uint64_t* wfull = bars;
    uint64_t* xfull = wfull + PST;
    uint64_t* sempty = xfull + PST;
    uint64_t* accfull = sempty + PST;
    uint64_t* accempty = accfull + 2;
    uint64_t* drain = accempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* s_last = reinterpret_cast<int*>(s_tmem + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < PST; ++i) {
            mbar_init(smem_u32(&wfull[i]), 1);
            mbar_init(smem_u32(&xfull[i]), 1);
            mbar_init(smem_u32(&sempty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&accfull[i]), 1);
            mbar_init(smem_u32(&accempty[i]), 8);
        }
        mbar_init(smem_u32(drain), 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
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

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const bool wprod = (warp == 0);
            if (!wprod) {
                // the activations may come from the kernel launched just before;
                // every kernel of the library triggers its dependents only after
                // its own wait
                grid_dep_wait();
                grid_dep_launch();
            }
            const uint64_t pol = wprod ? policy_evict_first() : policy_evict_last();
            uint64_t* fullb = wprod ? wfull : xfull;
            int ps = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
                for (int kb = 0; kb < p.kb_per_split; ++kb) {
                    if (!mbar_wait_or_abort(smem_u32(&sempty[ps]), ph ^ 1u, s_abort)) {
                        ok = false;
                        break;
                    }
                    const int g = ks * p.kb_per_split + kb;
                    uint8_t* st = smem + ps * Tr::kStage;
                    const uint32_t fb = smem_u32(&fullb[ps]);
                    if (wprod) {
                        mbar_arrive_expect_tx(fb, Tr::kA);
                        tma_load_2d_hint(smem_u32(st), &tm_w, g * 128, nb * 128, fb, pol);
                    } else {
                        mbar_arrive_expect_tx(fb, Tr::kB);
                        tma_load_2d_hint(smem_u32(st + Tr::kA), &tm_x, g * 128, mt * BN, fb, pol);
                    }
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
                        mbar_wait(smem_u32(&fullb[s]), (last_par >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3_f32(128, BN);
            int ps = 0, it = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const int d = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait_or_abort(smem_u32(&accempty[d]), (use & 1u) ^ 1u, s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + static_cast<uint32_t>(d * BN);
                for (int kb = 0; kb < p.kb_per_split; ++kb) {
                    if (!mbar_wait_or_abort(smem_u32(&wfull[ps]), ph, s_abort) ||
                        !mbar_wait_or_abort(smem_u32(&xfull[ps]), ph, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + ps * Tr::kStage);
                    const uint32_t b0 = a0 + Tr::kA;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f8(dt, desc_kmajor_sw128(a0 + kk * 32), desc_kmajor_sw128(b0 + kk * 32), idesc,
                                (kb | kk) ? 1u : 0u);
                    umma_commit(smem_u32(&sempty[ps]));
                    if (++ps == PST) {
                        ps = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(smem_u32(&accfull[d]));
            }
            if (!ok) {
                fail();
                umma_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        grid_dep_wait();   // y, the partials and the counters belong to this call
        grid_dep_launch();
        const int q = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int c0 = hh * Tr::kHalf;
        const float scale = __ldg(p.sx) * __ldg(p.sw);
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
            const int d = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            const int n = nb * 128 + q * 32 + lane;
            if (ok && !mbar_wait_or_abort(smem_u32(&accfull[d]), use & 1u, s_abort)) {
                ok = false;
                fail();
            }
            if (ok) {
                tc_fence_after();
                const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(d * BN + c0);
#pragma unroll 1
                for (int ch = 0; ch < Tr::kHalf / Tr::kChunk; ++ch) {
                    uint32_t v[Tr::kChunk];
                    fp_ld_cols<Tr::kChunk>(tb + ch * Tr::kChunk, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < Tr::kChunk; ++c) {
                        const int m = mt * BN + c0 + ch * Tr::kChunk + c;
                        if (m < p.M) {
                            const float val = __uint_as_float(v[c]);
                            if (p.ksplit == 1)
                                p.y[static_cast<int64_t>(m) * p.N + n] = float_to_bf16_bits(val * scale);
                            else
                                p.ypart[(static_cast<int64_t>(ks) * p.M + m) * p.N + n] = val;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&accempty[d]));
            }
            if (p.ksplit == 1) {
                if (!ok)
                    break;
                continue;
            }
            // Split K: every epilogue warp reaches this barrier (a warp that
            // failed skipped its work), and all leave together if any failed.
            // The barrier orders the partial stores before one thread's fence
            // + counter increment (release); the CTA completing the count
            // fences (acquire) before a second barrier releases its threads.
            if (fp_bar_any(1, 256, !ok)) {
                ok = false;
                break;
            }
            if (threadIdx.x == 128) {
                __threadfence();
                const int old = atomicAdd(p.tile_cnt + nb * p.mt_count + mt, 1);
                const int last = (old == p.ksplit - 1);
                if (last)
                    __threadfence();
                *s_last = last;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (*s_last) {
                const int mrows = min(BN, p.M - mt * BN);
                const int64_t step = static_cast<int64_t>(p.M) * p.N;
                // 4 consecutive outputs per item (16-byte loads), every split
                // of an item requested before its sum, splits added in order
#pragma unroll 2
                for (int o = threadIdx.x - 128; o < 32 * mrows; o += 256) {
                    const int m = mt * BN + (o >> 5);
                    const int nn = nb * 128 + (o & 31) * 4;
                    const float4* src = reinterpret_cast<const float4*>(p.ypart + static_cast<int64_t>(m) * p.N + nn);
                    float4 vv[kFpMaxKsplit];
#pragma unroll
                    for (int s = 0; s < kFpMaxKsplit; ++s)
                        if (s < p.ksplit)
                            vv[s] = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + s * step));
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int s = 0; s < kFpMaxKsplit; ++s) {
                        if (s < p.ksplit) {
                            sum.x += vv[s].x;
                            sum.y += vv[s].y;
                            sum.z += vv[s].z;
                            sum.w += vv[s].w;
                        }
                    }
                    uint2 ob;
                    ob.x = float_to_bf16_bits(sum.x * scale) | (static_cast<uint32_t>(float_to_bf16_bits(sum.y * scale)) << 16);
                    ob.y = float_to_bf16_bits(sum.z * scale) | (static_cast<uint32_t>(float_to_bf16_bits(sum.w * scale)) << 16);
                    *reinterpret_cast<uint2*>(p.y + static_cast<int64_t>(m) * p.N + nn) = ob;
                }
                if (threadIdx.x == 128)
                    p.tile_cnt[nb * p.mt_count + mt] = 0;   // zero for the next call
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

static int fp_pick_bn(int M)
{
    return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

int fp8_ksplit_max(int M, int K)
{
    // split K only while the fp32 partials stay small next to the weights
    int s = K / (16 * (M < 1 ? 1 : M));
    return s < 1 ? 1 : s > kFpMaxKsplit ? kFpMaxKsplit : s;
}

FpConfig fp8_pick_config(int M, int N, int K, int num_sms)
{
    FpConfig c;
    c.bn = fp_pick_bn(M);
    const int KB = K / 128;
    const int base = (N / 128) * ((M + c.bn - 1) / c.bn);
    // cost of a split d: waves(d) * (K-blocks per tile + about one block of
    // fixed per-tile cost)
    const int kmax = fp8_ksplit_max(M, K);
    c.ksplit = 1;
    double best = 0.0;
    for (int d = 1; d <= kmax; ++d) {
        if (KB % d != 0 || (d > 1 && KB / d < 2))
            continue;
        const int64_t tiles = static_cast<int64_t>(base) * d;
        const int64_t waves = (tiles + num_sms - 1) / num_sms;
        const double cost = static_cast<double>(waves) * (static_cast<double>(KB / d) + 1.0);
        if (d == 1 || cost < best) {
            best = cost;
            c.ksplit = d;
        }
    }
    return c;
}

template <int BN, int PST>
static int launch_fp(const CUtensorMap& tw, const CUtensorMap& tx, const FpParams& prm, int grid, cudaStream_t s)
{
    using Tr = FpTraits<BN, PST>;
    auto kern = fp8_gemm_kernel<BN, PST>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmem) != cudaSuccess)
        return kErrLaunch;
    return launch_dependent(kern, dim3(grid), dim3(384), Tr::kSmem, s, tw, tx, prm) == cudaSuccess ? kOK
                                                                                                   : kErrLaunch;
}

int launch_fp8_linear(const FpLaunch& L, const FpConfig& cfg, int num_sms, cudaStream_t s)
{
    const int BN = cfg.bn;
    CUtensorMap tw, tx;
    if (!encode_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.w, L.K, L.N, L.K, 128, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.x, L.K, L.M, L.K, 128, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return kErrLaunch;
    FpParams p{};
    p.M = L.M;
    p.N = L.N;
    p.K = L.K;
    p.KB = L.K / 128;
    p.ksplit = cfg.ksplit;
    p.kb_per_split = p.KB / cfg.ksplit;
    p.mt_count = (L.M + BN - 1) / BN;
    p.nb_count = L.N / 128;
    p.sx = L.sx;
    p.sw = L.sw;
    p.ypart = L.ypart;
    p.tile_cnt = L.tile_cnt;
    p.y = L.y;
    p.err = L.err;
    const int64_t tiles = static_cast<int64_t>(p.nb_count) * p.mt_count * p.ksplit;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    switch (BN) {
    case 16: return launch_fp<16, 10>(tw, tx, p, grid, s);
    case 32: return launch_fp<32, 10>(tw, tx, p, grid, s);
    case 64: return launch_fp<64, 8>(tw, tx, p, grid, s);
    case 128: return launch_fp<128, 6>(tw, tx, p, grid, s);
    default: return launch_fp<256, 4>(tw, tx, p, grid, s);
    }
}

}  // namespace w4a8
