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
// NBUF TMEM partial buffers let the MMAs run up to NBUF K-blocks ahead of the
// fold.
//
// Roles (4 + 4*NFW warps): warp 0 streams the weight tiles [WN x 128] (it
// starts before the dependency wait: no kernel of the call writes the
// weights), warp 2 the activation tiles [BN x 128] and, into a ring of their
// own that only the epilogue releases, the BN activation scales of each
// K-block; warp 1 owns TMEM and with warp 3 (one issuer when the ring
// depth is odd) issues the MMAs of alternate K-blocks, whose commit alone
// frees a weight/activation slot; warps 4.. fold (NFW
// warps per 32-lane TMEM quadrant, each a share of the partial product's
// columns).
//
// Two orientations. Up to 64 tokens (decode-sized calls) the MMA is
// M = 128 weight rows x N = BN tokens: a lane holds a weight row and its
// columns are tokens, so each column has its own activation scale (read from
// the scale slot as pairs and multiplied by the block's Wsi). For 128-token
// tiles the tokens are the MMA's M (the TMEM lanes) and N = WN weight rows
// (256 where N allows, else 128): every column a warp folds lies in one
// weight block, so a lane needs one combined scale per K-block,
// xs[m, g] * Wsi[n/128, g], and the fold is a TMEM load and one packed FMA
// per pair of columns. With 256 weight rows each fold warp then writes its
// [32 x 128] block through shared memory with TMA stores (a ring of 3 stages
// leaves room for the staging and measured as fast as 4); with 128 each lane
// writes its token's row segment with 32-byte stores (one whole L2 sector
// each). Both are marked evict-first in L2. Against the weight-row
// orientation at 128 tokens this took the [16384, 2560] projection of 4096
// tokens from 330 to about 185 us: that fold was bound by its per-column
// scale loads.
//
// When K is split over several CTAs, each writes its fp32 partial and bumps a
// per-tile counter; the CTA that completes the count sums the partials in
// split order and writes the bf16 tile (the counters are zeroed by the
// activation-quantization kernel of the same call).
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

constexpr int kBlkMaxKsplit = 16;   // largest split of K

struct BlkParams {
    int M, N, K, KB;
    int kb_per_split, ksplit, mt_count, nb_count;
    const float* wsi;   // [N/128, K/128]
    float* ypart;       // [ksplit, M, N] when ksplit > 1
    int* tile_cnt;      // [nb_count * mt_count] when ksplit > 1, zero at entry
    uint16_t* y;        // [M, N]
    uint32_t* err;
};

template <int BN, int PST, int NFW, int WN>
struct BlkTraits {
    // 128-token tiles put the tokens on the TMEM lanes (MMA M = 128 tokens,
    // N = WN weight rows); smaller token tiles are the MMA's N (M = 128
    // weight rows)
    static constexpr bool TL = (BN == 128);
    static constexpr int kA = WN * 128;                   // weight tile (WN rows)
    static constexpr int kB = BN * 128;                   // activation tile
    static constexpr int kStage = kA + kB;
    static constexpr int kCols = TL ? WN : BN;            // TMEM columns of one partial product
    static constexpr int kNbuf = (512 / kCols) < 8 ? (512 / kCols) : 8;   // TMEM partial buffers
    static constexpr int kNs = PST + kNbuf;               // scale ring depth
    static constexpr int kSBytes = BN * 4;                               // one scale slot's copy
    static constexpr int kSStride = ((kSBytes + 127) / 128) * 128;       // TMA destinations: 128-byte aligned
    static constexpr int kFold = 4 * NFW;                 // fold warps
    static constexpr int kHalf = kCols / NFW;             // columns per fold warp
    // 256-row weight tiles write their output through shared memory with TMA
    // stores: per fold warp a [32 rows x kHalf] bf16 block, as boxes of 64
    // columns (128 bytes, 128-byte swizzle)
    static constexpr bool kTmaOut = TL && WN == 256;
    static constexpr int kOutWarp = kTmaOut ? 32 * kHalf * 2 : 0;
    static constexpr int kSRing = ((kNs * kSStride + 1023) / 1024) * 1024;
    static constexpr int kData = PST * kStage + kSRing + kFold * kOutWarp;
    static constexpr int kBars = 3 * PST + 2 * kNs + 2 * kNbuf + 2;
    // With an even ring depth the two MMA-issuing threads (warps 1 and 3) take
    // alternate K-blocks: every ring slot and partial buffer must always
    // belong to the same thread (parity waits). An odd ring has one issuer.
    static constexpr int kIssuers = (PST % 2 == 0) ? 2 : 1;
    static_assert(kNbuf % kIssuers == 0, "partial buffers per issuer");
    static constexpr int kSmem = 1024 + kData + kBars * 8 + 32;
    static constexpr int kTmemNeed = kNbuf * kCols;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kThreads = 32 * (4 + kFold);
    static constexpr int kChunk = kHalf < 32 ? kHalf : (TL && WN == 256 ? 16 : 32);
    static_assert(NFW == 2 || NFW == 4, "fold warps per TMEM lane quadrant");
    static_assert(WN == 128 || (TL && WN == 256), "weight tiles of 128 rows, or 256 with tokens on the lanes");
    static_assert(kHalf <= 128 && 128 % kHalf == 0, "a fold warp's columns lie in one weight block");
    static_assert(kHalf >= 8 && kHalf % 8 == 0, "fold columns per warp");
    static_assert(!TL || kHalf % 16 == 0, "tokens on the lanes: 32-byte output stores");
    static_assert(!kTmaOut || kHalf % 64 == 0, "TMA output boxes of 64 columns");
    static_assert(kB % 1024 == 0, "stage alignment");
    static_assert((PST * kStage) % 1024 == 0 && kSStride % 128 == 0, "TMA destination alignment");
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kTmemNeed <= 512, "tensor memory budget");
};

// Packed pairs of fp32 (low word = first element) and the sm_100-family
// paired arithmetic on them; each lane rounds exactly like the scalar op.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// 32-byte store (address 32-byte aligned) with an L2 cache policy and no L1
// allocation.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t (&v)[8], uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(
                     dst),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "l"(pol)
                 : "memory");
}

// Barrier over `nthreads` threads (named barrier `id`) that returns whether
// any of them passed pred = true.
__device__ __forceinline__ bool bar_any(int id, int nthreads, bool pred)
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

template <int BN, int PST, int NFW, int WN>
__global__ void __launch_bounds__(32 * (4 + 4 * NFW), 1)
    blk_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_y,
                    const BlkParams p)
{
    using Tr = BlkTraits<BN, PST, NFW, WN>;
    constexpr bool TL = Tr::TL;
    constexpr int NBUF = Tr::kNbuf;
    // token tiles of 128 are used only without a K split (the host picks
    // ksplit = 1 for them), so their reduction needs no register array
    constexpr int kRed = BN >= 128 ? 1 : kBlkMaxKsplit;
    constexpr int NS = Tr::kNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sring = smem + PST * Tr::kStage;
    uint8_t* sout = sring + Tr::kSRing;    // output staging, kOutWarp bytes per fold warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kData);
    uint64_t* wfull = bars;             // weight tile landed
    uint64_t* xfull = wfull + PST;      // activation tile landed
    uint64_t* sempty = xfull + PST;     // weight + activation slot free (MMA commit)
    uint64_t* sfull = sempty + PST;     // scales landed  [NS]
    uint64_t* sfree = sfull + NS;       // scales consumed by the fold  [NS]
    uint64_t* dfull = sfree + NS;       // partial product ready  [NBUF]
    uint64_t* dempty = dfull + NBUF;    // partial buffer folded  [NBUF]
    uint64_t* drain = dempty + NBUF;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 2);   // one drain barrier per issuer
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
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&sfull[i]), 1);
            mbar_init(smem_u32(&sfree[i]), Tr::kFold);
        }
        for (int i = 0; i < NBUF; ++i) {
            mbar_init(smem_u32(&dfull[i]), 1);
            mbar_init(smem_u32(&dempty[i]), Tr::kFold);
        }
        mbar_init(smem_u32(&drain[0]), 1);
        mbar_init(smem_u32(&drain[1]), 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_s);
        if constexpr (Tr::kTmaOut)
            prefetch_tmap(&tm_y);
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

    // The producers and MMA issuers wait with a suspend hint (2 us): when the
    // fold warps set the pace these threads would otherwise spin on their
    // barriers and take issue slots from the fold (measured 2 % faster at
    // M = 4096 and M <= 8); the fold warps' own waits stay plain.
    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const bool wprod = (warp == 0);
            if (!wprod) {
                // activations and their scales come from the quantization kernel
                // launched just before; every kernel of the call triggers its
                // dependents only after its own wait
                grid_dep_wait();
                grid_dep_launch();
            }
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int ps = 0, ss = 0;
            uint32_t ph = 0, sph = 0, issued = 0, last_par = 0, s_issued = 0, s_last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
                for (int kb = 0; kb < p.kb_per_split; ++kb) {
                    const int g = ks * p.kb_per_split + kb;
                    if (!mbar_wait_or_abort<2000u>(smem_u32(&sempty[ps]), ph ^ 1u, s_abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + ps * Tr::kStage;
                    if (wprod) {
                        const uint32_t fb = smem_u32(&wfull[ps]);
                        mbar_arrive_expect_tx(fb, Tr::kA);
                        tma_load_2d_hint(smem_u32(st), &tm_w, g * 128, nb * WN, fb, pol_w);
                    } else {
                        const uint32_t fb = smem_u32(&xfull[ps]);
                        mbar_arrive_expect_tx(fb, Tr::kB);
                        tma_load_2d_hint(smem_u32(st + Tr::kA), &tm_x, g * 128, mt * BN, fb, pol_x);
                        if (!mbar_wait_or_abort<2000u>(smem_u32(&sfree[ss]), sph ^ 1u, s_abort)) {
                            ok = false;
                            issued |= 1u << ps;
                            last_par = (last_par & ~(1u << ps)) | (ph << ps);
                            break;
                        }
                        const uint32_t sb = smem_u32(&sfull[ss]);
                        mbar_arrive_expect_tx(sb, Tr::kSBytes);
                        tma_load_2d(smem_u32(sring + ss * Tr::kSStride), &tm_s, mt * BN, g, sb);
                        s_issued |= 1u << ss;
                        s_last_par = (s_last_par & ~(1u << ss)) | (sph << ss);
                        if (++ss == NS) {
                            ss = 0;
                            sph ^= 1u;
                        }
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
                // let every issued copy land before the CTA's shared memory goes away
                uint64_t* fullb = wprod ? wfull : xfull;
                for (int s = 0; s < PST; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait(smem_u32(&fullb[s]), (last_par >> s) & 1u);
                for (int s = 0; s < NS; ++s)
                    if ((s_issued >> s) & 1u)
                        mbar_wait(smem_u32(&sfull[s]), (s_last_par >> s) & 1u);
            }
        }
    } else if (warp == 1 || (Tr::kIssuers == 2 && warp == 3)) {
        // ------------------------------------------------------------ MMA issuers
        // Every K-block has its own partial buffer, so two threads can issue:
        // warp 1 takes the even K-blocks of the CTA's sequence, warp 3 the odd
        // ones, which hides each thread's barrier waits behind the other's MMAs
        // (short N = 16..64 MMAs). With an odd ring depth warp 1 issues them all.
        if (lane == 0) {
            const int me = (warp == 1) ? 0 : 1;
            const uint32_t idesc = idesc_e4m3_f32(128, Tr::kCols);
            int ps = 0;
            uint32_t ph = 0, kc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.kb_per_split; ++kb, ++kc) {
                    if (static_cast<int>(kc % Tr::kIssuers) != me) {
                        if (++ps == PST) {
                            ps = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    const int d = static_cast<int>(kc % NBUF);
                    const uint32_t use = kc / NBUF;
                    if (!mbar_wait_or_abort<2000u>(smem_u32(&dempty[d]), (use & 1u) ^ 1u, s_abort) ||
                        !mbar_wait_or_abort<2000u>(smem_u32(&wfull[ps]), ph, s_abort) ||
                        !mbar_wait_or_abort<2000u>(smem_u32(&xfull[ps]), ph, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // TL: the token tile is the MMA's A (128 TMEM lanes), the
                    // weight tile its B; otherwise the other way round
                    const uint32_t wt = smem_u32(smem + ps * Tr::kStage);
                    const uint32_t a0 = TL ? wt + Tr::kA : wt;
                    const uint32_t b0 = TL ? wt : wt + Tr::kA;
                    const uint32_t dt = tmem + static_cast<uint32_t>(d * Tr::kCols);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f8(dt, desc_kmajor_sw128(a0 + kk * 32), desc_kmajor_sw128(b0 + kk * 32),
                                idesc, kk ? 1u : 0u);
                    umma_commit(smem_u32(&sempty[ps]));
                    umma_commit(smem_u32(&dfull[d]));
                    if (++ps == PST) {
                        ps = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                fail();
                umma_commit(smem_u32(&drain[me]));
                mbar_wait(smem_u32(&drain[me]), 0);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ fold + store
        grid_dep_wait();   // the partials and counters are this call's workspace
        grid_dep_launch();
        const int q = warp & 3;
        const int hh = (warp - 4) >> 2;          // column group of this warp
        const int c0 = hh * Tr::kHalf;
        constexpr int kFoldThreads = 32 * Tr::kFold;
        int ss = 0;
        uint32_t sph = 0, kc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const int nb = t / per_nb, r = t % per_nb, mt = r / p.ksplit, ks = r % p.ksplit;
            // column pairs, folded with packed fp32x2 arithmetic (each lane of a
            // pair rounds exactly like the scalar fmaf(p, sc, acc), sc = xs * ws)
            uint64_t acc2[Tr::kHalf / 2];
#pragma unroll
            for (int c = 0; c < Tr::kHalf / 2; ++c)
                acc2[c] = 0ull;
            for (int kb = 0; kb < p.kb_per_split; ++kb, ++kc) {
                const int d = static_cast<int>(kc % NBUF);
                const uint32_t use = kc / NBUF;
                if (!mbar_wait_or_abort(smem_u32(&dfull[d]), use & 1u, s_abort) ||
                    !mbar_wait_or_abort(smem_u32(&sfull[ss]), sph, s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int g = ks * p.kb_per_split + kb;
                // the weight block of this warp's columns
                const int wb = TL ? (nb * WN + c0) >> 7 : nb;
                const float ws = __ldg(p.wsi + static_cast<int64_t>(wb) * p.KB + g);
                const uint64_t ws2 = f2_pack(ws, ws);
                const float* xs = reinterpret_cast<const float*>(sring + ss * Tr::kSStride);
                const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(d * Tr::kCols + c0);
                // TL: this lane's token has one scale for the warp's row of
                // partial products (all its columns are rows of weight block wb)
                float sc_row = 0.0f;
                if constexpr (TL)
                    sc_row = xs[q * 32 + lane] * ws;
                const uint64_t sc_row2 = f2_pack(sc_row, sc_row);
#pragma unroll
                for (int ch = 0; ch < Tr::kHalf / Tr::kChunk; ++ch) {
                    uint32_t v[Tr::kChunk];
                    tmem_ld_cols<Tr::kChunk>(tb + ch * Tr::kChunk, v);
                    tmem_ld_wait();
                    const uint64_t* xs2 = reinterpret_cast<const uint64_t*>(xs + c0 + ch * Tr::kChunk);
#pragma unroll
                    for (int c = 0; c < Tr::kChunk / 2; ++c) {
                        const uint64_t sc = TL ? sc_row2 : f2_mul(xs2[c], ws2);
                        const uint64_t pv = f2_pack(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
                        acc2[ch * Tr::kChunk / 2 + c] = f2_fma(pv, sc, acc2[ch * Tr::kChunk / 2 + c]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&dempty[d]));
                    mbar_arrive(smem_u32(&sfree[ss]));
                }
                if (++ss == NS) {
                    ss = 0;
                    sph ^= 1u;
                }
            }
            float acc[Tr::kHalf];
#pragma unroll
            for (int c = 0; c < Tr::kHalf / 2; ++c)
                f2_unpack(acc2[c], acc[2 * c], acc[2 * c + 1]);
            if constexpr (TL) {
                // one token row per lane, kHalf consecutive outputs of it:
                // 32-byte stores (one whole L2 sector) of 16 bf16 each (never
                // split over K), marked first to leave L2, where the weights
                // and activations of the tiles in flight are reused
                if (!ok)
                    break;
                if constexpr (Tr::kTmaOut) {
                    // Through shared memory: the warp's [32 x kHalf] block as
                    // boxes of 64 columns, 128-byte swizzled (16-byte chunk j of
                    // row r at position j ^ (r % 8): conflict-free writes), then
                    // TMA stores of whole rows (rows past M are not written).
                    uint8_t* stg = sout + (warp - 4) * Tr::kOutWarp;
                    if (lane == 0)
                        bulk_wait_read_all();   // the previous tile's stores have read it
                    __syncwarp();
#pragma unroll
                    for (int b = 0; b < Tr::kHalf / 64; ++b) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float* a8v = acc + 64 * b + 8 * j;
                            uint4 o;
                            o.x = float_to_bf16_bits(a8v[0]) | (static_cast<uint32_t>(float_to_bf16_bits(a8v[1])) << 16);
                            o.y = float_to_bf16_bits(a8v[2]) | (static_cast<uint32_t>(float_to_bf16_bits(a8v[3])) << 16);
                            o.z = float_to_bf16_bits(a8v[4]) | (static_cast<uint32_t>(float_to_bf16_bits(a8v[5])) << 16);
                            o.w = float_to_bf16_bits(a8v[6]) | (static_cast<uint32_t>(float_to_bf16_bits(a8v[7])) << 16);
                            *reinterpret_cast<uint4*>(stg + b * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
                        }
                    }
                    fence_proxy_async_smem();   // the writes, before the async proxy reads them
                    __syncwarp();
                    if (lane == 0) {
                        const uint64_t pol_y = policy_evict_first();
#pragma unroll
                        for (int b = 0; b < Tr::kHalf / 64; ++b)
                            tma_store_2d_hint(&tm_y, nb * WN + c0 + 64 * b, mt * BN + q * 32, smem_u32(stg + b * 4096),
                                              pol_y);
                        bulk_commit_group();
                    }
                    continue;
                }
                const int m = mt * BN + q * 32 + lane;
                if (m < p.M) {
                    const uint64_t pol_y = policy_evict_first();
                    uint16_t* dst = p.y + static_cast<int64_t>(m) * p.N + nb * WN + c0;
#pragma unroll
                    for (int c = 0; c < Tr::kHalf / 16; ++c) {
                        uint32_t o[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            o[j] = float_to_bf16_bits(acc[16 * c + 2 * j]) |
                                   (static_cast<uint32_t>(float_to_bf16_bits(acc[16 * c + 2 * j + 1])) << 16);
                        st_global_v8(dst + 16 * c, o, pol_y);
                    }
                }
                continue;
            }
            const int n = nb * 128 + q * 32 + lane;
            if (p.ksplit == 1) {
                if (!ok)
                    break;
#pragma unroll
                for (int c = 0; c < Tr::kHalf; ++c) {
                    const int m = mt * BN + c0 + c;
                    if (m < p.M)
                        p.y[static_cast<int64_t>(m) * p.N + n] = float_to_bf16_bits(acc[c]);
                }
                continue;
            }
            if (ok) {
#pragma unroll
                for (int c = 0; c < Tr::kHalf; ++c) {
                    const int m = mt * BN + c0 + c;
                    if (m < p.M)
                        p.ypart[(static_cast<int64_t>(ks) * p.M + m) * p.N + n] = acc[c];
                }
            }
            // publish the partial; the CTA that completes the tile's count sums
            // the splits in order. Every fold warp reaches this barrier (a warp
            // whose wait failed skipped its remaining K-blocks), and all of them
            // leave together if any failed. The barrier orders the fold
            // threads' stores before one thread's fence + counter increment
            // (release); the CTA that completes the count fences (acquire)
            // before a second barrier releases its threads to read.
            if (bar_any(1, kFoldThreads, !ok)) {
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
            asm volatile("bar.sync 1, %0;" ::"r"(kFoldThreads) : "memory");
            if (*s_last) {
                // the tile's outputs are spread over the fold threads (n
                // fastest: coalesced); each requests all of an output's split
                // partials before adding them in split order
                const int mrows = min(BN, p.M - mt * BN);
                const int64_t step = static_cast<int64_t>(p.M) * p.N;
                // 4 consecutive outputs per item (16-byte loads), every split
                // of an item requested before its sum, splits added in order
#pragma unroll 2
                for (int o = threadIdx.x - 128; o < 32 * mrows; o += kFoldThreads) {
                    const int m = mt * BN + (o >> 5);
                    const int nn = nb * 128 + (o & 31) * 4;
                    const float4* src = reinterpret_cast<const float4*>(p.ypart + static_cast<int64_t>(m) * p.N + nn);
                    float4 vv[kRed];
#pragma unroll
                    for (int s = 0; s < kRed; ++s)
                        if (s < p.ksplit)
                            vv[s] = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + s * step));
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int s = 0; s < kRed; ++s) {
                        if (s < p.ksplit) {
                            sum.x += vv[s].x;
                            sum.y += vv[s].y;
                            sum.z += vv[s].z;
                            sum.w += vv[s].w;
                        }
                    }
                    uint2 ob;
                    ob.x = float_to_bf16_bits(sum.x) | (static_cast<uint32_t>(float_to_bf16_bits(sum.y)) << 16);
                    ob.y = float_to_bf16_bits(sum.z) | (static_cast<uint32_t>(float_to_bf16_bits(sum.w)) << 16);
                    *reinterpret_cast<uint2*>(p.y + static_cast<int64_t>(m) * p.N + nn) = ob;
                }
            }
        }
        if (!ok)
            fail();
        if constexpr (Tr::kTmaOut) {
            // the staging must outlive the stores that read it
            if (lane == 0)
                bulk_wait_all();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Tr::kTmemCols);
    }
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
    if (s > kBlkMaxKsplit)
        s = kBlkMaxKsplit;
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
    c.ksplit = 1;
    // Splitting K costs a partial round trip and a per-tile counter hand-off
    // on the fold path; measured on the block-FP8 shapes it pays only when
    // the unsplit tiles leave most SMs idle (e.g. N = 2560 at M <= 64: 20
    // tiles for 152 SMs). Tiles of 128 tokens are never split.
    if (2 * base >= num_sms || c.bn >= 128)
        return c;
    const int kmax = blk_ksplit_max(M, K);
    double best_eff = 0.0;
    for (int d = 1; d <= kmax; ++d) {
        if (KB % d != 0 || KB / d < 2)
            continue;
        const int64_t tiles = static_cast<int64_t>(base) * d;
        const int64_t waves = (tiles + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(tiles) / static_cast<double>(waves * num_sms);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            c.ksplit = d;
        }
    }
    return c;
}

template <int BN, int PST, int NFW, int WN>
static int launch_blk(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts, const CUtensorMap& ty,
                      const BlkParams& prm, int grid, cudaStream_t s)
{
    using Tr = BlkTraits<BN, PST, NFW, WN>;
    auto kern = blk_gemm_kernel<BN, PST, NFW, WN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmem) != cudaSuccess)
        return kErrLaunch;
    return launch_dependent(kern, dim3(grid), dim3(Tr::kThreads), Tr::kSmem, s, tw, tx, ts, ty, prm) == cudaSuccess
               ? kOK
               : kErrLaunch;
}

int launch_block_gemm(const BlkLaunch& L, const BlkConfig& cfg, int num_sms, cudaStream_t s)
{
    const int BN = cfg.bn;
    const int KB = L.K / 128;
    // 128-token tiles take 256 weight rows where N allows: the same bytes per
    // stage feed twice the MMA work of a 128-row tile
    const int WN = (BN == 128 && L.N % 256 == 0) ? 256 : 128;
    CUtensorMap tw, tx, ts, ty;
    if (!encode_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.w, L.K, L.N, L.K, 128, WN,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.xq, L.K, L.M, L.K, 128, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, L.xs_t, L.ld_t, KB,
                       static_cast<uint64_t>(L.ld_t) * 4, BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return kErrLaunch;
    // bf16 output [M, N] for the TMA stores of 256-row weight tiles: boxes of
    // 64 columns x 32 rows, 128-byte swizzle (unused by the other shapes)
    if (WN == 256) {
        if (!encode_map_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_UINT16, L.y, L.N, L.M, static_cast<uint64_t>(L.N) * 2, 64, 32,
                           CU_TENSOR_MAP_SWIZZLE_128B))
            return kErrLaunch;
    } else {
        ty = tx;
    }
    BlkParams p{};
    p.M = L.M;
    p.N = L.N;
    p.K = L.K;
    p.KB = KB;
    p.ksplit = cfg.ksplit;
    p.kb_per_split = KB / cfg.ksplit;
    p.mt_count = (L.M + BN - 1) / BN;
    p.nb_count = L.N / WN;
    p.wsi = L.wsi;
    p.ypart = L.ypart;
    p.tile_cnt = L.tile_cnt;
    p.y = L.y;
    p.err = L.err;
    if (BN >= 128 && cfg.ksplit > 1)
        return kErrLaunch;   // not produced by blk_pick_config
    const int64_t tiles = static_cast<int64_t>(p.nb_count) * p.mt_count * p.ksplit;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    switch (BN) {
    case 16: return launch_blk<16, 8, 2, 128>(tw, tx, ts, ty, p, grid, s);
    case 32: return launch_blk<32, 8, 2, 128>(tw, tx, ts, ty, p, grid, s);
    case 64: return launch_blk<64, 8, 2, 128>(tw, tx, ts, ty, p, grid, s);
    default:
        // 256-row tiles: a ring of 3 stages (the 4th measured no faster) and
        // 64 KB of output staging
        return WN == 256 ? launch_blk<128, 3, 2, 256>(tw, tx, ts, ty, p, grid, s)
                         : launch_blk<128, 6, 2, 128>(tw, tx, ts, ty, p, grid, s);
    }
}

}  // namespace w4a8
