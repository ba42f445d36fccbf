// W4A8 MoE forward on sm_103a: gather -> grouped gate_up GEMM (+SiLU/GELU
// gating, E4M3 requantization) -> grouped down GEMM -> weighted combine.
//
// "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm",
// description: the int4 MoE weights are upcast to float8 so that fp8 math is
// used; "ROCm: enable trillion-parameter MoE models with INT4-FP8 single
// node", Motivation: INT4 weights lower the memory bandwidth of decoding, the
// FP8 tensor cores do the math.
//
// Grouped GEMM design (one persistent CTA per SM, 4 + NCONV + NEPI warps):
//   warp 0      TMA producer of the packed INT4 weight tiles [128 rows x KC/2
//               bytes] into the W ring (starts before the dependency wait).
//   warp 2      TMA producer of the expert's activation tiles [BN x KC] into
//               the X ring.
//   warps 1, 3  TMEM owner and the MMA-issuing thread(s): with two issuers
//               they take alternate stages into separate partial sums.
//   warps 4..   converters: thread r owns A row r; it turns its packed nibbles
//               into E4M3 bytes, in TMEM (tcgen05.st) for token tiles up to 128,
//               else in the 128-byte-swizzled K-major shared-memory layout.
//   last NEPI   epilogue: tcgen05.ld of the fp32 accumulators (lane = weight
//               row, column = token), scales, activation, stores; with 8 warps
//               the two warps of a lane quadrant take alternate 32-column chunks.
// The MMA runs "swapped": M = 128 weight rows, N = the expert's tokens, so a
// decode step with a handful of tokens per expert still uses M = 128 and the
// weights stream through the SMs once.
//
// Launch modes (template MODE): 0 gate_up, 1 down, 2 gate_up with the
// dynamic intermediate scale (fp32 h and max|h| out), 3 gate_up and down in
// one launch (token tiles up to 128): the CTAs take the gate_up tiles and
// then the down tiles, and a down tile of expert e waits on a per-expert
// count of finished gate_up tiles, so no SM idles between the projections.
//
// K need not be a multiple of the stage width KC: when H or I is 128 more
// than a multiple of 256, the last stage of a tile reaches past K, TMA fills
// the activation (and packed weight) bytes beyond K with zeros, and those
// activation zeros make the extra products vanish (the exact row sums below
// cover the real K only).
//
// INT4 -> E4M3 upcast. A nibble n holds q = n - 16*(n >= 8). The byte
// o = n ^ 8 = q + 8 lies in 0..15, and the E4M3 codes 0x00..0x0F encode
// exactly o * 2^-9 (subnormals plus the first normal binade share the spacing
// 2^-9). So one AND+XOR per 4 weights yields operands worth (q + 8) * 2^-9 and
//   sum_h x_h q_h = 512 * sum_h x_h dec(o_h) - 8 * sum_h x_h,
// where the per-token sum_h x_h is exact integer bookkeeping (S0 below). The
// tensor-core product is the exact upcast the pages describe, shifted by a
// constant that the epilogue removes. That is the in-GEMM form (decode-sized
// calls). Prefill-sized calls unpack the weights once per call instead, to the
// E4M3 code of q itself (every INT4 value is exact in E4M3), and need no shift.
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace w4a8 {

struct MoeGemmParams {
    const int32_t* counts;   // [E]
    const int32_t* offsets;  // [E+1]
    int E;
    int rows_per_expert;     // 2I (gate_up) or H (down)
    int rt_count;            // 128-row weight tiles per expert
    int kblocks;             // pipeline stages per tile (KC elements each)
    int ksplit;              // splits of K (down only)
    int I, H, A;
    // gate_up epilogue
    const float* s_gu;       // [E, 2I]
    const float* a1;         // [1]
    const float* a2;         // [1]
    int act;
    const long long* s0x;    // [A] sum_h 512*dec(x) of the assignment's token
    uint8_t* hq;             // [A, I]
    unsigned long long* s0h; // [A] sum_i 512*dec(hq), accumulated by atomics
    // down epilogue
    float* ypart;            // [ksplit or nslots, A, H] raw accumulator (before shift removal)
    // gate_up with a dynamic intermediate scale (MODE 2): h goes to hf (fp32,
    // natural column order) and max|h| to *hmax (float bits) instead of hq / s0h
    int dynamic;
    float* hf;               // [A, I]
    unsigned int* hmax;
    int streamk;             // down only: equal stage ranges per CTA (see WorkIter)
    int nslots;              // stream-K: partial slots per output (unused ones zeroed)
    // MODE 3 runs both projections in one launch: the fields above
    // (rows_per_expert .. ksplit) describe its gate_up tiles, these its down tiles
    int rows_per_expert2, rt_count2, kblocks2, ksplit2;
    int* done;               // [E] gate_up tiles finished per expert, x4 (one per epilogue warp)
    int* claim;              // [2] MODE 3: tiles claimed, CTAs done claiming (both zero between launches)
    // tile-order bands inside an expert (0: none): gate_up walks all weight
    // rows for `band` token tiles at a time, down all token tiles for `band`
    // weight-row tiles at a time (band2: the down tiles of MODE 3)
    int band, band2;
    // prefill down GEMM: pacing counters (see kMoeSyncEvery), nullptr: none
    int* sync;
    uint32_t* err;
};

template <int MODE, int BN, int KC, int NW, int NX, int NXT, int NCONV, int NISS, int NB, int NEPI>
struct MoeTraits {
    static constexpr int kAtoms = KC / 128;                      // 128-byte K atoms of A and B
    static constexpr int kWBytes = 128 * KC / 2;                 // packed weights per stage
    static constexpr int kWBoxBytes = KC == 128 ? 64 : 128;      // bytes per row per TMA box
    static constexpr int kWBoxes = KC / 2 / kWBoxBytes;
    static constexpr int kBBytes = kAtoms * BN * 128;            // activations per stage
    static constexpr int kXBytes = kBBytes;                      // X slot in shared memory: B
    static constexpr int kASlot = kAtoms * 128 * 128;            // unpacked A of a shared-memory slot
    static constexpr int kACols = KC / 4;                        // unpacked A of a TMEM slot
    // X slots 0..NXT-1 keep their unpacked A in TMEM, slots NXT..NX-1 in
    // shared memory (after the B tiles). With NB != NX the activation tiles
    // have a ring of their own (NB slots), decoupled from the A slots: the
    // activation copies then run NB stages ahead instead of NX.
    static constexpr bool kSplitB = (NB != NX);
    // No converter warps (NCONV = 0): A arrives by TMA from weights unpacked
    // ahead of the GEMM (moe_upcast_kernel) into the shared-memory A slots,
    // loaded by warp 0 in place of the packed weight stream (no W ring). Those
    // hold the signed INT4 values as E4M3 codes, so the accumulators need no
    // shift and the intermediate no exact row sums.
    static constexpr bool kA8 = (NCONV == 0);
    static constexpr int kData = NW * kWBytes + NB * kXBytes + (NX - NXT) * kASlot;
    static constexpr int kBars = 2 * NW + 2 * NB + 2 * NX + 4 + 2 + 2 * kTileQ;   // + drain, tile queue
    static constexpr int kCtrl = kBars * 8 + 16 + 4 * (256 + 260 + 260 + 260 + kTileQ);
    // MODE 3 tile queue: every role but the weight producer frees each entry
    static constexpr int kTileReaders = 1 + NISS + NCONV + NEPI;
    static constexpr int kSmem = 1024 + kData + kCtrl;
    // two accumulator buffers (tile i / tile i+1), each with one partial sum
    // per MMA-issuing thread
    static constexpr int kDCols = 2 * NISS * BN;
    static constexpr int kTmemNeed = kDCols + NXT * kACols;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kThreads = 32 * (4 + NCONV + NEPI);
    static constexpr int kEpi0 = 4 + NCONV;                      // first epilogue warp
    static constexpr int kPar = NCONV >= 4 ? NCONV / 4 : 1;     // converter warps per quadrant
    static_assert(kWBytes % 1024 == 0 && kXBytes % 1024 == 0 && kASlot % 1024 == 0, "stage alignment");
    static_assert(NXT >= 0 && NXT <= NX, "TMEM A slots");
    // where X slot x keeps its unpacked A; a compile-time constant unless the
    // slots are mixed (a runtime test in the hot loops costs real time)
    __device__ __forceinline__ static bool a_in_tmem(int x)
    {
        if constexpr (NXT == NX)
            return true;
        else if constexpr (NXT == 0)
            return false;
        else
            return x < NXT;
    }
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kTmemNeed <= 512, "tensor memory budget");
    static_assert(BN % 16 == 0 && BN <= 256, "token tile");
    static_assert((NCONV % 4 == 0 && NCONV >= 4) || (kA8 && NW == 0 && NXT == 0 && !kSplitB),
                  "converters cover the four TMEM lane quadrants; without them A comes by TMA into shared memory");
    static_assert(NEPI == 4 || NEPI == 8, "epilogue warps: one or two per TMEM lane quadrant");
    // Converter warp w takes the stages g with g % kPar == (w - 4) / 4 and waits
    // on the rings' barriers by phase parity. A parity wait cannot tell phase r
    // from r + 2, so every warp must see every round of each slot it serves:
    // both ring depths must be multiples of kPar (then a slot always maps to
    // the same warp).
    static_assert(NW % kPar == 0 && NX % kPar == 0, "ring depths must be multiples of the converter warps per quadrant");
    // MMA issuer i takes the stages g with g % NISS == i and waits on afull by
    // parity as well, so the X ring depth must be a multiple of NISS.
    static_assert((NISS == 1 || NISS == 2) && NX % NISS == 0, "MMA issuers");
    // a separate activation ring is waited on by the issuers (by parity) and
    // holds only activation tiles: its depth is a multiple of the issuers, and
    // every A slot lives in tensor memory
    static_assert(!kSplitB || (NB % NISS == 0 && NB > 0 && NXT == NX), "activation ring");
};

struct TileInfo {
    int e, rt, tt, ks, tok0, ntok;
};

// Tile t of the CTA-shared tile list -> (expert, 128-row weight tile, token
// tile, K split). Tiles run in expert order. Inside an expert, gate_up walks
// weight rows outermost (the expert's gathered activations stay in L2 while its
// weight tiles stream once); down walks token tiles outermost, so the CTAs
// working at the same time share a few token tiles of the intermediate
// activation and stream the weight rows, whose deeper ring hides HBM latency.
// With a band (prefill, where one expert's activations exceed what L2 keeps):
// gate_up takes `band` token tiles at a time and walks all weight rows over
// them, down takes `band` weight-row tiles at a time and walks all token tiles
// over them, so both operands of the tiles in flight are reused from L2.
template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(int t, const int* s_cnt, const int* s_off,
                                                const int* s_pre, int E, int BN, int ksplit, int rt_count, int band)
{
    TileInfo ti;
    int e = 0;
    while (e + 1 < E && s_pre[e + 1] <= t)
        ++e;
    const int local = t - s_pre[e];
    const int c = s_cnt[e];
    const int ntt = (c + BN - 1) / BN;
    ti.e = e;
    if (MODE != 1) {   // gate_up (static or dynamic scale)
        const int tb = band > 0 ? band : ntt;               // token tiles per band
        const int per_band = rt_count * tb * ksplit;        // tiles of a full band
        const int bi = local / per_band;
        const int rem = local - bi * per_band;
        const int w = min(tb, ntt - bi * tb);               // token tiles of this band
        const int per_rt = w * ksplit;
        ti.rt = rem / per_rt;
        const int r2 = rem - ti.rt * per_rt;
        ti.tt = bi * tb + r2 / ksplit;
        ti.ks = r2 - (r2 / ksplit) * ksplit;
    } else {
        const int rb = band > 0 ? band : rt_count;          // weight-row tiles per band
        const int per_band = rb * ntt * ksplit;
        const int bi = local / per_band;
        const int rem = local - bi * per_band;
        const int w = min(rb, rt_count - bi * rb);          // row tiles of this band
        const int per_tt = w * ksplit;
        ti.tt = rem / per_tt;
        const int r2 = rem - ti.tt * per_tt;
        ti.rt = bi * rb + r2 / ksplit;
        ti.ks = r2 - (r2 / ksplit) * ksplit;
    }
    ti.tok0 = s_off[e] + ti.tt * BN;
    ti.ntok = min(BN, c - ti.tt * BN);
    return ti;
}

// MODE 3 (both projections in one launch): the CTA-shared list holds the
// gate_up tiles [0, n_gu) followed by the down tiles. Every CTA takes its
// tiles in increasing order, so all of its gate_up tiles come before any of
// its down tiles; a down tile of expert e waits (once per CTA and expert)
// until every gate_up tile of e has been written.
template <int MODE>
__device__ __forceinline__ bool tile_is_gate_up(int t, int n_gu)
{
    if constexpr (MODE == 3)
        return t < n_gu;
    else
        return MODE != 1;
}

template <int MODE>
__device__ __forceinline__ TileInfo decode_any(int t, bool gu, const int* s_cnt, const int* s_off, const int* s_pre,
                                               const int* s_pre2, int n_gu, int BN, const MoeGemmParams& p)
{
    if constexpr (MODE == 3) {
        return gu ? decode_tile<0>(t, s_cnt, s_off, s_pre, p.E, BN, 1, p.rt_count, p.band)
                  : decode_tile<1>(t - n_gu, s_cnt, s_off, s_pre2, p.E, BN, p.ksplit2, p.rt_count2, p.band2);
    } else {
        (void)gu;
        (void)s_pre2;
        (void)n_gu;
        return decode_tile<MODE>(t, s_cnt, s_off, s_pre, p.E, BN, p.ksplit, p.rt_count, p.band);
    }
}

// Nibbles -> E4M3 operand bytes worth (q + 8) * 2^-9. The two output words
// hold the weights of one packed word in the order [0,2,4,6 | 1,3,5,7]: the
// K order inside every group of 8 is permuted, and the activation operands
// (gathered x, and hq written by the gate_up epilogue) are stored with the same
// permutation, so the dot products are unchanged and the unpack costs one
// shift and two AND/XOR per 8 weights.
__device__ __forceinline__ void unpack8(uint32_t w, uint32_t& lo4, uint32_t& hi4)
{
    lo4 = (w & 0x0F0F0F0Fu) ^ 0x08080808u;          // codes 0,2,4,6
    hi4 = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // codes 1,3,5,7
}

// Position of element i inside its group of 8 in the permuted K order.
__device__ __forceinline__ int kperm(int i)
{
    return (i & ~7) | ((i & 7) >> 1) | ((i & 1) << 2);
}

// SiLU: z * sigmoid(z). GELU (tanh form): 0.5 z (1 + tanh(u)) with
// u = sqrt(2/pi) (z + 0.044715 z^3), written as z * sigmoid(2u) (the same
// function). The result is quantized to E4M3 next (3 mantissa bits), so the
// error of the fast exponential and reciprocal is far below that rounding step.
__device__ __forceinline__ float act_fn(float z, int act)
{
    float t = -z;
    if (act != 0) {
        const float c2 = 1.5957691216057308f;  // 2 sqrt(2/pi)
        t = -c2 * fmaf(0.044715f * z, z * z, z);
    }
    return __fdividef(z, 1.0f + __expf(t));
}

// Two rings, both indexed by the global stage number g of this CTA.
//   W ring (NW slots, shared memory): packed weights. TMA -> wfull[w];
//     converters read the slot and free it at once (wfree[w]), so a weight slot
//     is held only for the HBM latency plus the conversion.
//   X ring (NX slots): the activation tile (shared memory, TMA -> bfull[x])
//     and the unpacked weights (TMEM, or shared memory, converters ->
//     afull[x]); the MMA's commit frees both (xfree[x]).
// Warp 0 issues weight copies as far ahead as the W ring allows; warp 2 issues
// activation copies, gated by xfree. A converter waits on bfull[x] as well,
// which both guarantees its A slot is free (bfull round r follows xfree round
// r-1) and lets the MMA wait on afull alone: one wait and one commit per stage
// in the single MMA thread.
// With a separate activation ring (NB != NX; the unpacked weights all in
// TMEM): activation tile b = g % NB arrives on bfull[b] and is freed by the
// MMA's commit to bfree[b]; A slot x = g % NX is freed by its commit to
// xfree[x], which the converters wait on; the MMA waits on afull[x] and
// bfull[b].
template <int MODE, int BN, int KC, int NW, int NX, int NXT, int NCONV, int NISS, int NB, int NEPI>
__global__ void __launch_bounds__(32 * (4 + NCONV + NEPI), 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_b2,
                    const MoeGemmParams p)
{
    using Tr = MoeTraits<MODE, BN, KC, NW, NX, NXT, NCONV, NISS, NB, NEPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* wring = smem;
    uint8_t* xring = smem + NW * Tr::kWBytes;
    uint8_t* aring = xring + NB * Tr::kXBytes;       // unpacked A of X slots NXT..NX-1
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kData);
    uint64_t* wfull = bars;
    uint64_t* wfree = wfull + NW;
    uint64_t* bfull = wfree + NW;                   // NB entries
    uint64_t* afull = bfull + NB;
    uint64_t* xfree = afull + NX;
    uint64_t* bfree = xfree + NX;                   // NB entries (separate activation ring only)
    uint64_t* accfull = bfree + NB;
    uint64_t* accempty = accfull + 2;
    uint64_t* drain = accempty + 2;                 // one per MMA issuer
    uint64_t* tq_full = drain + 2;                  // MODE 3 tile queue
    uint64_t* tq_free = tq_full + kTileQ;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tq_free + kTileQ);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* s_cnt = reinterpret_cast<int*>(s_tmem + 4);
    int* s_off = s_cnt + 256;
    int* s_pre = s_off + 260;
    int* s_pre2 = s_pre + 260;   // MODE 3: the down tiles' prefix over experts
    volatile int* s_tq = s_pre2 + 260;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // prefill tiles (A by TMA) wait with a suspend hint: their epilogue warps
    // wait through whole tiles and would otherwise take issue slots
    constexpr uint32_t kHint = Tr::kA8 ? 20000u : 0u;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NW; ++i) {
            mbar_init(smem_u32(&wfull[i]), 1);
            mbar_init(smem_u32(&wfree[i]), 4);   // one converter warp per lane quadrant
        }
        for (int i = 0; i < NX; ++i) {
            mbar_init(smem_u32(&afull[i]), Tr::kA8 ? 1 : 4);   // TMA of A, or one converter warp per quadrant
            mbar_init(smem_u32(&xfree[i]), 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(smem_u32(&bfull[i]), 1);
            mbar_init(smem_u32(&bfree[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&accfull[i]), NISS);
            mbar_init(smem_u32(&accempty[i]), NEPI);
        }
        mbar_init(smem_u32(&drain[0]), 1);
        mbar_init(smem_u32(&drain[1]), 1);
        for (int i = 0; i < kTileQ; ++i) {
            mbar_init(smem_u32(&tq_full[i]), 1);
            mbar_init(smem_u32(&tq_free[i]), Tr::kTileReaders);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_b);
        if constexpr (MODE == 3) {
            prefetch_tmap(&tm_w2);
            prefetch_tmap(&tm_b2);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), Tr::kTmemCols);
        tmem_relinquish();
    }
    // Programmatic launch: every kernel of the forward chain lets its
    // dependents launch only after its own griddepcontrol.wait returned, so
    // when this kernel runs, every kernel before its immediate predecessor has
    // completed -- in particular the router that wrote counts and offsets.
    // Those are read here without waiting, and the weight stream (which no
    // kernel writes) starts at once; only the activation producer and the
    // epilogue, which read or overwrite the predecessor's buffers, wait.
    if (threadIdx.x == 64) {
        int acc = 0, acc2 = 0;
        for (int e = 0; e < p.E; ++e) {
            const int c = p.counts[e];
            s_cnt[e] = c;
            s_off[e] = p.offsets[e];
            s_pre[e] = acc;
            acc += p.rt_count * ((c + BN - 1) / BN) * p.ksplit;
            if constexpr (MODE == 3) {
                s_pre2[e] = acc2;
                acc2 += p.rt_count2 * ((c + BN - 1) / BN) * p.ksplit2;
            }
        }
        s_pre[p.E] = acc;
        s_pre2[p.E] = acc2;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tmem_a = tmem + Tr::kDCols;   // A of X slots 0..NXT-1
    const int n_gu = s_pre[p.E];                   // MODE 3: the gate_up tiles come first
    const int total = n_gu + (MODE == 3 ? s_pre2[p.E] : 0);
    const int kb_second = (MODE == 3) ? p.kblocks2 : 0;

    auto fail = [&]() {
        *s_abort = 1;
        set_error(p.err, kErrBitTimeout);
    };
    // role: 0 the weight producer, 1 another single-thread role, 2 a whole warp.
    // MODE 3 claims the last kClaimRounds rounds of tiles (and the remainder).
    constexpr int kClaimRounds = 2;
    const int n_static = max(0, total / static_cast<int>(gridDim.x) - kClaimRounds) * static_cast<int>(gridDim.x);
    auto start_seq = [&](TileSeq& sq, int role) {
        if constexpr (MODE == 3)
            sq.init_dynamic(role, p.claim, s_tq, smem_u32(tq_full), smem_u32(tq_free), s_abort, total, n_gu,
                            p.kblocks, kb_second, n_static);
        else
            sq.init_static(total, p.kblocks, p.streamk != 0, n_gu, kb_second);
    };

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        // warp 0: packed weights into the W ring; warp 2: activations into the X ring
        if (lane == 0) {
            const bool wprod = (warp == 0);
            if (!wprod) {
                grid_dep_wait();
                grid_dep_launch();
            }
            // warp 0 fills the W ring, or (no converters) the A slots of the X ring
            const int nslot = wprod ? (Tr::kA8 ? NX : NW) : NB;
            uint64_t* fullb = wprod ? (Tr::kA8 ? afull : wfull) : bfull;
            uint64_t* freeb = wprod ? (Tr::kA8 ? xfree : wfree) : (Tr::kSplitB ? bfree : xfree);
            const uint64_t pol = wprod ? policy_evict_first() : policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;       // bit s: slot s was filled at least once
            uint32_t last_par = 0;     // bit s: parity of the last fill of slot s
            bool ok = true;
            int seen = -1;   // MODE 3: experts up to this one have all their gate_up tiles written
            // prefill down GEMM pacing (weight producer): stages issued so far
            const bool pace = (MODE == 1) && wprod && p.sync != nullptr;
            uint32_t gst = 0;
            TileSeq wi;
            for (start_seq(wi, wprod ? 0 : 1); wi.valid() && ok;) {
                const int t = wi.t;
                const bool gu = tile_is_gate_up<MODE>(t, n_gu);
                const TileInfo ti = decode_any<MODE>(t, gu, s_cnt, s_off, s_pre, s_pre2, n_gu, BN, p);
                const bool second = (MODE == 3 && !gu);
                const int kbl = second ? p.kblocks2 : p.kblocks;
                const int rpe = second ? p.rows_per_expert2 : p.rows_per_expert;
                const CUtensorMap* mw = second ? &tm_w2 : &tm_w;
                const CUtensorMap* mb = second ? &tm_b2 : &tm_b;
                if constexpr (MODE == 3) {
                    // the down tile reads the intermediate of expert e (TMA): wait
                    // until the NEPI epilogue warps of each of e's gate_up tiles counted
                    if (!wprod && second && ti.e > seen) {
                        const int need = NEPI * (s_pre[ti.e + 1] - s_pre[ti.e]);
                        if (!counter_wait_or_abort(p.done + ti.e, need, s_abort)) {
                            ok = false;
                            break;
                        }
                        seen = ti.e;
                    }
                }
                for (int kb = wi.kb0; kb < wi.kb0 + wi.nkb; ++kb) {
                    if (wi.claim_here(kb, 4))
                        wi.claim_next();
                    if (pace && gst % kMoeSyncEvery == 0) {
                        const int c = static_cast<int>(gst / kMoeSyncEvery);
                        if (c < kMoeSyncInts - 1) {
                            if (c >= kMoeSyncSlack &&
                                !pace_wait_or_abort(p.sync + (c - kMoeSyncSlack), p.sync + (kMoeSyncInts - 1),
                                                    static_cast<int>(gridDim.x), s_abort)) {
                                ok = false;
                                break;
                            }
                            atomicAdd(p.sync + c, 1);
                        }
                    }
                    ++gst;
                    if (!mbar_wait_or_abort<kHint>(smem_u32(&freeb[s]), ph ^ 1u, s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&fullb[s]);
                    const int kel = (ti.ks * kbl + kb) * KC;  // first K element
                    if (Tr::kA8 && wprod) {
                        // unpacked weight rows, already in the tile's row order
                        mbar_arrive_expect_tx(fb, Tr::kASlot);
                        uint8_t* st = aring + (s - NXT) * Tr::kASlot;
                        const int r0 = ti.e * rpe + ti.rt * 128;
#pragma unroll
                        for (int a = 0; a < Tr::kAtoms; ++a)
                            tma_load_2d_hint(smem_u32(st + a * 128 * 128), mw, kel + a * 128, r0, fb, pol);
                    } else if (wprod) {
                        mbar_arrive_expect_tx(fb, Tr::kWBytes);
                        uint8_t* st = wring + s * Tr::kWBytes;
#pragma unroll
                        for (int wa = 0; wa < Tr::kWBoxes; ++wa) {
                            // one box = 128 rows x kWBoxBytes (gate_up: 64 gate + 64 up rows)
                            uint8_t* wd = st + wa * 128 * Tr::kWBoxBytes;
                            const int kx = kel / 2 + wa * Tr::kWBoxBytes;
                            if (gu) {   // gate_up (static or dynamic scale)
                                const int r0 = ti.e * rpe + ti.rt * 64;
                                tma_load_2d_hint(smem_u32(wd), mw, kx, r0, fb, pol);
                                tma_load_2d_hint(smem_u32(wd + 64 * Tr::kWBoxBytes), mw, kx, r0 + p.I, fb, pol);
                            } else {
                                const int r0 = ti.e * rpe + ti.rt * 128;
                                tma_load_2d_hint(smem_u32(wd), mw, kx, r0, fb, pol);
                            }
                        }
                    } else {
                        mbar_arrive_expect_tx(fb, Tr::kBBytes);
                        uint8_t* st = xring + s * Tr::kXBytes;
#pragma unroll
                        for (int a = 0; a < Tr::kAtoms; ++a)
                            tma_load_2d_hint(smem_u32(st + a * BN * 128), mb, kel + a * 128, ti.tok0, fb, pol);
                    }
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == nslot) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok)   // (after a failed wait nothing more is published)
                    wi.next();
            }
            if (pace)
                atomicAdd(p.sync + (kMoeSyncInts - 1), 1);   // this CTA's weight stream is done
            if constexpr (MODE == 3) {
                if (wprod) {
                    // this CTA makes no further claim; the last CTA to get here
                    // leaves the claim counters zero for the next launch (off
                    // the kernel's tail: the weight stream ends before the
                    // CTA's last tile does)
                    __threadfence();
                    if (atomicAdd(p.claim + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                        atomicExch(p.claim, 0);
                        atomicExch(p.claim + 1, 0);
                    }
                }
            }
            ok = ok && wi.ok;
            if (!ok) {
                fail();
                // let every issued copy land before the CTA's shared memory goes away
                for (int i = 0; i < nslot; ++i)
                    if ((issued >> i) & 1u)
                        mbar_wait(smem_u32(&fullb[i]), (last_par >> i) & 1u);
            }
        }
    } else if (warp == 1 || (NISS == 2 && warp == 3)) {
        // ------------------------------------------------------------ MMA issuers
        // One thread issues tcgen05.mma at a bounded rate; with NISS = 2 a
        // second thread (warp 3) takes every other stage into its own partial
        // accumulator, which nearly doubles the MMA issue rate for the narrow
        // (few-token) tiles of decoding.
        if (lane == 0) {
            const int me = (warp == 1) ? 0 : 1;
            int x = 0, b = 0;
            uint32_t ph = 0, bph = 0;
            uint32_t g = 0;
            int it = 0;
            bool ok = true;
            TileSeq wi;
            for (start_seq(wi, 1); wi.valid() && ok; wi.next(), ++it) {
                const TileInfo ti = decode_any<MODE>(wi.t, tile_is_gate_up<MODE>(wi.t, n_gu), s_cnt, s_off, s_pre,
                                                     s_pre2, n_gu, BN, p);
                const int nmma = max(16, (ti.ntok + 15) & ~15);
                const uint32_t idesc = idesc_e4m3_f32(128, nmma);
                const int d = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait_or_abort<kHint>(smem_u32(&accempty[d]), (use & 1u) ^ 1u, s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + static_cast<uint32_t>((d * NISS + me) * BN);
                bool first = true;
                for (int kb = 0; kb < wi.nkb; ++kb, ++g) {
                    if (static_cast<int>(g % NISS) == me) {
                        if (!mbar_wait_or_abort<kHint>(smem_u32(&afull[x]), ph, s_abort) ||
                            ((Tr::kSplitB || Tr::kA8) && !mbar_wait_or_abort<kHint>(smem_u32(&bfull[b]), bph, s_abort))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint8_t* st = xring + (Tr::kSplitB ? b : x) * Tr::kXBytes;
                        const uint64_t bd0 = desc_kmajor_sw128(smem_u32(st));
                        const bool a_tmem = Tr::a_in_tmem(x);
                        const uint64_t ad0 =
                            a_tmem ? 0 : desc_kmajor_sw128(smem_u32(aring + (x - NXT) * Tr::kASlot));
#pragma unroll
                        for (int kk = 0; kk < KC / 32; ++kk) {
                            const int atom = kk >> 2, sub = kk & 3;
                            // start-address field advances in 16-byte units
                            const uint64_t bd = bd0 + static_cast<uint64_t>((atom * BN * 128 + sub * 32) >> 4);
                            const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                            if (a_tmem) {
                                umma_f8_ta(dt, tmem_a + static_cast<uint32_t>(x * Tr::kACols + kk * 8), bd, idesc,
                                           acc);
                            } else {
                                const uint64_t ad = ad0 + static_cast<uint64_t>((atom * 128 * 128 + sub * 32) >> 4);
                                umma_f8(dt, ad, bd, idesc, acc);
                            }
                        }
                        first = false;
                        umma_commit(smem_u32(&xfree[x]));
                        if constexpr (Tr::kSplitB)
                            umma_commit(smem_u32(&bfree[b]));
                    }
                    if (++x == NX) {
                        x = 0;
                        ph ^= 1u;
                    }
                    if (++b == NB) {
                        b = 0;
                        bph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(smem_u32(&accfull[d]));   // (an issuer with no stage in this tile arrives at once)
            }
            ok = ok && wi.ok;
            if (!ok) {
                fail();
                umma_commit(smem_u32(&drain[me]));  // wait for MMAs in flight before TMEM goes away
                mbar_wait(smem_u32(&drain[me]), 0);
            }
        }
    } else if (warp >= 4 && warp < Tr::kEpi0) {
        // ------------------------------------------------------------ converters
        // Warp w covers TMEM lane quadrant w % 4 (rows 32q..32q+31); with
        // NCONV = 8 the two warps of a quadrant take alternate stages.
        const int q = warp & 3;
        const int par = (warp - 4) >> 2;
        const int r = 32 * q + lane;  // A row == TMEM lane
        // gate_up: lanes 0-15 of each quadrant take gate rows, lanes 16-31 the
        // matching up rows (so one warp holds both halves of a gated pair)
        const int src_gu = (lane < 16) ? (16 * q + lane) : (64 + 16 * q + (lane - 16));
        int w = 0, x = 0;
        uint32_t wph = 0, xph = 0;
        uint32_t g = 0;
        bool ok = true;
        TileSeq wi;
        for (start_seq(wi, 2); wi.valid() && ok; wi.next()) {
            const int src = tile_is_gate_up<MODE>(wi.t, n_gu) ? src_gu : r;
            for (int kb = 0; kb < wi.nkb; ++kb, ++g) {
                if (static_cast<int>(g % Tr::kPar) == par) {
                    // the A slot is free once the MMAs of its previous round
                    // completed: seen through that round's activation copy
                    // (shared ring), or the MMA's commit (separate ring)
                    if (!mbar_wait_or_abort<kHint>(smem_u32(&wfull[w]), wph, s_abort) ||
                        !mbar_wait_or_abort<kHint>(smem_u32(Tr::kSplitB ? &xfree[x] : &bfull[x]),
                                            Tr::kSplitB ? (xph ^ 1u) : xph, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* wst = wring + w * Tr::kWBytes;
#pragma unroll
                    for (int half = 0; half < KC / 128; ++half) {
                        uint32_t o[32];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int c = half * 4 + c4;  // packed 16-byte chunk (32 weights)
                            // undo the TMA swizzle: 64-byte boxes (KC = 128) XOR chunk
                            // bits with row bits 1-2, 128-byte boxes with row bits 0-2
                            const uint8_t* wp =
                                (KC == 128) ? wst + src * 64 + ((c ^ ((src >> 1) & 3)) << 4)
                                            : wst + (c >> 3) * (128 * 128) + src * 128 + (((c & 7) ^ (src & 7)) << 4);
                            const uint4 w4 = *reinterpret_cast<const uint4*>(wp);
                            unpack8(w4.x, o[8 * c4 + 0], o[8 * c4 + 1]);
                            unpack8(w4.y, o[8 * c4 + 2], o[8 * c4 + 3]);
                            unpack8(w4.z, o[8 * c4 + 4], o[8 * c4 + 5]);
                            unpack8(w4.w, o[8 * c4 + 6], o[8 * c4 + 7]);
                        }
                        if (Tr::a_in_tmem(x)) {
                            tmem_st32(tmem_a + (static_cast<uint32_t>(q * 32) << 16) +
                                          static_cast<uint32_t>(x * Tr::kACols + half * 32),
                                      o);
                        } else {
                            uint8_t* arow = aring + (x - NXT) * Tr::kASlot + half * (128 * 128) + r * 128;
#pragma unroll
                            for (int c16 = 0; c16 < 8; ++c16)
                                *reinterpret_cast<uint4*>(arow + ((c16 ^ (r & 7)) << 4)) =
                                    make_uint4(o[4 * c16], o[4 * c16 + 1], o[4 * c16 + 2], o[4 * c16 + 3]);
                        }
                    }
                    // the packed slot has been read: hand it back to the producer now
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&wfree[w]));
                    if (Tr::a_in_tmem(x)) {
                        tmem_st_wait();
                        tc_fence_before();
                    } else {
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&afull[x]));
                }
                if (++w == NW) {
                    w = 0;
                    wph ^= 1u;
                }
                if (++x == NX) {
                    x = 0;
                    xph ^= 1u;
                }
            }
        }
        ok = ok && wi.ok;
        if (!ok)
            fail();
    } else if (warp >= Tr::kEpi0) {
        // ------------------------------------------------------------ epilogue
        // Prefill: the intermediate and the fp32 partial sums are read back by
        // later kernels, long after L2 could hold them, so their stores are
        // marked first to leave L2 (it keeps the operand panels the tiles in
        // flight share). The one-launch decode reads both back from L2 soon
        // after: plain stores there.
        const uint64_t pol_out = policy_evict_first();
        const int q = warp & 3;
        const int sub = (warp - Tr::kEpi0) >> 2;   // chunk phase: 32-column chunks sub, sub + NEPI/4, ...
        constexpr int kChStep = NEPI / 4;
        grid_dep_wait();
        grid_dep_launch();
        const float a1 = __ldg(p.a1);
        const float a2 = __ldg(p.a2);
        uint32_t gsum = 0;   // global stage index of the tile's first stage
        int it = 0;
        bool ok = true;
        TileSeq wi;
        for (start_seq(wi, 2); wi.valid() && ok; wi.next(), ++it) {
            const bool gu = tile_is_gate_up<MODE>(wi.t, n_gu);
            const TileInfo ti = decode_any<MODE>(wi.t, gu, s_cnt, s_off, s_pre, s_pre2, n_gu, BN, p);
            const int d = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait_or_abort<kHint>(smem_u32(&accfull[d]), use & 1u, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(d * NISS * BN);
            // partial sum of issuer i is valid when the issuer had a stage in
            // this tile: always when the tile has two or more stages
            const bool v0 = NISS == 1 || wi.nkb >= 2 || (gsum % NISS) == 0;
            const bool v1 = NISS == 2 && (wi.nkb >= 2 || (gsum % NISS) == 1);
            gsum += wi.nkb;
            auto load_acc = [&](int c, uint32_t (&v)[32]) {
                if (v0) {
                    tmem_ld32(tbase + c, v);
                } else {
#pragma unroll
                    for (int xx = 0; xx < 32; ++xx)
                        v[xx] = 0u;
                }
                if (v1) {
                    uint32_t w2[32];
                    tmem_ld32(tbase + BN + c, w2);
                    tmem_ld_wait();
#pragma unroll
                    for (int xx = 0; xx < 32; ++xx)
                        v[xx] = __float_as_uint(__uint_as_float(v[xx]) + __uint_as_float(w2[xx]));
                }
                tmem_ld_wait();
            };
            const int nchunks = (ti.ntok + 31) >> 5;
            if (gu) {   // gate_up (static or dynamic scale)
                const int half = lane >> 4;  // 0: gate lane, 1: up lane
                const int i = ti.rt * 64 + 16 * q + (lane & 15);
                const float sg = a1 * __ldg(p.s_gu + static_cast<int64_t>(ti.e) * 2 * p.I + i);
                const float su = a1 * __ldg(p.s_gu + static_cast<int64_t>(ti.e) * 2 * p.I + p.I + i);
                for (int ch = sub; ch < nchunks; ch += kChStep) {
                    // lane l fetches the exact shift of column ch*32 + l up front
                    // (the loop below hands it around by shuffle), so no load
                    // waits behind the byte stores of the loop; weights unpacked
                    // ahead (A by TMA) carry their signed values, no shift
                    const int mycol = ch * 32 + lane;
                    const long long my_s0x =
                        (!Tr::kA8 && mycol < ti.ntok) ? __ldg(p.s0x + ti.tok0 + mycol) : 0LL;
                    uint32_t v[32];
                    load_acc(ch * 32, v);
                    const float my_shift = static_cast<float>(my_s0x) * (1.0f / 64.0f);
                    float s512[16];   // 512 * dec(hq): integers, summed exactly in fp32
                    float hmax_l = 0.0f;
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        // gate lanes finish column cc, up lanes column 16+cc
                        const float send = __uint_as_float(half ? v[cc] : v[cc + 16]);
                        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
                        const float pg = half ? recv : __uint_as_float(v[cc]);
                        const float pu = half ? __uint_as_float(v[cc + 16]) : recv;
                        const int col = ch * 32 + cc + 16 * half;
                        const float shift = Tr::kA8 ? 0.0f : __shfl_sync(0xFFFFFFFFu, my_shift, cc + 16 * half);
                        s512[cc] = 0.0f;
                        if (col < ti.ntok) {
                            const int pos = ti.tok0 + col;
                            const float G = Tr::kA8 ? pg : fmaf(512.0f, pg, -shift);
                            const float U = Tr::kA8 ? pu : fmaf(512.0f, pu, -shift);
                            const float h = act_fn(sg * G, p.act) * (su * U);
                            if constexpr (MODE == 2) {
                                p.hf[static_cast<int64_t>(pos) * p.I + i] = h;
                                hmax_l = fmaxf(hmax_l, fabsf(h));
                            } else {
                                // hq = E4M3(h / a2): IEEE division, then one RNE rounding
                                const uint32_t code = cvt_e4m3(__fdiv_rn(h, a2));
                                uint8_t* dst = p.hq + static_cast<int64_t>(pos) * p.I + kperm(i);
                                if constexpr (Tr::kA8)
                                    st_u8_hint(dst, code, pol_out);
                                else
                                    *dst = static_cast<uint8_t>(code);
                                if constexpr (!Tr::kA8)
                                    s512[cc] = e4m3_times512_f32(code);
                            }
                        }
                    }
                    if constexpr (MODE == 2) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1)
                            hmax_l = fmaxf(hmax_l, __shfl_xor_sync(0xFFFFFFFFu, hmax_l, o));
                        if (lane == 0 && hmax_l > 0.0f)   // non-negative floats order like their bits
                            atomicMax(p.hmax, __float_as_uint(hmax_l));
                    } else if constexpr (!Tr::kA8) {   // the down GEMM's shift: exact row sums of hq
                        // reduce-scatter over the 16 lanes of each half: lane ends
                        // with the sum of column ch*32 + lane over this warp's rows
#pragma unroll
                        for (int m = 8; m >= 1; m >>= 1) {
                            const bool upper = (lane & m) != 0;
#pragma unroll
                            for (int x = 0; x < m; ++x) {
                                const float send = upper ? s512[x] : s512[x + m];
                                const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, m);
                                s512[x] = (upper ? s512[x + m] : s512[x]) + recv;
                            }
                        }
                        // |sum| <= 16 * 229376 < 2^24: exact, and exactly an integer
                        const int col = ch * 32 + lane;
                        if (col < ti.ntok && s512[0] != 0.0f)
                            atomicAdd(p.s0h + ti.tok0 + col,
                                      static_cast<unsigned long long>(static_cast<long long>(s512[0])));
                    }
                }
                if constexpr (MODE == 3) {
                    // publish this warp's quarter of the tile to the down tiles
                    // (which read it with TMA, in other CTAs): every lane's
                    // stores are made visible before lane 0 counts
                    __threadfence();
                    fence_proxy_async_global();
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        atomicAdd(p.done + ti.e, 1);
                    }
                }
            } else {
                const int n = ti.rt * 128 + q * 32 + lane;
                int slot = p.streamk ? wi.slot : ti.ks;
                if (p.streamk && slot >= p.nslots) {   // excluded by the host's bound
                    set_error(p.err, kErrBitTimeout);
                    slot = -1;
                }
                float* yb = p.ypart + (static_cast<int64_t>(slot) * p.A + ti.tok0) * p.H + n;
                if (p.streamk && wi.last && sub == 0) {
                    // the tile's last segment: slots no CTA writes hold zero
                    for (int sl = wi.slot + 1; sl < p.nslots; ++sl)
                        for (int col = 0; col < ti.ntok; ++col)
                            p.ypart[(static_cast<int64_t>(sl) * p.A + ti.tok0 + col) * p.H + n] = 0.0f;
                }
                for (int ch = sub; ch < nchunks; ch += kChStep) {
                    uint32_t v[32];
                    load_acc(ch * 32, v);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const int col = ch * 32 + cc;
                        if (col < ti.ntok && slot >= 0) {
                            if constexpr (Tr::kA8)
                                st_f32_hint(yb + static_cast<int64_t>(col) * p.H, __uint_as_float(v[cc]), pol_out);
                            else
                                yb[static_cast<int64_t>(col) * p.H] = __uint_as_float(v[cc]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&accempty[d]));
        }
        ok = ok && wi.ok;
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

// ---------------------------------------------------------------------------
// Gather: xp[pos] = x[sorted[pos] / k] (bytes in the permuted K order of
// unpack8); s0x[pos] = sum_h 512*dec(x) (exact);
// s0h[pos] = 0 (the gate_up epilogue accumulates into it).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) moe_gather_kernel(const uint8_t* __restrict__ xq, int H, int k,
                                                         const int32_t* __restrict__ sorted_ids,
                                                         int A, uint8_t* __restrict__ xp,
                                                         long long* __restrict__ s0x,
                                                         unsigned long long* __restrict__ s0h,
                                                         unsigned int* __restrict__ hmax, int* __restrict__ done,
                                                         int E, int sums, int* __restrict__ sync)
{
    // one block per assignment row: every 16-byte chunk of the row is in
    // flight at once. sums = 0 (weights unpacked ahead as signed codes): the
    // GEMMs need no exact row sums, and only the copy is done.
    __shared__ long long red[4];
    grid_dep_wait();
    grid_dep_launch();
    if (hmax && blockIdx.x == 0 && threadIdx.x == 0)
        *hmax = 0u;   // max|h| of the dynamic intermediate scale starts at zero
    if (done && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            done[e] = 0;   // per-expert gate_up progress of the one-launch forward
    if (sync && blockIdx.x == 1 % gridDim.x)
        for (int i = threadIdx.x; i < kMoeSyncInts; i += blockDim.x)
            sync[i] = 0;   // the prefill down GEMM's pacing counters
    const int pos = blockIdx.x;
    const int t = __ldg(sorted_ids + pos) / k;
    const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<int64_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<int64_t>(pos) * H);
    if (!sums) {
        // rows of at most 4 chunks per thread: all loads issued first
        constexpr int U = 4;
        for (int c0 = threadIdx.x; c0 < H / 16; c0 += U * blockDim.x) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + u * static_cast<int>(blockDim.x) < H / 16)
                    v[u] = __ldg(src + c0 + u * blockDim.x);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * static_cast<int>(blockDim.x);
                if (c < H / 16)
                    dst[c] = make_uint4(prmt(v[u].x, v[u].y, 0x6420u), prmt(v[u].x, v[u].y, 0x7531u),
                                        prmt(v[u].z, v[u].w, 0x6420u), prmt(v[u].z, v[u].w, 0x7531u));
            }
        }
        return;
    }
    int s = 0;
    for (int c = threadIdx.x; c < H / 16; c += blockDim.x) {
        const uint4 v = __ldg(src + c);
        // permuted K order inside each group of 8 (see unpack8)
        dst[c] = make_uint4(prmt(v.x, v.y, 0x6420u), prmt(v.x, v.y, 0x7531u), prmt(v.z, v.w, 0x6420u),
                            prmt(v.z, v.w, 0x7531u));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int b = 0; b < 4; ++b)
                s += e4m3_times512((u[j] >> (8 * b)) & 0xFFu);
    }
    long long sum = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long total = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w)
            total += red[w];
        s0x[pos] = total;
        s0h[pos] = 0ull;
    }
}

// ---------------------------------------------------------------------------
// Prefill: the INT4 weights of every expert with tokens, unpacked once per call
// into E4M3 codes of their signed values q (every INT4 value is exact in E4M3),
// codes of a packed word in the K order of unpack8, so that the GEMM loads A by
// TMA and its tiles each reuse it instead of unpacking it again for every token
// tile; with signed values the products need no offset correction. gate_up rows
// are stored in tile order: 128-row tile rt holds, for each TMEM lane quadrant
// q, gate rows rt*64 + 16q + 0..15 and then the matching up rows (the pairing of
// the gated epilogue). One thread per 16 packed bytes (32 weights) of a row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3_of_int4_pair4(uint32_t w, int first)
{
    // nibbles first, first + 2, first + 4, first + 6 of w -> their E4M3 codes
    float f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        f[j] = static_cast<float>(static_cast<int32_t>(w << (28 - 4 * (first + 2 * j))) >> 28);
    return static_cast<uint32_t>(cvt_e4m3x2(f[1], f[0])) | (static_cast<uint32_t>(cvt_e4m3x2(f[3], f[2])) << 16);
}
__device__ __forceinline__ void unpack8_signed(uint32_t w, uint32_t& lo4, uint32_t& hi4)
{
    lo4 = e4m3_of_int4_pair4(w, 0);   // codes 0,2,4,6
    hi4 = e4m3_of_int4_pair4(w, 1);   // codes 1,3,5,7
}

__global__ void __launch_bounds__(256) moe_upcast_kernel(const int32_t* __restrict__ w_gu,
                                                         const int32_t* __restrict__ w_d, int E, int H, int I,
                                                         const int32_t* __restrict__ counts,
                                                         uint8_t* __restrict__ a_gu, uint8_t* __restrict__ a_d)
{
    grid_dep_wait();
    grid_dep_launch();
    const int64_t gu_chunks = static_cast<int64_t>(E) * 2 * I * (H / 32);   // 16-byte chunks of packed gate_up
    const int64_t d_chunks = static_cast<int64_t>(E) * H * (I / 32);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < gu_chunks + d_chunks;
         c += stride) {
        const bool gu = c < gu_chunks;
        const int64_t cc = gu ? c : c - gu_chunks;
        const int K = gu ? H : I;
        const int rows = gu ? 2 * I : H;
        const int per_row = K / 32;
        const int64_t row = cc / per_row;             // expert * rows + output row
        const int j = static_cast<int>(cc - row * per_row);
        const int e = static_cast<int>(row / rows);
        if (__ldg(counts + e) == 0)
            continue;
        const int R = static_cast<int>(row - static_cast<int64_t>(e) * rows);
        int src = R;
        if (gu) {
            const int rt = R >> 7, r = R & 127, q = r >> 5, l = r & 31;
            src = (l < 16) ? rt * 64 + 16 * q + l : I + rt * 64 + 16 * q + (l - 16);
        }
        const int32_t* w = gu ? w_gu : w_d;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(w + (static_cast<int64_t>(e) * rows + src) * (K / 8)) + j);
        uint32_t o[8];
        unpack8_signed(v.x, o[0], o[1]);
        unpack8_signed(v.y, o[2], o[3]);
        unpack8_signed(v.z, o[4], o[5]);
        unpack8_signed(v.w, o[6], o[7]);
        uint4* dst = reinterpret_cast<uint4*>((gu ? a_gu : a_d) + row * K) + 2 * j;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ---------------------------------------------------------------------------
// Dynamic intermediate scale: a2 = max|h| / 448 over every assignment of the
// call (1 if all h are zero), then hq = E4M3(h / a2) (IEEE division) in the permuted K order
// of unpack8 and the exact row sums s0h[pos] = sum_i 512*dec(hq). One block per
// assignment row; 8 consecutive h per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_hquant_kernel(const float* __restrict__ hf, int I,
                                                         const unsigned int* __restrict__ hmax,
                                                         float* __restrict__ a2_out,
                                                         uint8_t* __restrict__ hq,
                                                         unsigned long long* __restrict__ s0h)
{
    grid_dep_wait();
    grid_dep_launch();
    __shared__ long long red[8];
    const float mx = __uint_as_float(__ldcg(hmax));
    const float s2 = (mx > 0.0f && mx <= 3.4028234663852886e38f) ? __fdiv_rn(mx, 448.0f) : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *a2_out = s2;
    const int pos = blockIdx.x;
    const float4* row = reinterpret_cast<const float4*>(hf + static_cast<int64_t>(pos) * I);
    uint2* dst = reinterpret_cast<uint2*>(hq + static_cast<int64_t>(pos) * I);
    long long sum = 0;
    for (int g = threadIdx.x; g < I / 8; g += blockDim.x) {
        const float4 a = __ldcg(row + 2 * g), b = __ldcg(row + 2 * g + 1);
        const float h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = cvt_e4m3(__fdiv_rn(h[j], s2));
            sum += e4m3_times512(c[j]);
        }
        // byte order inside the group: elements 0,2,4,6 then 1,3,5,7
        uint2 o;
        o.x = c[0] | (c[2] << 8) | (c[4] << 16) | (c[6] << 24);
        o.y = c[1] | (c[3] << 8) | (c[5] << 16) | (c[7] << 24);
        dst[g] = o;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long t = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w)
            t += red[w];
        s0h[pos] = static_cast<unsigned long long>(t);
    }
}

// ---------------------------------------------------------------------------
// Combine: out[t, n] = bf16( sum_j w[t,j] * a2 * S_d[e,n] * D ),
// D = 512 * sum_splits P - s0h/64 (weights with the +8 offset, unpacked in the
// GEMM), or D = sum_splits P (signed weights unpacked ahead: s0h = null,
// pmul = 1), in j then split order (deterministic).
// The routing arrays come from a kernel at least two launches back and S_d
// and a2 from no kernel of this forward (or, for the dynamic scale, two
// launches back), so they are fetched before the dependency wait; only the
// partial sums and s0h, which the GEMM writes, are read after it.
// ---------------------------------------------------------------------------

template <int KS_MAX>
__device__ __forceinline__ void fin_accumulate(float (&acc)[4], int pos, float wt, float4 sd, float a2, int A, int H,
                                               int n, int ksplit, const float* __restrict__ ypart,
                                               const unsigned long long* __restrict__ s0h, float pmul)
{
    // all split partials (at most KS_MAX) are requested before the first one
    // is added, then summed in split order
    float4 v[KS_MAX];
#pragma unroll
    for (int s = 0; s < KS_MAX; ++s)
        if (s < ksplit)
            v[s] = __ldg(reinterpret_cast<const float4*>(ypart + (static_cast<int64_t>(s) * A + pos) * H + n));
    const float shift = s0h ? static_cast<float>(static_cast<long long>(__ldg(s0h + pos))) * (1.0f / 64.0f) : 0.0f;
    float4 P = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < KS_MAX; ++s) {
        if (s < ksplit) {
            P.x += v[s].x;
            P.y += v[s].y;
            P.z += v[s].z;
            P.w += v[s].w;
        }
    }
    const float Pv[4] = {P.x, P.y, P.z, P.w};
    const float Sv[4] = {sd.x, sd.y, sd.z, sd.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float D = fmaf(pmul, Pv[c], -shift);
        acc[c] = fmaf(wt, a2 * Sv[c] * D, acc[c]);
    }
}

// KPRE: assignments per token fetched before the dependency wait (the rest,
// for k > KPRE, after it); sized by k so that the registers of unused slots
// do not cost occupancy (a memory-bound pass needs its loads in flight).
template <int KS_MAX, int KPRE>
__global__ void __launch_bounds__(256) moe_finalize_kernel(
    int T, int H, int k, int A, int ksplit, const int32_t* __restrict__ ids,
    const float* __restrict__ topk_w, const int32_t* __restrict__ inv,
    const float* __restrict__ ypart, const unsigned long long* __restrict__ s0h, float pmul,
    const float* __restrict__ s_d, const float* __restrict__ a2p, uint16_t* __restrict__ out)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int per_row = H / 4;
    const bool live = idx < static_cast<int64_t>(T) * per_row;
    const int t = live ? static_cast<int>(idx / per_row) : 0;
    const int n = live ? static_cast<int>(idx % per_row) * 4 : 0;
    int pos_p[KPRE];
    float wt_p[KPRE];
    float4 sd_p[KPRE];
    float a2 = 0.0f;
    if (live) {
        a2 = __ldg(a2p);
#pragma unroll
        for (int j = 0; j < KPRE; ++j) {
            if (j < k) {
                const int a = t * k + j;
                pos_p[j] = __ldg(inv + a);
                wt_p[j] = __ldg(topk_w + a);
                const int e = __ldg(ids + a);
                sd_p[j] = __ldg(reinterpret_cast<const float4*>(s_d + static_cast<int64_t>(e) * H + n));
            }
        }
    }
    grid_dep_wait();
    grid_dep_launch();
    if (!live)
        return;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (KS_MAX == 1) {
        // one partial per assignment: every assignment's partial requested
        // before the first is added
        float4 v[KPRE];
#pragma unroll
        for (int j = 0; j < KPRE; ++j)
            if (j < k)
                v[j] = __ldg(reinterpret_cast<const float4*>(ypart + static_cast<int64_t>(pos_p[j]) * H + n));
#pragma unroll
        for (int j = 0; j < KPRE; ++j) {
            if (j < k) {
                const float shift =
                    s0h ? static_cast<float>(static_cast<long long>(__ldg(s0h + pos_p[j]))) * (1.0f / 64.0f) : 0.0f;
                const float Pv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                const float Sv[4] = {sd_p[j].x, sd_p[j].y, sd_p[j].z, sd_p[j].w};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[c] = fmaf(wt_p[j], a2 * Sv[c] * fmaf(pmul, Pv[c], -shift), acc[c]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < KPRE; ++j)
            if (j < k)
                fin_accumulate<KS_MAX>(acc, pos_p[j], wt_p[j], sd_p[j], a2, A, H, n, ksplit, ypart, s0h, pmul);
    }
    for (int j = KPRE; j < k; ++j) {
        const int a = t * k + j;
        const int e = __ldg(ids + a);
        fin_accumulate<KS_MAX>(acc, __ldg(inv + a), __ldg(topk_w + a),
                               __ldg(reinterpret_cast<const float4*>(s_d + static_cast<int64_t>(e) * H + n)), a2, A,
                               H, n, ksplit, ypart, s0h, pmul);
    }
    uint2 o;
    o.x = static_cast<uint32_t>(float_to_bf16_bits(acc[0])) |
          (static_cast<uint32_t>(float_to_bf16_bits(acc[1])) << 16);
    o.y = static_cast<uint32_t>(float_to_bf16_bits(acc[2])) |
          (static_cast<uint32_t>(float_to_bf16_bits(acc[3])) << 16);
    *reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * H + n) = o;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int moe_ksplit_max(int T, int k)
{
    const int64_t A = static_cast<int64_t>(T) * k;
    if (A <= 128)
        return kMaxKsplit;
    if (A <= 1024)
        return 4;
    return 1;
}

static int pick_bn(int T)
{
    if (T <= 32)
        return 32;
    if (T <= 64)
        return 64;
    if (T <= 128)
        return 128;
    return 256;
}

// One launch for both projections (static intermediate scale, token tiles
// up to 128): the CTAs take the gate_up tiles and then the down tiles round
// robin, so an SM that runs out of gate_up tiles streams down weights at once
// instead of idling until the slowest gate_up CTA ends. The down split is
// picked for the balance of that whole list, assuming the T*k assignments
// spread evenly over min(E, T*k) experts: the cost of a split d is the most
// stages any CTA gets (plus one per tile, the accumulator hand-off) plus the
// reduction of the d partial sums, counted in stage times of the whole GPU.
static int fused_ksplit(int T, int H, int I, int E, int k, int bn, int kc, int num_sms)
{
    const int64_t A = static_cast<int64_t>(T) * k;
    const int64_t act = A < E ? A : E;
    const int64_t per = (A + act - 1) / act;
    const int64_t ntt = (per + bn - 1) / bn;
    const int64_t n_gu = act * (I / 64) * ntt;
    const int kb_gu = (H + kc - 1) / kc, kb_all = (I + kc - 1) / kc;
    const int kmax = moe_ksplit_max(T, k);
    const int64_t G = num_sms;
    const double stage_bytes = static_cast<double>(G) * 128 * kc / 2;   // one stage on every SM
    int best = 1;
    double best_cost = 0.0;
    for (int d = 1; d <= kmax; ++d) {
        if (kb_all % d != 0 || kb_all / d < 2)
            continue;
        const int kb_dn = kb_all / d;
        const int64_t n = n_gu + act * (H / 128) * ntt * d;
        int64_t worst = 0;
        for (int64_t c = 0; c < G && c < n; ++c) {
            const int64_t mine = (n - c + G - 1) / G;
            const int64_t mine_gu = c < n_gu ? (n_gu - c + G - 1) / G : 0;
            const int64_t cost = mine_gu * (kb_gu + 1) + (mine - mine_gu) * (kb_dn + 1);
            worst = cost > worst ? cost : worst;
        }
        // partial sums: written once, read once by the combine
        const double red = 2.0 * d * static_cast<double>(A) * H * 4 / stage_bytes;
        const double cost = static_cast<double>(worst) + (d > 1 ? red : 0.0);
        if (d == 1 || cost < best_cost) {
            best_cost = cost;
            best = d;
        }
    }
    return best;
}

bool moe_unpack_once(int T) { return T > 128; }

// Prefill tile-order band (see decode_tile): 16 token tiles of 256 tokens
// (about 25 MB of gathered activations at hidden 6144) for gate_up, 16
// weight-row tiles for down.
constexpr int kPrefillBand = 16;

MoeConfig moe_pick_config(int T, int H, int I, int E, int k, int num_sms, bool one_launch)
{
    MoeConfig c;
    c.bn = pick_bn(T);
    c.kc = (c.bn <= 128) ? 256 : 128;
    c.fused = 0;
    c.a8 = moe_unpack_once(T) ? 1 : 0;
    if (one_launch && c.kc == 256) {
        c.fused = 1;
        c.ksplit = fused_ksplit(T, H, I, E, k, c.bn, c.kc, num_sms);
        c.streamk = 0;
        c.nslots = 0;
        return c;
    }
    // Split the down projection's K so that its tiles fill the SMs: the cost
    // of a split d is waves(d) * (stages per tile + a fixed per-tile cost of
    // about one stage: the accumulator hand-off and the epilogue tail).
    const int kblocks = (I + c.kc - 1) / c.kc;
    const int base_tiles = E * (H / 128);
    const int kmax = moe_ksplit_max(T, k);
    int best = 1;
    double best_cost = 0.0;
    for (int d = 1; d <= kmax; ++d) {
        if (kblocks % d != 0 || kblocks / d < 2)
            continue;
        const int64_t tiles = static_cast<int64_t>(base_tiles) * d;
        const int64_t waves = (tiles + num_sms - 1) / num_sms;
        const double cost = static_cast<double>(waves) * (static_cast<double>(kblocks / d) + 1.0);
        if (d == 1 || cost < best_cost) {
            best_cost = cost;
            best = d;
        }
    }
    c.ksplit = best;
    // With at most E assignments (T*k <= E) most experts may be idle, and the
    // split above (chosen for E active experts) would leave SMs without work:
    // the down GEMM then runs stream-K, equal K-block ranges per CTA over the
    // tiles that exist, at most `nslots` segments per tile. (Measured: with
    // every expert active it is no faster than the split.) The slot bound
    // takes the fewest active experts (k): a CTA's range is then
    // S/G >= k * (H/128) * K-blocks / G stages.
    c.streamk = 0;
    c.nslots = 0;
    if (T <= 128 && static_cast<int64_t>(T) * k <= E) {
        const int rt = H / 128;
        const int need = (num_sms + k * rt - 1) / (k * rt) + 2;
        // every CTA range must be non-empty (then the CTA boundaries are
        // distinct and a tile's segments take consecutive slots)
        const bool ranges_nonempty = static_cast<int64_t>(k) * rt * kblocks >= num_sms;
        if (need <= kmax && ranges_nonempty) {
            c.streamk = 1;
            c.nslots = need;
        }
    }
    return c;
}

template <int MODE, int BN, int KC, int NW, int NX, int NXT, int NCONV, int NISS, int NB = NX, int NEPI = 4>
static int launch_gemm(const CUtensorMap& tw, const CUtensorMap& tb, const CUtensorMap& tw2, const CUtensorMap& tb2,
                       const MoeGemmParams& prm, int grid, cudaStream_t s)
{
    using Tr = MoeTraits<MODE, BN, KC, NW, NX, NXT, NCONV, NISS, NB, NEPI>;
    auto kern = moe_gemm_kernel<MODE, BN, KC, NW, NX, NXT, NCONV, NISS, NB, NEPI>;
    // attribute set on every launch: cheap, and correct for every device
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmem) != cudaSuccess)
        return kErrLaunch;
    return launch_dependent(kern, dim3(grid), dim3(Tr::kThreads), Tr::kSmem, s, tw, tb, tw2, tb2, prm) == cudaSuccess
               ? kOK
               : kErrLaunch;
}

// Token tile -> pipeline shape. Up to 128 tokens (decode) the weights are
// unpacked inside the GEMM into tensor memory, which leaves shared memory to a
// deep TMA ring: A and the activation tile share one ring of K = 256 stages.
// Above (prefill) each weight tile meets many token tiles: the weights are
// unpacked once per call by moe_upcast_kernel and the GEMM runs 256-token
// tiles (two fp32 accumulators of 256 columns fill the 512 TMEM columns) with
// A and the activations both loaded by TMA into shared memory, 128-wide
// stages, 4 deep, and eight epilogue warps. (Measured on the Grok-1 prefill
// layer: with the unpack inside the GEMM, each weight tile was unpacked again
// for every token tile -- about 43 times at 192-token tiles -- and the
// converter and gated-epilogue warps, not the tensor pipe, set the pace.)
// MODE 3 (both projections in one launch) exists for the decode shapes only.
template <int MODE>
static int dispatch_gemm(const MoeConfig& cfg, const CUtensorMap& tw, const CUtensorMap& tb, const CUtensorMap& tw2,
                         const CUtensorMap& tb2, const MoeGemmParams& prm, int grid, cudaStream_t s)
{
    switch (cfg.bn) {
    case 32: return launch_gemm<MODE, 32, 256, 10, 6, 6, 8, 2>(tw, tb, tw2, tb2, prm, grid, s);
    case 64: return launch_gemm<MODE, 64, 256, 8, 4, 4, 8, 2>(tw, tb, tw2, tb2, prm, grid, s);
    case 128: return launch_gemm<MODE, 128, 256, 4, 4, 4, 8, 1>(tw, tb, tw2, tb2, prm, grid, s);
    default:
        if constexpr (MODE == 3)
            return kErrLaunch;
        else
            return launch_gemm<MODE, 256, 128, 0, 4, 0, 0, 1, 4, 8>(tw, tb, tw2, tb2, prm, grid, s);
    }
}

int launch_moe_forward(const MoeLaunch& L, const MoeConfig& cfg, int num_sms, cudaStream_t s)
{
    const int A = L.T * L.k;
    const int BN = cfg.bn, KC = cfg.kc;
    const bool a8 = cfg.a8 != 0;
    // prefill: the weights of the experts with tokens, unpacked once
    if (a8 && launch_dependent(moe_upcast_kernel, dim3(static_cast<unsigned>(num_sms * 8)), dim3(256), 0, s,
                               L.w_gu, L.w_d, L.E, L.H, L.I, L.counts, L.wq8, L.wq8 + static_cast<int64_t>(L.E) * 2 *
                                                                                        L.I * L.H) != cudaSuccess)
        return kErrLaunch;
    // activations: gather (+ exact per-token sums for the in-GEMM unpack)
    const bool fused = cfg.fused && !L.dynamic;
    if (launch_dependent(moe_gather_kernel, dim3(A), dim3(128), 0, s, L.xq, L.H, L.k, L.sorted_ids, A, L.xp,
                         L.s0x, L.s0h, L.dynamic ? L.hmax : nullptr, fused ? L.done : nullptr, L.E,
                         a8 ? 0 : 1, (a8 && !fused) ? L.sync : nullptr) != cudaSuccess)
        return kErrLaunch;

    // weight boxes: 64-byte rows (64-byte swizzle) for KC = 128, else 128-byte rows
    const CUtensorMapSwizzle wsw = (KC == 128) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const uint32_t wbox = (KC == 128) ? 64u : 128u;
    CUtensorMap tw_gu, tb_gu, tw_d, tb_d;
    const uint8_t* wq8_d = a8 ? L.wq8 + static_cast<int64_t>(L.E) * 2 * L.I * L.H : nullptr;
    if (a8) {
        // unpacked weights: rows of E4M3 bytes, 128 x 128 boxes, 128-byte swizzle
        if (!encode_map_2d(&tw_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.wq8, L.H, static_cast<uint64_t>(L.E) * 2 * L.I,
                           L.H, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map_2d(&tw_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq8_d, L.I, static_cast<uint64_t>(L.E) * L.H, L.I,
                           128, 128, CU_TENSOR_MAP_SWIZZLE_128B))
            return kErrLaunch;
    } else if (!encode_map_2d(&tw_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.w_gu, L.H / 2,
                              static_cast<uint64_t>(L.E) * 2 * L.I, L.H / 2, wbox, 64, wsw) ||
               !encode_map_2d(&tw_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.w_d, L.I / 2,
                              static_cast<uint64_t>(L.E) * L.H, L.I / 2, wbox, 128, wsw)) {
        return kErrLaunch;
    }
    if (
!encode_map_2d(&tb_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.xp, L.H, A, L.H, 128, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&tb_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.hq, L.I, A, L.I, 128, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return kErrLaunch;

    const int64_t tok_tiles_max = (A + BN - 1) / BN + L.E;
    MoeGemmParams g{};
    g.counts = L.counts;
    g.offsets = L.offsets;
    g.E = L.E;
    g.I = L.I;
    g.H = L.H;
    g.A = A;
    g.s_gu = L.s_gu;
    g.a1 = L.a1;
    g.a2 = L.a2;
    g.act = L.act;
    g.s0x = L.s0x;
    g.hq = L.hq;
    g.s0h = L.s0h;
    g.ypart = L.ypart;
    g.done = L.done;
    g.claim = L.claim;
    g.err = L.err;

    auto mark = [&](int i) {
        if (L.events[i])
            cudaEventRecord(static_cast<cudaEvent_t>(L.events[i]), s);
    };
    if (fused) {
        // one launch: the gate_up tiles, then the down tiles (K split cfg.ksplit ways)
        MoeGemmParams f = g;
        f.rows_per_expert = 2 * L.I;
        f.rt_count = L.I / 64;
        f.kblocks = (L.H + KC - 1) / KC;
        f.ksplit = 1;
        f.rows_per_expert2 = L.H;
        f.rt_count2 = L.H / 128;
        f.ksplit2 = cfg.ksplit;
        f.kblocks2 = (L.I + KC - 1) / KC / cfg.ksplit;
        const int64_t tiles = static_cast<int64_t>(f.rt_count + f.rt_count2 * cfg.ksplit) * tok_tiles_max;
        const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
        mark(0);
        const int st = dispatch_gemm<3>(cfg, tw_gu, tb_gu, tw_d, tb_d, f, grid, s);
        if (st != kOK)
            return st;
        mark(1);
        mark(2);
    } else {
    // gate_up: 64 gated pairs (128 weight rows) per tile, full K = H
    mark(0);
    MoeGemmParams gu = g;
    gu.dynamic = L.dynamic;
    gu.hf = L.hf;
    gu.hmax = L.hmax;
    gu.rows_per_expert = 2 * L.I;
    gu.rt_count = L.I / 64;
    gu.kblocks = (L.H + KC - 1) / KC;
    gu.ksplit = 1;
    gu.band = a8 ? kPrefillBand : 0;
    int64_t tiles = static_cast<int64_t>(gu.rt_count) * tok_tiles_max;
    int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    int st = L.dynamic ? dispatch_gemm<2>(cfg, tw_gu, tb_gu, tw_gu, tb_gu, gu, grid, s)
                       : dispatch_gemm<0>(cfg, tw_gu, tb_gu, tw_gu, tb_gu, gu, grid, s);
    if (st != kOK)
        return st;
    if (L.dynamic &&
        launch_dependent(moe_hquant_kernel, dim3(A), dim3(256), 0, s, static_cast<const float*>(L.hf), L.I,
                         static_cast<const unsigned int*>(L.hmax), L.a2_out, L.hq, L.s0h) != cudaSuccess)
        return kErrLaunch;
    mark(1);

    // down: 128 output rows per tile, K = I split ksplit ways
    MoeGemmParams dn = g;
    dn.rows_per_expert = L.H;
    dn.rt_count = L.H / 128;
    dn.ksplit = cfg.streamk ? 1 : cfg.ksplit;
    dn.kblocks = (L.I + KC - 1) / KC / dn.ksplit;
    dn.streamk = cfg.streamk;
    dn.nslots = cfg.nslots;
    dn.band = a8 ? kPrefillBand : 0;
    dn.sync = a8 ? L.sync : nullptr;
    tiles = static_cast<int64_t>(dn.rt_count) * tok_tiles_max * dn.ksplit;
    grid = cfg.streamk ? num_sms : static_cast<int>(tiles < num_sms ? tiles : num_sms);
    st = dispatch_gemm<1>(cfg, tw_d, tb_d, tw_d, tb_d, dn, grid, s);
    if (st != kOK)
        return st;
    mark(2);
    }

    const int64_t nthreads = static_cast<int64_t>(L.T) * (L.H / 4);
    // the register array of split partials is sized for the split in use
    const int parts = (cfg.streamk && !fused) ? cfg.nslots : cfg.ksplit;
    auto fin = L.k <= 2 ? (parts == 1 ? moe_finalize_kernel<1, 2>
                           : parts <= 4 ? moe_finalize_kernel<4, 2>
                           : parts <= 8 ? moe_finalize_kernel<8, 2> : moe_finalize_kernel<kMaxKsplit, 2>)
                        : (parts == 1 ? moe_finalize_kernel<1, 8>
                           : parts <= 4 ? moe_finalize_kernel<4, 8>
                           : parts <= 8 ? moe_finalize_kernel<8, 8> : moe_finalize_kernel<kMaxKsplit, 8>);
    if (launch_dependent(fin, dim3(static_cast<unsigned>((nthreads + 255) / 256)), dim3(256), 0, s,
                         L.T, L.H, L.k, A, parts, L.ids, L.topk_w, L.inv, L.ypart,
                         // weights unpacked ahead carry signed values: no shift
                         a8 ? nullptr : static_cast<const unsigned long long*>(L.s0h), a8 ? 1.0f : 512.0f, L.s_d,
                         L.dynamic ? static_cast<const float*>(L.a2_out) : L.a2, L.out) != cudaSuccess)
        return kErrLaunch;
    mark(3);
    return kOK;
}

}  // namespace w4a8
