// Inline-PTX building blocks for sm_103a: mbarriers, TMA tile loads, tcgen05
// (TMEM allocation, FP8 MMA, commit, loads) and E4M3 conversion.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace w4a8 {

// Upper bound on any single wait for an mbarrier phase (~2 s at 2 GHz). A wait
// that runs out records an error word and makes the kernel unwind.
constexpr long long kWaitBudgetCycles = 4000000000LL;
constexpr uint32_t kWaitMaxPolls = 1u << 30;

// Error bits written to the device error word.
constexpr uint32_t kErrBitTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// HINT: suspend-time hint of a polling wait, in nanoseconds (0: none). With a
// hint a thread whose phase is incomplete sleeps until the phase completes or
// the hint runs out instead of re-issuing its test at once, which leaves the
// issue slots to the warps with work (measured: the prefill GEMM, whose
// epilogue warps wait through whole tiles, runs 7 % faster; the decode GEMM,
// where every wait is short, 2.6 % slower).
template <uint32_t HINT = 0>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (HINT == 0) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(HINT)
            : "memory");
    }
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete. Returns false
// when the budget (clock64 cycles) runs out: the caller records the error and
// unwinds.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, long long budget)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < kWaitMaxPolls; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (clock64() - t0 > budget)
            break;
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, kWaitBudgetCycles);
}

// Same, but also gives up as soon as another role of the CTA has set *abort
// (checked only while spinning, so a phase that is already complete costs one
// try_wait).
template <uint32_t HINT = 0>
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, const volatile int* abort)
{
    if (mbar_try_wait<HINT>(bar, parity))
        return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < kWaitMaxPolls; ++it) {
        if (*abort)
            return false;
        if (mbar_try_wait<HINT>(bar, parity))
            return true;
        if (clock64() - t0 > kWaitBudgetCycles)
            break;
    }
    return false;
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when the kernel was
// not launched as a dependent), and allow the next kernel to start launching.
// Every kernel of this library calls grid_dep_launch only after its own
// grid_dep_wait has returned, except the block-FP8 activation quantizer, whose
// only dependent (the block-FP8 GEMM) reads nothing but the weights before its
// own wait.
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *counter >= target, where other CTAs of the same grid count up
// after writing data that this thread will then read with TMA: the acquire
// load orders the reads after those writes, and the proxy fence orders this
// thread's later async-proxy (TMA) reads after its generic-proxy view. Gives
// up like mbar_wait_or_abort (budget, or *abort set by another role).
__device__ __forceinline__ bool counter_wait_or_abort(const int* counter, int target, const volatile int* abort)
{
    bool ok = ld_acquire_gpu(counter) >= target;
    if (!ok) {
        const long long t0 = clock64();
        for (uint32_t it = 0; it < kWaitMaxPolls && !ok; ++it) {
            if (*abort || clock64() - t0 > kWaitBudgetCycles)
                break;
            __nanosleep(64);
            ok = ld_acquire_gpu(counter) >= target;
        }
    }
    if (ok)
        fence_proxy_async_global();
    return ok;
}

// Bounded wait until *passed + *done >= target (both counters only grow).
__device__ __forceinline__ bool pace_wait_or_abort(const int* passed, const int* done, int target,
                                                   const volatile int* abort)
{
    bool ok = ld_acquire_gpu(passed) + ld_acquire_gpu(done) >= target;
    if (!ok) {
        const long long t0 = clock64();
        for (uint32_t it = 0; it < kWaitMaxPolls && !ok; ++it) {
            if (*abort || clock64() - t0 > kWaitBudgetCycles)
                break;
            __nanosleep(64);
            ok = ld_acquire_gpu(passed) + ld_acquire_gpu(done) >= target;
        }
    }
    return ok;
}

// ---------------------------------------------------------------- TMA
// 2-D tile load global -> shared, completion counted on an mbarrier in bytes.
// c0 is the innermost coordinate (elements), c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
// Same, with an L2 cache-policy hint (createpolicy result).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}
// TMA store of a 2-D tile from shared memory (bulk-group completion), with an
// L2 cache-policy hint. The innermost coordinate c0 times the element size
// must be a multiple of 16 bytes and neither coordinate may be negative; rows
// and columns past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, int c0, int c1, uint32_t src,
                                                  uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
        " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(src), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until the committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Global stores carrying an L2 cache policy (from createpolicy).
__device__ __forceinline__ void st_u8_hint(uint8_t* dst, uint32_t v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.u8 [%0], %1, %2;" ::"l"(dst), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_f32_hint(float* dst, float v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both operands K-major, kind::f8f6f4.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same with the A operand in tensor memory (a_tmem: lane 0, first column of A;
// row m of A in lane m, 4 consecutive K elements of fp8 per 32-bit column).
__device__ __forceinline__ void umma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier when every tcgen05 async op issued so far by
// this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM
// lane (lane = 32 * (warp % 4) + laneid, encoded in taddr bits 31..16).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Each thread of the warp writes 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row groups 1024 bytes apart, group base
// 1024-byte aligned. The start address may be advanced by 32-byte steps along
// K inside a row (one MMA K-slice of fp8).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
    d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: 8-row group
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4: D fp32, A = B = E4M3, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4)                                    // D format: f32
           | (0u << 7) | (0u << 10)                     // A, B: e4m3
           | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// ---------------------------------------------------------------- numerics
// fp32 pair -> E4M3 pair, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float hi, float lo)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t cvt_e4m3(float v)
{
    return static_cast<uint32_t>(cvt_e4m3x2(0.0f, v)) & 0xFFu;
}
// 512 * value of an E4M3 code, as an exact integer (|.| <= 229376).
__device__ __forceinline__ int e4m3_times512(uint32_t c)
{
    const int e = (c >> 3) & 15;
    const int m = c & 7;
    const int mag = e ? ((8 + m) << (e - 1)) : m;
    return (c & 0x80u) ? -mag : mag;
}
// The same as an fp32 number: the hardware E4M3 -> f16 conversion is exact
// for every finite code, and 512 * value is an integer below 2^18, so sums of
// up to 64 of them stay exact in fp32.
__device__ __forceinline__ float e4m3_times512_f32(uint32_t c)
{
    float r;
    asm("{\n\t.reg .b32 t;\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.f16x2.e4m3x2 t, %1;\n\t"
        "mov.b32 {lo, hi}, t;\n\t"
        "cvt.f32.f16 %0, lo;\n\t}"
        : "=f"(r)
        : "h"(static_cast<uint16_t>(c & 0xFFu)));
    return r * 512.0f;
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits)
{
    if (err)
        atomicOr(err, bits);
}

}  // namespace w4a8
