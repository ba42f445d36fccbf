// Work schedules of the persistent GEMM kernels (device code).
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace w4a8 {

// The CTA's work as a sequence of segments (tile t, first K-block kb0, nkb
// K-blocks, partial slot). Round robin: tiles blockIdx.x, +gridDim.x, ...,
// whole (slot = K split). Stream-K (down GEMM of decode-sized layers): the
// K-blocks of all tiles form one sequence of S stages and CTA c takes
// [c*S/G, (c+1)*S/G), so every CTA streams the same number of weight bytes; a
// tile cut by CTA boundaries yields one segment per CTA, and a segment's slot
// is the number of boundaries before it inside its tile.
// A round-robin list may hold two kinds of tiles: [0, n1) with kbt K-blocks
// each, then [n1, total) with kbt2 each (gate_up and down in one launch).
struct WorkIter {
    int t, kb0, nkb, slot;
    bool last;            // the segment ends its tile
    int total, kbt, stride;
    int n1, kbt2;
    bool sk;
    int64_t s, s_end, S, G;
    __device__ __forceinline__ int64_t owner(int64_t x) const { return ((x + 1) * G - 1) / S; }
    __device__ __forceinline__ void load()
    {
        if (sk) {
            if (s >= s_end) {
                t = total;
                return;
            }
            t = static_cast<int>(s / kbt);
            kb0 = static_cast<int>(s - static_cast<int64_t>(t) * kbt);
            const int64_t left = s_end - s;
            nkb = static_cast<int>(left < kbt - kb0 ? left : kbt - kb0);
            slot = static_cast<int>(owner(s) - owner(static_cast<int64_t>(t) * kbt));
            last = (kb0 + nkb == kbt);
        }
    }
    __device__ __forceinline__ void init(int total_, int kbt_, bool streamk, int n1_ = -1, int kbt2_ = 0)
    {
        total = total_;
        kbt = kbt_;
        n1 = n1_ < 0 ? total_ : n1_;
        kbt2 = kbt2_;
        sk = streamk;
        stride = gridDim.x;
        if (sk) {
            S = static_cast<int64_t>(total) * kbt;
            G = gridDim.x;
            s = S * blockIdx.x / G;
            s_end = S * (blockIdx.x + 1) / G;
            load();
        } else {
            t = blockIdx.x;
            kb0 = 0;
            nkb = t < n1 ? kbt : kbt2;
            slot = 0;
            last = true;
        }
    }
    __device__ __forceinline__ bool valid() const { return t < total; }
    __device__ __forceinline__ void next()
    {
        if (sk) {
            s += nkb;
            load();
        } else {
            t += stride;
            nkb = t < n1 ? kbt : kbt2;
        }
    }
};

// The tile sequence of one role of a persistent GEMM CTA.
//   static:  the schedule of WorkIter (round robin or stream-K).
//   dynamic: the weight producer takes the tiles [0, n_static) round robin
//            and then claims tiles from a grid-wide counter (one atomicAdd per
//            tile), and publishes them, in that order, through a
//            shared-memory queue of kTileQ entries that every other role of
//            the CTA reads. A CTA still meets its tiles in increasing list
//            order. The round-robin part keeps the CTAs streaming neighbouring
//            weight tiles at the same time (measured faster than claiming
//            throughout); the claimed tail lets a faster SM take more of the
//            last tiles, so the CTAs finish within about one tile of each other.
constexpr int kTileQ = 8;

struct TileSeq {
    WorkIter wi;
    bool dyn;
    int role;                 // dynamic: 0 claims and publishes, 1 reads (one thread), 2 reads (a whole warp)
    int* claim;
    volatile int* q;
    uint32_t full0, free0;    // shared addresses of the queue's full[0] and free[0] mbarriers
    const volatile int* abort;
    int qi;
    uint32_t qph;
    int pending;              // role 0: the claim for the next tile, taken ahead (see claim_next)
    int next_static, n_static;
    int t, kb0, nkb, slot;
    bool last, ok;
    int total, n1, kbt, kbt2;

    __device__ __forceinline__ void copy()
    {
        t = wi.t;
        kb0 = wi.kb0;
        nkb = wi.nkb;
        slot = wi.slot;
        last = wi.last;
    }
    __device__ __forceinline__ void init_static(int total_, int kbt_, bool streamk, int n1_, int kbt2_)
    {
        dyn = false;
        ok = true;
        total = total_;
        wi.init(total_, kbt_, streamk, n1_, kbt2_);
        copy();
    }
    __device__ __forceinline__ void init_dynamic(int role_, int* claim_, volatile int* q_, uint32_t full0_,
                                                 uint32_t free0_, const volatile int* abort_, int total_, int n1_,
                                                 int kbt_, int kbt2_, int n_static_)
    {
        dyn = true;
        role = role_;
        claim = claim_;
        q = q_;
        full0 = full0_;
        free0 = free0_;
        abort = abort_;
        total = total_;
        n1 = n1_;
        kbt = kbt_;
        kbt2 = kbt2_;
        qi = 0;
        qph = 0;
        kb0 = 0;
        slot = 0;
        last = true;
        ok = true;
        n_static = n_static_;
        next_static = blockIdx.x;
        pending = 0;
        if (role == 0)
            claim_next();
        step();
    }
    // Role 0 takes the claim for its next tile (once the round-robin part is
    // used up) a few stages before the current tile is fully issued, so the
    // atomic's round trip does not stall the weight stream at the tile
    // boundary (the result is first used in step()).
    __device__ __forceinline__ void claim_next()
    {
        if (next_static >= n_static)
            pending = atomicAdd(claim, 1);
    }
    // the stage of the current tile at which role 0 takes its next claim
    __device__ __forceinline__ bool claim_here(int kb, int ahead) const
    {
        const int at = kb0 + nkb - ahead;
        return dyn && role == 0 && kb == (at > kb0 ? at : kb0);
    }
    __device__ __forceinline__ void step()
    {
        const uint32_t fb = full0 + 8u * static_cast<uint32_t>(qi);
        const uint32_t eb = free0 + 8u * static_cast<uint32_t>(qi);
        if (role == 0) {
            int c;
            if (next_static < n_static) {
                c = next_static;
                next_static += static_cast<int>(gridDim.x);
            } else {
                c = n_static + pending;
            }
            if (!mbar_wait_or_abort(eb, qph ^ 1u, abort)) {
                ok = false;
                t = total;
                return;
            }
            t = c < total ? c : total;   // total: the end of the sequence
            q[qi] = t;
            mbar_arrive(fb);
        } else {
            if (!mbar_wait_or_abort(fb, qph, abort)) {
                ok = false;
                t = total;
                return;
            }
            t = q[qi];
            if (role == 2)
                __syncwarp();
            if (role == 1 || (threadIdx.x & 31) == 0)
                mbar_arrive(eb);
        }
        nkb = t < n1 ? kbt : kbt2;
        if (++qi == kTileQ) {
            qi = 0;
            qph ^= 1u;
        }
    }
    __device__ __forceinline__ bool valid() const { return t < total; }
    __device__ __forceinline__ void next()
    {
        if (dyn) {
            step();
        } else {
            wi.next();
            copy();
        }
    }
};

// Segments of tile t under the stream-K schedule of `S` stages over `G` CTAs
// (the number of CTA ranges that intersect the tile's stages).
__device__ __forceinline__ int streamk_segments(int64_t t, int kbt, int64_t S, int64_t G)
{
    const int64_t first = t * kbt, last = first + kbt - 1;
    return static_cast<int>(((last + 1) * G - 1) / S - ((first + 1) * G - 1) / S) + 1;
}

}  // namespace w4a8
