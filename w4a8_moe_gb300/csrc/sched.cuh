// Work schedules of the persistent GEMM kernels (device code).
#pragma once

#include <stdint.h>

namespace w4a8 {

// The CTA's work as a sequence of segments (tile t, first K-block kb0, nkb
// K-blocks, partial slot). Round robin: tiles blockIdx.x, +gridDim.x, ...,
// whole (slot = K split). Stream-K (down GEMM of decode-sized layers): the
// K-blocks of all tiles form one sequence of S stages and CTA c takes
// [c*S/G, (c+1)*S/G), so every CTA streams the same number of weight bytes; a
// tile cut by CTA boundaries yields one segment per CTA, and a segment's slot
// is the number of boundaries before it inside its tile.
struct WorkIter {
    int t, kb0, nkb, slot;
    bool last;            // the segment ends its tile
    int total, kbt, stride;
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
    __device__ __forceinline__ void init(int total_, int kbt_, bool streamk)
    {
        total = total_;
        kbt = kbt_;
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
            nkb = kbt;
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
