// Copy of operand rows that the TMA cannot address in place (a base, row
// stride or row length that is not a multiple of 16 bytes) into a workspace
// whose rows start on 128-byte boundaries, zero-padded to the new stride.
// This is what lets tiles run over any M, N, K and leading dimensions: the
// hello-gpu ch.11 section 11.4 boundary handling and the ROCm blog's Step 4
// (tiles that need not divide the matrix), under TMA's alignment rules.
#pragma once

#include <cstdint>

namespace tn {

template <typename T>
struct RepackJob {
    const T *src;
    int64_t ld_src;
    T *dst;
    int64_t ld_dst;
    int64_t rows, K;
};

// Bytes [s, s + 16) of the 32-byte window w[0..7] (little-endian words),
// for a window offset of 4q + sh/8 bytes.
template <int q>
__device__ __forceinline__ uint4 window16(const uint32_t (&w)[8], uint32_t sh)
{
    return make_uint4(__funnelshift_r(w[q], w[q + 1], sh), __funnelshift_r(w[q + 1], w[q + 2], sh),
                      __funnelshift_r(w[q + 2], w[q + 3], sh), __funnelshift_r(w[q + 3], w[q + 4], sh));
}

constexpr int kRepackWarps = 8;        // warps per CTA
constexpr int kRepackUnroll = 4;       // 16-byte chunks per lane in flight
constexpr int kRepackSeg = 32 * kRepackUnroll;   // chunks of one warp's segment of a row

// Both operands in one launch: rows 0 .. j0.rows-1 come from job 0, the rest
// from job 1 (which may have no rows); the two share ld_dst.  Each warp copies
// one segment of kRepackSeg 16-byte destination chunks of one row.  A source
// row starts wherever its elements do, so a chunk is cut out of two aligned
// 16-byte loads (the row's offset from 16-byte alignment is one value for the
// whole warp); chunks whose aligned loads would leave the row's K elements
// (its first and last ones, and the zero padding) are gathered element by
// element instead, so no load touches a byte outside the source rows.
template <typename T>
__global__ void __launch_bounds__(kRepackWarps * 32) repack_rows_kernel(const RepackJob<T> j0, const RepackJob<T> j1,
                                                                        int64_t segs_per_row)
{
    constexpr int kVec = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kRepackWarps + (threadIdx.x >> 5);
    int64_t r = unit / segs_per_row;
    const int64_t c0 = (unit - r * segs_per_row) * kRepackSeg;
    const bool second = r >= j0.rows;
    const RepackJob<T> &j = second ? j1 : j0;
    if (second) r -= j0.rows;
    if (r >= j.rows) return;
    const T *src = j.src + r * j.ld_src;
    uint4 *dst = reinterpret_cast<uint4 *>(j.dst + r * j.ld_dst);
    const int64_t chunks = j.ld_dst / kVec;
    const int64_t kbytes = j.K * static_cast<int64_t>(sizeof(T));
    const uint32_t s = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
    const uint4 *aligned = reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(src) - s);
    uint4 lo[kRepackUnroll], hi[kRepackUnroll];
    bool vec[kRepackUnroll];
#pragma unroll
    for (int u = 0; u < kRepackUnroll; ++u) {
        const int64_t c = c0 + 32 * u + lane;
        // aligned loads cover bytes [16c - s, 16c - s + (s ? 32 : 16)) of the row
        vec[u] = c < chunks && (s == 0 ? 16 * (c + 1) <= kbytes : c >= 1 && 16 * c + 32 - s <= kbytes);
        if (vec[u]) {
            lo[u] = __ldcs(aligned + c);
            if (s != 0) hi[u] = __ldcs(aligned + c + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < kRepackUnroll; ++u) {
        const int64_t c = c0 + 32 * u + lane;
        if (c >= chunks) continue;
        uint4 out;
        if (vec[u]) {
            if (s == 0) {
                out = lo[u];
            } else {
                const uint32_t w[8] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w, hi[u].x, hi[u].y, hi[u].z, hi[u].w};
                const uint32_t sh = 8u * (s & 3u);
                switch (s >> 2) {   // one value per warp
                case 0: out = window16<0>(w, sh); break;
                case 1: out = window16<1>(w, sh); break;
                case 2: out = window16<2>(w, sh); break;
                default: out = window16<3>(w, sh); break;
                }
            }
        } else {
            union {
                T v[kVec];
                uint4 u4;
            } chunk;
#pragma unroll
            for (int i = 0; i < kVec; ++i) chunk.v[i] = c * kVec + i < j.K ? src[c * kVec + i] : T(0);
            out = chunk.u4;
        }
        dst[c] = out;
    }
}

}  // namespace tn
