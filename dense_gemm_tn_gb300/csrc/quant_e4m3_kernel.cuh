// quant_e4m3_kernel.cuh -- per-tensor E4M3 quantisation with the amax taken
// on the device: the step that turns an FP32 / FP16 / BF16 operand into the
// E4M3 codes and the dequantisation scale the FP8 GEMM consumes.
//
// The ROCm blog "FP16 GEMM optimization on AMD RDNA 3 and RDNA 4" closes
// ("Where we are") by announcing an FP8 port; the pages give no quantisation
// rule.  This kernel uses the plain per-tensor one:
//     amax = max_i |x_i|                    (exact: a maximum of stored values)
//     s_q  = 448 / amax                     (fp32, round to nearest even)
//     q_i  = e4m3(x_i * s_q)                (fp32 product; RNE, saturating to +-448)
//     scale = amax / 448                    (fp32; the GEMM multiplies by it)
// with s_q = 0 when amax = 0 and s_q = FLT_MAX when 448 / amax overflows.
//
// Two kernels, back to back on the caller's stream; both are bound by HBM.
// Their CTAs split the tensor into the same contiguous ranges of row segments
// ("units": one 16-byte chunk of x per thread).  The first takes the maximum
// of |x| over each range -- on the bit patterns, which for finite values
// order like the magnitudes -- and leaves it in a per-CTA slot.  The second is
// launched as a programmatic dependent of the first (its CTAs may be scheduled
// while the first drains; they wait in hardware for the first grid to
// complete and its writes to be visible), reads every slot, and quantises its
// range walking the units in the opposite order, so that what the first
// kernel read last -- still in L2 -- is read again first.  Each thread keeps
// kUnroll 16-byte loads in flight.  Neither kernel waits on another CTA.
#pragma once

#include <cfloat>
#include <cstdint>

namespace qz {

constexpr int kThreads = 256;
constexpr int kChunk = 16;                // bytes of x per thread and unit
constexpr int kUnroll = 4;                // units in flight per thread
constexpr int kMinBlocks = 4;             // CTAs per SM the register budget allows

// Input element types (the x_type values of gemm_quantize_e4m3).
constexpr int kInF32 = 0;
constexpr int kInF16 = 1;
constexpr int kInBF16 = 2;

__host__ __device__ constexpr int elem_bytes(int in) { return in == kInF32 ? 4 : 2; }
// Elements of one unit: kThreads chunks of 16 bytes.
__host__ __device__ constexpr int64_t unit_elems(int in) { return int64_t(kThreads) * (kChunk / elem_bytes(in)); }

struct QuantParams {
    const void *x;            // rows x cols, row stride ldx elements
    uint8_t *q;               // rows x cols E4M3 codes, row stride ldq bytes
    float *scale_out;         // amax / 448
    float *slots;             // one per CTA: the maximum of |x| over its units
    int64_t ldx, ldq, rows, cols;
    int64_t units_per_row, num_units;
    int vec;                  // rows of x start 16-byte aligned and rows of q 8-byte aligned
};

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h)
{
    float f;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "r"(h));
    return f;
}

// Two E4M3 codes, `lo` in the low byte (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// L2 eviction policies for the loads of x: the part of a CTA's range that the
// quantising pass reads first is kept (evict_last) by the maximum-finding
// pass; everything else, and every load of the quantising pass (its data is
// dead afterwards), goes first (evict_first).
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t policy)
{
    uint4 v;
    asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(policy));
    return v;
}

// Per input type: the running maximum of |x| kept on bit patterns (for 16-bit
// types two halfword maxima in one word), and the decode to fp32.
template <int kIn>
struct In;

template <>
struct In<kInF32> {
    static constexpr int kVec = 4;
    __device__ static uint32_t acc_chunk(uint32_t m, const uint4 &w)
    {
        m = max(m, w.x & 0x7FFFFFFFu);
        m = max(m, w.y & 0x7FFFFFFFu);
        m = max(m, w.z & 0x7FFFFFFFu);
        return max(m, w.w & 0x7FFFFFFFu);
    }
    __device__ static uint32_t bits(const void *row, int64_t c) { return static_cast<const uint32_t *>(row)[c]; }
    __device__ static uint32_t acc_one(uint32_t m, uint32_t b) { return max(m, b & 0x7FFFFFFFu); }
    __device__ static float amax(uint32_t m) { return __uint_as_float(m); }
    __device__ static float decode(uint32_t b) { return __uint_as_float(b); }
};

template <int kIn>
struct In16 {
    static constexpr int kVec = 8;
    __device__ static uint32_t acc_chunk(uint32_t m, const uint4 &w)
    {
        m = __vmaxu2(m, w.x & 0x7FFF7FFFu);
        m = __vmaxu2(m, w.y & 0x7FFF7FFFu);
        m = __vmaxu2(m, w.z & 0x7FFF7FFFu);
        return __vmaxu2(m, w.w & 0x7FFF7FFFu);
    }
    __device__ static uint32_t bits(const void *row, int64_t c) { return static_cast<const uint16_t *>(row)[c]; }
    __device__ static uint32_t acc_one(uint32_t m, uint32_t b) { return __vmaxu2(m, b & 0x7FFFu); }
    __device__ static float decode(uint32_t b)
    {
        return kIn == kInF16 ? f16_bits_to_f32(b) : __uint_as_float(b << 16);
    }
    __device__ static float amax(uint32_t m) { return decode(max(m & 0xFFFFu, m >> 16)); }
};

template <>
struct In<kInF16> : In16<kInF16> {};
template <>
struct In<kInBF16> : In16<kInBF16> {};

// Position of a unit: row r, segment seg of that row.  Consecutive units of a
// CTA's range are visited by stepping, so there is one division per CTA.
struct UnitPos {
    int64_t r, seg;
};

__device__ __forceinline__ UnitPos unit_pos(const QuantParams &p, int64_t u)
{
    const int64_t r = u / p.units_per_row;
    return {r, u - r * p.units_per_row};
}

__device__ __forceinline__ void step_fwd(UnitPos &s, int64_t upr)
{
    if (++s.seg == upr) {
        s.seg = 0;
        ++s.r;
    }
}

__device__ __forceinline__ void step_back(UnitPos &s, int64_t upr)
{
    if (s.seg-- == 0) {
        s.seg = upr - 1;
        --s.r;
    }
}

// This CTA's range of units (the same in both kernels).
__device__ __forceinline__ void unit_range(const QuantParams &p, int64_t &ub, int64_t &ue)
{
    ub = int64_t(blockIdx.x) * p.num_units / gridDim.x;
    ue = int64_t(blockIdx.x + 1) * p.num_units / gridDim.x;
}

__device__ __forceinline__ float block_max(float m, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();                      // red[] may still be read by an earlier call
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = lane < kThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

template <int kIn>
__global__ void __launch_bounds__(kThreads, kMinBlocks) quant_amax_kernel(const __grid_constant__ QuantParams p)
{
    using T = In<kIn>;
    constexpr int kB = elem_bytes(kIn);
    __shared__ float red[kThreads / 32];
    // Launched as a programmatic dependent of the previous kernel on the
    // stream (which may still read the slot array, or write x): nothing below
    // touches global memory before that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int64_t ub, ue;
    unit_range(p, ub, ue);
    const int64_t unit = unit_elems(kIn);
    const int64_t c0 = int64_t(threadIdx.x) * T::kVec;
    const uint8_t *x = static_cast<const uint8_t *>(p.x);
    uint32_t acc = 0;
    UnitPos pos = unit_pos(p, ub);
    const int64_t keep_from = ub + (ue - ub) / 2;          // the second half is read again first
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    for (int64_t u = ub; u < ue; u += kUnroll) {
        uint4 raw[kUnroll];
        bool loaded[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            loaded[k] = false;
            if (u + k < ue) {
                const int64_t c = pos.seg * unit + c0;
                const uint8_t *row = x + pos.r * p.ldx * kB;
                if (p.vec && c + T::kVec <= p.cols) {
                    raw[k] = ld_stream_v4(row + c * kB, u + k >= keep_from ? pol_last : pol_first);
                    loaded[k] = true;
                } else {
                    for (int j = 0; j < T::kVec; ++j)
                        if (c + j < p.cols) acc = T::acc_one(acc, T::bits(row, c + j));
                }
                step_fwd(pos, p.units_per_row);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
            if (loaded[k]) acc = T::acc_chunk(acc, raw[k]);
    }
    const float m = block_max(T::amax(acc), red);
    if (threadIdx.x == 0) p.slots[blockIdx.x] = m;
    // Every CTA is done with its slot: the quantising grid may be scheduled.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Codes of one 16-byte chunk (8 or 4 elements) packed little-endian.
template <int kIn>
__device__ __forceinline__ uint2 codes_of(const uint4 &w, float s_q)
{
    using T = In<kIn>;
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    if constexpr (T::kVec == 8) {
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            c[j] = e4m3x2(__fmul_rn(T::decode(v[j] & 0xFFFFu), s_q), __fmul_rn(T::decode(v[j] >> 16), s_q));
        return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    } else {
        const uint32_t lo = e4m3x2(__fmul_rn(T::decode(v[0]), s_q), __fmul_rn(T::decode(v[1]), s_q));
        const uint32_t hi = e4m3x2(__fmul_rn(T::decode(v[2]), s_q), __fmul_rn(T::decode(v[3]), s_q));
        return make_uint2(lo | (hi << 16), 0u);
    }
}

template <int kIn>
__global__ void __launch_bounds__(kThreads, kMinBlocks) quant_store_kernel(const __grid_constant__ QuantParams p)
{
    using T = In<kIn>;
    constexpr int kB = elem_bytes(kIn);
    __shared__ float red[kThreads / 32];
    // Returns once the maximum-finding grid has completed and its slots are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float amax = 0.0f;
    for (unsigned b = threadIdx.x; b < gridDim.x; b += kThreads) amax = fmaxf(amax, p.slots[b]);
    amax = block_max(amax, red);

    float s_q = 0.0f;
    if (amax > 0.0f) {
        s_q = 448.0f / amax;
        if (s_q > FLT_MAX) s_q = FLT_MAX;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.scale_out = amax / 448.0f;

    int64_t ub, ue;
    unit_range(p, ub, ue);
    if (ue <= ub) return;
    const int64_t unit = unit_elems(kIn);
    const int64_t c0 = int64_t(threadIdx.x) * T::kVec;
    const uint8_t *x = static_cast<const uint8_t *>(p.x);
    const uint64_t pol_first = policy_evict_first();
    UnitPos pos = unit_pos(p, ue - 1);
    for (int64_t u = ue - 1; u >= ub; u -= kUnroll) {      // last unit first
        uint4 raw[kUnroll];
        uint8_t *dst[kUnroll];
        bool loaded[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            loaded[k] = false;
            dst[k] = nullptr;
            if (u - k >= ub) {
                const int64_t c = pos.seg * unit + c0;
                const uint8_t *row = x + pos.r * p.ldx * kB;
                uint8_t *qrow = p.q + pos.r * p.ldq;
                if (p.vec && c + T::kVec <= p.cols) {
                    raw[k] = ld_stream_v4(row + c * kB, pol_first);
                    dst[k] = qrow + c;
                    loaded[k] = true;
                } else {
                    for (int j = 0; j < T::kVec; ++j)
                        if (c + j < p.cols)
                            qrow[c + j] = static_cast<uint8_t>(
                                e4m3x2(__fmul_rn(T::decode(T::bits(row, c + j)), s_q), 0.0f) & 0xFFu);
                }
                step_back(pos, p.units_per_row);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            if (!loaded[k]) continue;
            const uint2 cw = codes_of<kIn>(raw[k], s_q);
            if constexpr (T::kVec == 8)
                *reinterpret_cast<uint2 *>(dst[k]) = cw;
            else
                *reinterpret_cast<uint32_t *>(dst[k]) = cw.x;
        }
    }
}

}  // namespace qz
