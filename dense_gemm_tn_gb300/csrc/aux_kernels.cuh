// aux_kernels.cuh -- the small kernels around the GEMM: the reduce pass of
// the split-reduce mode, and the fills of the K == 0 case.
#pragma once

#include <cstdint>

#include "tn_gemm_kernel.cuh"

namespace tn {

// kSplitReduce, second launch: C[m, n] = the sum over parts, in part order,
// of the FP32 partials of (m, n) -- stored, like the GEMM epilogue, as FP16
// or as bf16(sum * scale_a * scale_b).  One thread per 8 consecutive m of one
// column n: 32-byte reads of each partial, a 16-byte store of C.  Launched as
// a programmatic dependent of the GEMM; waits for it to complete first.
template <class Kind, int kGroup, int kTileRows = kTileM>
__global__ void __launch_bounds__(256) split_reduce_kernel(const float *__restrict__ ws, int parts, int64_t tiles_n,
                                                           int32_t M, int32_t N, void *c_ptr, int64_t ldc,
                                                           float scale, const float *scale_a, const float *scale_b)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next kernel on the stream (typically the next GEMM) may start its
    // setup now; it waits for this grid to complete before touching memory.
    // It starts once every CTA of this grid has got here, so all of them are
    // resident by then.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const float s = scale_a ? __fmul_rn(__ldg(scale_a), __ldg(scale_b)) : scale;
    constexpr int64_t kRows = 128;                       // rows n of one CTA's partial
    const int64_t part_stride = static_cast<int64_t>(kGroup) * kRows * kTileRows;
    const int64_t groups_m = (M + 7) / 8;
    const bool vec_c = (ldc * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(c_ptr) % 16 == 0;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < groups_m * N;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / groups_m;
        const int64_t m = (i - n * groups_m) * 8;
        const int64_t tm = m / kTileRows, tn = n / (kRows * kGroup);
        const int64_t pos = (n / kRows) % kGroup, row = n % kRows;
        const float *src = ws + ((tm * tiles_n + tn) * parts * kGroup + pos) * kRows * kTileRows + row * kTileRows +
                           (m % kTileRows);
        float v[8];
        {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(src));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(src) + 1);
            v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
        }
        for (int k = 1; k < parts; ++k) {
            const float4 *q = reinterpret_cast<const float4 *>(src + k * part_stride);
            const float4 a = __ldcg(q), b = __ldcg(q + 1);
            v[0] += a.x, v[1] += a.y, v[2] += a.z, v[3] += a.w, v[4] += b.x, v[5] += b.y, v[6] += b.z, v[7] += b.w;
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = Kind::pack(v[2 * j], v[2 * j + 1], s);
        uint16_t *col = static_cast<uint16_t *>(c_ptr) + n * ldc;
        if (vec_c && m + 8 <= M) {
            *reinterpret_cast<uint4 *>(col + m) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (m + j < M) col[m + j] = static_cast<uint16_t>((w[j / 2] >> (16 * (j & 1))) & 0xFFFFu);
        }
    }
}

// C[m + n*ldc] = +0 for m < M, n < N (the K == 0 case).
__global__ void zero_fill_kernel(uint16_t *__restrict__ c, int64_t ldc, int64_t M, int64_t N, uint16_t value)
{
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / M;
        c[(i - n * M) + n * ldc] = value;
    }
}

// Softmax statistics of an all-zero score matrix (K = 0): max 0, sum N.
__global__ void fill_stats_kernel(float *__restrict__ row_max, float *__restrict__ row_sum, int64_t M, float n)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        row_max[i] = 0.0f;
        row_sum[i] = n;
    }
}

}  // namespace tn
