// tn_skinny_kernel: the TN GEMM for few columns n (N <= 64) and many rows m,
// C[m + n ldc] = sum_k A[m lda + k] B[k + n ldb], FP32 accumulation.
//
// The general kernel puts n on the MMA's M side (128 rows of B per CTA), so a
// problem with N = 16 fills 16 of its 128 rows, loads 112 rows of zero fill
// per stage, and with few tiles must cut K into ranges that it adds up through
// distributed shared memory.  Here the operands swap sides: the MMA's M side
// is 128 rows m of A, its N side the problem's n columns (N rounded up to 16,
// at most 64), so a stage holds 16 KiB of A and at most 8 KiB of B, and eight
// stages keep 128 KiB of A in flight per SM.
//
// Work units: 128-row m tiles, each cut into `parts` (1, 2 or 4) ranges of
// its k blocks so that the grid fills the SMs.  With several ranges every
// unit writes its 128 x N FP32 partial to a workspace and takes the tile's
// ticket; the unit that arrives last adds all the partials in range order
// (its own from registers) and stores C, so the result is the same whatever
// the order of arrival.  No CTA ever waits for another.
//
// The roles, barriers, bounded waits and programmatic-dependent-launch
// protocol are the general kernel's: warp 0 loads (TMA), warp 1 allocates
// TMEM and one of its threads issues the MMAs, warps 2-5 read the accumulator
// (TMEM lanes = rows m) and store.  [ch11] §11.1 (the sum), §11.4 (store
// only valid outputs).
#pragma once

#include "tn_gemm_kernel.cuh"

namespace tn {

constexpr int kSkRowsM = 128;                   // rows m per tile = MMA M
constexpr int kSkMaxN = 64;                     // largest MMA N (columns n of a tile)
constexpr int kSkStages = 8;
constexpr int kSkABytes = kSkRowsM * kBlockKBytes;          // 16 KiB: one 128-byte K atom of 128 rows
constexpr int kSkBBytes = kSkMaxN * kBlockKBytes;           // 8 KiB: room for 64 rows of B
constexpr int kSkStageBytes = kSkABytes + kSkBBytes;
constexpr int kSkAccCols = kSkMaxN;                         // TMEM columns of one accumulator
constexpr uint32_t kSkTmemCols = 2 * kSkAccCols;           // two accumulators
constexpr int kSkMaxParts = 4;
constexpr int kSkPrefetchKb = 4;                // k blocks prefetched into L2 before the dependency wait
// full[s], empty[s], accfull[2], accempty[2], never, drain
constexpr int kSkNumBarriers = 2 * kSkStages + 6;
constexpr int kSkSmemBytes = 1024 /* alignment slack */ + kSkStages * kSkStageBytes + kSkNumBarriers * 8 + 32;
static_assert(kSkSmemBytes <= 232448, "exceeds the 227 KiB shared memory of one CTA");

struct SkinnyParams {
    CUtensorMap tmap_a;      // A: dims {K', M}, box {kBlockKBytes / esz, 128}, 128B swizzle
    CUtensorMap tmap_b;      // B: dims {K', N}, box {kBlockKBytes / esz, n_mma}, 128B swizzle
    void *c_ptr;             // C base (direct stores)
    int64_t ldc;
    int32_t M, N;
    int32_t num_kb;          // 128-byte k blocks
    int32_t n_mma;           // MMA N: N rounded up to 16 (16 .. 64)
    int32_t tiles_m;
    int32_t parts;           // k ranges per tile (1, 2 or 4)
    int32_t kb_part;         // k blocks of each range (the last may have fewer)
    int32_t num_units;       // tiles_m * parts
    // parts > 1: [tile][part][n < n_mma][128 rows m] FP32 partials, and one
    // ticket per tile (0 between launches: the last unit resets it)
    float *split_ws;
    unsigned long long *tickets;
    float scale;             // epilogue multiplier (F8: scale_a * scale_b)
    const float *scale_a_ptr, *scale_b_ptr;   // F8 with device scales (else NULL)
    uint32_t flags;          // kFlagStall* (test hooks)
    uint64_t wait_limit_ns;
};

template <class Kind>
__global__ void __launch_bounds__(kThreads, 1) tn_skinny_kernel(const __grid_constant__ SkinnyParams p)
{
    constexpr int kBlockKElems = kBlockKBytes / Kind::kElemBytes;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_ring = ptx::smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSkStages * kSkStageBytes);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + kSkNumBarriers);
    volatile uint32_t *abort_flag = tmem_holder + 1;
    volatile uint32_t *last_flag = tmem_holder + 2;     // this unit arrived last at its tile's ticket
    const uint32_t abort_addr = ptx::smem_addr(const_cast<uint32_t *>(abort_flag));
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSkStages + s); };
    auto accfull_bar = [&](int b) { return bar0 + 8u * (2 * kSkStages + b); };
    auto accempty_bar = [&](int b) { return bar0 + 8u * (2 * kSkStages + 2 + b); };
    const uint32_t never_bar = bar0 + 8u * (2 * kSkStages + 4);   // nothing ever arrives (test stalls)
    const uint32_t drain_bar = bar0 + 8u * (2 * kSkStages + 5);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSkStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull_bar(b), 1);
            ptx::mbar_init(accempty_bar(b), kEpiWarps);
        }
        ptx::mbar_init(never_bar, 1);
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        *last_flag = 0u;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&p.tmap_a);
        ptx::prefetch_tensormap(&p.tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc<1>(ptx::smem_addr(tmem_holder), kSkTmemCols);
        ptx::tmem_relinquish_alloc_permit<1>();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    const Waiter w{abort_flag, abort_addr, 0u, 1u, p.wait_limit_ns};

    // Units of this CTA: blockIdx.x, + gridDim.x, ...  Unit u is range
    // u % parts of tile u / parts.
    const int32_t nunits = p.num_units;
    auto kb_range = [&](int32_t u, int32_t &kb0, int32_t &nkb) {
        const int32_t part = u % p.parts;
        kb0 = part * p.kb_part;
        const int32_t end = kb0 + p.kb_part < p.num_kb ? kb0 + p.kb_part : p.num_kb;
        nkb = end - kb0;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, n_issued = 0;
            bool ok = true;
            if (p.flags & kFlagStallProducer0) ok = w.wait(never_bar, 0u, kSiteStall);
            // The first unit's first k blocks are prefetched into L2 while this CTA
            // may still wait for the previous kernel below (a prefetch returns no
            // data to the CTA: the loads after the wait read through L2, which that
            // kernel's writes reach first).
            if (ok && static_cast<int32_t>(blockIdx.x) < nunits) {
                int32_t kb0, nkb;
                kb_range(blockIdx.x, kb0, nkb);
                const int32_t m0 = (static_cast<int32_t>(blockIdx.x) / p.parts) * kSkRowsM;
                for (int32_t i = 0; i < nkb && i < kSkPrefetchKb; ++i) {
                    ptx::tma_prefetch_2d(&p.tmap_a, (kb0 + i) * kBlockKElems, m0);
                    ptx::tma_prefetch_2d(&p.tmap_b, (kb0 + i) * kBlockKElems, 0);
                }
            }
            const uint32_t fill = static_cast<uint32_t>(kSkABytes + p.n_mma * kBlockKBytes);
            for (int32_t u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                const int32_t m0 = (u / p.parts) * kSkRowsM;
                int32_t kb0, nkb;
                kb_range(u, kb0, nkb);
                for (int32_t i = 0; i < nkb; ++i) {
                    if (!w.wait(empty_bar(stage), phase ^ 1u, kSiteEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s_a = s_ring + stage * kSkStageBytes;
                    const int32_t k0 = (kb0 + i) * kBlockKElems;
                    if (n_issued == 0) ptx::griddep_wait();   // this thread's first global access
                    ptx::mbar_arrive_expect_tx(full_bar(stage), fill);
                    ptx::tma_load_2d(s_a, &p.tmap_a, full_bar(stage), k0, m0);
                    ptx::tma_load_2d(s_a + kSkABytes, &p.tmap_b, full_bar(stage), k0, 0);
                    ++n_issued;
                    if (++stage == kSkStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // no more loads from this CTA: the next kernel may start its setup
            if (n_issued == 0) ptx::griddep_wait();
            ptx::griddep_launch_dependents();
            // every issued load lands before the CTA can exit
            for (int s = 0; s < kSkStages; ++s) {
                const uint32_t passes =
                    n_issued / kSkStages + (static_cast<uint32_t>(s) < n_issued % kSkStages ? 1u : 0u);
                if (passes) w.drain(full_bar(s), (passes - 1) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued_any = false;
            if (p.flags & kFlagStallMma) ok = w.wait(never_bar, 0u, kSiteStall);
            const uint32_t idesc = ptx::idesc_f32acc(kSkRowsM, static_cast<uint32_t>(p.n_mma), Kind::kFmt, Kind::kFmt);
            for (int32_t u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                int32_t kb0, nkb;
                kb_range(u, kb0, nkb);
                if (!w.wait(accempty_bar(acc), acc_phase ^ 1u, kSiteAccEmpty)) break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kSkAccCols;
                for (int32_t i = 0; i < nkb; ++i) {
                    if (!w.wait(full_bar(stage), phase, kSiteLoaded)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t s_a = s_ring + stage * kSkStageBytes;
                    const uint64_t desc_a = ptx::desc_kmajor_sw128(s_a);
                    const uint64_t desc_b = ptx::desc_kmajor_sw128(s_a + kSkABytes);
#pragma unroll
                    for (int j = 0; j < kBlockKBytes / kMmaKBytes; ++j) {
                        // +32 bytes along K inside the 128-byte swizzle span = +2 in the address field
                        Kind::template mma<1>(d_tmem, desc_a + 2u * j, desc_b + 2u * j, idesc, (i | j) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    ptx::mma_commit<1>(empty_bar(stage));
                    if (++stage == kSkStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit<1>(accfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA this thread issued completes before TMEM is freed
            if (issued_any) {
                ptx::mma_commit<1>(drain_bar);
                w.drain(drain_bar, 0u);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31 are this warp's
        const int row = 32 * quarter + lane;      // this thread's row m within the tile
        ptx::griddep_wait();                      // (device scales, workspace, C: after the previous kernel)
        const float scale = p.scale_a_ptr ? __fmul_rn(__ldg(p.scale_a_ptr), __ldg(p.scale_b_ptr)) : p.scale;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint16_t *c = static_cast<uint16_t *>(p.c_ptr);
        const int32_t N = p.N;
        for (int32_t u = blockIdx.x; u < nunits; u += gridDim.x) {
            const int32_t tile = u / p.parts, part = u % p.parts;
            bool ok = __all_sync(0xffffffffu, w.wait(accfull_bar(acc), acc_phase, kSiteAccFull));
            if (!ok) break;
            ptx::tc_fence_after_sync();
            // all 64 columns of the accumulator (those past n_mma are not used)
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + acc * kSkAccCols;
            uint32_t r0[32], r1[32];
            ptx::tmem_ld_32x32b_x32(t_row, r0);
            ptx::tmem_ld_32x32b_x32(t_row + 32, r1);
            ptx::tmem_ld_wait(r0);
            ptx::reg_dependency(r1);
            float v[kSkMaxN];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v[j] = __uint_as_float(r0[j]);
                v[32 + j] = __uint_as_float(r1[j]);
            }
            // hand the accumulator back: its columns are in registers
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(accempty_bar(acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            const int64_t m = static_cast<int64_t>(tile) * kSkRowsM + row;
            if (p.parts > 1) {
                // This range's partial, column n at [n][row] (a warp writes 128 B per
                // n), in whole groups of 16 columns up to n_mma, so that every load
                // of a group below stays inside the partial.
                const int n_groups = p.n_mma / 16;
                const int64_t span = static_cast<int64_t>(p.n_mma) * kSkRowsM;      // one range's partial
                float *ws_tile = p.split_ws + static_cast<int64_t>(tile) * p.parts * span;
                float *mine = ws_tile + part * span + row;
#pragma unroll
                for (int gi = 0; gi < kSkMaxN / 16; ++gi)
                    if (gi < n_groups) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) mine[(16 * gi + j) * kSkRowsM] = v[16 * gi + j];
                    }
                ptx::named_barrier_sync(1, kEpiWarps * 32);
                if (warp == 2 && lane == 0) {
                    // releases this CTA's partial (the barrier orders every warp's
                    // writes before it) and acquires the others (the barrier below
                    // orders the reads after it)
                    unsigned long long *ticket = p.tickets + tile;
                    const bool last =
                        ptx::atom_add_acq_rel_gpu(ticket, 1ull) == static_cast<unsigned long long>(p.parts - 1);
                    if (last) atomicExch(ticket, 0ull);   // every range is in: ready for the next launch
                    *last_flag = last ? 1u : 0u;
                }
                ptx::named_barrier_sync(1, kEpiWarps * 32);
                if (*last_flag == 0u) continue;
                // The ranges added in order 0, 1, ... (this one's from registers).
                // A group's 16 loads are issued before any of them is used: with a
                // condition per column they went out one at a time (measured on
                // GB300: about 0.25 us each, 11 us for three partials of 16 columns).
#pragma unroll
                for (int gi = 0; gi < kSkMaxN / 16; ++gi) {
                    if (gi >= n_groups) break;
                    float sum[16];
#pragma unroll 1
                    for (int q = 0; q < p.parts; ++q) {
                        float x[16];
                        if (q == part) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) x[j] = v[16 * gi + j];
                        } else {
                            const float *src = ws_tile + q * span + (16 * gi) * kSkRowsM + row;
#pragma unroll
                            for (int j = 0; j < 16; ++j) x[j] = __ldcg(src + j * kSkRowsM);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) sum[j] = q == 0 ? x[j] : sum[j] + x[j];
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[16 * gi + j] = sum[j];
                }
            }
            if (m < p.M) {
#pragma unroll
                for (int n = 0; n < kSkMaxN; ++n)
                    if (n < N) c[n * p.ldc + m] = static_cast<uint16_t>(Kind::pack(v[n], v[n], scale) & 0xFFFFu);
            }
        }
    }

    __syncwarp();                // .aligned barriers below need converged warps
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<1>(tmem_base, kSkTmemCols);
    }
}

}  // namespace tn
