// tn_gemm_kernel.cuh -- the persistent, warp-specialised sm_103a TN GEMM.
//
// C = A x B with A row-major M x K, B column-major K x N (both K-contiguous)
// and C column-major with leading dimension ldc: the TN storage of the AMD
// ROCm blog "FP16 GEMM optimization on AMD RDNA 3 and RDNA 4" (section "What
// we compute"); the sum is the definition of hello-gpu ch.11 "GEMM-Like",
// section 11.1.  Accumulation is FP32 in tensor memory.
//
// Orientation.  C column-major is C^T row-major: row n of C^T (= column n of
// C) is contiguous in m.  The kernel therefore computes C^T = B^T A^T: the
// tensor core's first operand ("lanes") is a tile of B's columns, its second
// operand ("columns") a tile of A's rows.  TMEM lane i then holds one output
// column n and up to 256 consecutive m values per MMA, so every epilogue
// thread owns a contiguous run of C.
//
// Tiles (n x m): one CTA per 128 x 256 (MMA M128 N256); a CTA pair per
// 256 x 256 (cta_group::2, M256 N256); or a CTA pair per 256 x 512, two M256
// N256 halves that share the n-side rows (TileCfg below).
//
// The blog's RDNA design problems and their Blackwell re-solutions:
//   LDS padding / XOR permutation (its Step 3)   -> TMA 128-byte swizzle that
//       the tcgen05 shared-memory descriptor reads natively;
//   buffer-descriptor OOB-zero loads (Step 4)    -> TMA out-of-bounds zero
//       fill on loads, clipping on the TMA store, so M, N, K need not divide
//       the tile (hello-gpu ch.11, section 11.4);
//   double buffer + staged commit (Steps 2, 8)   -> a kStages-deep shared
//       memory ring with full/empty mbarriers;
//   deeper K slices (Step 5)                     -> 128- or 256-byte K stages
//       (64 / 128 fp16 or 128 / 256 e4m3 values), 4 or 8 MMAs per stage;
//   block reordering for cache reuse (Step 6)    -> persistent CTAs walking a
//       grouped raster (tile_coord below);
//   prefetch / WMMA interleave (Step 7)          -> warp specialisation: a TMA
//       producer warp, a single-thread MMA issuer, 4 epilogue warps; for tiles
//       up to 256 wide in m a double-buffered TMEM accumulator, so the
//       epilogue of tile i overlaps the main loop of tile i+1.
//
// Each launch is a programmatic dependent of the previous kernel on its
// stream: setup overlaps that kernel's end, and griddepcontrol.wait orders
// every global access after it.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace tn {

// ------------------------------------------------------------------ config
constexpr int kThreads = 192;               // warp 0 TMA, warp 1 TMEM + MMA (even CTA), warps 2-5 epilogue
constexpr int kBlockKBytes = 128;           // bytes of K per row of one swizzle atom (= one TMA box)
constexpr int kMmaKBytes = 32;              // K bytes per tcgen05.mma (16 fp16 / 32 e4m3)
constexpr int kEpiWarps = 4;
constexpr int kEpiBoxM = 64;                // m values per TMA store box (128 B of 16-bit C)
constexpr int kEpiBoxN = 32;                // n rows per box = one warp's TMEM lane quarter
constexpr int kEpiBufBytes = kEpiBoxN * kEpiBoxM * 2;       // 4 KiB
constexpr int kEpiBufs = 2;                 // per epilogue warp (ping-pong)
constexpr int kSmemEpi = kEpiWarps * kEpiBufs * kEpiBufBytes;
constexpr int kTileM = 256;                 // C rows m per tile = MMA N = TMEM columns per accumulator

// kGroup = 1: one CTA computes a 128 (n) x 256 (m) tile with M128 MMAs.
// kGroup = 2: a CTA pair (a cluster of two CTAs) computes a 256 (n) x 256 (m)
// tile with M256 MMAs issued by the pair's even CTA; each CTA holds 128 rows
// of each operand tile per stage and the accumulator rows of its own 128
// columns n.  Every CTA loads its own operand rows from global memory; no
// load is shared between CTAs.
//
// A stage holds kAtoms consecutive 128-byte K atoms of each operand (a pair:
// 256 bytes of K, 8 MMAs per stage), each atom its own 128B-swizzled block:
//   [B atom 0][B atom 1]...[A atom 0][A atom 1]...
// Fewer, longer stages halve the barrier waits, commits and TMA issues per
// MMA; measured on GB300 the MMA pipe then loses less time between stages.
//
// kWide (pairs only): a CTA pair computes a 256 (n) x 512 (m) tile as two M256
// N256 halves that share the n-side operand.  Each CTA holds, per stage, one
// 128-byte atom of its 128 B rows and of its 2 x 128 A rows (one block per
// half, the second at +kHalfABytes): 48 KiB, so four stages fit.  A quarter
// fewer bytes leave L2 per MMA, and four stages of 1024 MMA cycles hide more
// load latency than three of 2048 bytes per CTA and 1024 cycles.  The
// accumulator takes all 512 TMEM columns (half h at column 256 h), so it is
// not double-buffered: the next tile's MMAs on a half wait for the epilogue
// to have read that half (it hands the halves back one at a time).
// Measured on GB300 under the power cap (8192^3 FP16), the lower L2 traffic
// lets the SMs run at a 7-9 % higher clock for the same work per clock.
//
// kLean = 4 or 2 (single CTAs only): the configuration of launches whose units
// are all quarter-m (or half-m) units -- a grid of few tiles with a short K,
// each tile cut into four 64-row (two 128-row) ranges of m.  Its ring holds
// just such a unit's A rows (three stages of 24 KiB, or two of 32 KiB), its
// accumulators take 64 (128) TMEM columns each, and it is compiled for two
// CTAs per SM (at most 168 registers a thread), so that a launch's CTAs all
// become resident while the previous launch on the stream still runs and do
// their setup in its shadow.  With one 226 KiB CTA per SM, only the CTAs that
// found an idle SM started early; the rest entered as the previous launch's
// CTAs left and ran their first-time code (the parameter reads, the first
// unit's schedule) after the previous grid had completed.
template <int kGroup, bool kWide = false, int kLean = 0>
struct TileCfg {
    static_assert(!kWide || kGroup == 2, "256 x 512 tiles are CTA-pair tiles");
    static_assert(kLean == 0 || (kGroup == 1 && !kWide && (kLean == 2 || kLean == 4)),
                  "the lean configurations are single-CTA ones of half-m or quarter-m units");
    static constexpr int kCtas = kGroup;                   // CTAs per cluster
    static constexpr int kTileN = 128 * kGroup;            // C columns n per pair tile = MMA M
    static constexpr int kTileMRows = kWide ? 2 * kTileM : kTileM;   // C rows m per tile
    static constexpr int kHalves = kWide ? 2 : 1;           // MMA N = 256 halves per tile
    static constexpr int kRowsB = 128;                      // B rows (columns n) per CTA and stage
    static constexpr int kRowsA = kTileMRows / kGroup;      // A rows (m) per CTA and stage
    static constexpr int kAtoms = kGroup == 2 && !kWide ? 2 : 1;   // 128-byte K atoms per stage
    static constexpr int kStageKBytes = kAtoms * kBlockKBytes;
    static constexpr int kStages = kLean == 4 ? 3 : kLean == 2 ? 2 : kGroup == 2 && !kWide ? 3 : 4;
    static constexpr int kHalfABytes = kTileM / kGroup * kBlockKBytes;   // one half's A rows of one atom
    static constexpr int kRingRowsA = kLean ? kRowsA / kLean : kRowsA;   // A rows a stage has room for
    static constexpr int kAtomBBytes = kRowsB * kBlockKBytes;
    static constexpr int kAtomABytes = kRingRowsA * kBlockKBytes;
    static constexpr int kTileBBytes = kAtoms * kAtomBBytes;
    static constexpr int kTileABytes = kAtoms * kAtomABytes;
    static constexpr int kStageBytes = kTileBBytes + kTileABytes;
    static constexpr int kSmemRing = kStages * kStageBytes;
    // loaded[S][atoms], empty[S], accfull[2], accempty[2], drain, never, peers_free, received
    static constexpr int kNumBarriers = kStages * (kAtoms + 1) + 8;
    static constexpr int kSmemBytes = 1024 /* alignment slack */ + kSmemRing + kSmemEpi + kNumBarriers * 8 + 32;
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KiB shared memory of one CTA");
    // two CTAs per SM: 228 KiB of shared memory, 1 KiB of it reserved per CTA
    static_assert(!kLean || 2 * (kSmemBytes + 1024) <= 233472, "two lean CTAs must fit one SM");
    // TMEM columns of one accumulator (MMA N of a unit) and of the allocation
    // (two accumulators: a unit's epilogue overlaps the next unit's MMAs)
    static constexpr uint32_t kAccCols = kLean ? kTileM / kLean : kTileM;
    static constexpr uint32_t kTmemCols = 2 * kAccCols;
};

// How tiles are cut into several units each (split_parts of them): the tiles
// of a partly filled last wave, or every tile of a grid that fills at most
// half of the slots.
constexpr int32_t kTailNone = 0;
// split_parts (2 or 4) consecutive ranges of the tile's m rows, m_part_rows
// each (MMA N = 128 or 64); every unit reads all of the tile's B rows.
constexpr int32_t kTailMParts = 1;
constexpr int kMaxMParts = 4;
constexpr int32_t kTailSplitK = 2;   // two halves of the k blocks; partial sums meet in a workspace
// A grid of fewer tiles than half the slots, with a long K: every tile is cut
// into split_parts ranges of its k blocks; each unit stores its FP32 partial,
// and split_reduce_kernel (launched next) sums them and stores C.
constexpr int32_t kSplitReduce = 3;
// The same cut made inside a cluster: S = split_parts (2 to 4) single CTAs,
// or S CTA pairs, per tile, CTA (or pair) r computing k blocks
// [r kb_part, (r + 1) kb_part), one tile per cluster.  Of the tile's four
// 64-column chunks of m, range r reduces and stores those with c % S == r:
// the other ranges' CTAs write their FP32 partials of them into its shared
// memory (distributed shared memory), and it adds the S partials in range
// order.  No workspace, no second kernel.
constexpr int32_t kClusterReduce = 4;

constexpr uint32_t kFlagTmaStore = 1u;      // C rows m < m_tma are written with TMA stores
// Test hooks: the named thread first waits on a barrier nobody arrives on, so
// its bounded wait runs out and the kernel leaves through its abort path.
constexpr uint32_t kFlagStallMma = 2u;          // the MMA thread(s)
constexpr uint32_t kFlagStallProducer0 = 4u;    // the producer of cluster CTA 0 (or of the only CTA)
constexpr uint32_t kFlagStallProducer1 = 8u;    // the producer of cluster CTA 1 (the odd CTA of the first pair)
// FP16 scaled scores with softmax row statistics: C = fp16(scale * acc), and
// per row m the maximum and the sum of exp(score - maximum) over all n.
constexpr uint32_t kFlagStats = 16u;
// Whole tiles of odd waves (tile id / slots odd) walk their k blocks from the
// last to the first.  The tiles of one wave read their shared A and B panels
// in lockstep; the next wave shares panels with it (the grouped raster keeps
// its tile rows), and walking K the other way it starts on the k slices the
// previous wave read last, which are the likeliest to be still in L2.  The
// order of the FP32 sums changes, not their terms.
constexpr uint32_t kFlagAltK = 32u;

// L2 prefetch before griddepcontrol.wait (kClusterReduce launches): units of
// at least kPrefetchMinKb stages get their first kPrefetchAtoms 128-byte K
// atoms prefetched.
constexpr int kPrefetchMinKb = 16;
constexpr int kPrefetchAtoms = 4;

// Status word of the current device; set (never cleared) by a kernel whose
// bounded wait ran out: 4 (timeout) | site << 8.
__device__ int g_tn_status;

enum WaitSite : int {
    kSiteEmpty = 1, kSiteLoaded = 2, kSiteAccEmpty = 3, kSiteAccFull = 4, kSiteStall = 5, kSitePeerDone = 6,
    kSiteDrain = 7, kSiteReconcile = 8, kSitePeersFree = 9, kSiteReceived = 10
};

struct KernelParams {
    CUtensorMap tmap_a;      // A: dims {K', M}, box {kBlockKBytes / esz, kRowsA}, 128B swizzle
    CUtensorMap tmap_b;      // B: dims {K', N}, box {kBlockKBytes / esz, 128}, 128B swizzle
    CUtensorMap tmap_c;      // C: dims {m_tma, N}, box {kEpiBoxM, kEpiBoxN}, 128B swizzle
    CUtensorMap tmap_a_part; // kTailMParts: A with box {kBlockKBytes / esz, kRowsA / split_parts}
    void *c_ptr;             // C base (direct stores)
    int64_t ldc;
    int32_t M, N, K;
    int32_t m_tma;           // rows m < m_tma are written by TMA stores (a multiple of 8, or 0)
    int32_t tiles_m, tiles_n, num_tiles, num_kb, group;
    // Work units: tiles [0, tail_start) are whole units; each later tile is
    // split_parts units (so a last, partly filled wave of tiles becomes a full
    // wave of shorter units), cut as tail_mode says.  num_units counts both kinds.
    int32_t tail_start, num_units, tail_mode;
    int32_t kb_part;         // k blocks of each split unit: ceil(num_kb / parts), padded with zeros
    int32_t split_parts;     // units per cut tile: 2 (kTailSplitK), 2 or 4 (kTailMParts), 2..8 (kSplitReduce)
    int32_t m_part_rows;     // kTailMParts: rows m per unit, kTileM / split_parts
    float *split_ws;         // split-K partials: [tail tile][k half][CTA of pair][128 n][256 m] fp32
    // [tail tile][CTA of pair]: halves arrived so far; 0 between launches (the
    // second half resets it), so a captured graph can replay the launch.
    unsigned long long *split_tickets;
    float scale;             // epilogue multiplier (F8: scale_a * scale_b)
    // F8 with device-resident scales: when set, the epilogue multiplies by
    // (*scale_a_ptr) * (*scale_b_ptr) in FP32 instead of `scale`.
    const float *scale_a_ptr, *scale_b_ptr;
    // Softmax statistics (kFlagStats).  Every CTA that computes a tile writes,
    // per epilogue warp, the (max, sum) of its 32 columns n for each of the
    // tile's 256 rows m into stat_parts[tile_m][part][256] (a unit of a tile
    // cut along m writes its own rows of them).  The rows of one tile row and
    // m part are computed by stat_ctas CTAs; the last of them (counted in
    // stat_tickets[tile_m * kMaxMParts + m part], which the last resets to 0)
    // merges those rows' parts in a fixed order into row_max/row_sum.
    float *row_max, *row_sum;
    float2 *stat_parts;
    unsigned long long *stat_tickets;
    int32_t stat_ctas;                  // tiles_n * CTAs per tile
    uint32_t flags;
    uint64_t wait_limit_ns;
    // Optional (NULL: off): CTA 0's first thread adds the SM cycles and the
    // nanoseconds from its start (before griddepcontrol.wait) to its exit to
    // clock_probe[0] and [1], and 1 to [2]: [0] / [1] is the SM clock the
    // launches ran at.
    unsigned long long *clock_probe;
};

// ------------------------------------------------------------------ scheduler
// Grouped raster: `group` tile rows (m) form a tall region; consecutive ids
// walk down the region's rows for one tile column (n), then the next column.
// The last region is short when tiles_m % group != 0.  This is the GROUP_M
// mapping of hello-gpu ch.11 section 11.3.4 and the grouped block order of
// the ROCm blog's Step 6.
//
// The arithmetic is 32-bit (a 64-bit division is a long instruction sequence
// on the path to every unit's first load): grids have fewer than 2^31 tiles.
// group * tiles_n then fits too, except when tiles_m < group, where there is
// one group and every id lies in it.
__host__ __device__ __forceinline__ void tile_coord(int64_t id, int64_t tiles_m, int64_t tiles_n, int64_t group,
                                                    int64_t &tm, int64_t &tn)
{
    const uint32_t i = static_cast<uint32_t>(id), rows_m = static_cast<uint32_t>(tiles_m);
    const uint32_t gm = static_cast<uint32_t>(group);
    const uint32_t per_group = rows_m < gm ? 0xFFFFFFFFu : gm * static_cast<uint32_t>(tiles_n);
    const uint32_t g = i / per_group;
    const uint32_t first_m = g * gm;
    const uint32_t rows = (rows_m - first_m) < gm ? (rows_m - first_m) : gm;
    const uint32_t in_group = i - g * per_group;
    tm = first_m + in_group % rows;
    tn = in_group / rows;
}

// A work unit: a tile, or one part of a cut tile.
struct Unit {
    int64_t tile, tm, tn;    // tile id and coordinates
    int32_t mpart;           // -1: the whole m range; else that range of m_part_rows rows (kTailMParts)
    int32_t khalf;           // -1: all k blocks; 0 / 1: that half of them (kTailSplitK)
    int32_t kpart;           // -1: all k blocks; else this range of them (kSplitReduce)
    int32_t cpart;           // -1, or this CTA's k range of a tile reduced in the cluster (kClusterReduce)
    int32_t kb0, nkb;        // the unit's k blocks
    bool phantom;            // no such unit: loads out of bounds, computes zeros, stores nothing
};

__device__ __forceinline__ Unit unit_of(int64_t u, const KernelParams &p)
{
    Unit r{u, 0, 0, -1, -1, -1, -1, 0, p.num_kb, u >= p.num_units};
    if (r.phantom) return r;
    if (u >= p.tail_start) {
        const uint32_t v = static_cast<uint32_t>(u - p.tail_start), parts = static_cast<uint32_t>(p.split_parts);
        const int32_t part = static_cast<int32_t>(v % parts);
        r.tile = p.tail_start + static_cast<int64_t>(v / parts);
        if (p.tail_mode == kSplitReduce) {
            r.kpart = part;
            r.kb0 = part * p.kb_part;
            r.nkb = p.kb_part;
        } else if (p.tail_mode == kTailSplitK) {
            r.khalf = part;
            r.kb0 = part * p.kb_part;
            r.nkb = p.kb_part;
        } else {
            r.mpart = part;
        }
    }
    tile_coord(r.tile, p.tiles_m, p.tiles_n, p.group, r.tm, r.tn);
    return r;
}

// The units a work slot walks.  Slot s takes units s, s + nslots, ... of the
// whole tiles; if tiles were cut, slots s < split_parts * (tiles cut) first
// take unit tail_start + s, so its combine (split-K) overlaps the
// slot's later tiles instead of ending the launch.  (kSplitReduce launches at
// most one unit per slot: tail_start = 0, num_units <= slots.)
__device__ __forceinline__ bool slot_has_tail(int64_t slot, const KernelParams &p)
{
    return p.tail_mode != kTailNone && slot < p.num_units - p.tail_start;
}

__device__ __forceinline__ int64_t slot_iters(int64_t slot, int64_t nslots, const KernelParams &p)
{
    const int64_t whole = p.tail_start > slot ? static_cast<uint32_t>(p.tail_start - slot + nslots - 1) /
                                                    static_cast<uint32_t>(nslots)
                                              : 0;
    return whole + (slot_has_tail(slot, p) ? 1 : 0);
}

// Unit index of step `it` of slot `slot` (>= num_units: none, a phantom).
__device__ __forceinline__ int64_t slot_unit(int64_t slot, int64_t it, int64_t nslots, const KernelParams &p)
{
    if (slot_has_tail(slot, p)) {
        if (it == 0) return p.tail_start + slot;
        --it;
    }
    const int64_t u = slot + it * nslots;
    return u < p.tail_start ? u : p.num_units;   // past the whole tiles: none
}

// ------------------------------------------------------------------ waits
// Every wait is bounded: after `limit` ns the waiting thread raises the abort
// flag of every CTA of its cluster and the device status word, and returns
// false; the other roles see the flag and leave their loops.  drain() waits
// for copies already in flight and ignores the flag (those copies land).
struct Waiter {
    volatile uint32_t *abort_flag;
    uint32_t abort_addr;     // shared::cta address of the flag (the same offset in every CTA)
    uint32_t rank, ctas;     // this CTA's rank in its cluster, CTAs in the cluster
    uint64_t limit;

    __device__ __forceinline__ void raise(int site) const
    {
        *abort_flag = 1u;
        for (uint32_t q = 0; q < ctas; ++q)
            if (q != rank) ptx::st_shared_cluster_u32(ptx::mapa_shared(abort_addr, q), 1u);
        atomicCAS(&g_tn_status, 0, 4 | (site << 8));
    }

    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int site) const
    {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer();
        while (true) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > limit) {
                raise(site);
                return false;
            }
        }
    }

    // wait() with a cluster-scope acquire (data other CTAs published with a
    // cluster-scope release before arriving).
    __device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, int site) const
    {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer();
        while (true) {
            if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > limit) {
                raise(site);
                return false;
            }
        }
    }

    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const
    {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (ptx::globaltimer() - t0 > limit) {
                atomicCAS(&g_tn_status, 0, 4 | (kSiteDrain << 8));
                return false;
            }
        }
        return true;
    }
};

// ------------------------------------------------------------------ kinds
struct KindF16 {
    static constexpr bool kF8 = false;
    static constexpr int kElemBytes = 2;
    static constexpr uint32_t kFmt = 0;      // F16 (kind::f16)
    template <int kGroup>
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
    {
        ptx::mma_f16<kGroup>(d, a, b, idesc, acc);
    }
    __device__ static uint32_t pack(float lo, float hi, float) { return ptx::pack_f16x2(lo, hi); }
};

struct KindE4M3 {
    static constexpr bool kF8 = true;
    static constexpr int kElemBytes = 1;
    static constexpr uint32_t kFmt = 0;      // E4M3 (kind::f8f6f4)
    template <int kGroup>
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
    {
        ptx::mma_f8<kGroup>(d, a, b, idesc, acc);
    }
    // acc * (scale_a * scale_b) in FP32, one RNE rounding to bf16.
    __device__ static uint32_t pack(float lo, float hi, float s) { return ptx::pack_bf16x2(lo * s, hi * s); }
};

// ------------------------------------------------------------------ cluster drain
// Run by the even CTA of each pair once its own producer issues no more, so
// that no load feeding its loaded[] barriers is still in flight when the
// cluster leaves.  Loads go round the stages in order, and a stage can only
// be refilled after the pair's MMAs finished reading its previous fill (which
// needed all of that fill's bytes), so per stage the producers of the two
// CTAs are at most one fill apart.  For the last fill of each stage this CTA adds
// up the bytes really sent to it by the producers that issued that fill; if
// it armed the fill itself it cancels the bytes that will not come
// (mbarrier.complete_tx), otherwise it arms the fill for the bytes that will
// (arrive.expect_tx).  Then it waits for the phase.  On the normal path every
// producer issued every fill and each wait returns at once.
template <int kStages, int kAtoms, int kCtas, class LoadedBar, class Contribution>
__device__ __forceinline__ void drain_cluster_loads(const Waiter &w, LoadedBar loaded_bar, Contribution contribution,
                                                    uint32_t n_own, uint32_t count_addr, uint32_t done_addr,
                                                    uint32_t first)
{
    // the pair's CTAs: cluster ranks first .. first + kCtas - 1 (index q - first)
    uint32_t counts[kCtas];
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t q = first; q < first + kCtas; ++q) {
        if (q == w.rank) {
            counts[q - first] = n_own;
            continue;
        }
        bool stopped = true;
        while (ptx::ld_acquire_cluster_u32(ptx::mapa_shared(done_addr, q)) == 0u) {
            if (ptx::globaltimer() - t0 > w.limit) {
                atomicCAS(&g_tn_status, 0, 4 | (kSitePeerDone << 8));
                stopped = false;
                break;
            }
        }
        counts[q - first] = stopped ? ptx::ld_relaxed_cluster_u32(ptx::mapa_shared(count_addr, q)) : n_own;
    }
    for (int s = 0; s < kStages; ++s) {
        uint32_t lo = 0xffffffffu, hi = 0;
        uint32_t passes[kCtas];
        for (uint32_t q = 0; q < kCtas; ++q) {
            passes[q] = counts[q] / kStages + (static_cast<uint32_t>(s) < counts[q] % kStages ? 1u : 0u);
            lo = passes[q] < lo ? passes[q] : lo;
            hi = passes[q] > hi ? passes[q] : hi;
        }
        if (hi == 0) continue;
        if (hi > lo + 1) {      // cannot happen; never guess
            atomicCAS(&g_tn_status, 0, 4 | (kSiteReconcile << 8));
            continue;
        }
        const uint32_t fill = (hi - 1) * kStages + s;   // index of the stage's last fill
        uint32_t sent = 0, total = 0;
        for (uint32_t q = 0; q < kCtas; ++q) {
            const uint32_t c = contribution(q, fill);
            total += c;
            if (passes[q] == hi) sent += c;
        }
        // every atom of a fill carries the same share of its bytes, on its own barrier
        for (int t = 0; t < kAtoms; ++t) {
            if (passes[w.rank - first] == hi) {
                if (total > sent) ptx::mbar_complete_tx(loaded_bar(s, t), (total - sent) / kAtoms);
            } else {
                ptx::mbar_arrive_expect_tx(loaded_bar(s, t), sent / kAtoms);
            }
            w.drain(loaded_bar(s, t), (hi - 1) & 1u);
        }
    }
}

// ------------------------------------------------------------------ softmax statistics
// e^x for x <= 0 as 2^(x log2 e), with the PTX ex2.approx.ftz.f32
// instruction (the PTX ISA gives its maximum relative error as about 2^-22;
// results below 2^-126 flush to 0; e^-inf = 0).  Measured on GB300, the
// statistics epilogue ran 2.6x slower with CUDA's expf / __expf instead.
__device__ __forceinline__ float exp_nonpos(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// (max, sum) of two sets of values x, where sum = sum exp(x - max): the merge
// of the online softmax.  An empty set is (-inf, 0).
__device__ __forceinline__ void stat_merge(float &m, float &s, float m2, float s2)
{
    const float mx = fmaxf(m, m2);
    if (mx == -INFINITY) {
        m = mx;
        s = 0.0f;
        return;
    }
    s = s * exp_nonpos(m - mx) + s2 * exp_nonpos(m2 - mx);
    m = mx;
}

// (max, sum of exp(x - max)) of one row's 32 scores, held by one thread: the
// maximum by a tree of fmaxf, then the exponentials and their sum by a tree of
// adds.  Scores of absent columns are -inf (they add 0); a row with no score
// is (-inf, 0).
__device__ __forceinline__ float2 stat_row32(const float (&x)[32])
{
    float t[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) t[j] = x[j];
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    const float mx = t[0];
    if (mx == -INFINITY) return make_float2(mx, 0.0f);
#pragma unroll
    for (int j = 0; j < 32; ++j) t[j] = exp_nonpos(x[j] - mx);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = t[j] + t[j + w];
    return make_float2(mx, t[0]);
}

// ------------------------------------------------------------------ kernel
// kCluster: the kClusterReduce variant (launched in clusters of S single CTAs
// or S CTA pairs); kStats: the variant with the softmax-statistics epilogue
// (kFlagStats).  The other variants carry none of their code.  kLean = 4 or
// 2: the two-CTAs-per-SM configuration of TileCfg, launched only when every
// unit is a quarter-m (half-m) unit: kTailMParts with split_parts = kLean from
// the first tile.
template <class Kind, int kGroup, bool kWide = false, bool kCluster = false, bool kStats = false, int kLean = 0>
__global__ void __launch_bounds__(kThreads, kLean ? 2 : 1) tn_gemm_kernel(const __grid_constant__ KernelParams p)
{
    static_assert(!(kWide && kCluster), "256 x 512 tiles are not reduced in clusters");
    static_assert(!kStats || (!Kind::kF8 && !kWide && !kCluster), "the statistics are an FP16 epilogue of plain tiles");
    static_assert(!kLean || (!kCluster && !kStats), "the lean configurations are ones of plain m-part units");
    static_assert(kMaxMParts == 4, "m parts are halves or quarters");
    using Cfg = TileCfg<kGroup, kWide, kLean>;
    constexpr uint32_t kAccCols = Cfg::kAccCols;
    constexpr uint32_t kTmemCols = Cfg::kTmemCols;
    constexpr int kStages = Cfg::kStages;
    constexpr int kBlockKElems = kBlockKBytes / Kind::kElemBytes;   // K elements per atom
    constexpr uint32_t kIdesc = ptx::idesc_f32acc(Cfg::kTileN, kTileM, Kind::kFmt, Kind::kFmt);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_ring = ptx::smem_addr(smem);
    const uint32_t s_epi = s_ring + Cfg::kSmemRing;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kSmemRing + kSmemEpi);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + Cfg::kNumBarriers);
    volatile uint32_t *abort_flag = tmem_holder + 1;
    volatile uint32_t *issued_count = tmem_holder + 2;    // k-block loads this CTA's producer issued
    volatile uint32_t *producer_done = tmem_holder + 3;   // set once this CTA's producer issues no more
    const uint32_t abort_addr = ptx::smem_addr(const_cast<uint32_t *>(abort_flag));
    const uint32_t count_addr = ptx::smem_addr(const_cast<uint32_t *>(issued_count));
    const uint32_t done_addr = ptx::smem_addr(const_cast<uint32_t *>(producer_done));

    const uint32_t bar0 = ptx::smem_addr(bars);
    // loaded[s]: the stage's bytes (of both CTAs of a pair) have landed; used in even CTAs only
    // One loaded barrier per 128-byte atom of a stage, so the MMAs of an atom
    // start as soon as its own bytes have landed; one empty barrier per stage.
    constexpr int kAtoms = Cfg::kAtoms;
    constexpr int kLoadedBars = kStages * kAtoms;
    auto loaded_bar = [&](int s, int t) { return bar0 + 8u * (s * kAtoms + t); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kLoadedBars + s); };      // the MMAs have read the stage
    auto accfull_bar = [&](int b) { return bar0 + 8u * (kLoadedBars + kStages + b); };
    auto accempty_bar = [&](int b) { return bar0 + 8u * (kLoadedBars + kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (kLoadedBars + kStages + 4);
    const uint32_t never_bar = bar0 + 8u * (kLoadedBars + kStages + 5);        // nothing ever arrives
    // kClusterReduce: every other CTA of the cluster has announced that its ring
    // is free (peers_free), and has published its partials of this CTA's columns
    // (received)
    const uint32_t peers_free_bar = bar0 + 8u * (kLoadedBars + kStages + 6);
    const uint32_t received_bar = bar0 + 8u * (kLoadedBars + kStages + 7);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTAs per cluster: the pair (kGroup = 2), or one CTA; kCluster: those of
    // the k ranges of a tile reduced in the cluster (kClusterReduce)
    const uint32_t ctas = kCluster ? ptx::cluster_nctarank() : static_cast<uint32_t>(kGroup);
    const uint32_t rank = kGroup == 2 || kCluster ? ptx::cluster_ctarank() : 0u;
    const uint32_t pos = rank % kGroup;            // position within the pair
    const uint32_t lead = rank - pos;              // rank of the pair's even CTA
    const uint32_t part_rank = rank / kGroup;      // the pair's (or CTA's) k range under kClusterReduce
    const uint32_t parts = ctas / kGroup;          // k ranges per cluster (1 unless kClusterReduce)
    // One work slot per cluster, walking units slot, slot + nslots, ...
    const int64_t nslots = gridDim.x / ctas;
    const int64_t slot0 = blockIdx.x / ctas;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            for (int t = 0; t < kAtoms; ++t) ptx::mbar_init(loaded_bar(s, t), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull_bar(b), 1);
            ptx::mbar_init(accempty_bar(b), kEpiWarps * kGroup);
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(never_bar, 1);
        if (kCluster) {
            ptx::mbar_init(peers_free_bar, parts - 1);
            ptx::mbar_init(received_bar, parts - 1);
        }
        *abort_flag = 0u;
        *issued_count = 0u;
        *producer_done = 0u;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&p.tmap_a);
        ptx::prefetch_tensormap(&p.tmap_b);
        if (p.flags & kFlagTmaStore) ptx::prefetch_tensormap(&p.tmap_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc<kGroup>(ptx::smem_addr(tmem_holder), kTmemCols);
        ptx::tmem_relinquish_alloc_permit<kGroup>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (kGroup == 2 || kCluster)
        ptx::cluster_sync();     // every CTA's barriers initialised before any remote arrive
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // The kernel is launched as a programmatic dependent of whatever precedes
    // it on the stream, so the setup above (barriers, TMEM, descriptor
    // prefetch) overlaps the end of that kernel.  Every thread that touches
    // global memory first waits for that kernel to complete (griddepcontrol.wait):
    // the producer right before its first load, the epilogue warps as they
    // start; the MMA thread never touches global memory, and everything the
    // other roles do comes after the producer's loads.  So the schedule, the
    // first fill's barrier work and the code that does it (its first run)
    // overlap the previous kernel too.  Measured on GB300: computing the first
    // unit after a wait at the top put about 0.9 us between the wait and the
    // first load, and the rest of the first fill's work about 0.5 us more.
    // (The next kernel is let in by the producer once it has issued its last
    // load, below.)
    const Waiter w{abort_flag, abort_addr, rank, ctas, p.wait_limit_ns};
    // Single CTAs (no cluster reduce) free their TMEM as soon as the epilogue
    // has read the last accumulator (warp 1, below), not at the exit: the
    // free then overlaps the C stores and the bulk-store wait.  Measured on
    // GB300, tcgen05.dealloc takes about 230 cycles; back to back, 1024 x 1024
    // x 128 3.45 -> 3.38 us, 512^3 5.24 -> 5.13 us.  Not in the statistics
    // variant, whose epilogue's long reduction follows its last TMEM read:
    // there the waiting MMA thread cost more (1024 x 1024 x 128 7.04-7.19 ->
    // 7.37 us).
    constexpr bool kEarlyFree = kGroup == 1 && !kCluster && !kStats;
    bool tmem_freed = false;

    // The unit of step `it` of this CTA's slot (both CTAs of a pair run the same
    // one; the CTAs or pairs of a kClusterReduce cluster run its k ranges).
    auto slot_unit_at = [&](int64_t it) {
        Unit u = unit_of(slot_unit(slot0, it, nslots, p), p);
        if (kCluster && !u.phantom) {
            u.cpart = static_cast<int32_t>(part_rank);
            u.kb0 = static_cast<int32_t>(part_rank) * p.kb_part;
            u.nkb = p.kb_part;
        }
        return u;
    };
    const int64_t iters = slot_iters(slot0, nslots, p);
    // m-part units cover a half or a quarter of the tile's m range
    const bool quarter_m = p.m_part_rows == kTileM / 4;
    // A rows of this CTA per stage, and their bytes
    const int32_t part_rows_a = quarter_m ? Cfg::kRowsA / 4 : Cfg::kRowsA / 2;
    auto a_bytes = [&](const Unit &un) -> uint32_t {
        if constexpr (kLean != 0) return static_cast<uint32_t>(Cfg::kTileABytes);   // (every unit an m part)
        return un.mpart < 0 ? Cfg::kTileABytes : (quarter_m ? Cfg::kTileABytes / 4 : Cfg::kTileABytes / 2);
    };
    const Unit unit0 = slot_unit_at(0);      // (a phantom when the slot has no unit)
    auto unit_at = [&](int64_t it) { return it == 0 ? unit0 : slot_unit_at(it); };
    const uint32_t flags = p.flags;
    unsigned long long *const clock_probe = p.clock_probe;

    // Where this CTA's loads of a unit go: the A map and its first row m, B's
    // first row n, whether a whole wide tile loads A as two halves, and whether
    // the unit walks its k blocks from the last (odd waves, kFlagAltK).
    struct Boxes {
        const CUtensorMap *map_a;
        int32_t m0, nb;
        bool two_halves, rev;
    };
    auto boxes_of = [&](const Unit &un) {
        const bool cut_m = un.mpart >= 0;
        // A rows of this CTA: one box per stage, or (a whole wide tile) one per half,
        // the second kTileM rows further on.  A wide tile's A map has boxes of one
        // half's rows, which are also an m part's.
        const int32_t rows_a = kWide ? kTileM / kGroup : (cut_m ? part_rows_a : Cfg::kRowsA);
        Boxes b;
        b.map_a = cut_m && !kWide ? &p.tmap_a_part : &p.tmap_a;
        b.two_halves = kWide && !cut_m;
        b.rev = (flags & kFlagAltK) && !un.phantom && un.tile < p.tail_start &&
                ((static_cast<uint32_t>(un.tile) / static_cast<uint32_t>(nslots)) & 1u);
        // a phantom unit reads past the matrices: zero fill, the box's full byte count
        b.m0 = un.phantom ? p.M
                          : static_cast<int32_t>(un.tm * Cfg::kTileMRows + (cut_m ? un.mpart * p.m_part_rows : 0) +
                                                 pos * rows_a);
        b.nb = un.phantom ? p.N : static_cast<int32_t>(un.tn * Cfg::kTileN + pos * Cfg::kRowsB);
        return b;
    };

    // Two kinds of launch whose CTAs often wait below, as programmatic
    // dependents, while the previous kernel drains, prefetch their first fills
    // into L2 before that wait:
    //  - the k ranges of a tile reduced in a cluster (the small grids with a
    //    long K), whose work starts with a stream of its operands: the first
    //    kPrefetchAtoms K atoms of the boxes, if the unit has kPrefetchMinKb k
    //    blocks or more.  Measured on GB300, back to back: 8192 x 16 x 8192
    //    27.44 -> 26.23 us, 4096 x 512 x 8192 31.02 -> 30.63 us, 4096 x 256 x
    //    4096 19.14 -> 18.77 us.  With few k blocks per unit, e.g. 2048 x 2048
    //    x 512, it made calls 2-7 % slower: the prefetches queue ahead of the
    //    loads.
    //  - the lean launches, whose CTAs become resident while the previous
    //    launch runs: the first k block.  Back to back with inputs from HBM,
    //    1024 x 1024 x 128 3.56 -> 3.45 us, 512^3 5.50 -> 5.36 us; four k
    //    blocks gained no more, and with the inputs already in L2 (CUDA-graph
    //    replays) one block costs 0.04-0.1 us and four 0.05-0.2 us.
    // A prefetch returns no data to the CTA, so it cannot read ahead of the
    // previous kernel's writes: the loads after the wait read through L2, which
    // every write reaches first.
    if ((kCluster || kLean) && warp == 0 && lane == 0 && !unit0.phantom && (kLean || unit0.nkb >= kPrefetchMinKb)) {
        const Boxes bx = boxes_of(unit0);
        constexpr int kFills = kLean ? 1 : kPrefetchAtoms / Cfg::kAtoms;
        for (int i = 0; i < kFills; ++i) {
            const int kb = bx.rev ? unit0.kb0 + unit0.nkb - 1 - i : unit0.kb0 + i;
            if (kb >= p.num_kb) continue;   // (the zero-filled end of a last k range)
#pragma unroll
            for (int t = 0; t < Cfg::kAtoms; ++t) {
                const int32_t k0 = (kb * Cfg::kAtoms + t) * kBlockKElems;
                if (k0 >= p.K) break;
                if (bx.nb < p.N) ptx::tma_prefetch_2d(&p.tmap_b, k0, bx.nb);
                if (bx.m0 < p.M) ptx::tma_prefetch_2d(bx.map_a, k0, bx.m0);
                if (bx.two_halves && bx.m0 + kTileM < p.M) ptx::tma_prefetch_2d(bx.map_a, k0, bx.m0 + kTileM);
            }
        }
    }

    const bool probe_clock = clock_probe != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
    const uint64_t probe_c0 = probe_clock ? ptx::clock64() : 0, probe_t0 = probe_clock ? ptx::globaltimer() : 0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (every CTA)
        // 1 CTA: loads complete on the CTA's own loaded[s].  Pairs: every load
        // meant for a CTA completes on loaded[s] of that CTA's pair leader,
        // which its own producer arms with the bytes of the whole pair; the MMA
        // thread waits on that one barrier.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t n_issued = 0;
            bool ok = true;
            const uint32_t stall = rank == 0 ? kFlagStallProducer0 : (rank == 1 ? kFlagStallProducer1 : 0u);

            if (flags & stall) ok = w.wait(never_bar, 0u, kSiteStall);
            for (int64_t it = 0; ok && it < iters; ++it) {
                const Unit un = unit_at(it);
                const Boxes bx = boxes_of(un);
                const bool two_halves = bx.two_halves;
                const uint32_t fill = Cfg::kTileBBytes + a_bytes(un);
                const CUtensorMap *map_a = bx.map_a;
                const int32_t m0 = bx.m0, nb = bx.nb;
                for (int i = 0; i < un.nkb; ++i) {
                    const int kb = bx.rev ? un.kb0 + un.nkb - 1 - i : un.kb0 + i;
                    if (!w.wait(empty_bar(stage), phase ^ 1u, kSiteEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s_b = s_ring + stage * Cfg::kStageBytes;
                    const uint32_t s_a = s_b + Cfg::kTileBBytes;
                    if (n_issued == 0) ptx::griddep_wait();   // this thread's first global access
                    if constexpr (kGroup == 2) {
#pragma unroll
                        for (int t = 0; t < Cfg::kAtoms; ++t) {
                            if (pos == 0) ptx::mbar_arrive_expect_tx(loaded_bar(stage, t), 2 * fill / kAtoms);
                            const uint32_t lb = ptx::mapa_shared(loaded_bar(stage, t), lead);
                            const int32_t k0 = (kb * Cfg::kAtoms + t) * kBlockKElems;
                            ptx::tma_load_2d_pair(s_b + t * Cfg::kAtomBBytes, &p.tmap_b, lb, k0, nb);
                            ptx::tma_load_2d_pair(s_a + t * Cfg::kAtomABytes, map_a, lb, k0, m0);
                            if (two_halves)
                                ptx::tma_load_2d_pair(s_a + t * Cfg::kAtomABytes + Cfg::kHalfABytes, map_a, lb, k0,
                                                      m0 + kTileM);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < Cfg::kAtoms; ++t) {
                            const int32_t k0 = (kb * Cfg::kAtoms + t) * kBlockKElems;
                            ptx::mbar_arrive_expect_tx(loaded_bar(stage, t), fill / kAtoms);
                            ptx::tma_load_2d(s_b + t * Cfg::kAtomBBytes, &p.tmap_b, loaded_bar(stage, t), k0, nb);
                            ptx::tma_load_2d(s_a + t * Cfg::kAtomABytes, map_a, loaded_bar(stage, t), k0, m0);
                        }
                    }
                    *issued_count = ++n_issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // This CTA issues no more loads: the next kernel on the stream may
            // start its setup (it too waits for this grid to complete before it
            // touches memory).  Not earlier: a dependent's CTAs that wait on SMs
            // beside this grid's for a whole launch slowed it (by 2 % for a
            // 305 us FP8 GEMM followed by the quantiser).  A single thread's
            // signal counts for its CTA, else the CTA's exit does.  (A producer
            // that issued no load still waits first: this thread updates the
            // clock probe as the CTA leaves.)
            if (n_issued == 0) ptx::griddep_wait();
            ptx::griddep_launch_dependents();
            if constexpr (kGroup == 2) {
                // publish the final count (release: the count store is ordered before it)
                ptx::st_release_cluster_u32(ptx::mapa_shared(done_addr, rank), 1u);
                if (pos == 0) {
                    // bytes producer q sent to this leader for fill number i (both
                    // CTAs of the pair run the same unit, so the same bytes)
                    auto contribution = [&](uint32_t, uint32_t i) -> uint32_t {
                        // a split first step issues kb_part fills, every other step num_kb
                        const uint32_t first =
                            ((p.tail_mode == kTailSplitK || p.tail_mode == kSplitReduce) && slot_has_tail(slot0, p))
                                ? static_cast<uint32_t>(p.kb_part)
                                : static_cast<uint32_t>(p.num_kb);
                        const int64_t it = i < first ? 0 : 1 + static_cast<int64_t>((i - first) / p.num_kb);
                        return a_bytes(slot_unit_at(it)) + Cfg::kTileBBytes;
                    };
                    drain_cluster_loads<kStages, kAtoms, Cfg::kCtas>(w, loaded_bar, contribution, n_issued, count_addr,
                                                                     done_addr, lead);
                }
            } else {
                // Let every issued load land before the CTA can exit.
                for (int s = 0; s < kStages; ++s) {
                    const uint32_t passes =
                        n_issued / kStages + (static_cast<uint32_t>(s) < n_issued % kStages ? 1u : 0u);
                    for (int t = 0; t < kAtoms && passes; ++t) w.drain(loaded_bar(s, t), (passes - 1) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        bool free_now = false;
        if (lane == 0 && pos == 0) {
            // ------------------------------------------------ MMA issuer (even CTA of each pair)
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int64_t units_done = 0;        // accumulators committed
            bool ok = true, issued_any = false;
            const uint16_t all_mask = static_cast<uint16_t>(((1u << kGroup) - 1u) << lead);   // both CTAs of the pair
            const uint16_t pair_mask = all_mask;
            // m-part units: MMA N = m_part_rows
            constexpr uint32_t kIdescHalf = ptx::idesc_f32acc(Cfg::kTileN, kTileM / 2, Kind::kFmt, Kind::kFmt);
            constexpr uint32_t kIdescQuarter = ptx::idesc_f32acc(Cfg::kTileN, kTileM / 4, Kind::kFmt, Kind::kFmt);
            // (a wide tile's m parts are its halves: MMA N = 256)
            const uint32_t idesc_part = kWide ? kIdesc : (quarter_m ? kIdescQuarter : kIdescHalf);
            if (flags & kFlagStallMma) ok = w.wait(never_bar, 0u, kSiteStall);
            if constexpr (kWide) {
                // 256 x 512 tiles.  The epilogue hands the accumulator back one half at a
                // time (accempty[0], then accempty[1]), each as soon as it has read that
                // half into registers.  A whole tile's first MMAs need only half 0:
                // while half 1 is still being read, stages are held with only their
                // half-0 MMAs issued (at most kStages - 1, so the producer can always
                // fill the next one); once half 1 is back, the held stages' half-1 MMAs
                // are issued in order and each stage is freed after its own.  An m-part
                // unit uses half 0 only and waits for both halves.
                auto advance = [&](int &s, uint32_t &ph) {
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                };
                auto issue_half = [&](int s, int kk, int h) {
                    const uint32_t s_b = s_ring + s * Cfg::kStageBytes;
                    const uint64_t desc_b = ptx::desc_kmajor_sw128(s_b);
                    const uint64_t desc_a = ptx::desc_kmajor_sw128(s_b + Cfg::kTileBBytes + h * Cfg::kHalfABytes);
#pragma unroll
                    for (int j = 0; j < kBlockKBytes / kMmaKBytes; ++j)
                        Kind::template mma<kGroup>(tmem_base + h * kTileM, desc_b + 2u * j, desc_a + 2u * j, kIdesc,
                                                   (kk | j) != 0 ? 1u : 0u);
                };
                for (int64_t it = 0; ok && it < iters; ++it) {
                    const Unit un = unit_at(it);
                    const bool two = un.mpart < 0;
                    if (!w.wait(accempty_bar(0), acc_phase ^ 1u, kSiteAccEmpty)) break;
                    bool h1 = false;
                    if (!two) {
                        if (!w.wait(accempty_bar(1), acc_phase ^ 1u, kSiteAccEmpty)) break;
                        h1 = true;
                    }
                    ptx::tc_fence_after_sync();
                    int held = 0, h_stage = 0, h_kk = 0;
                    uint32_t h_phase = 0;
                    auto flush = [&]() {
                        ptx::tc_fence_after_sync();      // after the wait that returned half 1
                        for (int q = 0; q < held; ++q) {
                            issue_half(h_stage, h_kk + q, 1);
                            ptx::mma_commit<kGroup>(empty_bar(h_stage), all_mask);
                            advance(h_stage, h_phase);
                        }
                        held = 0;
                    };
                    for (int kk = 0; kk < un.nkb; ++kk) {
                        if (!w.wait(loaded_bar(stage, 0), phase, kSiteLoaded)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        issue_half(stage, kk, 0);
                        issued_any = true;
                        if (two && !h1) h1 = ptx::mbar_try_wait(accempty_bar(1), acc_phase ^ 1u);
                        if (two && !h1 && held + 1 < kStages) {
                            if (held == 0) {
                                h_stage = stage;
                                h_phase = phase;
                                h_kk = kk;
                            }
                            ++held;
                            advance(stage, phase);
                            continue;
                        }
                        if (two && !h1) {
                            if (!w.wait(accempty_bar(1), acc_phase ^ 1u, kSiteAccEmpty)) {
                                ok = false;
                                break;
                            }
                            h1 = true;
                        }
                        if (two) {
                            flush();
                            issue_half(stage, kk, 1);
                        }
                        ptx::mma_commit<kGroup>(empty_bar(stage), all_mask);   // stage free for every CTA that writes it
                        advance(stage, phase);
                    }
                    if (!ok) break;
                    if (held > 0) {                      // fewer k blocks than held stages: half 1 last
                        if (!h1 && !w.wait(accempty_bar(1), acc_phase ^ 1u, kSiteAccEmpty)) break;
                        flush();
                    }
                    ptx::mma_commit<kGroup>(accfull_bar(0), pair_mask);      // accumulator complete
                    acc_phase ^= 1u;
                }
            } else
            for (int64_t it = 0; ok && it < iters; ++it) {
                const Unit un = unit_at(it);
                const uint32_t idesc = un.mpart >= 0 ? idesc_part : kIdesc;
                if (!w.wait(accempty_bar(acc), acc_phase ^ 1u, kSiteAccEmpty)) break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kAccCols;
                for (int kk = 0; kk < un.nkb; ++kk) {
                    const uint32_t s_b = s_ring + stage * Cfg::kStageBytes;
                    const uint32_t s_a = s_b + Cfg::kTileBBytes;
#pragma unroll
                    for (int t = 0; t < Cfg::kAtoms; ++t) {
                        if (!w.wait(loaded_bar(stage, t), phase, kSiteLoaded)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        const uint64_t desc_b = ptx::desc_kmajor_sw128(s_b + t * Cfg::kAtomBBytes);
                        // a whole wide tile: both halves (the second half's A rows and
                        // accumulator columns follow the first's); otherwise one
                        const int halves = kWide && un.mpart < 0 ? 2 : 1;
#pragma unroll
                        for (int h = 0; h < Cfg::kHalves; ++h) {
                            if (h >= halves) break;
                            const uint64_t desc_a =
                                ptx::desc_kmajor_sw128(s_a + t * Cfg::kAtomABytes + h * Cfg::kHalfABytes);
#pragma unroll
                            for (int j = 0; j < kBlockKBytes / kMmaKBytes; ++j) {
                                // +32 bytes along K inside the 128-byte swizzle span = +2 in the address field
                                Kind::template mma<kGroup>(d_tmem + h * kTileM, desc_b + 2u * j, desc_a + 2u * j, idesc,
                                                           (kk | t | j) != 0 ? 1u : 0u);
                            }
                        }
                        issued_any = true;
                    }
                    if (!ok) break;
                    ptx::mma_commit<kGroup>(empty_bar(stage), all_mask);   // stage free for every CTA that writes it
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit<kGroup>(accfull_bar(acc), pair_mask);      // accumulator complete
                ++units_done;
                if (kWide || ++acc == 2) {          // a wide tile's accumulator is not double-buffered
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // All MMAs this thread issued must finish before TMEM is freed.
            bool drained = true;
            if (issued_any) {
                ptx::mma_commit<kGroup>(drain_bar, static_cast<uint16_t>(1u << rank));
                drained = w.drain(drain_bar, 0u);
            }
            if constexpr (kEarlyFree) {
                // Wait for the epilogue's last release of each accumulator buffer:
                // buffer b held units b, b + 2, ..., so its release number u_b
                // completes phase u_b - 1 of accempty[b] (this thread has seen
                // release u_b - 1 already, before the buffer's last use).
                free_now = ok && drained && units_done == iters;
                for (int b = 0; b < 2 && free_now; ++b) {
                    const int64_t uses = (units_done + 1 - b) / 2;
                    if (uses > 0)
                        free_now = w.wait(accempty_bar(b), static_cast<uint32_t>((uses - 1) & 1), kSiteAccEmpty);
                }
            }
        }
        if constexpr (kEarlyFree) {
            // every TMEM read of the epilogue is done: free the columns now
            free_now = __shfl_sync(0xffffffffu, free_now, 0);
            if (free_now) {
                ptx::tc_fence_after_sync();
                ptx::tmem_dealloc<kGroup>(tmem_base, kTmemCols);
                tmem_freed = true;
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, every CTA)
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31 are this warp's
        const int ew = warp - 2;
        const int row = 32 * quarter + lane;      // this thread's TMEM lane = output column within the CTA
        const bool tma_store = (flags & kFlagTmaStore) != 0;
        volatile uint32_t *second_flag = tmem_holder + 4;   // split-K: this CTA's half came second
        // The device scales may have been written by the previous kernel (the
        // quantiser): these warps wait for it before their first global access.
        ptx::griddep_wait();
        const float scale = p.scale_a_ptr ? __fmul_rn(__ldg(p.scale_a_ptr), __ldg(p.scale_b_ptr)) : p.scale;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t chunk_ctr = 0;

        // Hands accumulator barrier b's TMEM columns back to the MMA thread (after
        // their last TMEM read).
        auto release_bar = [&](int b) {
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (kGroup == 2)
                    ptx::mbar_arrive_remote(ptx::mapa_shared(accempty_bar(b), lead));
                else
                    ptx::mbar_arrive(accempty_bar(b));
            }
        };
        // The whole accumulator: a wide tile's is two halves with a barrier each.
        auto release_acc = [&]() {
            if constexpr (kWide) {
                release_bar(0);
                release_bar(1);
            } else {
                release_bar(acc);
            }
        };
        // Reads 64 accumulator columns (this thread's lane) starting at column `col`.
        auto load_chunk = [&](uint32_t t_row, int col, float (&v)[64]) {
            uint32_t r0[32], r1[32];
            ptx::tmem_ld_32x32b_x32(t_row + col, r0);
            ptx::tmem_ld_32x32b_x32(t_row + col + 32, r1);
            ptx::tmem_ld_wait(r0);
            ptx::reg_dependency(r1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v[j] = __uint_as_float(r0[j]);
                v[32 + j] = __uint_as_float(r1[j]);
            }
        };
        // Converts 64 values of rows mc .. mc+63 of output column (nw + lane) to
        // 16-bit pairs, and stores them: TMA store for m < m_tma, direct stores
        // for the rest.
        auto pack_chunk = [&](const float (&v)[64], uint32_t (&packed)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) packed[j] = Kind::pack(v[2 * j], v[2 * j + 1], scale);
        };
        auto store_packed = [&](const uint32_t (&packed)[32], int32_t mc, int32_t nw) {
            if (tma_store && mc < p.m_tma) {
                const uint32_t buf = s_epi + (ew * kEpiBufs + (chunk_ctr & 1u)) * kEpiBufBytes;
                if (lane == 0) ptx::bulk_wait_group_read<kEpiBufs - 1>();   // buffer's previous store has read it
                __syncwarp();
                // row = lane (one output column n), 8 chunks of 16 B, 128-byte swizzle
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t addr = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
                    ptx::st_shared_v4(addr, packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&p.tmap_c, buf, mc, nw);   // clipped at m_tma and N
                    ptx::bulk_commit_group();
                }
                ++chunk_ctr;
            }
            if (mc + kEpiBoxM > p.m_tma) {
                // Direct stores with bounds: rows m_tma <= m < M (the ragged tail TMA cannot
                // clip at element granularity, or all of C when C is not TMA-addressable).
                const int64_t n = nw + lane;
                const int32_t lo = mc > p.m_tma ? mc : p.m_tma;
                if (n < p.N) {
                    uint16_t *col = static_cast<uint16_t *>(p.c_ptr) + n * p.ldc;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int32_t m = mc + 2 * j;
                        if (m >= lo && m < p.M) col[m] = static_cast<uint16_t>(packed[j] & 0xFFFFu);
                        if (m + 1 >= lo && m + 1 < p.M) col[m + 1] = static_cast<uint16_t>(packed[j] >> 16);
                    }
                }
            }
        };
        auto store_chunk = [&](const float (&v)[64], int32_t mc, int32_t nw) {
            uint32_t packed[32];
            pack_chunk(v, packed);
            store_packed(packed, mc, nw);
        };

        for (int64_t it = 0; it < iters; ++it) {
            const Unit un = unit_at(it);
            bool ok = w.wait(accfull_bar(acc), acc_phase, kSiteAccFull);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            __syncwarp();
            ptx::tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + acc * kAccCols;
            const int32_t m_in_tile = un.mpart >= 0 ? un.mpart * p.m_part_rows : 0;   // the unit's first row m
            const int32_t m0 = static_cast<int32_t>(un.tm * Cfg::kTileMRows) + m_in_tile;
            // this warp's first output column
            const int32_t nw = static_cast<int32_t>(un.tn * Cfg::kTileN + pos * Cfg::kRowsB) + 32 * quarter;
            if (un.phantom) {
                release_acc();   // nothing to store
            } else if (kCluster && un.cpart >= 0) {
                // kClusterReduce: this CTA holds the partial sum of k range `me` of its
                // 128 rows n of the tile (a CTA pair's tile has two such CTAs, one per
                // position; the exchange runs between the CTAs of one position).  Of
                // the tile's four 64-column chunks of m, chunk c belongs to range
                // c % S, whose CTA adds the S partials of it in range order and stores
                // it.  This CTA's shared-memory ring is free once its MMAs are done;
                // slot j of it receives the owned chunks' partials of the range with
                // the j-th index other than `me` (per chunk 128 rows n of 64 floats,
                // 16-byte units swizzled by row).  Only rows n < N are sent; the
                // others are never stored.
                const uint32_t S = parts, me = part_rank;
                auto peer = [&](uint32_t q) { return q * kGroup + pos; };   // the CTA of range q
                constexpr uint32_t kChunkBytes = Cfg::kRowsB * kEpiBoxM * 4;       // 32 KiB
                const uint32_t slot_bytes = ((kTileM / kEpiBoxM + S - 1) / S) * kChunkBytes;
                const uint32_t row_off = static_cast<uint32_t>(row * kEpiBoxM * 4);
                const bool valid_n = nw + lane < p.N;
                // Whether any of this warp's 32 columns n is below N.  A warp with none
                // (the 8192 x 16 problem: three of four) sends, adds and stores nothing,
                // which leaves the CTA's shared-memory bandwidth to the warp that does.
                const bool warp_rows = nw < p.N;
                auto swz = [&](int c16) { return static_cast<uint32_t>((c16 ^ (row & 7)) << 4); };
                if (warp == 2 && lane == 0) {
                    // the ring was last written by TMA and read by the tensor cores
                    ptx::fence_proxy_async_smem();
                    for (uint32_t q = 0; q < S; ++q)
                        if (q != me) ptx::mbar_arrive_remote(ptx::mapa_shared(peers_free_bar, peer(q)));
                }
                bool fine = __all_sync(0xffffffffu, w.wait(peers_free_bar, 0u, kSitePeersFree));
                if (fine) {
                    for (uint32_t d = 1; warp_rows && d < S; ++d) {
                        const uint32_t q = (me + d) % S;
                        const uint32_t j = me < q ? me : me - 1;    // this CTA's slot in q's ring
                        const uint32_t dst = ptx::mapa_shared(s_ring + j * slot_bytes + row_off, peer(q));
#pragma unroll 1
                        for (uint32_t c = q, oc = 0; c < kTileM / kEpiBoxM; c += S, ++oc) {
                            float v[64];
                            load_chunk(t_row, static_cast<int>(c) * kEpiBoxM, v);
                            if (valid_n) {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    ptx::st_shared_cluster_v4(dst + oc * kChunkBytes + swz(i), v[4 * i], v[4 * i + 1],
                                                              v[4 * i + 2], v[4 * i + 3]);
                            }
                        }
                    }
                    // every epilogue thread's stores are ordered before one
                    // cluster-scope release per peer
                    ptx::named_barrier_sync(1, kEpiWarps * 32);
                    if (warp == 2 && static_cast<uint32_t>(lane) < S && static_cast<uint32_t>(lane) != me)
                        ptx::mbar_arrive_remote_release_cluster(ptx::mapa_shared(received_bar, peer(lane)));
                    fine = __all_sync(0xffffffffu, w.wait_cluster(received_bar, 0u, kSiteReceived));
                }
                if (!fine) {
                    release_acc();
                    break;
                }
                if (!warp_rows) release_acc();   // (the loop below is this warp's last read otherwise)
#pragma unroll 1
                for (uint32_t c = me, oc = 0; warp_rows && c < kTileM / kEpiBoxM; c += S, ++oc) {
                    const int col = static_cast<int>(c) * kEpiBoxM;
                    float v[64];
                    // the S partials added in range order
#pragma unroll 1
                    for (uint32_t q = 0; q < S; ++q) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float t[32];
                            if (q == me) {
                                uint32_t x[32];
                                ptx::tmem_ld_32x32b_x32(t_row + col + 32 * h, x);
                                ptx::tmem_ld_wait(x);
#pragma unroll
                                for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(x[i]);
                            } else {
                                const uint32_t src =
                                    s_ring + (q - (q > me ? 1u : 0u)) * slot_bytes + oc * kChunkBytes + row_off;
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float4 f = ptx::ld_shared_v4_f32(src + swz(8 * h + i));
                                    t[4 * i] = f.x;
                                    t[4 * i + 1] = f.y;
                                    t[4 * i + 2] = f.z;
                                    t[4 * i + 3] = f.w;
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[32 * h + i] = q == 0 ? t[i] : v[32 * h + i] + t[i];
                        }
                    }
                    if (c + S >= kTileM / kEpiBoxM) release_acc();   // this CTA's last read of its accumulator
                    store_chunk(v, m0 + col, nw);
                }
            } else if (un.kpart >= 0) {
                // Split-reduce part: store this part's FP32 partial; the reduce
                // kernel that follows sums the parts in order and stores C.  Only
                // the columns n < N (a few rows of a skinny problem's partial): the
                // reduce kernel reads no others.  A wide tile hands each half of
                // its accumulator back once read.
                constexpr int kRowM = Cfg::kTileMRows;          // floats of one column n's partial
                constexpr int kChunks = kRowM / kEpiBoxM;
                const int64_t span = static_cast<int64_t>(Cfg::kRowsB) * kRowM;
                float *mine = p.split_ws +
                              (((un.tm * p.tiles_n + un.tn) * p.split_parts + un.kpart) * kGroup + pos) * span +
                              row * kRowM;
                const bool valid_n = nw + lane < p.N;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    float v[64];
                    load_chunk(t_row, c * kEpiBoxM, v);
                    if (kWide && c == kChunks / 2 - 1) release_bar(0);
                    if (c == kChunks - 1) {
                        if constexpr (kWide)
                            release_bar(1);
                        else
                            release_acc();
                    }
                    if (valid_n) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            reinterpret_cast<float4 *>(mine + c * kEpiBoxM)[j] =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
            } else if (!kWide && un.khalf >= 0) {
                // Split-K half: store this half's FP32 partial, then take the tile's
                // ticket.  The half that comes second adds the other half's partial
                // (fp32 addition commutes, so either order gives the same C) and
                // stores C; no CTA ever waits for another.  One thread's
                // acquire-release add releases this CTA's partial (the barrier orders
                // every warp's writes before it) and acquires the other half's (the
                // barrier orders the reads after it).
                const int64_t t = un.tile - p.tail_start;
                const int64_t span = static_cast<int64_t>(Cfg::kRowsB) * kTileM;
                float *mine = p.split_ws + ((t * 2 + un.khalf) * kGroup + pos) * span + row * kTileM;
                const float *other = p.split_ws + ((t * 2 + (un.khalf ^ 1)) * kGroup + pos) * span + row * kTileM;
#pragma unroll 1
                for (int c = 0; c < kTileM / kEpiBoxM; ++c) {
                    float v[64];
                    load_chunk(t_row, c * kEpiBoxM, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        reinterpret_cast<float4 *>(mine + c * kEpiBoxM)[j] =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
                ptx::named_barrier_sync(1, kEpiWarps * 32);
                if (warp == 2 && lane == 0) {
                    unsigned long long *ticket = p.split_tickets + t * kGroup + pos;
                    const bool second = ptx::atom_add_acq_rel_gpu(ticket, 1ull) == 1ull;
                    if (second) atomicExch(ticket, 0ull);     // both halves are in: ready for the next launch
                    *second_flag = second ? 1u : 0u;
                }
                ptx::named_barrier_sync(1, kEpiWarps * 32);
                if (*second_flag == 0u) {
                    release_acc();
                } else {
#pragma unroll 1
                    for (int c = 0; c < kTileM / kEpiBoxM; ++c) {
                        float v[64];
                        load_chunk(t_row, c * kEpiBoxM, v);
                        if (c == kTileM / kEpiBoxM - 1) release_acc();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float4 o = ptx::ld_global_cg_v4(other + c * kEpiBoxM + 4 * j);
                            v[4 * j] += o.x;
                            v[4 * j + 1] += o.y;
                            v[4 * j + 2] += o.z;
                            v[4 * j + 3] += o.w;
                        }
                        store_chunk(v, m0 + c * kEpiBoxM, nw);
                    }
                }
            } else {
                // (a wide tile's m parts are its 256-row halves)
                const int n_chunks = un.mpart < 0 ? Cfg::kTileMRows / kEpiBoxM
                                                  : (kWide ? kTileM : (quarter_m ? kTileM / 4 : kTileM / 2)) / kEpiBoxM;
                const bool stats = kStats && (flags & kFlagStats) != 0;
                if (kWide && un.mpart < 0) {
                    // A whole wide tile, half by half: the first two chunks of the half go
                    // through the staging buffers, the last two are read into registers
                    // (16-bit pairs); then the half is handed back, so the next tile's MMAs
                    // on it can start while this warp stores those two.
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const int c0 = 4 * h;
#pragma unroll 1
                        for (int c = c0; c < c0 + 2; ++c) {
                            float v[64];
                            load_chunk(t_row, c * kEpiBoxM, v);
                            store_chunk(v, m0 + c * kEpiBoxM, nw);
                        }
                        uint32_t pk0[32], pk1[32];
                        {
                            float v[64];
                            load_chunk(t_row, (c0 + 2) * kEpiBoxM, v);
                            pack_chunk(v, pk0);
                        }
                        {
                            float v[64];
                            load_chunk(t_row, (c0 + 3) * kEpiBoxM, v);
                            pack_chunk(v, pk1);
                        }
                        release_bar(h);
                        store_packed(pk0, m0 + (c0 + 2) * kEpiBoxM, nw);
                        store_packed(pk1, m0 + (c0 + 3) * kEpiBoxM, nw);
                    }
                } else
#pragma unroll 1
                for (int c = 0; c < n_chunks; ++c) {
                    float v[64];
                    load_chunk(t_row, c * kEpiBoxM, v);
                    if (c == n_chunks - 1) release_acc();   // last read of this accumulator
                    if constexpr (!Kind::kF8) {
                        if (stats) {
#pragma unroll
                            for (int j = 0; j < 64; ++j) v[j] = __fmul_rn(v[j], p.scale);
                        }
                    }
                    bool stored = false;
                    if constexpr (!Kind::kF8) {
                        if (stats) {
                            // C's 16-bit values first: the FP32 scores are dead once staged below.
                            uint32_t packed[32];
                            pack_chunk(v, packed);
                            // This warp's (max, sum) over its 32 columns n, for each of the chunk's
                            // 64 rows m, through its two staging buffers (8 KiB): each lane (a
                            // column n) writes its 64 scores as one row, then lane l reduces rows
                            // l and 32 + l over the 32 columns in registers.  The 16-byte unit i
                            // of row n sits at unit i ^ (n & 15), so neither the row writes nor
                            // the column reads meet a bank conflict.  (Measured on GB300, the same
                            // reduction by halving shuffle exchanges took 0.96 us per 32 rows.)
                            const bool valid = nw + lane < p.N;
                            const uint32_t sbuf = s_epi + ew * kEpiBufs * kEpiBufBytes;
                            if (lane == 0) ptx::bulk_wait_group_read<0>();   // earlier C stores have read both
                            __syncwarp();
                            constexpr uint32_t kNegInf = 0xFF800000u;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const uint32_t a = sbuf + lane * (kEpiBoxM * 4) + ((i ^ (lane & 15)) << 4);
                                ptx::st_shared_v4(a, valid ? __float_as_uint(v[4 * i]) : kNegInf,
                                                  valid ? __float_as_uint(v[4 * i + 1]) : kNegInf,
                                                  valid ? __float_as_uint(v[4 * i + 2]) : kNegInf,
                                                  valid ? __float_as_uint(v[4 * i + 3]) : kNegInf);
                            }
                            __syncwarp();
                            float2 *part = p.stat_parts +
                                           (static_cast<int64_t>(un.tm) * p.stat_ctas * kEpiWarps +
                                            (un.tn * kGroup + pos) * kEpiWarps + quarter) * kTileM;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int m = 32 * h + lane;     // this lane's row within the chunk
                                float x[32];
#pragma unroll
                                for (int n = 0; n < 32; ++n)
                                    x[n] = ptx::ld_shared_f32(sbuf + n * (kEpiBoxM * 4) + (((m >> 2) ^ (n & 15)) << 4) +
                                                              (m & 3) * 4);
                                part[m_in_tile + c * kEpiBoxM + m] = stat_row32(x);
                            }
                            __syncwarp();   // every lane's reads are done before the C store reuses the buffers
                            store_packed(packed, m0 + c * kEpiBoxM, nw);
                            stored = true;
                        }
                    }
                    if (!stored) store_chunk(v, m0 + c * kEpiBoxM, nw);
                }
                if constexpr (!Kind::kF8) {
                    if (stats) {
                        // Take the ticket of this unit's rows (its tile row and m part); the CTA
                        // that comes last merges every part of those rows in a fixed order, so
                        // no CTA waits for another.  One thread's acquire-release add releases
                        // the CTA's parts (the barrier orders every warp's writes before it)
                        // and acquires the other CTAs' for the merge (the barrier orders the
                        // merge after it).  Measured on GB300, fences on both sides of a
                        // relaxed add cost 0.75 us more per 1024 x 1024 x 128 call.
                        ptx::named_barrier_sync(1, kEpiWarps * 32);
                        if (warp == 2 && lane == 0) {
                            unsigned long long *ticket =
                                p.stat_tickets + un.tm * kMaxMParts + (un.mpart >= 0 ? un.mpart : 0);
                            const bool last = ptx::atom_add_acq_rel_gpu(ticket, 1ull) ==
                                              static_cast<unsigned long long>(p.stat_ctas - 1);
                            if (last) atomicExch(ticket, 0ull);   // the rows are complete: ready for the next launch
                            *second_flag = last ? 1u : 0u;
                        }
                        ptx::named_barrier_sync(1, kEpiWarps * 32);
                        if (*second_flag != 0u) {
                            const int nparts = p.stat_ctas * kEpiWarps;
                            const float2 *row_parts =
                                p.stat_parts + static_cast<int64_t>(un.tm) * nparts * kTileM;
                            // thread t merges rows m_in_tile + t (+ 128): 32 parts of a row in flight
                            const int rows = un.mpart >= 0 ? p.m_part_rows : kTileM;
                            constexpr int kBatch = 32;
                            const int t = ew * 32 + lane;
#pragma unroll 1
                            for (int r = t; r < rows; r += kEpiWarps * 32) {
                                const int row = m_in_tile + r;
                                float mx = -INFINITY, sm = 0.0f;
#pragma unroll 1
                                for (int q0 = 0; q0 < nparts; q0 += kBatch) {
                                    float2 buf[kBatch];
#pragma unroll
                                    for (int i = 0; i < kBatch; ++i)
                                        buf[i] = q0 + i < nparts
                                                     ? __ldcg(row_parts + static_cast<int64_t>(q0 + i) * kTileM + row)
                                                     : make_float2(-INFINITY, 0.0f);
#pragma unroll
                                    for (int i = 0; i < kBatch; ++i) stat_merge(mx, sm, buf[i].x, buf[i].y);
                                }
                                const int64_t m = static_cast<int64_t>(un.tm) * kTileM + row;
                                if (m < p.M) {
                                    p.row_max[m] = mx;
                                    p.row_sum[m] = sm;
                                }
                            }
                        }
                    }
                }
            }
            if (kWide || ++acc == 2) {          // a wide tile's accumulator is not double-buffered
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // Before the CTA leaves, its staging buffers must have been read by the
        // TMA stores; the stores themselves complete before the grid does.
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
    }

    __syncwarp();                // .aligned barriers below need converged warps
    ptx::tc_fence_before_sync();
    if constexpr (kGroup == 2 || kCluster)
        ptx::cluster_sync();     // no CTA leaves while another may still touch its shared memory
    else
        __syncthreads();
    if (warp == 1 && !tmem_freed) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<kGroup>(tmem_base, kTmemCols);
    }
    if (probe_clock) {
        atomicAdd(&clock_probe[0], static_cast<unsigned long long>(ptx::clock64() - probe_c0));
        atomicAdd(&clock_probe[1], static_cast<unsigned long long>(ptx::globaltimer() - probe_t0));
        atomicAdd(&clock_probe[2], 1ull);
    }
}

}  // namespace tn
