// tn_gemm.cu -- host side of the C ABI declared in include/tn_gemm.h:
// argument validation, per-device state, TMA tensor-map encoding, the
// repack path for operands TMA cannot address, and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <memory>
#include <mutex>
#include <shared_mutex>
#include <unordered_map>
#include <vector>

#include "tn_gemm.h"
#include "tn_gemm_kernel.cuh"
#include "skinny_kernel.cuh"
#include "aux_kernels.cuh"
#include "repack_kernel.cuh"
#include "quant_e4m3_kernel.cuh"

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 256;   // TMA coordinates are signed 32-bit
constexpr int kMaxDevices = 64;
constexpr int kGroupM = 8;                               // tile rows per raster group
// The lean configuration (two CTAs per SM) for launches of m-part units
// that fill more than half of the slots, up to this many k blocks: quarters
// (a ring of three stages) and halves (two stages).  Measured on GB300, back
// to back with inputs from HBM, full -> lean: 1024 x 1024 x 128 3.89 -> 3.40
// us, x 512 5.64 -> 5.30, but x 1984 12.11 -> 13.44; 2048 x 1024 x 128 4.24
// -> 3.74, x 256 4.86 -> 4.73, but x 512 6.01 -> 6.85.  Launches of at most
// half the slots leave room for the next launch's CTAs beside them anyway,
// and there the deeper ring of the full configuration was as fast or faster
// (512^3 5.20 -> 5.32, 1024 x 512 x 1024 7.46 -> 7.96).
constexpr int kLeanQuarterMaxKb = 8;
// The skinny kernel (N <= 64) by default up to this many 128-byte k blocks.
// Measured on GB300, back to back with inputs from HBM, general -> skinny:
// 8192 x 8 x 2048 14.64 -> 10.52 us, 8192 x 16 x 512 8.61 -> 6.86, 32768 x 16
// x 1024 16.29 -> 14.54, 4096 x 16 x 4096 12.27 -> 11.40, 1024 x 16 x 1024
// 7.40 -> 6.53; but with 128 k blocks 8192 x 16 x 8192 26.02 -> 26.58, 8192 x
// 64 x 8192 28.43 -> 30.23, 2048 x 16 x 8192 13.23 -> 14.25.
constexpr int kSkinnyMaxKb = 64;
constexpr int kLeanHalfMaxKb = 4;
// Odd waves walk K backwards (kFlagAltK).  Measured on GB300 at 8192^3 (256 x
// 512 tiles, FP16, under the power cap): DRAM reads 815 -> 684 MB per launch,
// 1612 -> 1626 TFLOP/s; E4M3 3212 -> 3225.
constexpr bool kAltKDefault = true;

// replays, GPU time only) 1024 x 1024 x 128 4.19 -> 4.31 us, 512^3 6.07 ->

thread_local char t_last_error[512] = "";

gemm_status_t fail(gemm_status_t s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return s;
}

struct DeviceState {
    bool ready = false;
    int sms = 0, major = 0, minor = 0;
    // per kernel, indexed [kind: f16, e4m3][1: one CTA, 2: CTA pairs, 3: CTA pairs with 256 x 512 tiles,
    // 4 / 5: one CTA / CTA pairs in k-range clusters]
    bool smem_attr[2][10] = {};
    int max_clusters[2][10] = {};     // co-resident clusters of the kernel's own size (0 = not queried yet)
    // co-resident clusters of S single CTAs or S CTA pairs (kClusterReduce), by kind, CTAs per tile and S
    // (0 = not queried, -1 = none)
    int cluster_slots[2][3][5] = {};
    // Split-K partial sums of the last wave, one buffer per stream (calls on
    // one stream are ordered, so they may share it): [tickets | partials].
    struct Split {
        void *ptr = nullptr;
        size_t bytes = 0, ticket_bytes = 0;
        bool dirty = false;      // a launch may have stopped part-way (timeout): clear the tickets first
    };
    std::unordered_map<cudaStream_t, Split> split;
    // Per-CTA maxima of the quantiser, one array per stream.
    std::unordered_map<cudaStream_t, Split> quant;
    // Row copies of operands the TMA cannot address in place, one workspace
    // per stream, so calls on different streams may copy at the same time.
    std::unordered_map<cudaStream_t, Split> repack;
    // Softmax statistics: [tickets per tile row | parts], one buffer per stream.
    std::unordered_map<cudaStream_t, Split> stats;
    int quant_blocks[3] = {};         // co-resident quantiser CTAs per SM, by input type (0 = not queried)
    bool skinny_attr[2] = {};         // tn_skinny_kernel's shared-memory attribute set, by kind
    // One lock per stream, held by a call from its first buffer lookup through
    // its last launch: a call is several launches (row copy, GEMM, reduce),
    // and two host threads' calls on one stream must not interleave them.
    std::unordered_map<cudaStream_t, std::unique_ptr<std::mutex>> stream_locks;
};

std::mutex g_mutex;
// Held shared by every call from its first workspace lookup through its last
// launch, and exclusively by gemm_release_workspace: the buffers a call looked
// up stay allocated until its kernels are enqueued.
std::shared_mutex g_workspace_lock;

// The calling call's lock of `stream` on device state d (see stream_locks).
std::unique_lock<std::mutex> lock_stream(DeviceState &d, cudaStream_t stream);
DeviceState g_devices[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_force_cta_group{0};
std::atomic<int> g_force_wide{0};       // 0: the cost estimate decides; 1: always; -1: never
std::atomic<int> g_raster_group{0};     // tile rows per raster group; 0: kGroupM
std::atomic<int> g_k_order{0};          // 0: the library's choice; 1: every tile forward; 2: odd waves reversed
std::atomic<unsigned long long *> g_clock_probe{nullptr};   // gemm_debug_set_clock_probe
std::atomic<int> g_long_k{0};           // small grids with a long K: 0 the library's choice; 1 split-reduce; 2 cluster
std::atomic<int> g_lean{0};             // m-part launches: 0 the library's choice; 1 never lean; 2 lean where units allow
std::atomic<int> g_skinny{0};           // N <= 64: 0 the library's choice; 1 never the skinny kernel; 2 always
// The last launch on this host thread, for gemm_debug_last_launch: the
// numbers are kept and formatted only when asked for (formatting every call
// cost host time on the path of back-to-back small GEMMs).
struct LaunchRecord {
    const char *name = nullptr;     // nullptr: nothing launched yet
    bool quant = false;
    int G = 0, wide = 0, grid = 0, clusters = 0, slots = 0;
    int tiles = 0, units = 0, tail_start = 0, tail_mode = 0, split_parts = 0, vec = 0, cluster = 0, lean = 0;
    int skinny = 0;
    long long qgrid = 0, qunits = 0;
};
thread_local LaunchRecord t_rec;
thread_local char t_last_launch[256] = "";

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Current device's state, initialised on first use (caller holds no lock).
// The device whose primary context this host thread has made current.
thread_local int t_context_dev = -1;

gemm_status_t device_state(DeviceState **out, int *dev_out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    if (t_context_dev != dev) {
        // A host thread that has made no runtime call yet has no current
        // context, and the driver calls made here (tensor-map encoding) need
        // one: make the device's primary context current, once per thread.
        if ((e = cudaSetDevice(dev)) != cudaSuccess)
            return fail(GEMM_ERR_CUDA, "cudaSetDevice(%d): %s", dev, cudaGetErrorString(e));
        t_context_dev = dev;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail(GEMM_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        d.ready = true;
    }
    if (d.major != 10 || d.minor != 3)
        return fail(GEMM_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                    d.major, d.minor);
    *out = &d;
    if (dev_out) *dev_out = dev;
    return GEMM_OK;
}


// The key of a stream's buffers.  cudaStreamPerThread is one handle value
// that names a different stream on every host thread, so it is keyed per
// thread: small odd-shifted values no stream object has as its address.
cudaStream_t stream_key(cudaStream_t stream)
{
    if (stream != cudaStreamPerThread) return stream;
    static std::atomic<uint64_t> next_thread{1};
    thread_local const uint64_t thread_index = next_thread.fetch_add(1);
    return reinterpret_cast<cudaStream_t>(static_cast<uintptr_t>((thread_index << 8) | 0x2u));
}

// A per-stream buffer of `map` that starts with `zeroed_bytes` of words
// cleared when it is (re)allocated, followed by `extra_bytes`; grown on demand.
// The calls on one stream are ordered, and the caller holds the stream's lock
// (lock_stream) from here through its last launch, so calls on one stream
// share its buffers whatever host thread issues them; it also holds
// g_workspace_lock (shared).
gemm_status_t stream_buffer(DeviceState &, std::unordered_map<cudaStream_t, DeviceState::Split> &map,
                            cudaStream_t stream, size_t zeroed_bytes, size_t extra_bytes, const char *what,
                            uint8_t **base, size_t *zeroed_out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState::Split &w = map[stream_key(stream)];
    const size_t tb = (zeroed_bytes + 255) & ~size_t(255);
    if (w.ticket_bytes < tb || w.bytes < w.ticket_bytes + extra_bytes) {
        const size_t new_tb = tb > w.ticket_bytes ? tb : w.ticket_bytes;
        const size_t need = new_tb + extra_bytes;
        if (w.ptr) cudaFree(w.ptr);      // synchronises the device: earlier users are done
        w.ptr = nullptr;
        w.bytes = w.ticket_bytes = 0;
        cudaError_t e = cudaMalloc(&w.ptr, need);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return fail(GEMM_ERR_CUDA, "cudaMalloc(%zu) for %s: %s", need, what, cudaGetErrorString(e));
        }
        // the ticket words count arrivals within one launch and start from zero
        e = cudaMemsetAsync(w.ptr, 0, new_tb, stream);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "clearing %s: %s", what, cudaGetErrorString(e));
        w.bytes = need;
        w.ticket_bytes = new_tb;
        w.dirty = false;
    } else if (w.dirty) {
        cudaError_t e = cudaMemsetAsync(w.ptr, 0, w.ticket_bytes, stream);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "clearing %s: %s", what, cudaGetErrorString(e));
        w.dirty = false;
    }
    *base = static_cast<uint8_t *>(w.ptr);
    *zeroed_out = w.ticket_bytes;
    return GEMM_OK;
}

std::unique_lock<std::mutex> lock_stream(DeviceState &d, cudaStream_t stream)
{
    std::mutex *m;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        std::unique_ptr<std::mutex> &slot = d.stream_locks[stream_key(stream)];
        if (!slot) slot.reset(new std::mutex);
        m = slot.get();
    }
    return std::unique_lock<std::mutex>(*m);
}

// The stream's split-K buffer with room for `tickets` ticket words and
// `partial_bytes` of partial sums.
gemm_status_t split_workspace(DeviceState &d, cudaStream_t stream, size_t tickets, size_t partial_bytes,
                              unsigned long long **ticket_ptr, float **partial_ptr)
{
    uint8_t *base = nullptr;
    size_t zeroed = 0;
    gemm_status_t st = stream_buffer(d, d.split, stream, tickets * sizeof(unsigned long long), partial_bytes,
                                     "split-K partials", &base, &zeroed);
    if (st != GEMM_OK) return st;
    *ticket_ptr = reinterpret_cast<unsigned long long *>(base);
    *partial_ptr = reinterpret_cast<float *>(base + zeroed);
    return GEMM_OK;
}

// Tensor maps are a pure function of their arguments (address, sizes, stride,
// box, type), so encoded maps are cached and reused: repeated calls on the
// same buffers skip cuTensorMapEncodeTiled (about a microsecond of host time
// each, three per call).  A hash map holds up to kMaxEntries of them, enough
// for callers that cycle through many buffers (a serving loop over many
// weights, or a benchmark's rotating inputs); when it is full, the older half
// (by last use) goes at once, so eviction costs O(1) per insertion on average.
struct MapKey {
    uintptr_t base;
    uint64_t inner, outer, row_bytes;
    uint32_t box_inner, box_outer;
    int type;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
               box_inner == o.box_inner && box_outer == o.box_outer && type == o.type;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        // 64-bit multiplicative mixing of the fields
        uint64_t h = 0x9E3779B97F4A7C15ull;
        const uint64_t f[6] = {static_cast<uint64_t>(k.base), k.inner, k.outer, k.row_bytes,
                               (static_cast<uint64_t>(k.box_inner) << 32) | k.box_outer,
                               static_cast<uint64_t>(static_cast<uint32_t>(k.type))};
        for (uint64_t x : f) {
            h ^= x + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
            h *= 0xBF58476D1CE4E5B9ull;
        }
        return static_cast<size_t>(h ^ (h >> 31));
    }
};

struct MapCache {
    static constexpr size_t kMaxEntries = 8192;
    struct Entry {
        CUtensorMap map;
        uint64_t used_at;
    };
    std::unordered_map<MapKey, Entry, MapKeyHash> entries;
    uint64_t clock = 0;
    std::mutex mutex;
};
MapCache g_maps;

gemm_status_t encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        const char *what)
{
    const MapKey key{reinterpret_cast<uintptr_t>(base), inner, outer, row_bytes, box_inner, box_outer,
                     static_cast<int>(type)};
    {
        std::lock_guard<std::mutex> lock(g_maps.mutex);
        auto it = g_maps.entries.find(key);
        if (it != g_maps.entries.end()) {
            it->second.used_at = ++g_maps.clock;
            *map = it->second.map;
            return GEMM_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = fn(map, type, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    std::lock_guard<std::mutex> lock(g_maps.mutex);
    if (g_maps.entries.size() >= MapCache::kMaxEntries) {
        std::vector<uint64_t> ages;
        ages.reserve(g_maps.entries.size());
        for (const auto &kv : g_maps.entries) ages.push_back(kv.second.used_at);
        std::nth_element(ages.begin(), ages.begin() + ages.size() / 2, ages.end());
        const uint64_t cut = ages[ages.size() / 2];
        for (auto it = g_maps.entries.begin(); it != g_maps.entries.end();)
            it = it->second.used_at < cut ? g_maps.entries.erase(it) : std::next(it);
    }
    g_maps.entries[key] = MapCache::Entry{*map, ++g_maps.clock};
    return GEMM_OK;
}

// gemm_debug_inject_stall modes -> kernel flags.
uint32_t stall_flags(int mode)
{
    switch (mode) {
    case 1: return tn::kFlagStallMma;
    case 2: return tn::kFlagStallProducer0;
    case 3: return tn::kFlagStallProducer1;
    default: return 0u;
    }
}

// Launches repack_rows_kernel for one or two operands (a job with 0 rows is
// skipped); ld_dst, common to both, is a multiple of 16 bytes.
template <typename T>
void launch_repack(const tn::RepackJob<T> &j0, const tn::RepackJob<T> &j1, cudaStream_t stream)
{
    constexpr int64_t kVec = 16 / sizeof(T);
    const int64_t ld_dst = j0.rows ? j0.ld_dst : j1.ld_dst;
    const int64_t segs = (ld_dst / kVec + tn::kRepackSeg - 1) / tn::kRepackSeg;
    const int64_t units = (j0.rows + j1.rows) * segs;
    const unsigned blocks = static_cast<unsigned>((units + tn::kRepackWarps - 1) / tn::kRepackWarps);
    tn::repack_rows_kernel<T><<<blocks, tn::kRepackWarps * 32, 0, stream>>>(j0, j1, segs);
}

// Estimated length, in 256 x 256 tile times, of a persistent launch of `tiles`
// tiles of `tile` times each on `slots` slots.  A last partial wave that fills
// at most half of the slots is cut in two (`half` each); another one costs a
// whole tile.
double launch_estimate(int64_t tiles, int64_t slots, double tile, double half)
{
    const int64_t waves = tiles / slots, rem = tiles % slots;
    if (rem == 0) return waves * tile;
    return waves * tile + (waves >= 1 && 2 * rem <= slots ? half : tile);
}

// Tile times for the choice between 256 x 256 and 256 x 512 pair tiles, in
// units of a 256 x 256 tile's time; kb is the tile's number of 256-byte k
// stages.  Fitted to sustained A/B timings on GB300 under the power cap (FP16
// shapes from 3072^2 x 8192 to 16384^2 x 1024, and E4M3 ones):
//  - a 256 x 512 tile: two 256 x 256 tiles' work at 0.913 each (a quarter
//    fewer bytes out of L2 buys a higher clock), plus the part of its
//    epilogue that the next tile's MMAs wait for (a half of the accumulator
//    is handed back once read): a fixed time, 0.6 tile times at kb = 1;
//  - one m half of one, run in the wide stages: 1.36 (see below);
//  - a cut half of a 256 x 256 tile in a last partial wave: 0.9, not 0.5;
//    the partial sums cost more than a launch with few waves can hide.
// One family of shapes is still missed: 16384 x 8192 with 8 k stages, where
// 256 x 256 tiles are 4-5 % faster (FP16 and E4M3); 8192^2 with 8 stages,
// 7 % faster on wide tiles, rules out a larger epilogue term.
// Cutting 8192^3's last 56 wide tiles into 76 m halves and 72 k-half quarters
// made the launch 4 % slower than leaving them whole, which puts a half plus
// a quarter above one wide tile; so only m halves are used, at 1.36.
double wide_tile_cost(double kb) { return 2.0 * 0.913 + 0.6 / kb; }
constexpr double kWideHalfCost = 1.36;
constexpr double kNarrowHalfCost = 0.9;

int launch_grid(int64_t work, int cap)
{
    int64_t g = (work + 255) / 256;
    if (g > cap) g = cap;
    return g < 1 ? 1 : static_cast<int>(g);
}

// What A's tensor maps are made of; the map for units that cover part of a
// tile's m range is encoded once the number of parts is known.
struct ASource {
    CUtensorMapDataType type;
    const void *base;
    uint64_t inner, outer, row_bytes;
    uint32_t box_k, rows;      // rows: A rows per CTA of a whole tile
};

// Co-resident slots of tn_gemm_kernel<Kind, G, W, C, St, Ln>: clusters of its
// own size (one CTA, or a pair), or with C clusters of G * clusters_of CTAs (S
// pairs or S single CTAs), queried once per device (the kernel's shared-memory
// attribute is set first).
template <class Kind, int G, bool W, bool C = false, bool St = false, int Ln = 0>
gemm_status_t kernel_slots(DeviceState &dev, int clusters_of, int *out)
{
    using Cfg = tn::TileCfg<G, W, Ln>;
    auto kernel = tn::tn_gemm_kernel<Kind, G, W, C, St, Ln>;
    const int ki = Kind::kF8 ? 1 : 0;
    const int ks = Ln == 4 ? 8 : Ln == 2 ? 9 : W ? 3 : C ? 3 + G : St ? 5 + G : G;   // kernel index of the per-device caches
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!dev.smem_attr[ki][ks]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        dev.smem_attr[ki][ks] = true;
    }
    const int cl = G * clusters_of;
    int &n = clusters_of == 1 ? dev.max_clusters[ki][ks] : dev.cluster_slots[ki][G][clusters_of];
    if (n == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(tn::kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(cl * (dev.sms / cl), 1, 1);
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess || n <= 0) {
            cudaGetLastError();
            // one slot per SM (pair) for the kernel's own size; no cluster reduce otherwise
            n = clusters_of == 1 ? dev.sms / G : -1;
        }
    }
    *out = n;
    return GEMM_OK;
}

// The number of k ranges S (2 to 4) of a kClusterReduce launch of
// tn_gemm_kernel<Kind, G> for num_tiles tiles of num_kb k blocks on `slots`
// co-resident slots, or 1 for none: a grid of at most half the slots with a
// long K, cut as the split-reduce would cut it (as many ranges as the slots
// allow, at most 8, each at least 16 k blocks) when that is at most 4 (or
// always, when the call may not allocate the split-reduce's buffer), with
// one cluster of G * S CTAs per tile co-resident.
template <class Kind, int G>
int cluster_reduce_parts(DeviceState &dev, int64_t num_tiles, int64_t num_kb, int slots, bool allow_alloc,
                         int long_k)
{
    if (long_k == 1 || 2 * num_tiles > slots || num_kb < 32) return 1;
    int64_t S = slots / num_tiles;
    if (S > 8) S = 8;
    if (S > num_kb / 16) S = num_kb / 16;
    if (S < 2 || !(S <= 4 || long_k == 2 || !allow_alloc)) return 1;
    for (int Sc = S < 4 ? static_cast<int>(S) : 4; Sc >= 2; --Sc) {
        int n = 0;
        if (kernel_slots<Kind, G, false, true>(dev, Sc, &n) != GEMM_OK) return 1;
        if (n >= num_tiles) return Sc;
    }
    return 1;
}

// Launches the persistent kernel: one CTA (or one CTA pair, a 2-CTA cluster)
// per co-resident slot, each walking the tile raster with a stride of the
// grid.  W: CTA pairs with 256 x 512 tiles (never with the softmax statistics
// or a split K).
template <class Kind, int G, bool W = false>
gemm_status_t launch(const char *name, tn::KernelParams &prm, DeviceState &dev, bool allow_alloc,
                     const ASource &asrc, cudaStream_t stream)
{
    static_assert(!W || G == 2, "256 x 512 tiles are CTA-pair tiles");
    using Cfg = tn::TileCfg<G, W>;
    void (*kernel)(tn::KernelParams) = tn::tn_gemm_kernel<Kind, G, W>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(tn::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int slots = 0;
    {
        gemm_status_t st = kernel_slots<Kind, G, W>(dev, 1, &slots);
        if (st != GEMM_OK) return st;
    }
    // A grid of at most half the slots with a long K leaves most SMs idle:
    // every tile is cut into S ranges of its k blocks (as many as the slots
    // allow, at most 8, each at least 16 k blocks).  Single CTAs and CTA pairs
    // (not 256 x 512 tiles) do it in a cluster of S <= 4 CTAs or pairs per
    // tile, which add their partials up through distributed shared memory
    // (kClusterReduce: no workspace, one kernel); otherwise the units store
    // FP32 partials, and a reduce kernel sums them in order and stores C
    // (kSplitReduce).
    const int cap = slots;
    const bool stats = (prm.flags & tn::kFlagStats) != 0;
    if constexpr (!W && !Kind::kF8) {
        if (stats) {
            // the statistics variant (its own shared-memory attribute, the same slots)
            gemm_status_t st = kernel_slots<Kind, G, false, false, true>(dev, 1, &slots);
            if (st != GEMM_OK) return st;
        }
    }
    const int long_k = g_long_k.load();
    int reduce_parts = 1, cluster_parts = 1;
    if (!W && !stats) cluster_parts = cluster_reduce_parts<Kind, G>(dev, prm.num_tiles, prm.num_kb, cap, allow_alloc, long_k);
    if (cluster_parts == 1 && !stats && allow_alloc && long_k != 2 && 2 * prm.num_tiles <= cap && prm.num_kb >= 32) {
        int S = cap / prm.num_tiles;
        if (S > 8) S = 8;
        if (S > prm.num_kb / 16) S = prm.num_kb / 16;
        if (S >= 2) reduce_parts = S;
    }
    // A grid of at most half the slots with a shorter K: every tile's m range
    // is cut into 2 or 4 parts (MMA N = 128 or 64).  Such a launch is bound by
    // latency, mostly the epilogue's TMEM -> shared memory -> TMA store
    // round trips, and each unit stores a half or a quarter of a tile.
    int m_parts = 1;
    if (!W && reduce_parts == 1 && cluster_parts == 1 && 2 * prm.num_tiles <= cap)
        m_parts = tn::kMaxMParts * prm.num_tiles <= cap ? tn::kMaxMParts : 2;
    const int units0 = prm.num_tiles * reduce_parts * m_parts;
    // (kClusterReduce: one tile per cluster of cluster_parts CTAs, never more --
    // a CTA's ring takes the other CTAs' partials once its own MMAs are done)
    const int clusters = cluster_parts > 1 ? prm.num_tiles : units0 < slots ? units0 : slots;
    if (cluster_parts > 1) attr[0].val.clusterDim.x = G * cluster_parts;
    // A programmatic dependent of the previous kernel on the stream: the
    // kernel waits for it (griddepcontrol.wait) before touching memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(G * cluster_parts * clusters, 1, 1);
    // A last wave that fills at most half of the slots is run as twice as
    // many half-length units, so every slot finishes at about the same time:
    // each of those tiles is split into two halves of its k blocks whose
    // partial sums meet in a per-stream workspace, or -- without the
    // workspace, or with few k blocks -- into two halves of its m range.
    const int waves = prm.num_tiles / clusters, rem = prm.num_tiles % clusters;
    prm.tail_mode = tn::kTailNone;
    prm.tail_start = prm.num_tiles;
    prm.num_units = prm.num_tiles;
    prm.split_parts = 1;
    prm.m_part_rows = 0;
    if (cluster_parts > 1) {
        prm.tail_mode = tn::kClusterReduce;
        prm.split_parts = cluster_parts;
        prm.kb_part = (prm.num_kb + cluster_parts - 1) / cluster_parts;
    } else if (reduce_parts > 1) {
        const size_t partial = size_t(prm.num_tiles) * reduce_parts * G * Cfg::kRowsB * Cfg::kTileMRows * sizeof(float);
        uint8_t *base = nullptr;
        size_t zeroed = 0;
        gemm_status_t st = stream_buffer(dev, dev.split, stream, 0, partial, "split-K partials", &base, &zeroed);
        if (st != GEMM_OK) return st;
        prm.tail_mode = tn::kSplitReduce;
        prm.tail_start = 0;
        prm.num_units = units0;
        prm.split_parts = reduce_parts;
        prm.kb_part = (prm.num_kb + reduce_parts - 1) / reduce_parts;
        prm.split_ws = reinterpret_cast<float *>(base + zeroed);
    } else if (m_parts > 1) {
        prm.tail_mode = tn::kTailMParts;
        prm.tail_start = 0;
        prm.num_units = units0;
        prm.split_parts = m_parts;
    } else if (waves >= 1 && rem > 0 && 2 * rem <= clusters && !stats) {
        // (The softmax statistics count one kind of unit per tile row.)
        prm.tail_start = waves * clusters;
        prm.num_units = prm.tail_start + 2 * rem;
        prm.tail_mode = tn::kTailMParts;
        prm.split_parts = 2;
        if (!W && allow_alloc && prm.num_kb >= 4) {
            const size_t partial = size_t(rem) * 2 * G * Cfg::kRowsB * tn::kTileM * sizeof(float);
            unsigned long long *tickets = nullptr;
            float *partials = nullptr;
            gemm_status_t st = split_workspace(dev, stream, size_t(rem) * G, partial, &tickets, &partials);
            if (st != GEMM_OK) return st;
            prm.tail_mode = tn::kTailSplitK;
            prm.kb_part = (prm.num_kb + 1) / 2;
            prm.split_ws = partials;
            prm.split_tickets = tickets;
        }
    }
    if (prm.tail_mode == tn::kTailMParts) {
        prm.m_part_rows = Cfg::kTileMRows / prm.split_parts;
        // (a wide tile's parts are its halves, whose rows the A map's boxes already are)
        gemm_status_t st = W ? GEMM_OK
                             : encode_2d(&prm.tmap_a_part, asrc.type, asrc.base, asrc.inner, asrc.outer,
                                         asrc.row_bytes, asrc.box_k, asrc.rows / prm.split_parts, "A part");
        if (st != GEMM_OK) return st;
    }
    // Every unit a quarter-m (half-m) unit of a single CTA -- a grid of at
    // most a quarter (half) of the slots' tiles with a short K -- and more
    // units than half the slots, so that the next launch's CTAs would not
    // find idle SMs: the lean configuration, two CTAs per SM, whose CTAs
    // become resident beside the previous launch's and do their setup while
    // it runs (up to kLeanQuarterMaxKb / kLeanHalfMaxKb k blocks).  Not with
    // the softmax statistics: their epilogue, the longer part of such a
    // launch, ran slower under the lean register limit and with two CTAs on
    // an SM.
    int lean = 0;
    if constexpr (G == 1 && !W) {
        const int mode = g_lean.load();
        if (prm.tail_mode == tn::kTailMParts && prm.tail_start == 0 && !stats && mode != 1) {
            const bool crowded = 2 * prm.num_units > slots;
            if (prm.split_parts == 4 && (mode == 2 || (crowded && prm.num_kb <= kLeanQuarterMaxKb)))
                lean = 4;
            else if (prm.split_parts == 2 && (mode == 2 || (crowded && prm.num_kb <= kLeanHalfMaxKb)))
                lean = 2;
        }
        if (lean) {
            int n = 0;
            gemm_status_t st = lean == 4 ? kernel_slots<Kind, 1, false, false, false, 4>(dev, 1, &n)
                                         : kernel_slots<Kind, 1, false, false, false, 2>(dev, 1, &n);
            if (st != GEMM_OK) return st;
            cfg.dynamicSmemBytes =
                lean == 4 ? tn::TileCfg<1, false, 4>::kSmemBytes : tn::TileCfg<1, false, 2>::kSmemBytes;
        }
    }
    t_rec.name = name;
    t_rec.quant = false;
    t_rec.lean = lean;
    t_rec.skinny = 0;
    t_rec.G = G;
    t_rec.wide = W ? 1 : 0;
    t_rec.grid = G * cluster_parts * clusters;
    t_rec.cluster = G * cluster_parts;
    t_rec.clusters = clusters;
    t_rec.slots = slots;
    t_rec.tiles = prm.num_tiles;
    t_rec.units = prm.num_units;
    t_rec.tail_start = prm.tail_start;
    t_rec.tail_mode = prm.tail_mode;
    t_rec.split_parts = prm.split_parts;
    if constexpr (!W) {
        if (cluster_parts > 1) kernel = tn::tn_gemm_kernel<Kind, G, false, true>;
        if constexpr (!Kind::kF8) {
            if (stats) kernel = tn::tn_gemm_kernel<Kind, G, false, false, true>;
        }
    }
    if constexpr (G == 1 && !W) {
        if (lean == 4) kernel = tn::tn_gemm_kernel<Kind, 1, false, false, false, 4>;
        if (lean == 2) kernel = tn::tn_gemm_kernel<Kind, 1, false, false, false, 2>;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: launch: %s", name, cudaGetErrorString(e));
    if (prm.tail_mode == tn::kSplitReduce) {
        // the reduce kernel, as a programmatic dependent: its launch overlaps the GEMM's end
        cudaLaunchConfig_t rcfg = {};
        cudaLaunchAttribute rattr[1];
        rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        rattr[0].val.programmaticStreamSerializationAllowed = 1;
        const int64_t work = (int64_t(prm.M) + 7) / 8 * prm.N;
        rcfg.gridDim = dim3(static_cast<unsigned>(launch_grid(work, dev.sms * 8)), 1, 1);
        rcfg.blockDim = dim3(256, 1, 1);
        rcfg.stream = stream;
        rcfg.attrs = rattr;
        rcfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&rcfg, tn::split_reduce_kernel<Kind, G, Cfg::kTileMRows>,
                               static_cast<const float *>(prm.split_ws),
                               static_cast<int>(prm.split_parts), static_cast<int64_t>(prm.tiles_n), prm.M, prm.N,
                               prm.c_ptr, prm.ldc, prm.scale, prm.scale_a_ptr, prm.scale_b_ptr);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: split reduce launch: %s", name, cudaGetErrorString(e));
    }
    return GEMM_OK;
}

// Launches tn_skinny_kernel for N <= 64: 128-row m tiles, their k blocks cut
// into 1, 2 or 4 ranges (each of at least 4 blocks) so that the grid fills
// the SMs; with several ranges the partials meet in the per-stream split
// workspace (none when the call may not allocate: then one range per tile).
template <class Kind>
gemm_status_t launch_skinny(const char *name, int64_t M, int64_t N, int64_t K, const void *a, int64_t ka,
                            int64_t lda_bytes, const void *b, int64_t kb, int64_t ldb_bytes, void *C, int64_t ldc,
                            float scale, const float *dscale_a, const float *dscale_b, DeviceState &dev,
                            bool allow_alloc, cudaStream_t stream)
{
    constexpr int64_t esz = Kind::kElemBytes;
    tn::SkinnyParams prm;
    memset(&prm, 0, sizeof(prm));
    const CUtensorMapDataType in_type = Kind::kF8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint32_t box_k = tn::kBlockKBytes / esz;
    const int32_t n_mma = static_cast<int32_t>((N + 15) / 16 * 16);
    gemm_status_t st;
    if ((st = encode_2d(&prm.tmap_a, in_type, a, ka, M, lda_bytes, box_k, tn::kSkRowsM, "A")) != GEMM_OK) return st;
    if ((st = encode_2d(&prm.tmap_b, in_type, b, kb, N, ldb_bytes, box_k, static_cast<uint32_t>(n_mma), "B")) !=
        GEMM_OK)
        return st;
    const int64_t tiles_m = (M + tn::kSkRowsM - 1) / tn::kSkRowsM;
    const int64_t num_kb = (K * esz + tn::kBlockKBytes - 1) / tn::kBlockKBytes;
    const int slots = dev.sms;                 // one CTA per SM (about 194 KiB of shared memory each)
    int parts = 1;
    for (int q = tn::kSkMaxParts; q >= 2 && allow_alloc; q /= 2)
        if (tiles_m * q <= slots && num_kb >= 4 * q) {
            parts = q;
            break;
        }
    if (tiles_m * parts > INT32_MAX) return fail(GEMM_ERR_UNSUPPORTED, "%s: too many output tiles", name);
    prm.c_ptr = C;
    prm.ldc = ldc;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.num_kb = static_cast<int32_t>(num_kb);
    prm.n_mma = n_mma;
    prm.tiles_m = static_cast<int32_t>(tiles_m);
    prm.parts = parts;
    prm.kb_part = static_cast<int32_t>((num_kb + parts - 1) / parts);
    prm.num_units = static_cast<int32_t>(tiles_m * parts);
    if (parts > 1) {
        const size_t partial = size_t(tiles_m) * parts * size_t(n_mma) * tn::kSkRowsM * sizeof(float);
        if ((st = split_workspace(dev, stream, size_t(tiles_m), partial, &prm.tickets, &prm.split_ws)) != GEMM_OK)
            return st;
    }
    prm.scale = scale;
    prm.scale_a_ptr = dscale_a;
    prm.scale_b_ptr = dscale_b;
    prm.flags = stall_flags(g_inject_stall.load());
    prm.wait_limit_ns = g_wait_limit_ns.load();

    auto kernel = tn::tn_skinny_kernel<Kind>;
    const int ki = Kind::kF8 ? 1 : 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!dev.skinny_attr[ki]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tn::kSkSmemBytes);
            if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            dev.skinny_attr[ki] = true;
        }
    }
    const int64_t grid = prm.num_units < slots ? prm.num_units : slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    // a programmatic dependent of the previous kernel on the stream, like the general kernel
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(tn::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tn::kSkSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    t_rec = LaunchRecord{};
    t_rec.name = name;
    t_rec.G = 1;
    t_rec.grid = static_cast<int>(grid);
    t_rec.cluster = 1;
    t_rec.clusters = static_cast<int>(grid);
    t_rec.slots = slots;
    t_rec.tiles = prm.tiles_m;
    t_rec.units = prm.num_units;
    t_rec.split_parts = parts;
    t_rec.skinny = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: launch: %s", name, cudaGetErrorString(e));
    return GEMM_OK;
}

template <class Kind>
gemm_status_t run_gemm(const char *name, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                       const void *B, int64_t ldb, void *C, int64_t ldc, float scale, cudaStream_t stream,
                       bool allow_alloc = true, const float *dscale_a = nullptr, const float *dscale_b = nullptr,
                       float *row_max = nullptr, float *row_sum = nullptr)
{
    const bool stats = row_max != nullptr;
    constexpr int64_t esz = Kind::kElemBytes;
    const int64_t kmin = K > 1 ? K : 1;
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "%s: negative size (M=%lld N=%lld K=%lld)", name, (long long)M,
                    (long long)N, (long long)K);
    if (lda < kmin) return fail(GEMM_ERR_INVALID_ARG, "%s: lda=%lld < max(1,K)", name, (long long)lda);
    if (ldb < kmin) return fail(GEMM_ERR_INVALID_ARG, "%s: ldb=%lld < max(1,K)", name, (long long)ldb);
    if (ldc < (M > 1 ? M : 1)) return fail(GEMM_ERR_INVALID_ARG, "%s: ldc=%lld < max(1,M)", name, (long long)ldc);
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || lda > kMaxDim || ldb > kMaxDim || ldc > kMaxDim)
        return fail(GEMM_ERR_UNSUPPORTED, "%s: a size or leading dimension exceeds 2^31-256", name);
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "%s: C is NULL", name);
    if (reinterpret_cast<uintptr_t>(C) % 2) return fail(GEMM_ERR_INVALID_ARG, "%s: C is not 2-byte aligned", name);
    if (K > 0) {
        if (!A || !B) return fail(GEMM_ERR_INVALID_ARG, "%s: A or B is NULL", name);
        if (reinterpret_cast<uintptr_t>(A) % esz || reinterpret_cast<uintptr_t>(B) % esz)
            return fail(GEMM_ERR_INVALID_ARG, "%s: A or B is not aligned to its element size", name);
    }
    // buffers looked up below stay allocated until this call's launches are enqueued
    std::shared_lock<std::shared_mutex> workspace_guard(g_workspace_lock);
    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev, nullptr);
    if (st != GEMM_OK) return st;
    // this call's launches go onto the stream together (no other host thread's in between)
    std::unique_lock<std::mutex> stream_guard = lock_stream(*dev, stream);

    if (K == 0) {
        // every sum is +0; scaled scores are scale * +0 (-0 for a negative scale)
        const uint16_t fill = stats && std::signbit(scale) ? 0x8000u : 0u;
        tn::zero_fill_kernel<<<launch_grid(M * N, dev->sms * 8), 256, 0, stream>>>(static_cast<uint16_t *>(C), ldc,
                                                                                 M, N, fill);
        if (stats)
            tn::fill_stats_kernel<<<launch_grid(M, dev->sms), 256, 0, stream>>>(row_max, row_sum, M,
                                                                              static_cast<float>(N));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: zero fill launch: %s", name, cudaGetErrorString(e));
        return GEMM_OK;
    }

    // Tile shape.  One CTA per 128 x 256 tile when N <= 128 (a pair's second
    // half would idle); else a CTA pair per 256 x 256 tile.  A problem of at most half a wave of pair tiles runs on single CTAs: it
    // is latency-bound, and a CTA without a partner skips the cluster
    // barriers (measured on GB300: 1024 x 1024 x 128 5.8 -> 4.3 us per
    // kernel, 512^3 9.1 -> 6.0 us).
    int ctas = N > 128 ? 2 : 1;
    if (ctas == 2 && 2 * (((M + 255) / 256) * ((N + 255) / 256)) <= dev->sms / 2) ctas = 1;
    // Small grids with a long K, their k ranges reduced in clusters: CTA pairs
    // need two thirds of the operand bytes per MMA of single CTAs (64 against
    // 96 bytes per SM cycle), so pairs run them where their clusters keep at
    // least as many SMs busy.  Measured on GB300 (single CTAs -> pairs):
    // 4096 x 512 x 8192 35.7 -> 31.7 us, 8192 x 256 x 8192 39.4 -> 35.2,
    // 2048 x 1024 x 8192 33.0 -> 30.0; with fewer SMs busy, pairs lost
    // (1024^2 x 8192 on 96 instead of 128 SMs: 24.4 -> 27.3).
    if (ctas == 1 && N > 128 && !stats && K * esz >= 32 * 256) {    // (at least 32 k blocks of a pair)
        const int long_k = g_long_k.load();
        const int64_t rows = (M + tn::kTileM - 1) / tn::kTileM;
        const int64_t t1 = rows * ((N + 127) / 128), t2 = rows * ((N + 255) / 256);
        int s1 = 0, s2 = 0;
        if ((st = kernel_slots<Kind, 1, false>(*dev, 1, &s1)) != GEMM_OK) return st;
        if ((st = kernel_slots<Kind, 2, false>(*dev, 1, &s2)) != GEMM_OK) return st;
        const int p1 = cluster_reduce_parts<Kind, 1>(*dev, t1, (K * esz + 127) / 128, s1, allow_alloc, long_k);
        const int p2 = cluster_reduce_parts<Kind, 2>(*dev, t2, (K * esz + 255) / 256, s2, allow_alloc, long_k);
        if (p1 > 1 && p2 > 1 && 2 * t2 * p2 >= t1 * p1) ctas = 2;
    }
    if (const int forced = g_force_cta_group.load()) ctas = forced;
    const int cta_group = ctas >= 2 ? 2 : 1;
    const int64_t tiles_n = (N + 128 * cta_group - 1) / (128 * cta_group);
    // 256 x 512 pair tiles (two N = 256 halves that share the n-side rows) move
    // a quarter fewer bytes out of L2 per MMA.  Under the power cap that buys a
    // 7-9 % higher SM clock at about the same work per clock (8192^3 FP16 on
    // GB300).  But there are half as many of them, a last partial wave can
    // only be cut into m halves, and their accumulator is not double-buffered.
    // They are used where an estimate of the launch's length says so.
    bool wide = false;
    if (cta_group == 2 && !stats) {
        const int force = g_force_wide.load();
        const int64_t slots = dev->sms / 2;
        const int64_t tiles256 = (M + tn::kTileM - 1) / tn::kTileM * tiles_n;
        const int64_t tiles512 = (M + 2 * tn::kTileM - 1) / (2 * tn::kTileM) * tiles_n;
        const int64_t kb = (K * esz + 255) / 256;                       // 256-byte k stages
        const double t_wide = launch_estimate(tiles512, slots, wide_tile_cost(double(kb)), kWideHalfCost);
        const double t_narrow = launch_estimate(tiles256, slots, 1.0, kNarrowHalfCost);
        wide = force > 0 || (force == 0 && t_wide < t_narrow);
    }
    const int64_t tile_m_rows = wide ? 2 * tn::kTileM : tn::kTileM;
    const int64_t tiles_m = (M + tile_m_rows - 1) / tile_m_rows;
    if (tiles_m * tiles_n > INT32_MAX) return fail(GEMM_ERR_UNSUPPORTED, "%s: too many output tiles", name);

    // The TMA reads an operand in place only when its base, its row stride and
    // its row length K are all multiples of 16 bytes (a row that ends inside a
    // 16-byte unit is not clipped element by element).  Other operands are
    // first copied to a workspace with a padded stride and zero-filled pad,
    // and the padded length becomes the tensor's inner dimension.  The padded
    // stride is a multiple of 128 bytes, so that every row of every TMA box
    // (one 128-byte swizzle atom) is one aligned 128-byte line; with a stride
    // that is only 16-byte aligned each box row straddles two lines, which
    // measured 13 % slower on 3000 x 12289 x 4097.
    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb, ka = K, kb = K;
    const bool k_aligned = (K * esz) % 16 == 0;
    const bool repack_a = !k_aligned || (lda * esz) % 16 != 0 || reinterpret_cast<uintptr_t>(A) % 16 != 0;
    const bool repack_b = !k_aligned || (ldb * esz) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0;
    if (repack_a || repack_b) {
        constexpr int64_t kPad = tn::kBlockKBytes / esz;       // elements per 128 bytes
        const int64_t ldp = (K + kPad - 1) / kPad * kPad;
        const size_t bytes_a = repack_a ? ((size_t(M) * ldp * esz + 255) & ~size_t(255)) : 0;
        const size_t bytes_b = repack_b ? ((size_t(N) * ldp * esz + 255) & ~size_t(255)) : 0;
        uint8_t *ws = nullptr;
        size_t zeroed = 0;
        if ((st = stream_buffer(*dev, dev->repack, stream, 0, bytes_a + bytes_b, "the row-copy workspace", &ws,
                                &zeroed)) != GEMM_OK)
            return st;
        using T = typename std::conditional<esz == 2, uint16_t, uint8_t>::type;
        tn::RepackJob<T> ja{static_cast<const T *>(A), lda, reinterpret_cast<T *>(ws), ldp, repack_a ? M : 0, K};
        tn::RepackJob<T> jb{static_cast<const T *>(B), ldb, reinterpret_cast<T *>(ws + bytes_a), ldp,
                            repack_b ? N : 0, K};
        launch_repack<T>(ja, jb, stream);       // one launch for both operands
        if (repack_a) {
            a_use = ws;
            lda_use = ka = ldp;
        }
        if (repack_b) {
            b_use = ws + bytes_a;
            ldb_use = kb = ldp;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: repack launch: %s", name, cudaGetErrorString(e));
    }

    // Few columns n: the kernel with the operands on the other MMA sides, up to
    // kSkinnyMaxKb k blocks of 128 bytes (beyond that, with the operand stream
    // at the DRAM roofline in both kernels, the general kernel's cluster
    // reduce measured as fast or faster).
    {
        const int mode = g_skinny.load();
        const int64_t num_kb = (K * esz + tn::kBlockKBytes - 1) / tn::kBlockKBytes;
        // (a test hook that forces the general kernel's tile shape or k cut keeps it)
        const bool forced = g_force_cta_group.load() != 0 || g_force_wide.load() != 0 || g_long_k.load() != 0;
        if (!stats && N <= tn::kSkMaxN && (mode == 2 || (mode == 0 && !forced && num_kb <= kSkinnyMaxKb)))
            return launch_skinny<Kind>(name, M, N, K, a_use, ka, lda_use * esz, b_use, kb, ldb_use * esz, C, ldc,
                                       scale, dscale_a, dscale_b, *dev, allow_alloc, stream);
    }

    tn::KernelParams prm;
    memset(&prm, 0, sizeof(prm));
    const CUtensorMapDataType in_type = Kind::kF8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapDataType out_type = Kind::kF8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint32_t box_k = tn::kBlockKBytes / esz;
    const uint32_t rows_a = static_cast<uint32_t>(tn::kTileM / cta_group);
    if ((st = encode_2d(&prm.tmap_a, in_type, a_use, ka, M, lda_use * esz, box_k, rows_a, "A")) != GEMM_OK)
        return st;
    if ((st = encode_2d(&prm.tmap_b, in_type, b_use, kb, N, ldb_use * esz, box_k, 128, "B")) != GEMM_OK)
        return st;
    // TMA stores cover rows m < M rounded down to 8 (16 bytes); the kernel
    // writes the ragged rest, or all of C when C's base or stride is unaligned.
    const int64_t m_tma = M & ~int64_t(7);
    const bool tma_c = (ldc * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(C) % 16 == 0 && m_tma > 0;
    if (tma_c &&
        (st = encode_2d(&prm.tmap_c, out_type, C, m_tma, N, ldc * 2, tn::kEpiBoxM, tn::kEpiBoxN, "C")) != GEMM_OK)
        return st;
    prm.m_tma = tma_c ? static_cast<int32_t>(m_tma) : 0;
    prm.c_ptr = C;
    prm.ldc = ldc;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.tiles_m = static_cast<int32_t>(tiles_m);
    prm.tiles_n = static_cast<int32_t>(tiles_n);
    prm.num_tiles = static_cast<int32_t>(tiles_m * tiles_n);
    const int64_t stage_k = wide ? tn::TileCfg<2, true>::kStageKBytes
                                 : cta_group == 2 ? tn::TileCfg<2>::kStageKBytes : tn::TileCfg<1>::kStageKBytes;
    prm.num_kb = static_cast<int32_t>((K * esz + stage_k - 1) / stage_k);   // k blocks = stages per tile
    {
        const int rg = g_raster_group.load();
        prm.group = rg > 0 ? rg : kGroupM;
    }
    prm.scale = scale;
    prm.scale_a_ptr = dscale_a;
    prm.scale_b_ptr = dscale_b;
    if (stats) {
        prm.flags |= tn::kFlagStats;
        prm.row_max = row_max;
        prm.row_sum = row_sum;
        prm.stat_ctas = static_cast<int32_t>(tiles_n * cta_group);
        const size_t parts = size_t(tiles_m) * prm.stat_ctas * tn::kEpiWarps * tn::kTileM * sizeof(float2);
        uint8_t *base = nullptr;
        size_t zeroed = 0;
        // one ticket per tile row and m part
        const size_t tickets = size_t(tiles_m) * tn::kMaxMParts * sizeof(unsigned long long);
        if ((st = stream_buffer(*dev, dev->stats, stream, tickets, parts, "softmax statistics", &base, &zeroed)) !=
            GEMM_OK)
            return st;
        prm.stat_tickets = reinterpret_cast<unsigned long long *>(base);
        prm.stat_parts = reinterpret_cast<float2 *>(base + zeroed);
    }
    prm.flags |= (tma_c ? tn::kFlagTmaStore : 0u) | stall_flags(g_inject_stall.load());
    {
        const int ko = g_k_order.load();
        if (ko == 2 || (ko == 0 && kAltKDefault)) prm.flags |= tn::kFlagAltK;
    }
    prm.wait_limit_ns = g_wait_limit_ns.load();
    prm.clock_probe = g_clock_probe.load();

    const ASource asrc{in_type, a_use, static_cast<uint64_t>(ka), static_cast<uint64_t>(M),
                       static_cast<uint64_t>(lda_use * esz), box_k, rows_a};
    if (wide) return launch<Kind, 2, true>(name, prm, *dev, allow_alloc, asrc, stream);
    if (cta_group == 2) return launch<Kind, 2>(name, prm, *dev, allow_alloc, asrc, stream);
    return launch<Kind, 1>(name, prm, *dev, allow_alloc, asrc, stream);
}

// Per-tensor E4M3 quantisation (quant_e4m3_kernel.cuh): the maximum-finding
// kernel, then the quantising kernel as its programmatic dependent, both with
// the same grid; the per-CTA maxima go through the stream's slot array.
template <int kIn>
gemm_status_t launch_quant(DeviceState &dev, qz::QuantParams &prm, cudaStream_t stream)
{
    auto amax_kernel = qz::quant_amax_kernel<kIn>;
    auto store_kernel = qz::quant_store_kernel<kIn>;
    int per_sm;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (dev.quant_blocks[kIn] == 0) {
            int n1 = 0, n2 = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, amax_kernel, qz::kThreads, 0);
            if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n2, store_kernel, qz::kThreads, 0);
            if (e != cudaSuccess || n1 <= 0 || n2 <= 0)
                return fail(GEMM_ERR_CUDA, "gemm_quantize_e4m3: occupancy query: %s", cudaGetErrorString(e));
            dev.quant_blocks[kIn] = n1 < n2 ? n1 : n2;    // both grids resident in one wave
        }
        per_sm = dev.quant_blocks[kIn];
    }
    int64_t grid = int64_t(per_sm) * dev.sms;
    if (grid > prm.num_units) grid = prm.num_units;
    if (grid < 1) grid = 1;
    uint8_t *slots = nullptr;
    size_t zeroed = 0;
    gemm_status_t st = stream_buffer(dev, dev.quant, stream, 0, size_t(grid) * sizeof(float), "quantiser slots",
                                     &slots, &zeroed);
    if (st != GEMM_OK) return st;
    prm.slots = reinterpret_cast<float *>(slots + zeroed);
    t_rec.name = "gemm_quantize_e4m3";
    t_rec.quant = true;
    t_rec.qgrid = grid;
    t_rec.qunits = prm.num_units;
    t_rec.vec = prm.vec;

    // Both kernels are programmatic dependents of the kernel before them on
    // the stream, and wait for it (griddepcontrol.wait) before any access.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(qz::kThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, amax_kernel, prm);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "gemm_quantize_e4m3: launch (amax): %s", cudaGetErrorString(e));
    e = cudaLaunchKernelEx(&cfg, store_kernel, prm);
    if (e != cudaSuccess)
        return fail(GEMM_ERR_CUDA, "gemm_quantize_e4m3: launch (quantise): %s", cudaGetErrorString(e));
    return GEMM_OK;
}

gemm_status_t run_quant(const void *x, int x_type, int64_t rows, int64_t cols, int64_t ldx, void *q, int64_t ldq,
                        float *scale, cudaStream_t stream)
{
    const char *name = "gemm_quantize_e4m3";
    if (x_type < qz::kInF32 || x_type > qz::kInBF16)
        return fail(GEMM_ERR_INVALID_ARG, "%s: unknown input type %d", name, x_type);
    const int64_t esz = x_type == qz::kInF32 ? 4 : 2;
    if (rows < 0 || cols < 0) return fail(GEMM_ERR_INVALID_ARG, "%s: negative size", name);
    const int64_t cmin = cols > 1 ? cols : 1;
    if (ldx < cmin || ldq < cmin) return fail(GEMM_ERR_INVALID_ARG, "%s: ldx or ldq < max(1, cols)", name);
    if (!scale) return fail(GEMM_ERR_INVALID_ARG, "%s: scale is NULL", name);
    if (reinterpret_cast<uintptr_t>(scale) % 4) return fail(GEMM_ERR_INVALID_ARG, "%s: scale is not 4-byte aligned", name);
    if (rows > 0 && cols > 0) {
        if (!x || !q) return fail(GEMM_ERR_INVALID_ARG, "%s: x or q is NULL", name);
        if (reinterpret_cast<uintptr_t>(x) % esz)
            return fail(GEMM_ERR_INVALID_ARG, "%s: x is not aligned to its element size", name);
    }
    if (rows > (int64_t(1) << 40) / cmin)
        return fail(GEMM_ERR_UNSUPPORTED, "%s: more than 2^40 elements", name);
    std::shared_lock<std::shared_mutex> workspace_guard(g_workspace_lock);
    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev, nullptr);
    if (st != GEMM_OK) return st;
    std::unique_lock<std::mutex> stream_guard = lock_stream(*dev, stream);
    if (rows == 0 || cols == 0) {
        // no elements: amax = 0, so the dequantisation scale is 0
        cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), stream);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: clearing scale: %s", name, cudaGetErrorString(e));
        return GEMM_OK;
    }
    qz::QuantParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.x = x;
    prm.q = static_cast<uint8_t *>(q);
    prm.scale_out = scale;
    if (ldx == cols && ldq == cols) {      // contiguous: one long row
        prm.rows = 1;
        prm.cols = rows * cols;
    } else {
        prm.rows = rows;
        prm.cols = cols;
    }
    prm.ldx = ldx;
    prm.ldq = ldq;
    const int64_t unit = qz::unit_elems(x_type);
    prm.units_per_row = (prm.cols + unit - 1) / unit;
    prm.num_units = prm.rows * prm.units_per_row;
    // 16-byte loads of x and 8-byte stores of q need every row start aligned
    // (a single row starts at the bases).
    prm.vec = reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(q) % 8 == 0 &&
              (prm.rows == 1 || ((ldx * esz) % 16 == 0 && ldq % 8 == 0));
    switch (x_type) {
    case qz::kInF32: return launch_quant<qz::kInF32>(*dev, prm, stream);
    case qz::kInF16: return launch_quant<qz::kInF16>(*dev, prm, stream);
    default: return launch_quant<qz::kInBF16>(*dev, prm, stream);
    }
}

}  // namespace

extern "C" {

gemm_status_t gemm_f16_tn(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                          void *C, int64_t ldc, void *stream)
{
    t_last_error[0] = '\0';
    return run_gemm<tn::KindF16>("gemm_f16_tn", M, N, K, A, lda, B, ldb, C, ldc, 1.0f,
                                 static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f8e4m3_tn(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                             int64_t ldb, void *C, int64_t ldc, float scale_a, float scale_b, void *stream)
{
    t_last_error[0] = '\0';
    return run_gemm<tn::KindE4M3>("gemm_f8e4m3_tn", M, N, K, A, lda, B, ldb, C, ldc, scale_a * scale_b,
                                  static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f8e4m3_tn_dscale(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                                    int64_t ldb, void *C, int64_t ldc, const float *scale_a, const float *scale_b,
                                    void *stream)
{
    t_last_error[0] = '\0';
    if (!scale_a || !scale_b) return fail(GEMM_ERR_INVALID_ARG, "gemm_f8e4m3_tn_dscale: a scale pointer is NULL");
    if (reinterpret_cast<uintptr_t>(scale_a) % 4 || reinterpret_cast<uintptr_t>(scale_b) % 4)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_f8e4m3_tn_dscale: a scale pointer is not 4-byte aligned");
    return run_gemm<tn::KindE4M3>("gemm_f8e4m3_tn_dscale", M, N, K, A, lda, B, ldb, C, ldc, 1.0f,
                                  static_cast<cudaStream_t>(stream), true, scale_a, scale_b);
}

gemm_status_t gemm_f16_tn_softmax_stats(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                                        int64_t ldb, void *C, int64_t ldc, float scale, float *row_max,
                                        float *row_sum, void *stream)
{
    t_last_error[0] = '\0';
    if (M > 0 && N > 0) {
        if (!row_max || !row_sum)
            return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_tn_softmax_stats: row_max or row_sum is NULL");
        if (reinterpret_cast<uintptr_t>(row_max) % 4 || reinterpret_cast<uintptr_t>(row_sum) % 4)
            return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_tn_softmax_stats: row_max or row_sum is not 4-byte aligned");
        if (!std::isfinite(scale))
            return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_tn_softmax_stats: scale is not finite");
    }
    return run_gemm<tn::KindF16>("gemm_f16_tn_softmax_stats", M, N, K, A, lda, B, ldb, C, ldc, scale,
                                 static_cast<cudaStream_t>(stream), true, nullptr, nullptr,
                                 M > 0 && N > 0 ? row_max : nullptr, row_sum);
}

gemm_status_t gemm_quantize_e4m3(const void *x, int x_type, int64_t rows, int64_t cols, int64_t ldx, void *q,
                                 int64_t ldq, float *scale, void *stream)
{
    t_last_error[0] = '\0';
    return run_quant(x, x_type, rows, cols, ldx, q, ldq, scale, static_cast<cudaStream_t>(stream));
}

const char *gemm_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

const char *gemm_last_error(void) { return t_last_error; }

gemm_status_t gemm_poll_device_status(void *stream)
{
    t_last_error[0] = '\0';
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, tn::g_tn_status, sizeof(int));
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(tn::g_tn_status, &zero, sizeof(int));
        // A kernel that gave up may have left ticket counts part-way: the next
        // call on each stream clears them before use.
        int dev = -1;
        if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
            std::lock_guard<std::mutex> lock(g_mutex);
            for (auto &kv : g_devices[dev].split) kv.second.dirty = true;
            for (auto &kv : g_devices[dev].stats) kv.second.dirty = true;
        }
        return fail(GEMM_ERR_TIMEOUT, "a kernel's bounded wait ran out (site %d)", v >> 8);
    }
    return GEMM_OK;
}

void gemm_release_workspace(void)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    // waits for calls on other threads to have enqueued their launches
    std::unique_lock<std::shared_mutex> workspace_guard(g_workspace_lock);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    for (auto &kv : d.repack)
        if (kv.second.ptr) cudaFree(kv.second.ptr);
    d.repack.clear();
    for (auto &kv : d.split)
        if (kv.second.ptr) cudaFree(kv.second.ptr);
    d.split.clear();
    for (auto &kv : d.quant)
        if (kv.second.ptr) cudaFree(kv.second.ptr);
    d.quant.clear();
    for (auto &kv : d.stats)
        if (kv.second.ptr) cudaFree(kv.second.ptr);
    d.stats.clear();

}

int gemm_tile_coord(int64_t tiles_m, int64_t tiles_n, int64_t group, int64_t id, int64_t *tile_m, int64_t *tile_n)
{
    if (tiles_m <= 0 || tiles_n <= 0 || group <= 0 || group > INT32_MAX || tiles_m > INT32_MAX / tiles_n || id < 0 ||
        id >= tiles_m * tiles_n || !tile_m || !tile_n)
        return -1;
    tn::tile_coord(id, tiles_m, tiles_n, group, *tile_m, *tile_n);
    return 0;
}

void gemm_set_wait_limit_ns(uint64_t limit_ns) { g_wait_limit_ns.store(limit_ns ? limit_ns : 2000000000ull); }

void gemm_debug_inject_stall(int mode) { g_inject_stall.store(mode >= 0 && mode <= 3 ? mode : 1); }

int gemm_debug_force_cta_group(int group)
{
    if (group != 0 && group != 1 && group != 2) return -1;
    g_force_cta_group.store(group);
    return 0;
}

int gemm_debug_force_wide_tiles(int mode)
{
    if (mode < -1 || mode > 1) return -1;
    g_force_wide.store(mode);
    return 0;
}

int gemm_debug_set_raster_group(int rows)
{
    if (rows < 0 || rows > 64 || rows % 2) return -1;
    g_raster_group.store(rows);
    return 0;
}

int gemm_debug_set_k_order(int mode)
{
    if (mode < 0 || mode > 2) return -1;
    g_k_order.store(mode);
    return 0;
}

void gemm_debug_set_clock_probe(unsigned long long *counters) { g_clock_probe.store(counters); }

int gemm_debug_set_long_k_mode(int mode)
{
    if (mode < 0 || mode > 2) return -1;
    g_long_k.store(mode);
    return 0;
}

int gemm_debug_set_skinny_mode(int mode)
{
    if (mode < 0 || mode > 2) return -1;
    g_skinny.store(mode);
    return 0;
}

int gemm_debug_set_lean_mode(int mode)
{
    if (mode < 0 || mode > 2) return -1;
    g_lean.store(mode);
    return 0;
}

const char *gemm_debug_last_launch(void)
{
    const LaunchRecord &r = t_rec;
    if (!r.name)
        t_last_launch[0] = '\0';
    else if (r.quant)
        snprintf(t_last_launch, sizeof(t_last_launch), "%s: grid=%lld units=%lld vec=%d", r.name, r.qgrid, r.qunits,
                 r.vec);
    else
        snprintf(t_last_launch, sizeof(t_last_launch),
                 "%s: ctas_per_cluster=%d wide=%d grid=%d clusters=%d slots=%d tiles=%d units=%d tail_start=%d "
                 "tail_mode=%d split_parts=%d lean=%d skinny=%d",
                 r.name, r.cluster, r.wide, r.grid, r.clusters, r.slots, r.tiles, r.units,
                 r.tail_start, r.tail_mode, r.split_parts, r.lean, r.skinny);
    return t_last_launch;
}

const char *gemm_build_info(void)
{
    static char info[768];
    snprintf(info, sizeof(info),
             "dense_gemm_tn sm_103a: CTA-pair tile 256x256 in 2-CTA clusters, %d stages of %d B "
             "of K, %d B smem; CTA-pair tile 256x512, %d stages of %d B of K, %d B smem; 1-CTA tile 128x256, "
             "%d stages of %d B of K, %d B smem; TMEM %u cols; lean 1-CTA quarter-m units, %d stages, %d B smem, "
             "TMEM %u cols; half-m units, %d stages, %d B smem, TMEM %u cols; N <= %d: 128-row m tiles, %d stages, "
             "%d B smem, TMEM %u cols; raster group %d",
             tn::TileCfg<2>::kStages, tn::TileCfg<2>::kStageKBytes, tn::TileCfg<2>::kSmemBytes,
             tn::TileCfg<2, true>::kStages, tn::TileCfg<2, true>::kStageKBytes, tn::TileCfg<2, true>::kSmemBytes,
             tn::TileCfg<1>::kStages, tn::TileCfg<1>::kStageKBytes, tn::TileCfg<1>::kSmemBytes, tn::TileCfg<1>::kTmemCols,
             tn::TileCfg<1, false, 4>::kStages, tn::TileCfg<1, false, 4>::kSmemBytes,
             tn::TileCfg<1, false, 4>::kTmemCols, tn::TileCfg<1, false, 2>::kStages,
             tn::TileCfg<1, false, 2>::kSmemBytes, tn::TileCfg<1, false, 2>::kTmemCols, tn::kSkMaxN, tn::kSkStages,
             tn::kSkSmemBytes, tn::kSkTmemCols, kGroupM);
    return info;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_f16_tn_noalloc: the FP16 entry point for callers that must not have the
// library allocate device memory.  Where gemm_f16_tn would grow its repack
// workspace with cudaMalloc, this variant copies the operand(s) into a fixed
// array that is part of the library's device image.  Once repacked, the
// operands are 16-byte aligned with a padded K (zero filled), so the ordinary
// FP16 path runs on them without touching its own workspace.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB on every device that loads the library

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself: on the host it names a stand-in, not device memory).
void *g_noalloc_scratch_ptr[kMaxDevices] = {};

// Held from a call's copy into the array through its GEMM launch, so that two
// host threads' calls on one stream do not enqueue copy, copy, GEMM, GEMM.
std::mutex g_noalloc_issue;

gemm_status_t noalloc_scratch(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_noalloc_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(GEMM_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_noalloc_scratch_ptr[dev] = p;
    }
    *out = g_noalloc_scratch_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_f16_tn_noalloc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                             const void *B, int64_t ldb, void *C, int64_t ldc, void *stream)
{
    t_last_error[0] = '\0';
    const char *name = "gemm_f16_tn_noalloc";
    constexpr int64_t esz = 2;
    const int64_t kmin = K > 1 ? K : 1;
    // Arguments the ordinary path would reject are handed to it unchanged so
    // the caller sees the same status and message; nothing is copied for them.
    const bool plain = M <= 0 || N <= 0 || K <= 0 || lda < kmin || ldb < kmin || ldc < (M > 1 ? M : 1) ||
                       M > kMaxDim || N > kMaxDim || K > kMaxDim || lda > kMaxDim || ldb > kMaxDim ||
                       ldc > kMaxDim || !A || !B || !C || reinterpret_cast<uintptr_t>(A) % esz ||
                       reinterpret_cast<uintptr_t>(B) % esz;
    if (plain)
        return run_gemm<tn::KindF16>(name, M, N, K, A, lda, B, ldb, C, ldc, 1.0f,
                                     static_cast<cudaStream_t>(stream), false);

    const bool k_aligned = (K * esz) % 16 == 0;
    const bool repack_a = !k_aligned || (lda * esz) % 16 != 0 || reinterpret_cast<uintptr_t>(A) % 16 != 0;
    const bool repack_b = !k_aligned || (ldb * esz) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0;
    if (!repack_a && !repack_b)
        return run_gemm<tn::KindF16>(name, M, N, K, A, lda, B, ldb, C, ldc, 1.0f,
                                     static_cast<cudaStream_t>(stream), false);

    const int64_t ldp = (K + 7) / 8 * 8;
    const size_t bytes_a = repack_a ? ((size_t(M) * ldp * esz + 255) & ~size_t(255)) : 0;
    const size_t bytes_b = repack_b ? ((size_t(N) * ldp * esz + 255) & ~size_t(255)) : 0;
    if (bytes_a + bytes_b > kNoAllocScratchBytes)
        return fail(GEMM_ERR_INVALID_ARG,
                    "%s: the repacked operands need %zu bytes, more than the fixed %zu-byte scratch array", name,
                    bytes_a + bytes_b, kNoAllocScratchBytes);

    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev, nullptr);
    if (st != GEMM_OK) return st;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != GEMM_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    std::lock_guard<std::mutex> issue_guard(g_noalloc_issue);
    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb;
    tn::RepackJob<uint16_t> ja{static_cast<const uint16_t *>(A), lda, reinterpret_cast<uint16_t *>(ws), ldp,
                               repack_a ? M : 0, K};
    tn::RepackJob<uint16_t> jb{static_cast<const uint16_t *>(B), ldb, reinterpret_cast<uint16_t *>(ws + bytes_a), ldp,
                               repack_b ? N : 0, K};
    launch_repack<uint16_t>(ja, jb, s);
    if (repack_a) {
        a_use = ws;
        lda_use = ldp;
    }
    if (repack_b) {
        b_use = ws + bytes_a;
        ldb_use = ldp;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "%s: repack launch: %s", name, cudaGetErrorString(e));
    // When K is not a multiple of 8 both operands were repacked with zeros in
    // columns K..ldp-1; those extra products are +0 and leave every sum as is.
    const int64_t k_use = k_aligned ? K : ldp;
    st = run_gemm<tn::KindF16>(name, M, N, k_use, a_use, lda_use, b_use, ldb_use, C, ldc, 1.0f, s, false);
    if (st != GEMM_OK) return st;
    return GEMM_OK;
}
