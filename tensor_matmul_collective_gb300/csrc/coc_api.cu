// Host side of the C ABI declared in include/coc.h: argument validation
// (before any CUDA call), TMA descriptor encoding, launch of the persistent
// fused kernel, and the device status buffer used by the bounded waits.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <utility>

#include <cudaTypedefs.h>

#include "coc_internal.h"

namespace coc {
namespace {

thread_local char g_err[512] = "";

coc_status_t fail(coc_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

coc_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(COC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<int> g_inject{0};
std::atomic<int> g_clock_slot{-1};         // coc_debug_clock_probe
std::atomic<long long> g_alloc_calls{0};   // device allocations made by the library (coc_debug_alloc_count)

// Scratch owned by the library for the calls made on one stream: the
// rank-split fp32 parts, the MoE routing tables, the w8A16 pre-pass weight.
// Allocated at the first call on the stream that needs it and grown only when
// a call needs more, so steady-state calls allocate nothing.  `last_use` is
// recorded after every call that used it and waited on by the next one, so a
// stream handle that is reused after cudaStreamDestroy can never overlap the
// previous owner's kernels.
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    cudaEvent_t last_use = nullptr;
};

struct DeviceState {
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned* status = nullptr;
    int max_pairs[NUM_OPS][2] = {{-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}};   // per op, per bf16; -1 = not queried
    int ts_pairs[2] = {-1, -1};     // co-resident pairs of the w8A16 tensor-memory kernel, per bf16
    int split_clusters[2][2][2] = {{{-1, -1}, {-1, -1}}, {{-1, -1}, {-1, -1}}};   // [RS][bf16][ksplit 4]: co-resident
    std::unordered_map<long long, int> slab_clusters;   // column-slab clusters co-resident, by launch shape
    cudaMemPool_t pool = nullptr;   // stream-ordered allocations of calls captured into CUDA graphs
    std::unordered_map<cudaStream_t, Workspace> ws;   // per-stream scratch of eager calls
};

std::mutex g_mu;
std::unordered_map<int, DeviceState> g_dev;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

coc_status_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(COC_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    DeviceState& st = g_dev[dev];
    if (st.status == nullptr) {
        if ((e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (st.cc_major != 10 || st.cc_minor != 3)
            return fail(COC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                        st.cc_major, st.cc_minor);
        void* p = nullptr;
        g_alloc_calls.fetch_add(1);
        if ((e = cudaMalloc(&p, STATUS_BLOCK_WORDS * sizeof(unsigned))) != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
        if ((e = cudaMemset(p, 0, STATUS_BLOCK_WORDS * sizeof(unsigned))) != cudaSuccess) {
            cudaFree(p);
            return cuda_fail(e, "cudaMemset(status)");
        }
        st.status = static_cast<unsigned*>(p);
    }
    if (st.pool == nullptr) {
        // the pool that captured calls allocate their scratch from; created
        // here, by the first call on the device, because creating it while a
        // stream is being captured would invalidate the capture
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = UINT64_MAX;   // keep freed memory for the next replay / capture
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return cuda_fail(e, "cudaMemPoolSetAttribute");
        }
        st.pool = pool;
    }
    *out = &st;
    return COC_OK;
}

// 2-D row-major tensor map: inner dimension `cols` (contiguous), `rows` rows of
// `pitch_bytes`, box of box_cols x box_rows.
coc_status_t encode(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                    uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(COC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llu x %llu, pitch %llu", static_cast<int>(r),
                    static_cast<unsigned long long>(rows), static_cast<unsigned long long>(cols),
                    static_cast<unsigned long long>(pitch_bytes));
    return COC_OK;
}

// 3-D view of a row-major matrix for stage-sized boxes: element (i, r, j) at
// base + (j d0 + i) * elem + r pitch, i.e. dims (d0 = one block of the inner
// dimension, rows, blocks), strides (pitch, d0 * elem).  Returns the driver's
// result without reporting (the caller falls back to 2-D boxes).
CUresult encode_blocked(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t rows,
                        uint64_t blocks, uint64_t pitch_bytes, uint32_t box0, uint32_t box_rows, uint32_t box_blocks) {
    const cuuint64_t dims[3] = {d0, rows, blocks};
    const cuuint64_t strides[2] = {pitch_bytes, d0 * 2};
    const cuuint32_t box[3] = {box0, box_rows, box_blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1024;

bool pow2_rank(int v) { return v == 1 || v == 2 || v == 4 || v == 8; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

coc_status_t check_common(int R, int chunks, coc_dtype_t dt, int deterministic) {
    (void)deterministic;
    if (!pow2_rank(R)) return fail(COC_ERR_INVALID_ARG, "R = %d; must be 1, 2, 4 or 8", R);
    if (!pow2_rank(chunks)) return fail(COC_ERR_INVALID_ARG, "chunks = %d; must be 1, 2, 4 or 8", chunks);
    if (dt != COC_FP16 && dt != COC_BF16) return fail(COC_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    return COC_OK;
}

coc_status_t check_dims(int64_t a, int64_t b, int64_t c) {
    if (a < 0 || b < 0 || c < 0) return fail(COC_ERR_SHAPE, "negative size");
    if (a > kMaxDim || b > kMaxDim || c > kMaxDim) return fail(COC_ERR_SHAPE, "size above 2^31 - 1024");
    return COC_OK;
}

// R device pointers; all non-null and 16-byte aligned when `needed`.
coc_status_t check_ptrs(const void* const* arr, int R, bool needed, const char* name, bool allow_null_entries = false) {
    if (arr == nullptr) return fail(COC_ERR_INVALID_ARG, "%s is NULL", name);
    if (!needed) return COC_OK;
    for (int r = 0; r < R; ++r) {
        if (arr[r] == nullptr) {
            if (allow_null_entries) continue;
            return fail(COC_ERR_INVALID_ARG, "%s[%d] is NULL", name, r);
        }
        if (!aligned16(arr[r])) return fail(COC_ERR_ALIGN, "%s[%d] is not 16-byte aligned", name, r);
    }
    return COC_OK;
}

int chunk_m_tiles(int64_t m, int chunks, int tile_m) {
    const int64_t rows = m / chunks;
    return (rows > 0 && rows % tile_m == 0) ? static_cast<int>(rows / tile_m) : 0;
}

// The 2-SM variant (a CTA pair per 256-row tile) is used once the output has
// more than one 128-row tile; the AllReduce and ReduceScatter keep single-CTA
// tiles up to two of them (twice the tiles over the same SMs: the 8-rank
// layer with n 8192, K 8 x 1024 at m 129-256 measured 45-46 us against 50-52
// with pairs; from 384 rows pairs are faster).  COC_PAIR=0/1 forces a
// variant (tuning only).
int pair_forced() {
    static const int forced = [] {
        const char* e = std::getenv("COC_PAIR");
        return e == nullptr ? -1 : (std::atoi(e) != 0 ? 1 : 0);
    }();
    return forced;
}

bool use_pair(int op, int64_t m) {
    if (pair_forced() >= 0) return pair_forced() == 1;
    if ((op == OP_AR || op == OP_RS) && m <= 2 * BM) return false;
    return m > BM;
}

// Largest divisor of chunk_mt whose A rows (row_tile_bytes each) fit in
// 32 MiB of L2; 0 (no grouping) when the whole chunk fits or nothing does.
int l2_group(int chunk_mt, int64_t row_tile_bytes) {
    constexpr int64_t kBudget = int64_t(32) << 20;
    if (chunk_mt <= 0 || row_tile_bytes <= 0 || chunk_mt * row_tile_bytes <= kBudget) return 0;
    for (int g = chunk_mt - 1; g >= 2; --g)
        if (chunk_mt % g == 0 && g * row_tile_bytes <= kBudget) return g;
    return 0;
}

// Row-parallel operators (AR/RS/w8A16): every (m-tile, n-tile) unit reads an
// X row tile of x_tile bytes (all ranks' shards) and a W column tile of
// w_tile bytes.  In m-tile-inner order the concurrently running units share
// W columns and need all of the chunk's X rows, which are re-read once per
// wave of units when they do not fit in L2.  Grouping G m-tiles (their X
// rows held in L2) reads X once but W once per group.  Returns the group
// size with the smaller modelled DRAM read volume, 0 for no grouping.
int row_group(int chunk_mt, int n_tiles, int64_t x_tile, int64_t w_tile, int concurrent) {
    constexpr int64_t kBudget = int64_t(32) << 20;
    if (chunk_mt <= 0 || x_tile <= 0 || chunk_mt * x_tile <= kBudget || concurrent <= 0) return 0;
    const int64_t waves = (static_cast<int64_t>(chunk_mt) * n_tiles + concurrent - 1) / concurrent;
    int64_t best = waves * chunk_mt * x_tile + n_tiles * w_tile;
    int best_g = 0;
    for (int g = chunk_mt - 1; g >= 2; --g) {
        if (chunk_mt % g != 0 || g * x_tile > kBudget) continue;
        const int64_t t = chunk_mt * x_tile + static_cast<int64_t>(chunk_mt / g) * n_tiles * w_tile;
        if (t < best) {
            best = t;
            best_g = g;
        }
    }
    return best_g;
}

int pairs_available(DeviceState* ds, int op, bool bf16) {
    std::lock_guard<std::mutex> lk(g_mu);
    int& v = ds->max_pairs[op][bf16 ? 1 : 0];
    if (v < 0) v = max_pairs(op, bf16);
    return v;
}

// ALL_GATHER_MATMUL's tile shape for m gathered rows and col_units (rank,
// n-tile) columns: 256-row pair tiles run about 15% faster per tile than
// 128-row single-CTA tiles, so pairs, unless the single-CTA tiles take
// clearly fewer rounds (tiles / co-resident pairs or CTAs, at least one):
// where a last pair tile would be at most half full among few row tiles.
// Measured (8 ranks, n_shard 7168, k 8192, 224 columns): m 384 269 against
// 296 us, m 640 413 against 447 single-CTA; m 512 / 768 / 1280 pairs (275 /
// 397 / 650 against 319 / 455 / 743).  The AllReduce and ReduceScatter, with
// 32 columns at n 8192, ran pairs faster at m 384 and 640 (56 / 98 against
// 66 / 116 us): both shapes fit one round there.
bool ag_use_pair(DeviceState* ds, int64_t m, int64_t col_units, bool bf16) {
    if (pair_forced() >= 0 || m <= 2 * BM) return use_pair(OP_AG, m);
    const int pairs = pairs_available(ds, OP_AG, bf16);
    if (pairs <= 0 || ds->sm_count <= 0) return true;
    const double rp = std::max(1.0, static_cast<double>((m + 2 * BM - 1) / (2 * BM)) * col_units / pairs);
    const double rs = std::max(1.0, static_cast<double>((m + BM - 1) / BM) * col_units / ds->sm_count);
    return !(rs < 0.85 * rp);
}

int largest_pow2_divisor_le(int64_t v, int cap) {
    int b = cap;
    while (b > 8 && v % b != 0) b >>= 1;
    return b;
}

CUtensorMapDataType tma_dtype(coc_dtype_t dt) {
    return dt == COC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

coc_status_t launch_checked(int op, bool bf16, bool pair, KParams& p, DeviceState* ds, cudaStream_t stream) {
    p.status = ds->status;
    p.inject_timeout = g_inject.load();
    p.clock_slot = g_clock_slot.load();
    int grid;
    if (pair) {
        const int pairs = pairs_available(ds, op, bf16);
        if (pairs <= 0) return fail(COC_ERR_CUDA, "no co-resident CTA pair fits on this device");
        grid = 2 * (p.units < pairs ? p.units : pairs);
    } else {
        grid = p.units < ds->sm_count ? p.units : ds->sm_count;
    }
    cudaError_t e = launch(op, bf16, pair, p, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return COC_OK;
}

coc_status_t device_pool(DeviceState* ds, cudaMemPool_t* out);

// Scratch for one call (see Workspace): a region of at least `bytes` bytes,
// usable by the kernels the call puts on `stream`.  Eager calls get the
// stream's persistent workspace (allocated or grown only when too small);
// calls captured into a CUDA graph get a stream-ordered allocation from the
// device pool, which becomes a memory node of the graph, so graph replays
// call no allocator either.  scratch_release ends the call's use.
struct Scratch {
    void* ptr = nullptr;
    bool captured = false;
    Workspace* w = nullptr;
};
constexpr size_t kWorkspaceCap = size_t(4) << 30;   // largest scratch one call may take
coc_status_t scratch_acquire(DeviceState* ds, cudaStream_t stream, size_t bytes, Scratch* out);
coc_status_t scratch_release(cudaStream_t stream, Scratch& sc, coc_status_t st);

// Rank split (AllReduce, ReduceScatter, single-CTA tiles: m <= 128): with at
// most half as many output tiles as SMs (decode-sized m), each tile's R shards
// are cut into ksplit parts of R / ksplit shards, one work unit each, so the
// weight stream is spread over ksplit times more SMs; ksplit is the largest
// power of two dividing R that keeps the units within one wave.  It depends
// on the shape only (never on chunks), so results stay bitwise
// chunk-independent.  Measured (8 ranks, n 8192, k_shard 1024, bf16, one
// call in a CUDA graph): m 1 / 16 / 64 / 128 take 48 / 42 / 42 / 49 us split
// in 4 against 70 / 62 / 55 / 60 us unsplit; for 256-row tiles (m > 128)
// splitting gained nothing (m 256: 54 us either way), so they are not split.
// COC_SPLIT_PATH=scratch forces the rank split through global scratch
// instead of a cluster's shared memory (tests and tuning only; both give the
// same bits: the same parts added in the same order).
bool split_cluster_allowed() {
    const char* e = std::getenv("COC_SPLIT_PATH");
    return !(e != nullptr && std::strcmp(e, "scratch") == 0);
}

int rank_split(int op, int R, int64_t ks, int64_t tiles, bool pair, int sm_count) {
    int ksplit = 1;
    if ((op == OP_AR || op == OP_RS) && ks > 0 && R > 1) {
        const char* e = std::getenv("COC_KSPLIT");   // forces the part count (tuning and tests only)
        if (e != nullptr) {
            const int f = std::atoi(e);
            while (ksplit * 2 <= f && ksplit < R) ksplit *= 2;
            return ksplit;
        }
        if (pair) return 1;
        while (ksplit < R && tiles * ksplit * 2 <= sm_count) ksplit *= 2;
    }
    return ksplit;
}

// Column-slab kernel (coc_slab.cu) for decode-sized m (m <= 128, one row
// tile).  Plan: 128-column slabs (256-byte weight rows: measured faster than
// 64 columns, whose 128-byte rows moved 30% less per SM), two k-blocks per
// stage (one TMA operation per 64-column group and one for X), and, while the
// slabs fill at most half of the SMs, each slab's contraction split over a
// cluster of 2 or 4 CTAs.  Taken for every m <= 128, even where the CTAs fill
// few SMs.  Measured (8 ranks, K 8 x 1024, bf16, CUDA graph): n 8192 at m 16
// / 64 / 96 / 128 takes 27.0 / 27.7 / 30.0 / 37.1 us against 34.1 / 34.4 /
// 37.0 / 41.5 us for the persistent kernel's rank split, and n 1024 / 2048 at
// m 16 13.5 / 13.6 against 33.9 / 33.8 us.  COC_SLAB=0 turns the kernel off;
// COC_SLAB=1 takes it whenever m <= 128, with COC_SLAB_BOXES, COC_SLAB_KPS
// and COC_SLAB_SPLIT overriding the plan (tests and tuning only).
struct SlabPlan {
    int boxes = 0, split = 1, kps = 1;
};
}  // namespace

bool pdl_launch() {
    static const bool on = [] {
        const char* e = std::getenv("COC_PDL");
        return e == nullptr || std::atoi(e) != 0;
    }();
    return on;
}

namespace {

int env_int(const char* name, int dflt) {
    const char* e = std::getenv(name);
    return e == nullptr ? dflt : std::atoi(e);
}
// The column-slab schedule of one slab width (64 boxes columns) and kps0
// k-blocks per stage (fewer where they do not divide the k-blocks or two
// stages do not fit); boxes = 0 where the slabs would not fill the SMs.
SlabPlan slab_plan_for(int op, int R, int64_t m, int64_t n, int64_t ks, int sm_count, int boxes, int kps0,
                       bool forced) {
    SlabPlan pl;
    const bool w8 = (op == OP_W8);
    const int64_t kblocks = (ks + BK - 1) / BK;
    int kps = kps0 >= 4 ? 4 : kps0 >= 2 ? 2 : 1;
    while (kps > 1 && kblocks % kps != 0) kps /= 2;
    // AllGather: R rank outputs of n columns, each slab's contraction the
    // whole k; otherwise one output, each slab summed over the R shards
    const int64_t slabs = (op == OP_AG ? R : 1) * ((n + 64 * boxes - 1) / (64 * boxes));
    const int64_t spu = static_cast<int64_t>(op == OP_AG ? 1 : R) * (kblocks / kps);   // stages per slab
    int split = 1;
    // (each part finalises 64 boxes / split >= 32 columns and sums at least one stage)
    const int max_split = boxes == 1 ? 2 : 4;
    while (split < max_split && slabs * split * 2 <= sm_count && split * 2 <= spu) split *= 2;
    const int fs = env_int("COC_SLAB_SPLIT", 0);
    if ((fs == 1 || fs == 2 || fs == 4) && fs <= max_split && fs <= spu) split = fs;
    (void)forced;   // (slabs that fill few SMs still beat the persistent kernel's rank split:
                    // 8 ranks, K 8 x 1024, m 16, n 1024 / 2048: 13.4 / 13.6 against 33.9 / 33.8 us)
    // two stages at least must fit in shared memory (w8A16 also holds the
    // 16-bit ring): fewer k-blocks per stage where they do not
    const int a_rows = static_cast<int>((m + 7) / 8 * 8);
    while (kps > 1 && slab_smem_bytes(2, a_rows, boxes, kps, split, w8) > kSlabSmemCap) kps /= 2;
    if (slab_smem_bytes(2, a_rows, boxes, kps, split, w8) > kSlabSmemCap) return pl;
    pl.boxes = boxes;
    pl.split = split;
    pl.kps = kps;
    return pl;
}

SlabPlan slab_plan(int op, int R, int64_t m, int64_t n, int64_t ks, int sm_count) {
    SlabPlan pl;
    if ((op != OP_AR && op != OP_RS && op != OP_W8 && op != OP_AG) || ks <= 0 || m <= 0 || m > BM) return pl;
    const int forced = env_int("COC_SLAB", -1);
    if (forced == 0) return pl;
    const int env_boxes = env_int("COC_SLAB_BOXES", 0);
    const int env_kps = env_int("COC_SLAB_KPS", 0);
    if (op == OP_W8 && env_boxes == 0) {
        // w8A16: the schedule with the most int8 weight bytes in flight over
        // all its CTAs (stages x int8 stage bytes x CTAs at once, per round;
        // ties: 128 columns), 256-column slabs counted a quarter more up to
        // 32 rows (their int8 rows are read as 256-byte segments; measured
        // fastest from 1 to 32 rows at n 8192, 30.4 against 32.5 us at m 1
        // with fewer bytes in flight per CTA; at m 64 128 columns, 34.6
        // against 36.9 us).  Every candidate keeps 16 KiB int8 boxes:
        // smaller ones stream far slower.
        const int a_rows = static_cast<int>((m + 7) / 8 * 8);
        long long best = 0;
        for (const auto& c : {std::pair<int, int>{2, 2}, {4, 1}, {1, 4}}) {
            const SlabPlan cand = slab_plan_for(op, R, m, n, ks, sm_count, c.first, c.second, forced == 1);
            if (cand.boxes == 0 || cand.kps != c.second) continue;
            const int st = slab_stages(a_rows, cand.boxes, cand.kps, cand.split, true);
            // CTAs working at once, averaged over the rounds the units take
            const long long units = (n + 64 * cand.boxes - 1) / (64 * cand.boxes) * cand.split;
            const long long ctas = units / ((units + sm_count - 1) / sm_count);
            const long long score = static_cast<long long>(st) * cand.kps * 64 * 64 * cand.boxes * ctas *
                                    ((cand.boxes == 4 && a_rows <= 32) ? 5 : 4);
            if (score > best) {
                best = score;
                pl = cand;
            }
        }
        return pl;
    }
    // 128-column slabs (64 with COC_SLAB_BOXES=1; w8A16 also 256 with 4).
    // k-blocks per stage: 4 for 64-column slabs, 2 for 128 (measured best; at
    // m = 128 two stages of 2 k-blocks beat five of 1: fewer TMA operations
    // in flight matter more than ring depth), 1 for 256
    const int boxes = env_boxes == 1 ? 1 : (op == OP_W8 && env_boxes >= 4) ? 4 : 2;
    const int kps = boxes == 4 ? 1 : (env_kps > 0 ? env_kps : boxes == 1 ? 4 : 2);
    return slab_plan_for(op, R, m, n, ks, sm_count, boxes, kps, forced == 1);
}

// A split slab takes one cluster for its whole life (the parts' reception
// areas are not reused), so every slab needs a resident cluster: where the
// clusters of `split` CTAs do not all fit at once, smaller ones are taken
// (measured, 8 ranks, n 4864, K 8 x 2048, m 16: 38 slabs in clusters of 4,
// of which only 32 fit at once, ran unsplit in 65.6 us; in clusters of 2
// they take 36.9 us).
int slab_resident_split(DeviceState* ds, bool bf16, bool w8, int boxes, int kps, int a_rows, int split, int units) {
    while (split > 1) {
        const int smem = slab_smem_bytes(slab_stages(a_rows, boxes, kps, split, w8), a_rows, boxes, kps, split, w8);
        const long long key = (static_cast<long long>(w8) << 41) | (static_cast<long long>(bf16) << 40) |
                              (static_cast<long long>(split) << 32) | smem;
        int clusters = 0;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            auto it = ds->slab_clusters.find(key);
            if (it == ds->slab_clusters.end())
                it = ds->slab_clusters.emplace(key, slab_max_clusters(bf16, w8, split, smem)).first;
            clusters = it->second;
        }
        if (clusters >= units) break;
        split /= 2;
    }
    return split;
}

// op OP_W8: the w8A16 AllReduce (int8 w, scales / zero points as for the
// persistent kernel).
coc_status_t slab_row_parallel(int op, int R, int64_t m, int64_t n, int64_t ks, const void* const* x,
                               const void* const* w, void* const* out, int n_out, coc_dtype_t dt, const SlabPlan& pl,
                               DeviceState* ds, cudaStream_t stream, bool w_nk, const void* const* scale,
                               coc_scale_t gran, int64_t group, const void* const* zero) {
    const bool w8 = (op == OP_W8);
    KParams p;
    std::memset(&p, 0, sizeof p);
    p.R = R;
    p.n_out = n_out;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(ks);
    p.num_kshards = R;
    p.kblocks = static_cast<int>((ks + BK - 1) / BK);
    p.m_tiles = 1;
    p.n_tiles = static_cast<int>((n + 64 * pl.boxes - 1) / (64 * pl.boxes));
    p.units = p.n_tiles;
    p.rows_per_rank = static_cast<int>(m / R);
    p.a_box_rows = static_cast<int>((m + 7) / 8 * 8);
    const int kps = pl.kps, boxes = pl.boxes;
    const int split = slab_resident_split(ds, dt == COC_BF16, w8, boxes, kps, p.a_box_rows, pl.split, p.units);
    p.slab_boxes = boxes;
    p.slab_kps = kps;
    p.slab_split = split;
    p.slab_stages = slab_stages(p.a_box_rows, boxes, kps, split, w8);
    if (slab_smem_bytes(p.slab_stages, p.a_box_rows, boxes, kps, split, w8) > kSlabSmemCap)
        return fail(COC_ERR_SHAPE, "column-slab schedule does not fit in shared memory (m = %lld)", (long long)m);
    p.b_kmajor = w_nk ? 1 : 0;
    const CUtensorMapDataType adt = tma_dtype(dt);
    coc_status_t st;
    // 3-D maps (one A box per stage; n x k B likewise) where the k-blocks tile
    // k_shard exactly, so that no box reads past a row's end
    bool a3d = kps > 1 && ks % BK == 0;
    for (int r = 0; a3d && r < R; ++r) {
        a3d = encode_blocked(&p.tm_a[r], adt, x[r], BK, m, ks / BK, ks * 2, BK, p.a_box_rows, kps) == CUDA_SUCCESS;
        if (a3d && w_nk)
            a3d = encode_blocked(&p.tm_b[r], adt, w[r], BK, n, ks / BK, ks * 2, BK, 64 * boxes, kps) == CUDA_SUCCESS;
    }
    p.slab_a3d = a3d ? 1 : 0;
    for (int r = 0; r < R; ++r) {
        if (!a3d) {
            if ((st = encode(&p.tm_a[r], adt, x[r], ks, m, ks * 2, BK, p.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
            if (w_nk && (st = encode(&p.tm_b[r], adt, w[r], ks, n, ks * 2, BK, 64 * boxes, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
        }
        if (w8) {
            // int8 W: one box of the slab's columns x the stage's k-blocks, unswizzled
            st = encode(&p.tm_b[r], CU_TENSOR_MAP_DATA_TYPE_UINT8, w[r], n, ks, n, 64 * boxes, BK * kps,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != COC_OK) return st;
        } else if (!w_nk &&
                   (st = encode(&p.tm_b[r], adt, w[r], n, ks, n * 2, 64, BK * kps, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK) {
            return st;
        }
    }
    if (w8) {
        p.gran = static_cast<int>(gran);
        p.group = static_cast<int>(group);
        for (int r = 0; r < R; ++r) p.scale[r] = static_cast<const uint16_t*>(scale[r]);
        if (zero != nullptr) {
            p.has_zero = 1;
            for (int r = 0; r < R; ++r) p.zero[r] = static_cast<const int8_t*>(zero[r]);
        }
    }
    for (int o = 0; o < (op == OP_RS ? R : n_out); ++o) p.outp[o] = static_cast<uint16_t*>(out[o]);
    p.status = ds->status;
    p.inject_timeout = g_inject.load();
    p.clock_slot = g_clock_slot.load();
    const int grid = split > 1 ? split * p.units : (p.units < ds->sm_count ? p.units : ds->sm_count);
    const cudaError_t e = launch_slab(w8 ? OP_AR : op, dt == COC_BF16, w8, p, grid, stream);
    return e == cudaSuccess ? COC_OK : cuda_fail(e, "kernel launch (column slabs)");
}

// ---- row-parallel family: AR, RS, W8, plain ----------------------------------
// w_nk: each W shard is stored n x k_shard (Megatron's [out, in]) instead of
// k_shard x n; the kernel then reads B K-major.
coc_status_t row_parallel(int op, int R, int64_t m, int64_t n, int64_t ks, const void* const* x,
                          const void* const* w, void* const* out, int n_out, coc_dtype_t dt, int chunks,
                          const void* const* scale, coc_scale_t gran, int64_t group, cudaStream_t stream,
                          bool w_nk = false, const void* const* zero = nullptr, bool allow_split = true) {
    KParams p;
    std::memset(&p, 0, sizeof p);
    p.b_kmajor = w_nk ? 1 : 0;
    p.R = R;
    p.n_out = n_out;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(ks);
    p.num_kshards = R;
    const bool pair = use_pair(op, m);
    const int tile_m = pair ? 2 * BM : BM;
    p.kblocks = static_cast<int>((ks + BK - 1) / BK);
    p.m_tiles = static_cast<int>((m + tile_m - 1) / tile_m);
    p.n_tiles = static_cast<int>((n + BN - 1) / BN);
    p.units = p.m_tiles * p.n_tiles;
    p.chunk_mt = chunk_m_tiles(m, chunks, tile_m);
    p.rows_per_rank = static_cast<int>(m / R);
    p.store_rows = 32;
    p.a_box_rows = BM;
    p.gran = static_cast<int>(gran);
    p.group = static_cast<int>(group);
    if (op == OP_RS) p.store_rows = largest_pow2_divisor_le(p.rows_per_rank, 32);

    DeviceState* ds = nullptr;
    coc_status_t st = device_state(&ds);
    if (st != COC_OK) return st;
    if (allow_split) {
        const SlabPlan pl = slab_plan(op, R, m, n, ks, ds->sm_count);
        if (pl.boxes > 0)
            return slab_row_parallel(op, R, m, n, ks, x, w, out, n_out, dt, pl, ds, stream, w_nk, scale, gran, group, zero);
    }

    const bool w8 = (op == OP_W8);
    const CUtensorMapDataType adt = tma_dtype(dt);
    {
        const int64_t k_total = static_cast<int64_t>(R) * ks;
        const int concurrent = pair ? pairs_available(ds, op, dt == COC_BF16) : ds->sm_count;
        p.group_mt = row_group(p.chunk_mt, p.n_tiles, int64_t(tile_m) * k_total * 2, int64_t(BN) * k_total * (w8 ? 1 : 2),
                               concurrent);
        if (p.group_mt > 0) p.a_hint = 2;   // the group's X rows stay in L2 while W streams past
    }
    if (ks > 0) {
        for (int r = 0; r < R; ++r) {
            if ((st = encode(&p.tm_a[r], adt, x[r], ks, m, ks * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK) return st;
            if (w8) {
                st = encode(&p.tm_b[r], CU_TENSOR_MAP_DATA_TYPE_UINT8, w[r], n, ks, n, pair ? BN / 2 : BN, BK,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
            } else if (w_nk) {
                st = encode(&p.tm_b[r], adt, w[r], ks, n, ks * 2, BK, pair ? BN / 2 : BN, CU_TENSOR_MAP_SWIZZLE_128B);
            } else {
                st = encode(&p.tm_b[r], adt, w[r], n, ks, n * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
            }
            if (st != COC_OK) return st;
        }
    }
    const int64_t out_rows = (op == OP_RS) ? m / R : m;
    for (int o = 0; o < n_out; ++o) {
        if ((st = encode(&p.tm_out[o], adt, out[o], n, out_rows, n * 2, EPI_COLS, p.store_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
            return st;
    }
    if (w8) {
        for (int r = 0; r < R; ++r) p.scale[r] = static_cast<const uint16_t*>(scale[r]);
        if (zero != nullptr) {
            p.has_zero = 1;
            for (int r = 0; r < R; ++r) p.zero[r] = static_cast<const int8_t*>(zero[r]);
        }
    }
    if ((op == OP_AR || op == OP_W8) && n_out > 1) {
        for (int o = 0; o < n_out; ++o) p.outp[o] = static_cast<uint16_t*>(out[o]);
        p.replica_stores = 1;
    }
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int ksplit = allow_split ? rank_split(op, R, ks, tiles, pair, ds->sm_count) : 1;
    if (ksplit == 1) return launch_checked(op, dt == COC_BF16, pair, p, ds, stream);

    p.ksplit = ksplit;
    p.units = static_cast<int>(tiles * ksplit);
    for (int o = 0; o < (op == OP_RS ? R : n_out); ++o) p.outp[o] = static_cast<uint16_t*>(out[o]);
    // rank split through distributed shared memory: the ksplit part-CTAs of a
    // tile are one cluster, one unit per CTA (all tiles' clusters co-resident)
    if (!pair && (ksplit == 2 || ksplit == 4) && split_cluster_allowed()) {
        int clusters = 0;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            int& v = ds->split_clusters[op == OP_RS ? 1 : 0][dt == COC_BF16 ? 1 : 0][ksplit == 4 ? 1 : 0];
            if (v < 0) v = max_split_clusters(op, dt == COC_BF16, ksplit);
            clusters = v;
        }
        if (clusters >= tiles) {
            p.split_cluster = 1;
            p.status = ds->status;
            p.inject_timeout = g_inject.load();
            p.clock_slot = g_clock_slot.load();
            const cudaError_t e = launch_split(op, dt == COC_BF16, p, p.units, ksplit, stream);
            return e == cudaSuccess ? COC_OK : cuda_fail(e, "kernel launch (rank split in clusters)");
        }
    }

    // rank split through global memory: fp32 parts and arrival counters in the
    // stream's workspace, the last part to arrive adds them
    const size_t part_bytes = static_cast<size_t>(tiles) * ksplit * tile_m * BN * sizeof(float);
    const size_t cnt_bytes = static_cast<size_t>(tiles) * (pair ? 2 : 1) * NUM_EPI_WARPS * sizeof(unsigned);
    Scratch sc;
    if ((st = scratch_acquire(ds, stream, part_bytes + cnt_bytes, &sc)) != COC_OK) return st;
    p.part = static_cast<float*>(sc.ptr);
    p.part_cnt = reinterpret_cast<unsigned*>(static_cast<char*>(sc.ptr) + part_bytes);
    const cudaError_t e = cudaMemsetAsync(p.part_cnt, 0, cnt_bytes, stream);
    st = (e != cudaSuccess) ? cuda_fail(e, "cudaMemsetAsync (rank-split counters)")
                            : launch_checked(op, dt == COC_BF16, pair, p, ds, stream);
    return scratch_release(stream, sc, st);
}

coc_status_t validate_row_parallel(int R, int64_t m, int64_t n, int64_t ks, const void* const* x, const void* const* w,
                                   const void* const* out, int n_out, coc_dtype_t dt, int chunks, int det,
                                   int w_elem_bytes) {
    coc_status_t st;
    if ((st = check_common(R, chunks, dt, det)) != COC_OK) return st;
    if ((st = check_dims(m, n, ks)) != COC_OK) return st;
    const bool empty = (m == 0 || n == 0);
    if ((st = check_ptrs(x, R, !empty && ks > 0, "x")) != COC_OK) return st;
    if ((st = check_ptrs(w, R, !empty && ks > 0, "w")) != COC_OK) return st;
    if ((st = check_ptrs(out, n_out, !empty, "out")) != COC_OK) return st;
    if (m % chunks != 0) return fail(COC_ERR_SHAPE, "m = %lld is not a multiple of chunks = %d", (long long)m, chunks);
    if ((ks * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "k_shard = %lld: rows of X must span a multiple of 16 bytes", (long long)ks);
    if ((n * 2) % 16 != 0 || (n * w_elem_bytes) % 16 != 0)
        return fail(COC_ERR_ALIGN, "n = %lld: rows of W and of the output must span a multiple of 16 bytes", (long long)n);
    return COC_OK;
}

// w8A16 schedule.  Three kernels compute the same bits: the persistent fused
// kernel whose dequant warps write the 16-bit weight tile to shared memory
// ("fused"), a streaming pre-pass that dequantises every weight element once
// into the stream's workspace followed by the fp16 AllReduce kernel
// ("prepass"), and one launch of the kernel that keeps the dequantised weight
// in tensor memory ("ts", coc_w8_ts.cu).  At m <= 128 the column-slab kernel
// ("slab", coc_slab.cu) streams the int8 weight over all SMs with its own
// dequant warps (the same bits unsplit; split over a cluster, the parts add
// in part order).  Default: the slab kernel up to 128 rows where its plan fits
// the shape, the fused kernel below kW8PrepassMinRows rows, the pre-pass from
// there (it repeats no conversion per row tile); COC_W8_PATH=
// fused|prepass|ts|slab forces one (tests, tuning).
enum class W8Path { TS, Fused, Prepass, Slab };
constexpr int64_t kW8PrepassMinRows = 2048;

W8Path w8_path(int64_t m) {
    const char* e = std::getenv("COC_W8_PATH");
    if (e != nullptr && std::strcmp(e, "fused") == 0) return W8Path::Fused;
    if (e != nullptr && std::strcmp(e, "prepass") == 0) return W8Path::Prepass;
    if (e != nullptr && std::strcmp(e, "ts") == 0) return W8Path::TS;
    if (e != nullptr && std::strcmp(e, "slab") == 0) return W8Path::Slab;
    if (m >= kW8PrepassMinRows) return W8Path::Prepass;
    return m <= BM ? W8Path::Slab : W8Path::Fused;
}

coc_status_t device_pool(DeviceState* ds, cudaMemPool_t* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (ds->pool == nullptr) return fail(COC_ERR_CUDA, "no memory pool on this device (coc_shutdown during a capture?)");
    *out = ds->pool;
    return COC_OK;
}

coc_status_t scratch_acquire(DeviceState* ds, cudaStream_t stream, size_t bytes, Scratch* out) {
    *out = Scratch{};
    if (bytes == 0) return COC_OK;
    if (bytes > kWorkspaceCap)
        return fail(COC_ERR_SHAPE, "the call needs %zu bytes of scratch, above the %zu-byte cap", bytes, kWorkspaceCap);
    bytes = (bytes + 255) & ~size_t(255);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone) {
        cudaMemPool_t pool = nullptr;
        coc_status_t st = device_pool(ds, &pool);
        if (st != COC_OK) return st;
        g_alloc_calls.fetch_add(1);
        if ((e = cudaMallocFromPoolAsync(&out->ptr, bytes, pool, stream)) != cudaSuccess)
            return cuda_fail(e, "cudaMallocFromPoolAsync (scratch of a captured call)");
        out->captured = true;
        return COC_OK;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = ds->ws[stream];
    if (w.last_use == nullptr && (e = cudaEventCreateWithFlags(&w.last_use, cudaEventDisableTiming)) != cudaSuccess) {
        w.last_use = nullptr;
        return cuda_fail(e, "cudaEventCreateWithFlags (workspace)");
    }
    if (w.bytes < bytes) {
        // grow: the previous buffer is freed once every kernel that used it is done
        if (w.ptr != nullptr) {
            if ((e = cudaEventSynchronize(w.last_use)) != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize (workspace)");
            if ((e = cudaFree(w.ptr)) != cudaSuccess) return cuda_fail(e, "cudaFree (workspace)");
            w.ptr = nullptr;
            w.bytes = 0;
        }
        const size_t want = std::max(bytes, (size_t(1) << 20));
        g_alloc_calls.fetch_add(1);
        if ((e = cudaMalloc(&w.ptr, want)) != cudaSuccess) {
            w.ptr = nullptr;
            return cuda_fail(e, "cudaMalloc (workspace)");
        }
        w.bytes = want;
    }
    // after the previous user of this workspace (this stream, or a destroyed
    // stream whose handle this one reuses)
    if ((e = cudaStreamWaitEvent(stream, w.last_use, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent (workspace)");
    out->ptr = w.ptr;
    out->w = &w;
    return COC_OK;
}

coc_status_t scratch_release(cudaStream_t stream, Scratch& sc, coc_status_t st) {
    cudaError_t e = cudaSuccess;
    if (sc.captured && sc.ptr != nullptr) e = cudaFreeAsync(sc.ptr, stream);
    else if (sc.w != nullptr) e = cudaEventRecord(sc.w->last_use, stream);
    sc = Scratch{};
    if (st == COC_OK && e != cudaSuccess) st = cuda_fail(e, "releasing the call's scratch");
    return st;
}

// Pre-pass path: dequantise all ranks' weights into the call's scratch, run
// the AllReduce on it, release the scratch in stream order.
coc_status_t w8_prepass_all_reduce(int R, int64_t m, int64_t n, int64_t ks, const void* const* x, const void* const* w,
                                   const void* const* scale, const void* const* zero, coc_scale_t gran, int64_t group,
                                   void* const* out, coc_dtype_t dt, int chunks, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    coc_status_t st = device_state(&ds);
    if (st != COC_OK) return st;
    const size_t per_rank = static_cast<size_t>(ks) * static_cast<size_t>(n);   // elements
    Scratch sc;
    if ((st = scratch_acquire(ds, stream, per_rank * 2 * R, &sc)) != COC_OK) return st;
    void* ws = sc.ptr;
    cudaError_t e;
    W8PrepassArgs a;
    std::memset(&a, 0, sizeof a);
    const void* wd[COC_MAX_RANKS] = {};
    for (int r = 0; r < R; ++r) {
        a.q[r] = static_cast<const int8_t*>(w[r]);
        a.scale[r] = static_cast<const uint16_t*>(scale[r]);
        a.zero[r] = zero ? static_cast<const int8_t*>(zero[r]) : nullptr;
        a.out[r] = static_cast<uint16_t*>(ws) + per_rank * r;
        wd[r] = a.out[r];
    }
    a.R = R;
    a.k = static_cast<int>(ks);
    a.n = static_cast<int>(n);
    a.gran = static_cast<int>(gran);
    a.group = static_cast<int>(group);
    e = launch_w8_prepass(a, dt == COC_BF16, ds->sm_count, stream);
    if (e != cudaSuccess) st = cuda_fail(e, "w8A16 pre-pass launch");
    // (unsplit, like the fused w8A16 kernel: both paths give the same bits)
    else st = row_parallel(OP_AR, R, m, n, ks, x, wd, out, R, dt, chunks, nullptr, COC_SCALE_TENSOR, 0, stream, false,
                           nullptr, false);
    return scratch_release(stream, sc, st);
}

// The default w8A16 path: Y^T = Wd^T X^T in one launch, the int8 weight
// dequantised in registers into tensor memory (the MMA's A operand).
coc_status_t w8_ts_all_reduce(int R, int64_t m, int64_t n, int64_t ks, const void* const* x, const void* const* w,
                              const void* const* scale, const void* const* zero, coc_scale_t gran, int64_t group,
                              void* const* out, coc_dtype_t dt, int chunks, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    coc_status_t st = device_state(&ds);
    if (st != COC_OK) return st;
    KParams p;
    std::memset(&p, 0, sizeof p);
    p.R = R;
    p.n_out = R;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(ks);
    p.num_kshards = R;
    p.kblocks = static_cast<int>((ks + BK - 1) / BK);
    // rows per unit (the MMA's N): the smallest power of two >= m in [32, 256],
    // so that decode-sized m does not pay for 256-row tiles
    int nr = 32;
    while (nr < TS_MAX_ROWS && nr < m) nr *= 2;
    p.unit_rows = nr;
    p.m_tiles = static_cast<int>((m + nr - 1) / nr);
    p.n_tiles = static_cast<int>((n + TS_UNIT_COLS - 1) / TS_UNIT_COLS);
    p.units = p.m_tiles * p.n_tiles;
    p.chunk_mt = chunk_m_tiles(m, chunks, nr);
    p.gran = static_cast<int>(gran);
    p.group = static_cast<int>(group);
    int pairs = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        int& v = ds->ts_pairs[dt == COC_BF16 ? 1 : 0];
        if (v < 0) v = w8_ts_max_pairs(dt == COC_BF16);
        pairs = v;
    }
    if (pairs <= 0) return fail(COC_ERR_CUDA, "no co-resident CTA pair of the w8A16 kernel fits on this device");
    {
        const int64_t k_total = static_cast<int64_t>(R) * ks;
        p.group_mt = row_group(p.chunk_mt, p.n_tiles, int64_t(nr) * k_total * 2, int64_t(TS_UNIT_COLS) * k_total, pairs);
        if (p.group_mt > 0) p.a_hint = 2;   // the group's X rows stay in L2 while W streams past
    }
    const CUtensorMapDataType adt = tma_dtype(dt);
    for (int r = 0; r < R; ++r) {
        if (ks > 0) {
            if ((st = encode(&p.tm_a[r], adt, x[r], ks, m, ks * 2, BK, nr / 2, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
            if ((st = encode(&p.tm_b[r], CU_TENSOR_MAP_DATA_TYPE_UINT8, w[r], n, ks, n, TS_UNIT_COLS / 2, BK,
                             CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
        }
        p.scale[r] = static_cast<const uint16_t*>(scale[r]);
        p.outp[r] = static_cast<uint16_t*>(out[r]);
    }
    if (zero != nullptr) {
        p.has_zero = 1;
        for (int r = 0; r < R; ++r) p.zero[r] = static_cast<const int8_t*>(zero[r]);
    }
    p.replica_stores = 1;
    p.status = ds->status;
    p.inject_timeout = g_inject.load();
    p.clock_slot = g_clock_slot.load();
    const int grid = 2 * (p.units < pairs ? p.units : pairs);
    const cudaError_t e = launch_w8_ts(p, dt == COC_BF16, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "w8A16 kernel launch");
    return COC_OK;
}

// Rows each destination buffer of the MoE dispatch needs in the worst case:
// all tokens of all ranks, each of the rank's eloc expert groups padded to a
// 256-row boundary.
int64_t moe_capacity(int R, int64_t T, int eloc) {
    const int64_t rows = static_cast<int64_t>(R) * T + static_cast<int64_t>(eloc) * (MOE_GROUP_ALIGN - 1);
    return (rows + MOE_GROUP_ALIGN - 1) / MOE_GROUP_ALIGN * MOE_GROUP_ALIGN;
}

}  // namespace
}  // namespace coc

using namespace coc;

#define COC_API extern "C" __attribute__((visibility("default")))

COC_API coc_status_t coc_matmul_all_reduce(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                           const void* const* w, void* const* out, coc_dtype_t dt, int chunks,
                                           int deterministic, coc_stream_t stream) {
    coc_status_t st = validate_row_parallel(R, m, n, k_shard, x, w, out, R, dt, chunks, deterministic, 2);
    if (st != COC_OK || m == 0 || n == 0) return st;
    return row_parallel(OP_AR, R, m, n, k_shard, x, w, out, R, dt, chunks, nullptr, COC_SCALE_TENSOR, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}

COC_API coc_status_t coc_matmul(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x, const void* const* w,
                                void* out, coc_dtype_t dt, coc_stream_t stream) {
    void* outs[1] = {out};
    coc_status_t st = validate_row_parallel(R, m, n, k_shard, x, w, outs, 1, dt, 1, 1, 2);
    if (st != COC_OK || m == 0 || n == 0) return st;
    return row_parallel(OP_AR, R, m, n, k_shard, x, w, outs, 1, dt, 1, nullptr, COC_SCALE_TENSOR, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}

COC_API coc_status_t coc_matmul_reduce_scatter(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                               const void* const* w, void* const* out, coc_dtype_t dt, int chunks,
                                               int deterministic, coc_stream_t stream) {
    coc_status_t st = validate_row_parallel(R, m, n, k_shard, x, w, out, R, dt, chunks, deterministic, 2);
    if (st != COC_OK) return st;
    if (m % R != 0) return fail(COC_ERR_SHAPE, "ReduceScatter: m = %lld is not a multiple of R = %d", (long long)m, R);
    if ((m / R) % 8 != 0) return fail(COC_ERR_SHAPE, "ReduceScatter: m / R = %lld is not a multiple of 8", (long long)(m / R));
    if (m == 0 || n == 0) return COC_OK;
    return row_parallel(OP_RS, R, m, n, k_shard, x, w, out, R, dt, chunks, nullptr, COC_SCALE_TENSOR, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}

COC_API coc_status_t coc_matmul_all_reduce_w8a16_ex(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                                    const void* const* w, const void* const* scale,
                                                    const void* const* zero, coc_scale_t gran, int64_t group_size,
                                                    void* const* out, coc_dtype_t dt, int chunks, int deterministic,
                                                    coc_stream_t stream) {
    if (dt != COC_FP16 && dt != COC_BF16) return fail(COC_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    coc_status_t st = validate_row_parallel(R, m, n, k_shard, x, w, out, R, dt, chunks, deterministic, 1);
    if (st != COC_OK) return st;
    if (gran != COC_SCALE_TENSOR && gran != COC_SCALE_CHANNEL && gran != COC_SCALE_GROUP)
        return fail(COC_ERR_INVALID_ARG, "unknown scale granularity %d", static_cast<int>(gran));
    if (scale == nullptr) return fail(COC_ERR_INVALID_ARG, "scale is NULL");
    const bool empty = (m == 0 || n == 0);
    for (int r = 0; r < R && !empty; ++r) {
        if (scale[r] == nullptr) return fail(COC_ERR_INVALID_ARG, "scale[%d] is NULL", r);
        if (gran != COC_SCALE_TENSOR && !aligned16(scale[r]))
            return fail(COC_ERR_ALIGN, "scale[%d] is not 16-byte aligned", r);
        if (gran == COC_SCALE_TENSOR && (reinterpret_cast<uintptr_t>(scale[r]) & 1u))
            return fail(COC_ERR_ALIGN, "scale[%d] is not 2-byte aligned", r);
        if (zero != nullptr) {
            if (zero[r] == nullptr) return fail(COC_ERR_INVALID_ARG, "zero[%d] is NULL", r);
            if (gran != COC_SCALE_TENSOR && !aligned16(zero[r]))
                return fail(COC_ERR_ALIGN, "zero[%d] is not 16-byte aligned", r);
        }
    }
    if (gran == COC_SCALE_GROUP) {
        if (group_size <= 0 || group_size % BK != 0)
            return fail(COC_ERR_SHAPE, "group_size = %lld must be a positive multiple of %d", (long long)group_size, BK);
        if (k_shard % group_size != 0)
            return fail(COC_ERR_SHAPE, "k_shard = %lld is not a multiple of group_size = %lld", (long long)k_shard,
                        (long long)group_size);
    }
    if (empty) return COC_OK;
    const W8Path path = w8_path(m);
    if (path == W8Path::TS)
        return w8_ts_all_reduce(R, m, n, k_shard, x, w, scale, zero, gran, group_size, out, dt, chunks,
                                reinterpret_cast<cudaStream_t>(stream));
    if (k_shard > 0 && path == W8Path::Prepass)
        return w8_prepass_all_reduce(R, m, n, k_shard, x, w, scale, zero, gran, group_size, out, dt, chunks,
                                     reinterpret_cast<cudaStream_t>(stream));
    // (the column-slab kernel where its plan fits the shape, else the fused kernel)
    return row_parallel(OP_W8, R, m, n, k_shard, x, w, out, R, dt, chunks, scale, gran, group_size,
                        reinterpret_cast<cudaStream_t>(stream), false, zero, path == W8Path::Slab);
}

COC_API coc_status_t coc_matmul_all_reduce_w8a16(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                                 const void* const* w, const void* const* scale, coc_scale_t gran,
                                                 int64_t group_size, void* const* out, int chunks, int deterministic,
                                                 coc_stream_t stream) {
    return coc_matmul_all_reduce_w8a16_ex(R, m, n, k_shard, x, w, scale, nullptr, gran, group_size, out, COC_FP16,
                                          chunks, deterministic, stream);
}

namespace coc {
namespace {

// An AllGather call can stack X (the R shards in rank order, m x k) into
// V2's first kept gathered output, or else into scratch under the workspace
// cap.  `kept`: V2's gathered outputs (entries may be NULL), NULL for V1.
bool ag_can_stack(int R, int64_t ms, int64_t k, void* const* kept) {
    for (int r = 0; kept != nullptr && r < R; ++r)
        if (kept[r] != nullptr) return true;
    return static_cast<size_t>(R) * static_cast<size_t>(ms) * static_cast<size_t>(k) * 2 <= kWorkspaceCap;
}

// The copy that stacks X (for calls where ag_can_stack holds): g->src the
// shards, g->dst the first kept gathered output or, with none, scratch taken
// into *sc (released by the caller with scratch_release).
coc_status_t ag_stack_target(DeviceState* ds, cudaStream_t stream, int R, int64_t ms, int64_t k, const void* const* x,
                             void* const* kept, AgGatherParams* g, Scratch* sc) {
    std::memset(g, 0, sizeof *g);
    g->R = R;
    g->shard_vecs = ms * k / 8;
    for (int r = 0; r < R; ++r) {
        g->src[r] = static_cast<const uint16_t*>(x[r]);
        if (kept != nullptr && g->dst == nullptr && kept[r] != nullptr) g->dst = static_cast<uint16_t*>(kept[r]);
    }
    if (g->dst != nullptr) return COC_OK;
    const coc_status_t st = scratch_acquire(ds, stream, static_cast<size_t>(R) * ms * k * 2, sc);
    g->dst = static_cast<uint16_t*>(sc->ptr);
    return st;
}

// ALL_GATHER_MATMUL(_V2) through the column-slab kernel (gathered m = R
// m_shard <= 128): first the gather kernel stacks the R shards of X into the
// first non-NULL gathered output (V2) or, with none, into the call's
// scratch; then the slab kernel reads A from that one m x k buffer (3-D
// boxes when k % 64 == 0) and B from each rank's W (k x n_s, or w_nk n_s x
// k), one unit per column slab of one rank's output, and copies the buffer
// into V2's other gathered outputs.
coc_status_t slab_all_gather(int R, int64_t ms, int64_t ns, int64_t k, const void* const* x, const void* const* w,
                             void* const* out, void* const* gathered, coc_dtype_t dt, const SlabPlan& pl,
                             DeviceState* ds, cudaStream_t stream, bool w_nk) {
    KParams p;
    std::memset(&p, 0, sizeof p);
    const int64_t m = static_cast<int64_t>(R) * ms;
    const int boxes = pl.boxes, kps = pl.kps;
    p.R = R;
    p.n_out = R;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(ns);
    p.k = static_cast<int>(k);
    p.num_kshards = 1;
    p.kblocks = static_cast<int>((k + BK - 1) / BK);
    p.m_tiles = 1;
    p.n_tiles = static_cast<int>((ns + 64 * boxes - 1) / (64 * boxes));   // slabs per rank output
    p.units = R * p.n_tiles;
    p.rows_per_rank = static_cast<int>(ms);
    p.a_box_rows = static_cast<int>(m);   // m_shard % 8 == 0
    const int split = slab_resident_split(ds, dt == COC_BF16, false, boxes, kps, p.a_box_rows, pl.split, p.units);
    p.slab_boxes = boxes;
    p.slab_kps = kps;
    p.slab_split = split;
    p.slab_stages = slab_stages(p.a_box_rows, boxes, kps, split, false);
    if (slab_smem_bytes(p.slab_stages, p.a_box_rows, boxes, kps, split, false) > kSlabSmemCap)
        return fail(COC_ERR_SHAPE, "column-slab schedule does not fit in shared memory (m = %lld)", (long long)m);
    p.b_kmajor = w_nk ? 1 : 0;

    // the gathered X the slab kernel reads (V2's first kept gathered output,
    // else scratch); the slab kernel copies it into V2's other kept outputs
    AgGatherParams g;
    Scratch sc;
    coc_status_t st = ag_stack_target(ds, stream, R, ms, k, x, gathered, &g, &sc);
    if (st != COC_OK) return scratch_release(stream, sc, st);
    for (int r = 0; gathered != nullptr && r < R; ++r) {
        if (gathered[r] != nullptr && gathered[r] != g.dst) {
            p.gdst[r] = static_cast<uint16_t*>(gathered[r]);
            p.has_gather = 1;
        }
    }
    const void* xg = g.dst;
    p.gsrc[0] = g.dst;
    const CUtensorMapDataType tdt = tma_dtype(dt);
    // 3-D maps (one A box per stage; n x k B likewise) where the k-blocks tile k exactly
    bool a3d = kps > 1 && k % BK == 0;
    if (a3d) a3d = encode_blocked(&p.tm_a[0], tdt, xg, BK, m, k / BK, k * 2, BK, m, kps) == CUDA_SUCCESS;
    for (int r = 0; a3d && w_nk && r < R; ++r)
        a3d = encode_blocked(&p.tm_b[r], tdt, w[r], BK, ns, k / BK, k * 2, BK, 64 * boxes, kps) == CUDA_SUCCESS;
    p.slab_a3d = a3d ? 1 : 0;
    st = a3d ? COC_OK : encode(&p.tm_a[0], tdt, xg, k, m, k * 2, BK, m, CU_TENSOR_MAP_SWIZZLE_128B);
    for (int r = 0; st == COC_OK && r < R; ++r) {
        if (w_nk && !a3d) st = encode(&p.tm_b[r], tdt, w[r], k, ns, k * 2, BK, 64 * boxes, CU_TENSOR_MAP_SWIZZLE_128B);
        else if (!w_nk) st = encode(&p.tm_b[r], tdt, w[r], ns, k, ns * 2, 64, BK * kps, CU_TENSOR_MAP_SWIZZLE_128B);
        p.outp[r] = static_cast<uint16_t*>(out[r]);
    }
    if (st == COC_OK) {
        p.status = ds->status;
        p.inject_timeout = g_inject.load();
        p.clock_slot = g_clock_slot.load();
        const int grid = split > 1 ? split * p.units : (p.units < ds->sm_count ? p.units : ds->sm_count);
        cudaError_t e = launch_ag_gather(g, ds->sm_count, stream);
        if (e != cudaSuccess) {
            st = cuda_fail(e, "kernel launch (AllGather copy)");
        } else {
            e = launch_slab(OP_AG, dt == COC_BF16, false, p, grid, stream);
            if (e != cudaSuccess) st = cuda_fail(e, "kernel launch (column slabs)");
        }
    }
    return scratch_release(stream, sc, st);
}

coc_status_t all_gather(int R, int64_t ms, int64_t ns, int64_t k, const void* const* x, const void* const* w,
                        void* const* out, void* const* gathered, bool v2, coc_dtype_t dt, int chunks, int det,
                        cudaStream_t stream, bool w_nk = false) {
    coc_status_t st;
    if ((st = check_common(R, chunks, dt, det)) != COC_OK) return st;
    if ((st = check_dims(ms, ns, k)) != COC_OK) return st;
    const int64_t m = static_cast<int64_t>(R) * ms;
    if (m > kMaxDim) return fail(COC_ERR_SHAPE, "gathered rows R * m_shard above 2^31 - 1024");
    if (v2 && gathered == nullptr) return fail(COC_ERR_INVALID_ARG, "gathered is NULL");
    const bool empty = (ms == 0 || ns == 0);
    if ((st = check_ptrs(x, R, ms > 0 && k > 0 && (ns > 0 || v2), "x")) != COC_OK) return st;
    if ((st = check_ptrs(w, R, !empty && k > 0, "w")) != COC_OK) return st;
    if ((st = check_ptrs(out, R, !empty, "out")) != COC_OK) return st;
    if (v2 && (st = check_ptrs(const_cast<const void* const*>(gathered), R, ms > 0 && k > 0, "gathered", true)) != COC_OK)
        return st;
    if (ms % 8 != 0) return fail(COC_ERR_SHAPE, "m_shard = %lld is not a multiple of 8", (long long)ms);
    if (m % chunks != 0) return fail(COC_ERR_SHAPE, "gathered m = %lld is not a multiple of chunks = %d", (long long)m, chunks);
    if ((k * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "k = %lld: rows must span a multiple of 16 bytes", (long long)k);
    if ((ns * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "n_shard = %lld: rows must span a multiple of 16 bytes", (long long)ns);
    if (v2 && ns == 0 && ms > 0) return fail(COC_ERR_SHAPE, "ALL_GATHER_MATMUL_V2 needs n_shard > 0");
    if (empty) return COC_OK;

    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != COC_OK) return st;
    void* const* kept = v2 ? gathered : nullptr;
    const bool can_stack = k > 0 && ag_can_stack(R, ms, k, kept);
    if (can_stack) {
        const SlabPlan pl = slab_plan(OP_AG, R, m, ns, k, ds->sm_count);
        if (pl.boxes > 0) return slab_all_gather(R, ms, ns, k, x, w, out, kept, dt, pl, ds, stream, w_nk);
    }
    KParams p;
    std::memset(&p, 0, sizeof p);
    p.R = R;
    p.n_out = R;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(ns);
    p.k = static_cast<int>(k);
    p.num_kshards = 1;
    const bool pair = ag_use_pair(ds, m, R * ((ns + BN - 1) / BN), dt == COC_BF16);
    const int tile_m = pair ? 2 * BM : BM;
    p.kblocks = static_cast<int>((k + BK - 1) / BK);
    p.m_tiles = static_cast<int>((m + tile_m - 1) / tile_m);
    p.n_tiles = static_cast<int>((ns + BN - 1) / BN);
    p.units = R * p.m_tiles * p.n_tiles;
    p.chunk_mt = chunk_m_tiles(m, chunks, tile_m);
    p.rows_per_rank = static_cast<int>(ms);
    p.a_box_rows = largest_pow2_divisor_le(ms, BM);
    p.store_rows = 32;
    p.has_gather = (v2 && k > 0) ? 1 : 0;
    p.b_kmajor = w_nk ? 1 : 0;
    // The gathered X is re-read by every (rank, n-tile) column.  Take the
    // row tiles in groups whose X rows fit comfortably in L2 (32 MiB) and
    // mark those loads evict-last, so W streams past a resident X slice:
    // W is then read once per group instead of X once per wave of columns.
    p.a_hint = 2;
    p.b_hint = 0;
    p.group_mt = l2_group(p.chunk_mt, static_cast<int64_t>(tile_m) * k * 2);

    // Shards that do not fill whole 128-row boxes would need several A boxes
    // per tile and k-block (one per shard piece, down to 8 rows), and a CTA's
    // operand stream is bound by its TMA operations: stack X once instead
    // (into V2's first kept copy, else into scratch under the workspace cap)
    // and read it as one shard of m rows (measured, 8 ranks, n_shard 7168, k
    // 8192: m_shard 24 / 48 took 738 / 847 us with 8 / 16-row boxes).
    const CUtensorMapDataType tdt = tma_dtype(dt);
    AgGatherParams g;
    std::memset(&g, 0, sizeof g);
    Scratch sc;
    if (can_stack && p.a_box_rows < BM && (st = ag_stack_target(ds, stream, R, ms, k, x, kept, &g, &sc)) != COC_OK)
        return scratch_release(stream, sc, st);
    const bool stacked = g.dst != nullptr;
    if (stacked) {
        // one shard covering every tile's rows, so that the kernel's shard
        // index (row / rows_per_rank) is 0 for all of them, also for the
        // rows of a ragged last tile past m (zero-filled); every map entry
        // holds the stacked map all the same
        p.rows_per_rank = p.m_tiles * tile_m;
        p.a_box_rows = BM;
        st = encode(&p.tm_a[0], tdt, g.dst, k, m, k * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
        for (int r = 1; r < R; ++r) p.tm_a[r] = p.tm_a[0];
        p.gsrc[0] = g.dst;
    }
    for (int r = 0; st == COC_OK && r < R; ++r) {
        if (k > 0) {
            if (!stacked && (st = encode(&p.tm_a[r], tdt, x[r], k, ms, k * 2, BK, p.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                break;
            st = w_nk ? encode(&p.tm_b[r], tdt, w[r], k, ns, k * 2, BK, pair ? BN / 2 : BN, CU_TENSOR_MAP_SWIZZLE_128B)
                      : encode(&p.tm_b[r], tdt, w[r], ns, k, ns * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
            if (st != COC_OK) break;
        }
        if ((st = encode(&p.tm_out[r], tdt, out[r], ns, m, ns * 2, EPI_COLS, p.store_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
            break;
        if (!stacked) p.gsrc[r] = static_cast<const uint16_t*>(x[r]);
        // (the stacking kernel already wrote the copy it stacked into)
        p.gdst[r] = v2 && gathered[r] != g.dst ? static_cast<uint16_t*>(gathered[r]) : nullptr;
    }
    if (st == COC_OK && stacked) {
        const cudaError_t e = launch_ag_gather(g, ds->sm_count, stream);
        if (e != cudaSuccess) st = cuda_fail(e, "kernel launch (AllGather copy)");
    }
    if (st == COC_OK) st = launch_checked(OP_AG, dt == COC_BF16, pair, p, ds, stream);
    return scratch_release(stream, sc, st);
}

}  // namespace
}  // namespace coc

COC_API coc_status_t coc_all_gather_matmul(int R, int64_t m_shard, int64_t n_shard, int64_t k, const void* const* x,
                                           const void* const* w, void* const* out, coc_dtype_t dt, int chunks,
                                           int deterministic, coc_stream_t stream) {
    return all_gather(R, m_shard, n_shard, k, x, w, out, nullptr, false, dt, chunks, deterministic,
                      reinterpret_cast<cudaStream_t>(stream));
}

COC_API coc_status_t coc_all_gather_matmul_v2(int R, int64_t m_shard, int64_t n_shard, int64_t k, const void* const* x,
                                              const void* const* w, void* const* out, void* const* gathered,
                                              coc_dtype_t dt, int chunks, int deterministic, coc_stream_t stream) {
    return all_gather(R, m_shard, n_shard, k, x, w, out, gathered, true, dt, chunks, deterministic,
                      reinterpret_cast<cudaStream_t>(stream));
}

namespace coc {
namespace {

// Weight gradient of a TP linear layer: dW_r = dY_r^T X_r for every rank r
// (no collective).  dY_r is inner x rows (tokens x out_features), X_r inner x
// cols (tokens x in_features), dW_r rows x cols.  Runs on the AllGather path
// of the kernel with A read per rank and MN-major.
coc_status_t weight_grad(int R, int64_t rows, int64_t cols, int64_t inner, const void* const* dy,
                         const void* const* x, void* const* out, coc_dtype_t dt, int chunks, int det,
                         cudaStream_t stream) {
    coc_status_t st;
    if ((st = check_common(R, chunks, dt, det)) != COC_OK) return st;
    if ((st = check_dims(rows, cols, inner)) != COC_OK) return st;
    const bool empty = (rows == 0 || cols == 0);
    if ((st = check_ptrs(dy, R, !empty && inner > 0, "x (dY)")) != COC_OK) return st;
    if ((st = check_ptrs(x, R, !empty && inner > 0, "w (X)")) != COC_OK) return st;
    if ((st = check_ptrs(out, R, !empty, "out")) != COC_OK) return st;
    if (rows % chunks != 0) return fail(COC_ERR_SHAPE, "rows = %lld is not a multiple of chunks = %d", (long long)rows, chunks);
    if ((rows * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "rows = %lld: dY rows must span a multiple of 16 bytes", (long long)rows);
    if ((cols * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "cols = %lld: X rows must span a multiple of 16 bytes", (long long)cols);
    if (empty) return COC_OK;

    KParams p;
    std::memset(&p, 0, sizeof p);
    const bool pair = use_pair(OP_AG, rows);
    const int tile_m = pair ? 2 * BM : BM;
    p.R = R;
    p.n_out = R;
    p.m = static_cast<int>(rows);
    p.n = static_cast<int>(cols);
    p.k = static_cast<int>(inner);
    p.num_kshards = 1;
    p.kblocks = static_cast<int>((inner + BK - 1) / BK);
    p.m_tiles = static_cast<int>((rows + tile_m - 1) / tile_m);
    p.n_tiles = static_cast<int>((cols + BN - 1) / BN);
    p.units = R * p.m_tiles * p.n_tiles;
    p.chunk_mt = chunk_m_tiles(rows, chunks, tile_m);
    p.rows_per_rank = static_cast<int>(rows);
    p.a_box_rows = BM;
    p.store_rows = 32;
    p.a_mnmajor = 1;

    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != COC_OK) return st;
    const CUtensorMapDataType tdt = tma_dtype(dt);
    for (int r = 0; r < R; ++r) {
        if (inner > 0) {
            if ((st = encode(&p.tm_a[r], tdt, dy[r], rows, inner, rows * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
            if ((st = encode(&p.tm_b[r], tdt, x[r], cols, inner, cols * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
                return st;
        }
        if ((st = encode(&p.tm_out[r], tdt, out[r], cols, rows, cols * 2, EPI_COLS, p.store_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != COC_OK)
            return st;
    }
    return launch_checked(OP_AG, dt == COC_BF16, pair, p, ds, stream);
}

}  // namespace
}  // namespace coc

COC_API coc_status_t coc_fused_matmul(coc_op_t op, int R, int64_t rows, int64_t cols, int64_t inner,
                                      const void* const* x, const void* const* w, coc_wlayout_t layout,
                                      void* const* out, void* const* gathered, coc_dtype_t dt, int chunks,
                                      int deterministic, coc_stream_t stream) {
    if (layout != COC_W_KN && layout != COC_W_NK)
        return fail(COC_ERR_INVALID_ARG, "unknown weight layout %d", static_cast<int>(layout));
    const bool nk = (layout == COC_W_NK);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    coc_status_t st;
    switch (op) {
        case COC_OP_ALL_REDUCE:
            st = validate_row_parallel(R, rows, cols, inner, x, w, out, R, dt, chunks, deterministic, 2);
            if (st != COC_OK || rows == 0 || cols == 0) return st;
            return row_parallel(OP_AR, R, rows, cols, inner, x, w, out, R, dt, chunks, nullptr, COC_SCALE_TENSOR, 0,
                                s, nk);
        case COC_OP_REDUCE_SCATTER:
            st = validate_row_parallel(R, rows, cols, inner, x, w, out, R, dt, chunks, deterministic, 2);
            if (st != COC_OK) return st;
            if (rows % R != 0) return fail(COC_ERR_SHAPE, "ReduceScatter: m = %lld is not a multiple of R = %d", (long long)rows, R);
            if ((rows / R) % 8 != 0)
                return fail(COC_ERR_SHAPE, "ReduceScatter: m / R = %lld is not a multiple of 8", (long long)(rows / R));
            if (rows == 0 || cols == 0) return COC_OK;
            return row_parallel(OP_RS, R, rows, cols, inner, x, w, out, R, dt, chunks, nullptr, COC_SCALE_TENSOR, 0,
                                s, nk);
        case COC_OP_ALL_GATHER:
            return all_gather(R, rows, cols, inner, x, w, out, nullptr, false, dt, chunks, deterministic, s, nk);
        case COC_OP_ALL_GATHER_V2:
            return all_gather(R, rows, cols, inner, x, w, out, gathered, true, dt, chunks, deterministic, s, nk);
        case COC_OP_WEIGHT_GRAD:
            if (nk) return fail(COC_ERR_INVALID_ARG, "the weight-gradient pass takes X as tokens x in_features (COC_W_KN)");
            return weight_grad(R, rows, cols, inner, x, w, out, dt, chunks, deterministic, s);
        default:
            return fail(COC_ERR_INVALID_ARG, "unknown operator %d", static_cast<int>(op));
    }
}

COC_API int64_t coc_moe_capacity(int R, int64_t tokens, int experts_per_rank) {
    if (R < 1 || R > COC_MAX_RANKS || tokens < 0 || experts_per_rank < 1) return -1;
    return moe_capacity(R, tokens, experts_per_rank);
}

// Shared by the dispatch-only and the dispatch + combine entry points: y
// (dispatched layout) or y_tok (token order on the source ranks) is NULL.
// k routing entries per token (entry i of rank r: token i / k, slot i % k).
// gates != NULL: weighted top-k combine after the grouped GEMM (y holds the
// dispatched expert outputs, y_tok receives the combined tokens); gates ==
// NULL with y_tok: the k = 1 combine fused into the grouped GEMM's epilogue.
static coc_status_t moe_impl(int R, int64_t tokens, int k, int64_t h, int64_t f, int experts_per_rank,
                             const void* const* x, const int32_t* const* idx, const float* const* gates, const void* w,
                             void* const* xd, void* const* y, void* const* y_tok, int64_t capacity, int32_t* counts,
                             int32_t* offsets, coc_dtype_t dt, coc_stream_t stream) {
    if (R < 1 || R > COC_MAX_RANKS) return fail(COC_ERR_INVALID_ARG, "R = %d outside [1, %d]", R, COC_MAX_RANKS);
    if (dt != COC_FP16 && dt != COC_BF16) return fail(COC_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    const int eloc = experts_per_rank;
    if (eloc < 1 || static_cast<int64_t>(R) * eloc > MOE_MAX_EXPERTS)
        return fail(COC_ERR_INVALID_ARG, "experts = R x %d must lie in [1, %d]", eloc, MOE_MAX_EXPERTS);
    if (k < 1 || k > 8) return fail(COC_ERR_INVALID_ARG, "top-k = %d outside [1, 8]", k);
    if (tokens < 0 || tokens * k > (int64_t(1) << 24)) return fail(COC_ERR_SHAPE, "tokens = %lld per rank", (long long)tokens);
    const int64_t entries = tokens * k;   // routing entries per rank
    if (h <= 0 || h % BK != 0) return fail(COC_ERR_SHAPE, "h = %lld must be a positive multiple of %d", (long long)h, BK);
    if (f <= 0 || (f * 2) % 16 != 0) return fail(COC_ERR_ALIGN, "f = %lld: rows of W and Y must span a multiple of 16 bytes", (long long)f);
    if (h > (int64_t(1) << 20) || f > (int64_t(1) << 20)) return fail(COC_ERR_SHAPE, "h or f too large");
    const int64_t need = moe_capacity(R, entries, eloc);
    if (capacity < need)
        return fail(COC_ERR_SHAPE, "capacity = %lld rows, needs %lld (coc_moe_capacity)", (long long)capacity, (long long)need);
    if (capacity > (int64_t(1) << 30)) return fail(COC_ERR_SHAPE, "capacity too large");
    if (counts == nullptr || offsets == nullptr) return fail(COC_ERR_INVALID_ARG, "counts / offsets is NULL");
    if ((reinterpret_cast<uintptr_t>(counts) | reinterpret_cast<uintptr_t>(offsets)) & 3u)
        return fail(COC_ERR_ALIGN, "counts / offsets not 4-byte aligned");
    coc_status_t st;
    if ((st = check_ptrs(xd, R, true, "xd")) != COC_OK) return st;
    if (y != nullptr && (st = check_ptrs(y, R, true, "y")) != COC_OK) return st;
    if (y_tok != nullptr && (st = check_ptrs(y_tok, R, true, "y_tok")) != COC_OK) return st;
    if (w == nullptr || !aligned16(w)) return fail(w == nullptr ? COC_ERR_INVALID_ARG : COC_ERR_ALIGN, "w is NULL or not 16-byte aligned");
    if (tokens > 0) {
        if ((st = check_ptrs(x, R, true, "x")) != COC_OK) return st;
        if (idx == nullptr) return fail(COC_ERR_INVALID_ARG, "idx is NULL");
        for (int r = 0; r < R; ++r)
            if (idx[r] == nullptr || (reinterpret_cast<uintptr_t>(idx[r]) & 3u))
                return fail(idx[r] == nullptr ? COC_ERR_INVALID_ARG : COC_ERR_ALIGN, "idx[%d] is NULL or misaligned", r);
        if (gates != nullptr)
            for (int r = 0; r < R; ++r)
                if (gates[r] == nullptr || (reinterpret_cast<uintptr_t>(gates[r]) & 3u))
                    return fail(gates[r] == nullptr ? COC_ERR_INVALID_ARG : COC_ERR_ALIGN, "gates[%d] is NULL or misaligned", r);
    }
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != COC_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int E = R * eloc;

    MoeRouteArgs ra;
    std::memset(&ra, 0, sizeof ra);
    void* ws = nullptr;
    Scratch sc;
    // routing table: R x tokens destination rows, then (combine) R x capacity source tokens
    const bool fused_combine = y_tok != nullptr && gates == nullptr;
    const size_t dest_ints = static_cast<size_t>(R) * entries;
    const size_t src_ints = fused_combine ? static_cast<size_t>(R) * capacity : 0;
    if (tokens > 0) {
        if ((st = scratch_acquire(ds, s, (dest_ints + src_ints) * sizeof(int32_t), &sc)) != COC_OK) return st;
        ws = sc.ptr;
        cudaError_t e;
        if (src_ints > 0 &&
            (e = cudaMemsetAsync(static_cast<int32_t*>(ws) + dest_ints, 0xFF, src_ints * sizeof(int32_t), s)) != cudaSuccess)
            return scratch_release(s, sc, cuda_fail(e, "cudaMemsetAsync (MoE source map)"));
    }
    for (int r = 0; r < R; ++r) ra.idx[r] = tokens > 0 ? idx[r] : nullptr;
    ra.dest = static_cast<int32_t*>(ws);
    ra.srcmap = (tokens > 0 && src_ints > 0) ? static_cast<int32_t*>(ws) + dest_ints : nullptr;
    ra.cap = static_cast<int>(capacity);
    ra.counts = counts;
    ra.offsets = offsets;
    ra.status = ds->status;
    ra.R = R;
    ra.T = static_cast<int>(entries);
    ra.E = E;
    ra.eloc = eloc;
    cudaError_t e = launch_moe_route(ra, s);
    if (e != cudaSuccess) st = cuda_fail(e, "MoE routing launch");
    if (st == COC_OK && tokens > 0) {
        MoePermuteArgs pa;
        std::memset(&pa, 0, sizeof pa);
        for (int r = 0; r < R; ++r) {
            pa.x[r] = static_cast<const uint16_t*>(x[r]);
            pa.xd[r] = static_cast<uint16_t*>(xd[r]);
            pa.idx[r] = idx[r];
        }
        pa.dest = ra.dest;
        pa.R = R;
        pa.T = static_cast<int>(entries);
        pa.h = static_cast<int>(h);
        pa.E = E;
        pa.eloc = eloc;
        pa.k = k;
        if ((e = launch_moe_permute(pa, ds->sm_count, s)) != cudaSuccess) st = cuda_fail(e, "MoE permute launch");
    }
    if (st == COC_OK && tokens > 0) {
        // grouped GEMM on the dispatched rows: units come from the device counts
        KParams p;
        std::memset(&p, 0, sizeof p);
        const bool pair = use_pair(OP_GMM, static_cast<int64_t>(R) * tokens);
        const int tile_m = pair ? 2 * BM : BM;
        // inside an expert, row tiles in groups whose token rows fit in 32 MiB
        // of L2 (held there, evict-last) while the expert's W streams past
        const int64_t row_tile_bytes = static_cast<int64_t>(tile_m) * h * 2;
        p.group_mt = static_cast<int>(std::max<int64_t>(1, (int64_t(32) << 20) / row_tile_bytes));
        p.a_hint = 2;
        p.R = R;
        p.n_out = 1;
        p.m = static_cast<int>(capacity);
        p.n = static_cast<int>(f);
        p.k = static_cast<int>(h);
        p.num_kshards = 1;
        p.kblocks = static_cast<int>(h / BK);
        p.n_tiles = static_cast<int>((f + BN - 1) / BN);
        p.units = 1 << 30;   // upper bound for the grid size; the kernel counts its units
        p.rows_per_rank = static_cast<int>(capacity);
        p.a_box_rows = BM;
        p.store_rows = 32;
        p.gmm_counts = counts;
        p.gmm_offsets = offsets;
        p.gmm_E = E;
        p.gmm_eloc = eloc;
        if (fused_combine) {
            // combine: the epilogue writes each row to its token's row of y_tok[source rank]
            p.gmm_srcmap = ra.srcmap;
            p.gmm_T = static_cast<int>(tokens);
            for (int r = 0; r < R; ++r) p.outp[r] = static_cast<uint16_t*>(y_tok[r]);
        }
        const CUtensorMapDataType tdt = tma_dtype(dt);
        for (int q = 0; q < R && st == COC_OK; ++q) {
            st = encode(&p.tm_a[q], tdt, xd[q], h, capacity, h * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
            if (st == COC_OK && y != nullptr)
                st = encode(&p.tm_out[q], tdt, y[q], f, capacity, f * 2, EPI_COLS, p.store_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (st == COC_OK)
            st = encode(&p.tm_b[0], tdt, w, f, static_cast<int64_t>(E) * h, f * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st == COC_OK) st = launch_checked(OP_GMM, dt == COC_BF16, pair, p, ds, s);
    }
    if (st == COC_OK && tokens > 0 && gates != nullptr) {
        MoeCombineArgs ca;
        std::memset(&ca, 0, sizeof ca);
        for (int r = 0; r < R; ++r) {
            ca.y[r] = static_cast<const uint16_t*>(y[r]);
            ca.idx[r] = idx[r];
            ca.gates[r] = gates[r];
            ca.out[r] = static_cast<uint16_t*>(y_tok[r]);
        }
        ca.dest = ra.dest;
        ca.R = R;
        ca.tokens = static_cast<int>(tokens);
        ca.k = k;
        ca.f = static_cast<int>(f);
        ca.E = E;
        ca.eloc = eloc;
        e = launch_moe_combine(ca, dt == COC_BF16, ds->sm_count, s);
        if (e != cudaSuccess) st = cuda_fail(e, "MoE top-k combine launch");
    }
    return scratch_release(s, sc, st);
}

COC_API coc_status_t coc_moe_dispatch_grouped_matmul(int R, int64_t tokens, int64_t h, int64_t f, int experts_per_rank,
                                                     const void* const* x, const int32_t* const* idx, const void* w,
                                                     void* const* xd, void* const* y, int64_t capacity,
                                                     int32_t* counts, int32_t* offsets, coc_dtype_t dt,
                                                     coc_stream_t stream) {
    if (y == nullptr) return fail(COC_ERR_INVALID_ARG, "y is NULL");
    return moe_impl(R, tokens, 1, h, f, experts_per_rank, x, idx, nullptr, w, xd, y, nullptr, capacity, counts, offsets, dt,
                    stream);
}

COC_API coc_status_t coc_moe_dispatch_grouped_matmul_combine(int R, int64_t tokens, int64_t h, int64_t f,
                                                             int experts_per_rank, const void* const* x,
                                                             const int32_t* const* idx, const void* w, void* const* xd,
                                                             void* const* y_tok, int64_t capacity, int32_t* counts,
                                                             int32_t* offsets, coc_dtype_t dt, coc_stream_t stream) {
    if (y_tok == nullptr) return fail(COC_ERR_INVALID_ARG, "y_tok is NULL");
    return moe_impl(R, tokens, 1, h, f, experts_per_rank, x, idx, nullptr, w, xd, nullptr, y_tok, capacity, counts,
                    offsets, dt, stream);
}

COC_API coc_status_t coc_moe_topk_grouped_matmul_combine(int R, int64_t tokens, int k, int64_t h, int64_t f,
                                                         int experts_per_rank, const void* const* x,
                                                         const int32_t* const* idx, const float* const* gates,
                                                         const void* w, void* const* xd, void* const* y,
                                                         void* const* y_tok, int64_t capacity, int32_t* counts,
                                                         int32_t* offsets, coc_dtype_t dt, coc_stream_t stream) {
    if (y == nullptr || y_tok == nullptr || gates == nullptr)
        return fail(COC_ERR_INVALID_ARG, "y, y_tok and gates are required");
    return moe_impl(R, tokens, k, h, f, experts_per_rank, x, idx, gates, w, xd, y, y_tok, capacity, counts, offsets,
                    dt, stream);
}

// Status words of the current device's library state, read and cleared; all
// zero (and nothing created) when no allocating call has run on the device.
static coc_status_t take_library_status(unsigned (&words)[STATUS_WORDS]) {
    std::memset(words, 0, sizeof words);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    unsigned* status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) status = it->second.status;
    }
    if (status == nullptr) return COC_OK;
    if ((e = cudaMemcpy(words, status, sizeof words, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    if (words[0] != 0 && (e = cudaMemset(status, 0, sizeof words)) != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    return COC_OK;
}

COC_API coc_status_t coc_sync_status(coc_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    // both status blocks: the library's (allocating entry points) and the
    // static one of the allocation-free entry point; neither read allocates
    unsigned lib_words[STATUS_WORDS], na_words[STATUS_WORDS];
    coc_status_t st = take_library_status(lib_words);
    if (st != COC_OK) return st;
    if ((st = noalloc_take_status(na_words)) != COC_OK) return st;
    const unsigned* words = lib_words[0] != 0 ? lib_words : na_words;
    if (words[0] != 0) {
        if (words[0] == DEV_ERR_BAD_INDEX)
            return fail(COC_ERR_INVALID_ARG, "MoE dispatch: an expert id was outside [0, E); those tokens were not dispatched");
        return fail(COC_ERR_TIMEOUT, "device wait timed out%s (flags 0x%x, first wait site 0x%x, block %u)",
                    words == na_words ? " in the allocation-free AllReduce" : "", words[0], words[1],
                    words[2] ? words[2] - 1 : 0);
    }
    return COC_OK;
}

COC_API const char* coc_status_string(coc_status_t s) {
    switch (s) {
        case COC_OK: return "COC_OK";
        case COC_ERR_INVALID_ARG: return "COC_ERR_INVALID_ARG";
        case COC_ERR_SHAPE: return "COC_ERR_SHAPE";
        case COC_ERR_ALIGN: return "COC_ERR_ALIGN";
        case COC_ERR_UNSUPPORTED: return "COC_ERR_UNSUPPORTED";
        case COC_ERR_CUDA: return "COC_ERR_CUDA";
        case COC_ERR_TIMEOUT: return "COC_ERR_TIMEOUT";
        default: return "COC_ERR_UNKNOWN";
    }
}

COC_API const char* coc_last_error(void) { return g_err; }

COC_API int coc_version(void) { return (1 << 16) | 0; }

COC_API coc_status_t coc_debug_inject_timeout(int enable) {
    g_inject.store(enable ? 1 : 0);
    return COC_OK;
}

COC_API int64_t coc_debug_alloc_count(void) { return static_cast<int64_t>(g_alloc_calls.load()); }

COC_API coc_status_t coc_debug_clock_probe(int slot) {
    if (slot < -1 || slot >= CLOCK_SLOTS) return fail(COC_ERR_INVALID_ARG, "clock slot %d outside [-1, %d)", slot, CLOCK_SLOTS);
    g_clock_slot.store(slot);
    return COC_OK;
}

COC_API coc_status_t coc_debug_clock_read(int slot, int64_t* cycles, int64_t* ns) {
    if (slot < 0 || slot >= CLOCK_SLOTS || cycles == nullptr || ns == nullptr)
        return fail(COC_ERR_INVALID_ARG, "clock slot %d outside [0, %d) or NULL output", slot, CLOCK_SLOTS);
    *cycles = 0;
    *ns = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    unsigned* status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) status = it->second.status;
    }
    if (status == nullptr) return COC_OK;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned long long v[2] = {0, 0};
    unsigned long long* src = reinterpret_cast<unsigned long long*>(status + STATUS_WORDS) + 2 * slot;
    if ((e = cudaMemcpy(v, src, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "cudaMemcpy(clock)");
    if ((e = cudaMemset(src, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "cudaMemset(clock)");
    *cycles = static_cast<int64_t>(v[0]);
    *ns = static_cast<int64_t>(v[1]);
    return COC_OK;
}

COC_API coc_status_t coc_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    coc_status_t st = COC_OK;
    for (auto& kv : g_dev) {
        if (!kv.second.ws.empty() && cudaSetDevice(kv.first) == cudaSuccess) {
            for (auto& w : kv.second.ws) {
                if (w.second.last_use != nullptr) {
                    cudaEventSynchronize(w.second.last_use);
                    cudaEventDestroy(w.second.last_use);
                }
                if (w.second.ptr != nullptr && cudaFree(w.second.ptr) != cudaSuccess)
                    st = fail(COC_ERR_CUDA, "could not free a workspace of device %d", kv.first);
            }
            kv.second.ws.clear();
        }
        if (kv.second.pool != nullptr) {
            if (cudaSetDevice(kv.first) == cudaSuccess && cudaMemPoolDestroy(kv.second.pool) == cudaSuccess)
                kv.second.pool = nullptr;
            else
                st = fail(COC_ERR_CUDA, "could not destroy the workspace pool of device %d", kv.first);
        }
        if (kv.second.status != nullptr) {
            if (cudaSetDevice(kv.first) == cudaSuccess && cudaFree(kv.second.status) == cudaSuccess)
                kv.second.status = nullptr;
            else
                st = fail(COC_ERR_CUDA, "could not free the status buffer of device %d", kv.first);
        }
    }
    if (have_cur) cudaSetDevice(cur);
    g_dev.clear();
    noalloc_forget_devices();
    return st;
}

// ---- helpers shared with the allocation-free entry point (coc_noalloc.cu) ----
namespace coc {

coc_status_t validate_all_reduce_args(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                      const void* const* w, void* const* out, coc_dtype_t dt, int chunks,
                                      int deterministic) {
    return validate_row_parallel(R, m, n, k_shard, x, w, out, R, dt, chunks, deterministic, 2);
}

coc_status_t report_error(coc_status_t st, const char* msg) { return fail(st, "%s", msg); }

int inject_timeout_enabled() { return g_inject.load(); }

}  // namespace coc
