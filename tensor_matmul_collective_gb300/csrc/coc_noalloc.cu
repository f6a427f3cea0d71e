// coc_matmul_all_reduce_noalloc: MATMUL_ALL_REDUCE without any device
// allocation by the library.
//
// Who needs it: callers that must not call cudaMalloc at the point where
// they run this operator — a serving runtime that carves all device memory
// into its own pools up front (and where a cudaMalloc would fail or
// fragment them), code on a latency-critical path where cudaMalloc's
// implicit device-wide synchronisation is unacceptable, and callers whose
// process policy routes every allocation through a custom allocator the
// library cannot see.  The allocating entry points create a small device
// status block the first time they run on a device; this one never does.
//
// The only device scratch the fused kernel needs is that status block (the
// words its bounded waits write when one runs out).  Here it lives in a
// file-scope __device__ array of fixed size, which every GPU that loads the
// library holds until the process exits.  Host code may not pass the array's
// name to a kernel (on the host it is only a stand-in symbol), so its device
// address is looked up with cudaGetSymbolAddress once per device, with that
// device current, on the first call on that device.
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "coc_internal.h"

// 256 bytes: room for the kernel's status block (STATUS_BLOCK_WORDS words).
constexpr int kNoallocScratchWords = 64;
static_assert(coc::STATUS_BLOCK_WORDS <= kNoallocScratchWords, "status block must fit the static scratch");

static __device__ __align__(256) unsigned g_noalloc_scratch[kNoallocScratchWords];

namespace coc {
namespace {

constexpr int kMaxDevices = 64;

struct NoallocDevice {
    bool ready = false;
    unsigned* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int sm_count = 0;
};

std::mutex g_mu;
NoallocDevice g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

coc_status_t cuda_error(cudaError_t e, const char* what) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return report_error(COC_ERR_CUDA, msg);
}

// One-time set-up for the current device.  Allocates nothing.
coc_status_t setup(NoallocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return report_error(COC_ERR_UNSUPPORTED, "device index beyond 63");
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode_fn == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return report_error(COC_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    NoallocDevice& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_error(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return report_error(COC_ERR_UNSUPPORTED, "this library is built for sm_103a");
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return cuda_error(e, "cudaGetSymbolAddress(scratch)");
        // the status block starts at zero; after this it is cleared only when
        // coc_sync_status reads a non-zero status, so a timeout stays visible
        // until it is reported (later calls do not wipe it)
        if ((e = cudaMemset(p, 0, sizeof g_noalloc_scratch)) != cudaSuccess) return cuda_error(e, "cudaMemset(scratch)");
        d.scratch = static_cast<unsigned*>(p);
        d.ready = true;
    }
    *out = &d;
    return COC_OK;
}

coc_status_t encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                       uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return report_error(COC_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    return COC_OK;
}

}  // namespace
}  // namespace coc

using namespace coc;

extern "C" __attribute__((visibility("default"))) coc_status_t coc_matmul_all_reduce_noalloc(
    int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x, const void* const* w, void* const* out,
    coc_dtype_t dt, int chunks, int deterministic, coc_stream_t stream) {
    coc_status_t st = validate_all_reduce_args(R, m, n, k_shard, x, w, out, dt, chunks, deterministic);
    if (st != COC_OK || m == 0 || n == 0) return st;
    // The kernel's scratch need is its status block, whatever the sizes; the
    // check stays so that a larger need can never overrun the static array.
    const size_t need_words = STATUS_WORDS;
    if (need_words > static_cast<size_t>(kNoallocScratchWords))
        return report_error(COC_ERR_SHAPE, "scratch need exceeds the 256-byte static scratch of the no-alloc path");

    NoallocDevice* d = nullptr;
    if ((st = setup(&d)) != COC_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    KParams p;
    std::memset(&p, 0, sizeof p);
    p.R = R;
    p.n_out = R;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k_shard);
    p.num_kshards = R;
    p.kblocks = static_cast<int>((k_shard + BK - 1) / BK);
    p.m_tiles = static_cast<int>((m + BM - 1) / BM);
    p.n_tiles = static_cast<int>((n + BN - 1) / BN);
    p.units = p.m_tiles * p.n_tiles;
    const int64_t chunk_rows = m / chunks;
    p.chunk_mt = (chunk_rows > 0 && chunk_rows % BM == 0) ? static_cast<int>(chunk_rows / BM) : 0;
    p.rows_per_rank = static_cast<int>(m / R);
    p.store_rows = 32;
    p.a_box_rows = BM;
    const CUtensorMapDataType tdt = dt == COC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    for (int r = 0; r < R; ++r) {
        if (k_shard > 0) {
            if ((st = encode_2d(&p.tm_a[r], tdt, x[r], k_shard, m, k_shard * 2, BK, BM)) != COC_OK) return st;
            if ((st = encode_2d(&p.tm_b[r], tdt, w[r], n, k_shard, n * 2, 64, BK)) != COC_OK) return st;
        }
        if ((st = encode_2d(&p.tm_out[r], tdt, out[r], n, m, n * 2, EPI_COLS, p.store_rows)) != COC_OK) return st;
    }
    p.status = d->scratch;
    p.inject_timeout = inject_timeout_enabled();
    p.clock_slot = -1;
    const int grid = p.units < d->sm_count ? p.units : d->sm_count;
    const cudaError_t e = launch(OP_AR, dt == COC_BF16, false, p, grid, s);
    if (e != cudaSuccess) return cuda_error(e, "kernel launch");
    return COC_OK;
}

namespace coc {

coc_status_t noalloc_take_status(unsigned (&words)[STATUS_WORDS]) {
    for (int i = 0; i < STATUS_WORDS; ++i) words[i] = 0u;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return COC_OK;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_devices[dev].ready) return COC_OK;   // never ran here: nothing to report, nothing set up
    }
    if ((e = cudaMemcpyFromSymbol(words, g_noalloc_scratch, sizeof words)) != cudaSuccess)
        return cuda_error(e, "cudaMemcpyFromSymbol(scratch)");
    if (words[0] != 0u) {
        const unsigned zero[STATUS_WORDS] = {};
        if ((e = cudaMemcpyToSymbol(g_noalloc_scratch, zero, sizeof zero)) != cudaSuccess)
            return cuda_error(e, "cudaMemcpyToSymbol(scratch)");
    }
    return COC_OK;
}

void noalloc_forget_devices() {
    std::lock_guard<std::mutex> lk(g_mu);
    for (NoallocDevice& d : g_devices) d = NoallocDevice{};
}

}  // namespace coc
