// w8A16 streaming pre-pass: every rank's int8 weight is dequantised once into
// a 16-bit buffer, Wd = rne((q - z) * s), which the AllReduce kernel then
// reads as an ordinary fp16/bf16 weight.  Used for large m, where the fused
// kernel would repeat the dequantisation of each weight tile once per row
// tile (m / 256 times) in shared memory; here each weight element is read
// once (1 byte) and written once (2 bytes).  The conversion is the fused
// kernel's own (coc_dequant.cuh), so both paths give the same bits.
#include "coc_dequant.cuh"
#include "coc_internal.h"

namespace coc {
namespace {

constexpr int kPrepassRows = 8;    // weight rows per thread: divides every group size (a multiple of 64)
constexpr int kPrepassThreads = 256;

// Thread i -> (rank, block of kPrepassRows rows, 16-column chunk), chunks
// fastest so that a warp reads 512 and writes 1024 contiguous bytes per row.
template <bool BF16>
__global__ void __launch_bounds__(kPrepassThreads) w8_prepass_kernel(const __grid_constant__ W8PrepassArgs a) {
    const int chunks = a.n / 16;
    const int rblocks = (a.k + kPrepassRows - 1) / kPrepassRows;
    const long long per_rank = static_cast<long long>(chunks) * rblocks;
    const long long total = per_rank * a.R;
    const W8Layout L{a.gran, a.group, a.n};
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / per_rank);
        const long long v = i - r * per_rank;
        const int rb = static_cast<int>(v / chunks);
        const int j0 = static_cast<int>(v - static_cast<long long>(rb) * chunks) * 16;
        const int t0 = rb * kPrepassRows;
        Dq<BF16> d0, d1;
        d0.load(L, a.scale[r], a.zero[r], t0, j0);
        d1.load(L, a.scale[r], a.zero[r], t0, j0 + 8);
        const int8_t* q = a.q[r] + static_cast<long long>(t0) * a.n + j0;
        uint16_t* o = a.out[r] + static_cast<long long>(t0) * a.n + j0;
        const int rows = min(kPrepassRows, a.k - t0);
        // every row's load in flight before the first conversion (the pass is
        // bound by HBM latency x bytes in flight)
        uint4 wv[kPrepassRows];
#pragma unroll
        for (int t = 0; t < kPrepassRows; ++t)
            wv[t] = (t < rows) ? __ldg(reinterpret_cast<const uint4*>(q + static_cast<long long>(t) * a.n))
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int t = 0; t < kPrepassRows; ++t) {
            if (t >= rows) break;
            uint4* dst = reinterpret_cast<uint4*>(o + static_cast<long long>(t) * a.n);
            dst[0] = d0.convert(make_uint2(wv[t].x, wv[t].y));
            dst[1] = d1.convert(make_uint2(wv[t].z, wv[t].w));
        }
    }
}

}  // namespace

cudaError_t launch_w8_prepass(const W8PrepassArgs& a, bool bf16, int sm_count, cudaStream_t stream) {
    const long long total = static_cast<long long>(a.n / 16) * ((a.k + kPrepassRows - 1) / kPrepassRows) * a.R;
    if (total <= 0) return cudaSuccess;
    long long blocks = (total + kPrepassThreads - 1) / kPrepassThreads;
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 64;
    if (blocks > cap) blocks = cap;   // grid-stride beyond 64 blocks per SM
    if (bf16)
        w8_prepass_kernel<true><<<static_cast<unsigned>(blocks), kPrepassThreads, 0, stream>>>(a);
    else
        w8_prepass_kernel<false><<<static_cast<unsigned>(blocks), kPrepassThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace coc
