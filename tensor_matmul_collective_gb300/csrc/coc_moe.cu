// MoE expert-parallel dispatch (the token all-to-all in front of the experts'
// GroupedMatMul; MindSpeed-LLM overlap blog, section 第二层MC2, "EP MC2").
// R ranks, E = R * eloc experts, expert e on rank e / eloc, top-1 routing.
// Destination rank q receives every token routed to one of its experts,
// grouped by expert (ascending), inside an expert by source rank, inside a
// source rank by token index; each expert's group starts on a 256-row
// boundary of q's buffer so that the grouped GEMM's row tiles never straddle
// two experts.
//
// moe_route_kernel    one CTA, 32 warps over contiguous segments of the source
//                     ranks' tokens: counts, offsets and every token's
//                     destination row (deterministic, stable)
// moe_permute_kernel  one warp per token row: the copy itself
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "coc_internal.h"

namespace coc {
namespace {

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

constexpr int kRouteAhead = 8;   // 32-token chunks of expert ids loaded ahead

// Expert id of token t of this warp's rank, -1 if t is past the end or the id
// is out of range (which is reported and the token not dispatched).
__device__ __forceinline__ int route_id(const MoeRouteArgs& a, const int32_t* idx, int t) {
    if (t >= a.T) return -1;
    const int e = __ldg(idx + t);
    if (e < 0 || e >= a.E) {
        atomicOr(a.status, DEV_ERR_BAD_INDEX);
        return -1;
    }
    return e;
}

// Each source rank's tokens are cut into S contiguous segments (S = 32 / R
// warps per rank, at least one); warp (r, s) counts and later places segment
// s of rank r.  Segment order within a rank is token order, so the placement
// is the same as one pass over the rank's tokens.
constexpr int kRouteWarps = 32;

__global__ void __launch_bounds__(32 * kRouteWarps) moe_route_kernel(const __grid_constant__ MoeRouteArgs a) {
    __shared__ int cnt[kRouteWarps][MOE_MAX_EXPERTS];   // per warp: tokens per expert, later its base
    __shared__ int off[MOE_MAX_EXPERTS];                 // group offset of expert e in its rank's buffer
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = kRouteWarps / a.R;                     // segments per rank (R <= 8)
    const int seg_len = ((a.T + S - 1) / S + 31) / 32 * 32;
    for (int i = threadIdx.x; i < kRouteWarps * MOE_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();

    const int r = warp / S, sgm = warp - r * S;
    const bool active = r < a.R;
    const int t_begin = sgm * seg_len, t_end = min(a.T, t_begin + seg_len);
    // 1. counts: warp w alone writes row w
    if (active) {
        const int32_t* idx = a.idx[r];
        for (int t0 = t_begin; t0 < t_end; t0 += 32 * kRouteAhead) {
            int e[kRouteAhead];
#pragma unroll
            for (int i = 0; i < kRouteAhead; ++i) {
                const int t = t0 + 32 * i + lane;
                e[i] = (t < t_end) ? route_id(a, idx, t) : -1;
            }
#pragma unroll
            for (int i = 0; i < kRouteAhead; ++i) {
                const uint32_t same = __match_any_sync(0xffffffffu, e[i]);
                if (e[i] >= 0 && lane == __ffs(same) - 1) cnt[warp][e[i]] += __popc(same);
                __syncwarp();
            }
        }
    }
    __syncthreads();

    // 2. per expert: group size and offset (groups of a rank padded to 256 rows)
    const int W = a.R * S;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int n = 0;
        for (int w = 0; w < W; ++w) n += cnt[w][e];
        int o = 0;
        for (int x = (e / a.eloc) * a.eloc; x < e; ++x) {
            int nx = 0;
            for (int w = 0; w < W; ++w) nx += cnt[w][x];
            o += (nx + MOE_GROUP_ALIGN - 1) / MOE_GROUP_ALIGN * MOE_GROUP_ALIGN;
        }
        off[e] = o;
        a.counts[e] = n;
        a.offsets[e] = o;
    }
    __syncthreads();
    // 3. within expert e, warp (r, s)'s tokens start after those of earlier
    //    ranks and of earlier segments of rank r
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            const int c = cnt[w][e];
            cnt[w][e] = run;
            run += c;
        }
    }
    __syncthreads();

    // 4. placement: after the earlier tokens of this segment routed to the
    //    same expert (match_any ranks equal ids inside a 32-token chunk)
    if (active) {
        const int32_t* idx = a.idx[r];
        const uint32_t lt = lanemask_lt();
        for (int t0 = t_begin; t0 < t_end; t0 += 32 * kRouteAhead) {
            int e[kRouteAhead];
#pragma unroll
            for (int i = 0; i < kRouteAhead; ++i) {
                const int t = t0 + 32 * i + lane;
                e[i] = (t < t_end) ? __ldg(idx + t) : -1;
                if (e[i] < 0 || e[i] >= a.E) e[i] = -1;
            }
#pragma unroll
            for (int i = 0; i < kRouteAhead; ++i) {
                const int t = t0 + 32 * i + lane;
                const uint32_t same = __match_any_sync(0xffffffffu, e[i]);
                const int pos = (e[i] >= 0) ? off[e[i]] + cnt[warp][e[i]] + __popc(same & lt) : -1;
                __syncwarp();
                if (e[i] >= 0 && lane == __ffs(same) - 1) cnt[warp][e[i]] += __popc(same);
                __syncwarp();
                if (t < t_end) {
                    a.dest[static_cast<long long>(r) * a.T + t] = pos;
                    if (a.srcmap != nullptr && pos >= 0)
                        a.srcmap[static_cast<long long>(e[i] / a.eloc) * a.cap + pos] = r * a.T + t;
                }
            }
        }
    }
}

// One warp per token row: 16-byte vectors of X_r[t] to xd[q][dest].
__global__ void __launch_bounds__(256) moe_permute_kernel(const __grid_constant__ MoePermuteArgs a) {
    const long long nrows = static_cast<long long>(a.R) * a.T;
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int vecs = a.h / 8;
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < nrows;
         w += warps) {
        const int r = static_cast<int>(w / a.T);
        const int t = static_cast<int>(w - static_cast<long long>(r) * a.T);
        const int dst_row = __ldg(a.dest + w);
        if (dst_row < 0) continue;
        const int q = __ldg(a.idx[r] + t) / a.eloc;
        const uint4* src = reinterpret_cast<const uint4*>(a.x[r] + static_cast<long long>(t / a.k) * a.h);
        uint4* dst = reinterpret_cast<uint4*>(a.xd[q] + static_cast<long long>(dst_row) * a.h);
        for (int v = lane; v < vecs; v += 32) dst[v] = __ldg(src + v);
    }
}

// Top-k combine: one warp per token, lanes over 8-column chunks; the k expert
// outputs are weighted and summed in fp32 in slot order, then rounded once.
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            const float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}
template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        } else {
            const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool BF16>
__global__ void __launch_bounds__(256) moe_combine_kernel(const __grid_constant__ MoeCombineArgs a) {
    const long long ntok = static_cast<long long>(a.R) * a.tokens;
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int vecs = a.f / 8;
    const long long entries = static_cast<long long>(a.tokens) * a.k;
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < ntok;
         w += warps) {
        const int r = static_cast<int>(w / a.tokens);
        const int t = static_cast<int>(w - static_cast<long long>(r) * a.tokens);
        uint16_t* dst = a.out[r] + static_cast<long long>(t) * a.f;
        for (int v = lane; v < vecs; v += 32) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < a.k; ++j) {
                const long long ent = static_cast<long long>(t) * a.k + j;
                const int row = __ldg(a.dest + r * entries + ent);
                if (row < 0) continue;
                const int q = __ldg(a.idx[r] + ent) / a.eloc;
                const float g = __ldg(a.gates[r] + ent);
                float yv[8];
                unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(a.y[q] + static_cast<long long>(row) * a.f) + v), yv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(g, yv[i], acc[i]);
            }
            reinterpret_cast<uint4*>(dst)[v] = pack8<BF16>(acc);
        }
    }
}

}  // namespace

cudaError_t launch_moe_combine(const MoeCombineArgs& a, bool bf16, int sm_count, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.R) * a.tokens;
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows + 7) / 8;
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (bf16)
        moe_combine_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    else
        moe_combine_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_moe_route(const MoeRouteArgs& a, cudaStream_t stream) {
    moe_route_kernel<<<1, 32 * kRouteWarps, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_moe_permute(const MoePermuteArgs& a, int sm_count, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.R) * a.T;
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows + 7) / 8;
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    moe_permute_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace coc
