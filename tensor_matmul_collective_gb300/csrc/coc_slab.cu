// Column-slab kernel: MATMUL_ALL_REDUCE, MATMUL_REDUCE_SCATTER and
// ALL_GATHER_MATMUL(_V2) at decode-sized m (CoC page, 融合算子实现: the same
// operators as the persistent kernel, for the few-row activations of token
// generation).
//
// At m <= 128 (one row tile) the operator reads the R weight shards (R x
// k_shard x n) once and does little arithmetic per weight byte, so its time
// is the weight stream.  The persistent kernel's 128 x 256 tiles are too few to spread that
// stream over the SMs, and cutting K across CTAs (the rank split) costs a
// cross-CTA reduction after the last weight byte arrives.  Here a work unit
// is one column slab of the output instead: all m rows by SN = 64 or 128
// columns, accumulated over the whole contraction (rank 0..R-1, k ascending)
// in one CTA, so n / SN units cover the SMs and nothing is reduced across
// CTAs.
//
//   stage          kps = 1, 2 or 4 k-blocks of 64 k, in as few TMA operations
//                  as the layouts allow: measured, a CTA's weight stream is
//                  bound by the TMA operations it has in flight, not by their
//                  bytes (one 8 KiB box per 64 k moved 26 GB/s per SM; the
//                  stream of the same weight in 32 KiB boxes is several times
//                  faster).
//   A (X shards)   per k-block a_rows = roundup(m, 8) rows x 64 k (128-byte
//                  swizzle, K-major): one 3-D box (k within the block, row,
//                  k-block) for the whole stage when k_shard % 64 == 0, else
//                  one 2-D box per k-block.  The MMA is M = 128, so it also
//                  reads the 128 - a_rows rows after a k-block's rows, which
//                  belong to the next k-blocks: those accumulator rows are
//                  never read back.
//   B (W shards)   k x n storage (MN-major): per 64-column group one box of
//                  64 columns x kps * 64 k; n x k storage (K-major): per
//                  k-block SN rows x 64 k, as one 3-D box for the stage when
//                  k_shard % 64 == 0.
//   AllGather      m = R m_shard gathered rows; a unit is one column slab
//                  of one rank's output (R x n_shard / SN units), its
//                  contraction the full k (no shard loop).  A is the gathered
//                  X, stacked beforehand by coc_ag_gather_kernel into one
//                  m x k buffer (V2's first gathered output, else the call's
//                  scratch) and loaded like one AllReduce shard; B comes from
//                  the unit's rank's W, and the slab is stored to that rank's
//                  output only.  V2's other gathered copies are written from
//                  that buffer by the epilogue warps while the first slab's
//                  mainloop runs.  (Loading A as one box per source rank and
//                  k-block instead measured 1.9x slower at 8 ranks: a CTA's
//                  stream is bound by its TMA operations, about 80 ns each.)
//   stages         as many as fit in shared memory (up to kSlabMaxStages).
//   accumulator    two TMEM buffers of SN fp32 columns, so a CTA with a
//                  second unit overlaps its epilogue with the next mainloop.
//
// Warp roles (192 threads, one CTA per SM, persistent over slabs):
//   warp 0      TMA producer; it initialised the barriers, so it starts
//               loading without waiting for the TMEM allocation
//   warp 1      TMEM owner + MMA issuer (tcgen05.mma kind::f16, M 128, N SN)
//   warps 2-5   epilogue: warp q drains accumulator lanes 32q..32q+31 (rows)
//               when they hold output rows, rounds them, transposes them
//               through a swizzled shared-memory buffer and writes coalesced
//               128-byte row segments: every rank output (AllReduce) or the
//               rank owning each row (ReduceScatter).
//
// Every mbarrier wait is bounded (COC_WAIT_NS); a wait that runs out sets
// the CTA abort flag and the device status word, every role leaves its loop,
// issued copies and MMAs are drained, TMEM is freed and the kernel returns.
#include <atomic>
#include <cstdlib>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "coc_dequant.cuh"
#include "coc_internal.h"
#include "coc_ptx.cuh"

namespace coc {
namespace {

constexpr int SLAB_DQ_WARPS = 8;                  // w8A16: dequantisation warps
constexpr int SLAB_DQ_GW = SLAB_DQ_WARPS / 2;      // ... in two groups taking alternate stages
// warps: producer, MMA, 4 epilogue; w8A16 adds the dequant warps
__host__ __device__ constexpr int slab_threads(bool w8) { return (6 + (w8 ? SLAB_DQ_WARPS : 0)) * 32; }
constexpr uint32_t kSlabBoxBytes = 64 * BK * 2;   // one 64 x 64 16-bit box
constexpr uint32_t kSlabStageBar = 3;             // named barrier of the set-up phase
static_assert(kSlabMaxStages <= 32, "the producer's fill masks hold one bit per stage");

__host__ __device__ constexpr uint32_t slab_bar_bytes(int stages, bool w8) {
    return static_cast<uint32_t>(8 * (2 * stages + (w8 ? 2 * kSlabW8BStages : 0) + 8) + 16);
}
// Reception area of a slab split over `split` CTAs: per other part, per row
// quadrant holding output rows (a_rows / 32 rounded up), 32 rows of the (64
// boxes / split) fp32 columns this CTA finalises.
__host__ __device__ constexpr uint32_t slab_recv_bytes(int boxes, int split, int a_rows) {
    return split > 1 ? static_cast<uint32_t>((split - 1) * ((a_rows + 31) / 32) * 32 * (64 * boxes / split) * 4) : 0u;
}
// Above 32 rows the reception area lies over the rings, which are idle once
// every part's last MMA has completed (the parts wait for that before they
// push): its room goes to more stages.  Measured, from 64 rows: bf16 m 128
// 36.1 -> 30.9 us, w8A16 m 128 44.8 -> 39.2 us; at m 16 the wait for the
// slowest part's mainloop cost more (0.2-1.1 us) than the extra stage gave.
__host__ __device__ constexpr bool slab_recv_over_rings(int split, int a_rows) { return split > 1 && a_rows > 32; }

// w8A16: bytes of one stage of the producer's ring: X of the stage (kps
// k-blocks x a_rows rows x 128 bytes, first: 1 KiB aligned for the swizzle),
// the int8 weight (kps k-blocks x 64 rows x 64 boxes columns) and its scale /
// zero-point table rows (kps rows of 64 boxes 16-bit scales, then kps rows of
// int8 zero points), rounded to 1 KiB.
__host__ __device__ constexpr int slab_raw_stage(int kps, int boxes, int a_rows) {
    return kps * a_rows * 128 + (kps * 64 * 64 * boxes + kps * 64 * boxes * 3 + 1023) / 1024 * 1024;
}

template <int V>
struct IntC {
    static constexpr int value = V;
};

// w8A16: one dequant thread's share of a stage of NB 64-column groups x KPS
// k-blocks: chunk cc (8 columns) of rows kr0, kr0 + R_STEP, ... of every
// k-block, from the int8 stage `raw` (rows of 64 NB bytes) into the 16-bit B
// stage (NB groups of KPS k-blocks x 64 rows x 128 bytes, 16-byte chunks
// XOR-ed with row % 8).  Up to 8 rows' loads are issued before their conversions.
// The scale and zero points of this thread's 8 columns from table slot
// `tab` of the stage (16-bit scales at tab, int8 zero points at ztab; zero
// points 0 when there are none, scales 0 past n, as for the global tables).
template <bool BF16>
__device__ __forceinline__ void dq_from_slot(Dq<BF16>& dq, const uint8_t* tab, const uint8_t* ztab, int cc, bool valid) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    int z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (valid) {
        const uint4 s4 = *reinterpret_cast<const uint4*>(tab + cc * 16);
        w[0] = s4.x; w[1] = s4.y; w[2] = s4.z; w[3] = s4.w;
        if (ztab != nullptr) {
            const uint2 z8 = *reinterpret_cast<const uint2*>(ztab + cc * 8);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                z[e] = static_cast<int8_t>((z8.x >> (8 * e)) & 0xFFu);
                z[4 + e] = static_cast<int8_t>((z8.y >> (8 * e)) & 0xFFu);
            }
        }
    }
    dq.set(w, z);
}

template <bool BF16, int NB, int KPS>
__device__ __forceinline__ void dequant_stage(const uint8_t* raw, uint8_t* bst, int kr0, int cc, int c16, Dq<BF16>& dq,
                                              const uint8_t* tab, const uint8_t* ztab, bool valid, bool per_group) {
    constexpr int W = 64 * NB;
    constexpr int R_STEP = (SLAB_DQ_GW * 32) / (W / 8);
    constexpr int RPK = BK / R_STEP;   // rows per k-block
    constexpr int ROWS = KPS * RPK;
    constexpr int RB = ROWS < 8 ? ROWS : 8;   // rows in flight (registers)
#pragma unroll
    for (int b0 = 0; b0 < ROWS; b0 += RB) {
        uint2 q8[RB];
#pragma unroll
        for (int j = 0; j < RB; ++j) {
            const int i = b0 + j;
            q8[j] = *reinterpret_cast<const uint2*>(raw + ((i / RPK) * BK + kr0 + (i % RPK) * R_STEP) * W + cc * 8);
        }
#pragma unroll
        for (int j = 0; j < RB; ++j) {
            const int i = b0 + j;
            if (per_group && i % RPK == 0)
                dq_from_slot<BF16>(dq, tab + (i / RPK) * W * 2, ztab != nullptr ? ztab + (i / RPK) * W : nullptr, cc, valid);
            const int kk = (i / RPK) * BK + kr0 + (i % RPK) * R_STEP;   // row of the stage
            *reinterpret_cast<uint4*>(bst + kk * 128 + ((c16 ^ (kk & 7)) << 4)) = dq.convert(q8[j]);
        }
    }
}

// AllGather-V2: the gathered X (m x k at gsrc[0], stacked before the kernel)
// into every non-NULL gdst.  Its 16-byte vectors are cut into `ctas`
// contiguous slices, one per CTA, shared by the CTA's epilogue warps (wi of
// NUM_EPI_WARPS) while the first slab's mainloop runs.
__device__ __forceinline__ void slab_copy_gathered(const KParams& p, int cta, int ctas, int wi, int lane) {
    const long long total = static_cast<long long>(p.m) * (p.k / 8);   // k % 8 == 0
    const long long lo = total * cta / ctas, hi = total * (cta + 1) / ctas;
    const long long a = lo + (hi - lo) * wi / NUM_EPI_WARPS, b = lo + (hi - lo) * (wi + 1) / NUM_EPI_WARPS;
    const uint4* src = reinterpret_cast<const uint4*>(p.gsrc[0]);
    for (long long v0 = a; v0 < b; v0 += 32 * 4) {
        uint4 d[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const long long v = v0 + j * 32 + lane;
            d[j] = v < b ? src[v] : make_uint4(0u, 0u, 0u, 0u);
        }
        for (int r = 0; r < p.R; ++r) {
            uint4* dst = reinterpret_cast<uint4*>(p.gdst[r]);
            if (dst == nullptr) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const long long v = v0 + j * 32 + lane;
                if (v < b) dst[v] = d[j];
            }
        }
    }
}

template <int OP, bool BF16, bool W8>
__global__ void __launch_bounds__(slab_threads(W8), 1) coc_slab_kernel(const __grid_constant__ KParams p) {
    constexpr int THREADS = slab_threads(W8);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // every kernel parameter the roles need, read once up front (the first
    // read of each parameter line is a long-latency miss)
    const int S = p.slab_stages;
    const int nb = p.slab_boxes;          // 64-column groups per slab
    const int kps = p.slab_kps;           // k-blocks per stage (divides kblocks)
    const int csplit = p.slab_split;      // CTAs (one cluster) per slab
    const int a_rows = p.a_box_rows;
    const int R = p.num_kshards;          // shards summed per slab (AllGather: 1)
    const int kblocks = p.kblocks;
    const int spr = p.n_tiles;            // AllGather: slabs per rank output
    const int units = p.units;
    const int m = p.m, n = p.n;
    const uint32_t a_kb = static_cast<uint32_t>(a_rows) * 128u;                 // A bytes per k-block
    const uint32_t a_stage = static_cast<uint32_t>(kps) * a_kb;
    const uint32_t b_group = static_cast<uint32_t>(kps) * kSlabBoxBytes;       // one 64-column group's k x 64
    const uint32_t b_stage = static_cast<uint32_t>(nb) * b_group;
    const int W = nb * 64;                // slab width
    const int ow = W / csplit;            // columns this CTA finalises (split: its share of the slab)
    // w8A16: the producer's ring carries X and the int8 W of each stage (one
    // barrier; freed by the dequant warps and the MMA, so X runs as far ahead
    // as the weight); the dequant warps write the 16-bit W into a second ring
    // of SB stages, freed by the MMA
    const uint32_t raw_stage = W8 ? static_cast<uint32_t>(slab_raw_stage(kps, nb, a_rows)) : 0u;
    constexpr int SB = W8 ? kSlabW8BStages : 0;

    // A first: the MMA reads 128 rows from a k-block's start, past the last
    // stage's A into the B ring (>= 16 KiB), never past the allocation.
    // bf16: S stages of A, then S of B; w8A16: S stages of (X, int8 W,
    // tables), then the SB 16-bit B stages.
    uint8_t* a_st = smem;                                      // bf16: S x a_stage
    uint8_t* raw_st = smem;                                    // w8A16: S x raw_stage (X at the start)
    uint8_t* b_st = W8 ? raw_st + S * raw_stage : a_st + S * a_stage;   // S (w8A16: SB) x b_stage
    // split: the other parts' fp32 sums of this CTA's columns, after the
    // staging buffers, or (over 32 rows) at the start of shared memory over
    // the rings, once every part's last MMA has completed (ring_free)
    const bool over_rings = slab_recv_over_rings(csplit, a_rows);
    const uint32_t ring_bytes = W8 ? S * raw_stage + SB * b_stage : S * (a_stage + b_stage);
    const uint32_t recv_bytes = slab_recv_bytes(nb, csplit, a_rows);
    uint8_t* stg = smem + (over_rings && recv_bytes > ring_bytes ? recv_bytes : ring_bytes);   // 4 warps x 4 KiB
    uint8_t* recv = over_rings ? smem : stg + NUM_EPI_WARPS * EPI_BUF_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(stg + NUM_EPI_WARPS * EPI_BUF_BYTES + (over_rings ? 0u : recv_bytes));   // [S]
    uint64_t* empty = full + S;                    // [S]  (w8A16: read by the stage's dequant warps and the MMA)
    uint64_t* bfull = empty + S;                   // [SB] w8A16: 16-bit B stage written (its dequant warps)
    uint64_t* bempty = bfull + SB;                 // [SB] w8A16: 16-bit B stage consumed by the MMA
    uint64_t* accf = bempty + SB;                  // [2] accumulator ready for the epilogue
    uint64_t* acce = accf + 2;                     // [2] accumulator drained (4 epilogue warps)
    uint64_t* never = acce + 2;                    // [1] nothing arrives here (fault-injection test)
    uint64_t* drain = never + 1;                   // [1] MMA drain before TMEM release
    uint64_t* red_full = drain + 1;                // [1] split: every other part pushed its sums here
    uint64_t* ring_free = red_full + 1;            // [1] split: every part's rings are idle
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring_free + 1);
    uint32_t* abort_word = tmem_slot + 1;
    const Ctl ctl{abort_word, p.status};
    const int nq = min(NUM_EPI_WARPS, (m + 31) / 32);   // epilogue warps holding output rows

    if (warp == 0 && lane < p.R && lane < COC_MAX_RANKS) {
        if (lane < R) prefetch_tmap(&p.tm_a[lane]);   // (AllGather: one A map)
        prefetch_tmap(&p.tm_b[lane]);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), W8 ? SLAB_DQ_GW + 1 : 1);
        }
        for (int b = 0; b < SB; ++b) {
            mbar_init(smem_u32(&bfull[b]), SLAB_DQ_GW);
            mbar_init(smem_u32(&bempty[b]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(never), 1);
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(red_full), csplit > 1 ? (csplit - 1) * nq : 1);
        mbar_init(smem_u32(ring_free), csplit > 1 ? csplit : 1);
        *abort_word = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    const uint32_t tmem_cols = static_cast<uint32_t>(2 * W);   // two W-column accumulators
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    // The producer warp (whose lane 0 initialised the barriers) only arrives
    // and starts loading; it waits for the cluster barrier at the end.  Split:
    // the cluster's barriers exist before any part pushes remotely.
    tc_fence_before();
    if (warp == 0) __syncwarp();
    if (csplit > 1) {
        cluster_arrive();
        if (warp != 0) cluster_wait();
    } else if (warp == 0) {
        named_arrive(kSlabStageBar, THREADS);
    } else {
        named_sync(kSlabStageBar, THREADS);
    }
    tc_fence_after();
    // Everything above touches only this CTA's shared and tensor memory and
    // the kernel parameters, so with a programmatic launch it overlaps the
    // previous kernel in the stream; global memory is touched only after it
    // has completed.  Every CTA of this grid is resident at once, so the next
    // kernel may then start on the SMs this one leaves free.
    grid_dependency_wait();
    grid_dependents_launch();
    const uint32_t tmem_base = warp == 0 ? 0u : *tmem_slot;
    const bool probe = p.clock_slot >= 0 && blockIdx.x == 0 && threadIdx.x == 0;
    uint64_t probe_clk = 0, probe_ns = 0;
    if (probe) {
        probe_clk = clock64();
        probe_ns = globaltimer();
    }
    // a unit is one slab (stage s of its contraction: shard s / spk, k-blocks
    // from (s % spk) kps).  Unsplit, CTA b takes slabs b, b + grid, ...;
    // split, cluster c takes slab c alone (the host launches one cluster per
    // slab: the reception areas are never reused), and its part `part` sums
    // stages [st_lo, st_hi), the parts adding up to the whole contraction.
    const uint32_t part = csplit > 1 ? cluster_rank() : 0u;
    const int first_u = static_cast<int>(blockIdx.x) / csplit;
    const int u_step = static_cast<int>(gridDim.x) / csplit;
    const int spk = kblocks / kps;            // stages per shard
    const int spu = R * spk;                  // stages per unit
    const int st_lo = (spu * static_cast<int>(part)) / csplit;
    const int st_hi = (spu * (static_cast<int>(part) + 1)) / csplit;

    if (warp == 0) {
        // ================================================= TMA producer ===
        const bool b_kmajor = p.b_kmajor != 0;
        const bool a3d = p.slab_a3d != 0;
        const uint64_t pol_a = make_l2_policy(2), pol_b = make_l2_policy(1);   // X reused, W streamed once
        uint32_t stage = 0, phase = 0, filled = 0, fill_parity = 0;
        bool ok = true;
        for (int u = first_u; ok && u < units; u += u_step) {
            const int ur = OP == OP_AG ? u / spr : 0;   // AllGather: the rank whose W and output
            const int col0 = (u - ur * spr) * W;
            for (int s = st_lo; s < st_hi; ++s) {
                const int ks = s / spk;
                const int kb = (s - ks * spk) * kps;
                ok = warp_wait(smem_u32(&empty[stage]), phase ^ 1u, ctl, 0x500u + stage);
                if (!ok) break;
                if (lane == 0) {
                    const CUtensorMap* am = &p.tm_a[ks];
                    const CUtensorMap* bm = &p.tm_b[OP == OP_AG ? ur : ks];
                    const uint32_t fb = smem_u32(&full[stage]);
                    // w8A16 per-group: the int8 box plus the in-range columns of the
                    // scale and zero-point rows of the stage's k-blocks (measured:
                    // per-group 50.9 -> 42.8 us at m 16; the per-tensor and
                    // per-channel constants change only per shard and come from
                    // global memory there, which measured faster than an extra
                    // copy per stage or per shard)
                    const int tab_cols = W8 ? min(W, n - col0) : 0;
                    const int tab_rows = (W8 && p.gran == COC_SCALE_GROUP) ? kps : 0;
                    const uint32_t tab_bytes = static_cast<uint32_t>(tab_rows * tab_cols * (p.has_zero ? 3 : 2));
                    mbar_expect_tx(fb, a_stage + (W8 ? static_cast<uint32_t>(kps * 64 * W) + tab_bytes : b_stage));
                    // X of the stage (w8A16: at the start of the int8 stage)
                    const uint32_t adst = W8 ? smem_u32(raw_st + stage * raw_stage) : smem_u32(a_st + stage * a_stage);
                    if (a3d) {
                        tma_load_3d_hint(adst, am, 0, 0, kb, fb, pol_a);
                    } else {
                        for (int t = 0; t < kps; ++t)
                            tma_load_2d_hint(adst + t * a_kb, am, (kb + t) * BK, 0, fb, pol_a);
                    }
                    const uint32_t bdst = smem_u32(b_st + stage * b_stage);
                    if constexpr (W8) {
                        // the int8 W of the stage after its X: W columns x kps k-blocks, one box
                        uint8_t* rs = raw_st + stage * raw_stage + a_stage;
                        tma_load_2d_hint(smem_u32(rs), bm, col0, kb * BK, fb, pol_b);
                        uint8_t* tab = rs + kps * 64 * W;   // scale rows, then zero-point rows
                        for (int t = 0; t < tab_rows; ++t) {
                            const long long row =
                                (p.gran == COC_SCALE_GROUP) ? static_cast<long long>((kb + t) * BK / p.group) * n : 0LL;
                            bulk_load_g2s(smem_u32(tab + t * W * 2), p.scale[ks] + row + col0,
                                          static_cast<uint32_t>(tab_cols * 2), fb);
                            if (p.has_zero)
                                bulk_load_g2s(smem_u32(tab + kps * W * 2 + t * W), p.zero[ks] + row + col0,
                                              static_cast<uint32_t>(tab_cols), fb);
                        }
                    } else if (b_kmajor) {
                        if (a3d) {
                            tma_load_3d_hint(bdst, bm, 0, col0, kb, fb, pol_b);
                        } else {
                            for (int t = 0; t < kps; ++t)
                                tma_load_2d_hint(bdst + t * (b_stage / kps), bm, (kb + t) * BK, col0, fb, pol_b);
                        }
                    } else {
                        for (int j = 0; j < nb; ++j)
                            tma_load_2d_hint(bdst + j * b_group, bm, col0 + 64 * j, kb * BK, fb, pol_b);
                    }
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                }
                __syncwarp();
                if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            // leave no TMA load in flight into shared memory
            for (int s = 0; s < S; ++s)
                if (filled & (1u << s)) drain_wait(smem_u32(&full[s]), (fill_parity >> s) & 1u, kDrainNs);
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer ===
        // B MN-major (k x n storage): 64-column groups b_group apart, k-block t
        // at +8 KiB t, +2 KiB per 16-k step; B K-major (n x k storage): k-block
        // t at +W x 128 bytes t, +32 bytes per 16-k step, and the "B
        // transposed" bit cleared
        const bool b_kmajor = p.b_kmajor != 0;
        const uint32_t idesc = make_idesc(BF16, BM, W) & (b_kmajor ? ~(1u << 16) : ~0u);
        const uint32_t b_lbo = b_kmajor ? 16u : b_group;
        const uint64_t b_step = b_kmajor ? 2u : 128u;
        const uint32_t b_kb = b_kmajor ? static_cast<uint32_t>(W) * 128u : kSlabBoxBytes;
        uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0;
        int acc_i = 0;
        bool ok = true;
        for (int u = first_u; ok && u < units; u += u_step) {
            const int buf = acc_i & 1;
            ok = warp_wait(smem_u32(&acce[buf]), ((acc_i >> 1) & 1) ^ 1u, ctl, 0x520u + buf);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * W);
            for (int i = 0; i < st_hi - st_lo; ++i) {
                // (w8A16: X landed with the int8 stage, the 16-bit W is in B stage bstage)
                ok = warp_wait(smem_u32(&full[stage]), phase, ctl, 0x540u + stage);
                if (W8 && ok) ok = warp_wait(smem_u32(&bfull[bstage]), bphase, ctl, 0x598u + bstage);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint8_t* a_s = W8 ? raw_st + stage * raw_stage : a_st + stage * a_stage;
                    const uint8_t* b_s = b_st + (W8 ? bstage : stage) * b_stage;
                    for (int t = 0; t < kps; ++t) {
                        const uint64_t ad = make_sdesc(smem_u32(a_s + t * a_kb), 16u, 1024u);
                        const uint64_t bd = make_sdesc(smem_u32(b_s + t * b_kb), b_lbo, 1024u);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            tc_mma_f16(d_tmem, ad + static_cast<uint64_t>(kk) * 2u,
                                       bd + static_cast<uint64_t>(kk) * b_step, idesc,
                                       (i > 0 || t > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (W8) tc_commit(smem_u32(&bempty[bstage]));
                    tc_commit(smem_u32(&empty[stage]));
                }
                __syncwarp();
                if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
                if (W8 && ++bstage == static_cast<uint32_t>(SB)) { bstage = 0; bphase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(smem_u32(&accf[buf]));
            __syncwarp();
            ++acc_i;
        }
        // every issued MMA must finish before TMEM is released
        if (lane == 0) {
            tc_commit(smem_u32(drain));
            drain_wait(smem_u32(drain), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp < 2 + NUM_EPI_WARPS) {
        // ================================================= epilogue ===
        const int q = warp & 3;                  // TMEM lane quadrant this warp may read
        const int row0 = 32 * q;
        const bool active = q < nq;
        uint8_t* buf_s = stg + (warp - 2) * EPI_BUF_BYTES;
        const int n_out = p.n_out, rpr = p.rows_per_rank;
        const uint32_t row_bytes = static_cast<uint32_t>(ow) * 4u;   // one row of a reception slot
        // Round 32 columns of this warp's rows (fp32 bits, lane = row) and
        // store them: row = lane into the staging buffer (64 bytes, 16-byte
        // chunk j at j ^ (row / 2 % 4)), read back so that lane l holds chunk
        // l % 4 of rows l / 4 + 8 i, then 16-byte stores to every rank output
        // (AllReduce) or to the rank owning the row (ReduceScatter).
        auto emit32 = [&](int col, int ur, const uint32_t (&v)[32]) {
            uint8_t* rowp = buf_s + lane * 64;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 w4;
                w4.x = pack2<BF16>(v[8 * j + 0], v[8 * j + 1]);
                w4.y = pack2<BF16>(v[8 * j + 2], v[8 * j + 3]);
                w4.z = pack2<BF16>(v[8 * j + 4], v[8 * j + 5]);
                w4.w = pack2<BF16>(v[8 * j + 6], v[8 * j + 7]);
                *reinterpret_cast<uint4*>(rowp + ((j ^ ((lane >> 1) & 3)) << 4)) = w4;
            }
            __syncwarp();
            const int ch = lane & 3;
            uint4 rv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rr = (lane >> 2) + 8 * i;
                rv[i] = *reinterpret_cast<const uint4*>(buf_s + rr * 64 + ((ch ^ ((rr >> 1) & 3)) << 4));
            }
            __syncwarp();   // the buffer is free for the next 32 columns
            const int c = col + ch * 8;   // n % 8 == 0: a chunk is wholly inside or outside
            if (c >= n) return;
            if constexpr (OP == OP_RS) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int g = row0 + (lane >> 2) + 8 * i;
                    if (g < m) {
                        const int dst = g / rpr;
                        *reinterpret_cast<uint4*>(p.outp[dst] + static_cast<long long>(g - dst * rpr) * n + c) = rv[i];
                    }
                }
            } else {
                // AllReduce: every rank output; AllGather: rank ur's
                const int o0 = OP == OP_AG ? ur : 0, o1 = OP == OP_AG ? ur + 1 : n_out;
                for (int o = o0; o < o1; ++o) {
                    uint16_t* base = p.outp[o] + c;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int g = row0 + (lane >> 2) + 8 * i;
                        if (g < m) *reinterpret_cast<uint4*>(base + static_cast<long long>(g) * n) = rv[i];
                    }
                }
            }
        };
        // reception slot row of source part `src` (not this CTA) for this warp's lane
        auto recv_row = [&](uint32_t src, uint32_t dst_part) {
            const uint32_t sidx = src < dst_part ? src : src - 1u;
            return smem_u32(recv) +
                   ((sidx * static_cast<uint32_t>(nq) + static_cast<uint32_t>(q)) * 32u + static_cast<uint32_t>(lane)) * row_bytes;
        };
        int acc_i = 0;
        bool ok = true;
        if constexpr (OP == OP_AG) {
            // AllGather-V2: this CTA's slice of the other gathered copies
            if (p.has_gather) slab_copy_gathered(p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), warp - 2, lane);
        }
        if (p.inject_timeout) ok = warp_wait(smem_u32(never), 0, ctl, 0x560u);
        for (int u = first_u; ok && u < units; u += u_step) {
            const int buf = acc_i & 1;
            ok = warp_wait(smem_u32(&accf[buf]), (acc_i >> 1) & 1, ctl, 0x570u + buf);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(row0) << 16) + static_cast<uint32_t>(buf * W);
            if (over_rings) {
                // this CTA's rings are idle (a split slab is its only unit, and its
                // last MMA has completed): tell every part, and push only once
                // every part's rings are idle
                if (warp == 2 && lane == 0)
                    for (int j = 0; j < csplit; ++j)
                        mbar_arrive_cluster(map_to_rank(smem_u32(ring_free), static_cast<uint32_t>(j)));
                if (active) {
                    ok = warp_wait<true>(smem_u32(ring_free), 0, ctl, 0x590u);
                    if (!ok) break;
                }
            }
            if (active && csplit > 1) {
                // push this part's sums of every other part's columns into that
                // part's reception area (16-byte chunk c of a row at c ^ (row % 8))
                for (int j = 0; j < csplit; ++j) {
                    if (j == static_cast<int>(part)) continue;
                    const uint32_t dst = map_to_rank(recv_row(part, static_cast<uint32_t>(j)), static_cast<uint32_t>(j));
                    for (int cc = 0; cc < ow; cc += 32) {
                        uint32_t v[32];
                        tmem_ld_32cols(t_row + j * ow + cc, v);
                        tmem_wait_ld();
                        if (row0 + lane < m) {
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                const uint32_t chunk = static_cast<uint32_t>(cc / 4 + jj);
                                asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};"
                                             ::"r"(dst + ((chunk ^ (lane & 7)) << 4)), "r"(v[4 * jj]), "r"(v[4 * jj + 1]),
                                               "r"(v[4 * jj + 2]), "r"(v[4 * jj + 3])
                                             : "memory");
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    for (int j = 0; j < csplit; ++j)
                        if (j != static_cast<int>(part))
                            mbar_arrive_cluster(map_to_rank(smem_u32(red_full), static_cast<uint32_t>(j)));
                ok = warp_wait<true>(smem_u32(red_full), acc_i & 1, ctl, 0x580u);
                if (!ok) break;
            }
            // this CTA's columns: the parts added in part order (its own from
            // TMEM), 32 at a time
            for (int cc = 0; cc < ow; cc += 32) {
                uint32_t v[32];
                if (active) {
                    tmem_ld_32cols(t_row + static_cast<int>(part) * ow + cc, v);
                    tmem_wait_ld();
                }
                if (cc + 32 >= ow) {
                    // the accumulator is free for the unit after next
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acce[buf]));
                }
                const int ur = OP == OP_AG ? u / spr : 0;
                const int col = (u - ur * spr) * W + static_cast<int>(part) * ow + cc;
                if (!active || col >= n) continue;
                if (csplit > 1) {
                    uint32_t own[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) own[i] = v[i];
                    for (int sp = 0; sp < csplit; ++sp) {
                        uint32_t w[32];
                        if (sp == static_cast<int>(part)) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) w[i] = own[i];
                        } else {
                            const uint32_t rb = recv_row(static_cast<uint32_t>(sp), part);
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                const uint32_t chunk = static_cast<uint32_t>(cc / 4 + jj);
                                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(w[4 * jj]), "=r"(w[4 * jj + 1]), "=r"(w[4 * jj + 2]), "=r"(w[4 * jj + 3])
                                             : "r"(rb + ((chunk ^ (lane & 7)) << 4))
                                             : "memory");
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = sp == 0 ? w[i] : __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
                    }
                }
                emit32(col, ur, v);
            }
            ++acc_i;
        }
    }

    if constexpr (W8) {
        if (warp >= 2 + NUM_EPI_WARPS) {
            // ================================================= w8A16 dequant ===
            // Per stage: once the MMA has freed the A and B stage (bempty) and the
            // int8 stage has landed (full), thread tt, which owns 8 consecutive
            // columns (chunk cc) of the slab and the stage rows kr0, kr0 + R_STEP, ... (dequant_stage), reads
            // their int8 bytes, dequantises them (coc_dequant.cuh, the fused
            // kernel's and the pre-pass's conversion) and writes the 16-bit B
            // stage in the MMA's MN-major 128-byte-swizzled layout.  Every warp
            // then arrives on the B stage's `bfull` and the int8 stage's `empty`.
            // Two groups of SLAB_DQ_GW warps take alternate stages (group g the
            // stages c with c % 2 == g, c counted over all units), so one group's
            // waits, fence and arrivals overlap the other's conversion.  Any ring
            // depth works: a slot is refilled (producer) or rewritten (16-bit
            // ring) only after the group that used it and the MMA are done with
            // it, so no wait can be two phases behind its barrier.
            const int dw = warp - 2 - NUM_EPI_WARPS;
            const int group = dw / SLAB_DQ_GW;
            const int tt = (dw % SLAB_DQ_GW) * 32 + lane;
            const int chunks = W / 8;
            const int cc = tt % chunks;
            const int kr0 = tt / chunks;
            const W8Layout w8l{p.gran, p.group, p.n};
            uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0, cnt = 0;
            bool ok = true;
            for (int u = first_u; ok && u < units; u += u_step) {
                const int j0 = u * W + cc * 8;   // this thread's first output column
                int dq_ks = -1;
                Dq<BF16> dq;
                const bool valid = j0 + 8 <= n;   // this thread's columns lie inside the output
                for (int s = st_lo; s < st_hi; ++s, ++cnt) {
                    if (static_cast<int>(cnt & 1u) != group) {   // the other group's stage
                        if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
                        if (++bstage == static_cast<uint32_t>(SB)) { bstage = 0; bphase ^= 1u; }
                        continue;
                    }
                    const int ks = s / spk;
                    // per-tensor / per-channel: the shard's constants from global memory
                    if (ks != dq_ks && p.gran != COC_SCALE_GROUP)
                        dq.load(w8l, p.scale[ks], p.has_zero ? p.zero[ks] : nullptr, 0, j0);
                    dq_ks = ks;
                    ok = warp_wait(smem_u32(&bempty[bstage]), bphase ^ 1u, ctl, 0x5C0u + bstage);
                    if (ok) ok = warp_wait(smem_u32(&full[stage]), phase, ctl, 0x5A0u + stage);
                    if (!ok) break;
                    const uint8_t* raw = raw_st + stage * raw_stage + a_stage;   // after the stage's X
                    const uint8_t* tab = raw + kps * 64 * W;
                    const uint8_t* ztab = p.has_zero ? tab + kps * W * 2 : nullptr;
                    uint8_t* bst = b_st + bstage * b_stage + (cc >> 3) * b_group;
                    const int c16 = cc & 7;
                    // this thread's rows of the stage, all loads first, then convert
                    // and store (slab width and stage depth fixed at compile time)
                    auto run = [&](auto nb_c, auto kps_c) {
                        dequant_stage<BF16, decltype(nb_c)::value, decltype(kps_c)::value>(
                            raw, bst, kr0, cc, c16, dq, tab, ztab, valid, p.gran == COC_SCALE_GROUP);
                    };
                    if (nb == 4) {
                        run(IntC<4>{}, IntC<1>{});   // (256-column slabs take one k-block per stage)
                    } else if (nb == 2) {
                        if (kps == 4) run(IntC<2>{}, IntC<4>{});
                        else if (kps == 2) run(IntC<2>{}, IntC<2>{});
                        else run(IntC<2>{}, IntC<1>{});
                    } else {
                        if (kps == 4) run(IntC<1>{}, IntC<4>{});
                        else if (kps == 2) run(IntC<1>{}, IntC<2>{});
                        else run(IntC<1>{}, IntC<1>{});
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bfull[bstage]));
                        mbar_arrive(smem_u32(&empty[stage]));
                    }
                    if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
                    if (++bstage == static_cast<uint32_t>(SB)) { bstage = 0; bphase ^= 1u; }
                }
            }
        }
    }
    if (csplit > 1) {
        // no CTA leaves while a part may still push into its shared memory
        if (warp == 0) cluster_wait();   // the set-up phase this warp only arrived at
        tc_fence_before();
        cluster_sync();
    } else {
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    if (probe) {
        unsigned long long* slot = reinterpret_cast<unsigned long long*>(p.status + STATUS_WORDS) + 2 * p.clock_slot;
        atomicAdd(slot, static_cast<unsigned long long>(clock64() - probe_clk));
        atomicAdd(slot + 1, static_cast<unsigned long long>(globaltimer() - probe_ns));
    }
}

// AllGather ahead of the column-slab kernel: the R shards' m_shard rows of k
// 16-bit values, stacked in rank order into dst (the slab kernel's A: V2's
// first gathered output, or the call's scratch).  One 16-byte vector per
// thread and grid-stride step.  A programmatic launch like the slab kernel:
// it waits for the previous kernel before reading X, and lets the slab kernel
// start its set-up at once (the slab kernel waits for this one to complete
// before its first load).
__global__ void __launch_bounds__(256) coc_ag_gather_kernel(const __grid_constant__ AgGatherParams g) {
    grid_dependency_wait();
    grid_dependents_launch();
    const long long total = g.shard_vecs * g.R;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    uint4* dst = reinterpret_cast<uint4*>(g.dst);
    for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride) {
        const long long sh = v / g.shard_vecs;   // the source rank of this row
        dst[v] = __ldg(reinterpret_cast<const uint4*>(g.src[sh]) + (v - sh * g.shard_vecs));
    }
}

constexpr int kMaxDevices = 64;

template <int OP, bool BF16, bool W8>
cudaError_t launch_slab_t(const KParams& p, int grid, cudaStream_t stream) {
    auto kern = coc_slab_kernel<OP, BF16, W8>;
    static std::atomic<unsigned char> smem_set[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !smem_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlabSmemCap);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) smem_set[dev].store(1, std::memory_order_release);
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(slab_threads(W8), 1, 1);
    cfg.dynamicSmemBytes = slab_smem_bytes(p.slab_stages, p.a_box_rows, p.slab_boxes, p.slab_kps, p.slab_split, W8);
    cfg.stream = stream;
    cfg.attrs = attr;
    if (p.slab_split > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = p.slab_split;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (pdl_launch()) {
        // may start its set-up while the previous kernel in the stream runs
        // (the kernel waits for it before touching global memory)
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int OP, bool BF16, bool W8>
int slab_max_clusters_t(int split, int smem) {
    auto kern = coc_slab_kernel<OP, BF16, W8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlabSmemCap) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(split, 1, 1);
    cfg.blockDim = dim3(slab_threads(W8), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int v = 0;
    if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess) return 0;
    return v;
}

}  // namespace

int slab_stages(int a_rows, int boxes, int kps, int split, bool w8) {
    int s = kSlabMaxStages;
    while (s > 2 && slab_smem_bytes(s, a_rows, boxes, kps, split, w8) > kSlabSmemCap) --s;
    return s;
}

int slab_smem_bytes(int stages, int a_rows, int boxes, int kps, int split, bool w8) {
    const int b_stage = boxes * kps * static_cast<int>(kSlabBoxBytes);   // 16-bit B of a stage
    const int raw_stage = slab_raw_stage(kps, boxes, a_rows);             // w8A16: X, int8 W and its tables
    const int a_stage = kps * a_rows * 128;
    const int rings = w8 ? stages * raw_stage + kSlabW8BStages * b_stage : stages * (a_stage + b_stage);
    const int recv = static_cast<int>(slab_recv_bytes(boxes, split, a_rows));
    const int area = slab_recv_over_rings(split, a_rows) ? (rings > recv ? rings : recv) : rings + recv;
    return 1024 + area + NUM_EPI_WARPS * EPI_BUF_BYTES + static_cast<int>(slab_bar_bytes(stages, w8));
}

cudaError_t launch_slab(int op, bool bf16, bool w8, const KParams& p, int grid, cudaStream_t stream) {
    if (w8) {
        if (op != OP_AR) return cudaErrorInvalidValue;
        return bf16 ? launch_slab_t<OP_AR, true, true>(p, grid, stream) : launch_slab_t<OP_AR, false, true>(p, grid, stream);
    }
    switch (op) {
        case OP_AR:
            return bf16 ? launch_slab_t<OP_AR, true, false>(p, grid, stream)
                        : launch_slab_t<OP_AR, false, false>(p, grid, stream);
        case OP_RS:
            return bf16 ? launch_slab_t<OP_RS, true, false>(p, grid, stream)
                        : launch_slab_t<OP_RS, false, false>(p, grid, stream);
        case OP_AG:
            return bf16 ? launch_slab_t<OP_AG, true, false>(p, grid, stream)
                        : launch_slab_t<OP_AG, false, false>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ag_gather(const AgGatherParams& g, int sm_count, cudaStream_t stream) {
    const long long total = g.shard_vecs * g.R;
    long long blocks = (total + 255) / 256;
    if (blocks > 8LL * sm_count) blocks = 8LL * sm_count;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    if (pdl_launch()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, coc_ag_gather_kernel, g);
}

int slab_max_clusters(bool bf16, bool w8, int split, int smem) {
    // the kernel's resources do not depend on the operator; ask one instance
    if (w8) return bf16 ? slab_max_clusters_t<OP_AR, true, true>(split, smem) : slab_max_clusters_t<OP_AR, false, true>(split, smem);
    return bf16 ? slab_max_clusters_t<OP_AR, true, false>(split, smem) : slab_max_clusters_t<OP_AR, false, false>(split, smem);
}

}  // namespace coc
