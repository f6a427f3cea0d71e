// Persistent fused matmul + collective kernel for GB300 (sm_103a).
//
// One kernel computes every operator of the CoC page's "fused-operator
// implementation" section (MindSpeed developer guide, compute-communication
// parallelism): MATMUL_ALL_REDUCE, MATMUL_REDUCE_SCATTER, ALL_GATHER_MATMUL
// (+V2) and the w8A16 MATMUL_ALL_REDUCE.  With the R tensor-parallel ranks held
// as R shard buffers on one GPU, the collective becomes part of the tile
// pipeline:
//
//   AllReduce      the contraction runs over all R shards into one TMEM
//                  accumulator (rank 0..R-1, k ascending) and the epilogue
//                  stores the rounded tile to all R rank outputs;
//   ReduceScatter  same accumulator, the epilogue routes each 8..32-row block
//                  to the rank that owns those rows;
//   AllGather      the producer routes each A tile from the shard holding its
//                  rows; V2 also copies the gathered rows out, spread over all
//                  work units;
//   w8A16          int8 weight tiles are dequantised in shared memory by
//                  dedicated warps and fed to the fp16 MMA.
//
// CoC chunking (page section 解决思路: split compute and communication into
// smaller sub-tasks and pipeline them) is the work-unit order: units are
// issued chunk by chunk along m, and the double-buffered TMEM accumulator lets
// one tile's epilogue (the "communication") run while the next tile's
// mainloop runs.
//
// At decode-sized m (few output tiles) AllReduce and ReduceScatter cut each
// tile's R shards into groups run as separate units (the rank split); the
// epilogue warp whose group completes a row slab adds the groups' fp32 sums
// in group order and stores the slab.
//
// Warp roles (one CTA per SM, persistent over work units):
//   warp 0      TMA producer: A/B tiles into a STAGES-deep smem ring
//   warp 1      TMEM owner + MMA issuer: tcgen05.mma N=256, K=16, M=128 per CTA
//               (M=256 over a cta_group::2 pair), fp32 accumulators in TMEM
//   warps 2-5   epilogue: tcgen05.ld -> round -> swizzled smem -> TMA store and
//               coalesced 16-byte stores to the other rank outputs
//   warps 6-13  (w8A16 only) int8 -> fp16 dequantisation into the B stage, in
//               two groups of 4 warps taking alternate k-blocks
//
// Every mbarrier wait is bounded (COC_WAIT_NS); a wait that runs out sets a
// CTA-wide abort flag and the device status word, every role leaves its loop,
// in-flight copies and MMAs are drained (again with bounded waits), TMEM is
// freed and the kernel returns.
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "coc_dequant.cuh"
#include "coc_internal.h"
#include "coc_ptx.cuh"

namespace coc {
namespace {

// Grouped GEMM (MoE dispatch): unit -> (expert e, global row tile mt, n-tile
// nt).  Experts in order; inside an expert, its row tiles are taken in L2
// groups of group_mt (the last group may be smaller) and inside a group the
// row tiles of one n-tile column are adjacent, so running CTAs share the
// expert's W tile while the group's token rows stay in L2; odd groups walk
// the columns backwards.  Each expert's group starts on a 256-row boundary of
// its rank's buffer, so a row tile never straddles two experts.  Counts and
// offsets come from the routing kernel.
__device__ __forceinline__ void gmm_decode(const KParams& p, int u, int tile_m, int& e, int& mt, int& nt) {
    int acc = 0;
    e = 0;
    mt = 0;
    nt = 0;
    for (int x = 0; x < p.gmm_E; ++x) {
        const int mte = (__ldg(p.gmm_counts + x) + tile_m - 1) / tile_m;
        const int ue = mte * p.n_tiles;
        if (u < acc + ue) {
            const int v = u - acc;
            const int G = (p.group_mt > 0 && p.group_mt < mte) ? p.group_mt : mte;
            const int g = v / (G * p.n_tiles);
            const int w = v - g * G * p.n_tiles;
            const int Gg = min(G, mte - g * G);   // rows tiles in this group
            int col = w / Gg;
            if (g & 1) col = p.n_tiles - 1 - col;
            e = x;
            nt = col;
            mt = __ldg(p.gmm_offsets + x) / tile_m + g * G + (w - (w / Gg) * Gg);
            return;
        }
        acc += ue;
    }
}
__device__ __forceinline__ int gmm_units(const KParams& p, int tile_m) {
    int acc = 0;
    for (int x = 0; x < p.gmm_E; ++x) acc += (__ldg(p.gmm_counts + x) + tile_m - 1) / tile_m * p.n_tiles;
    return acc;
}

// ALL_GATHER_MATMUL_V2: copy this unit's share of the m-tile's gathered rows
// to every rank's gather buffer.  The tile's rows are one contiguous run of
// the gathered matrix; it is cut into R * n_tiles equal pieces, one per work
// unit of this m-tile (so the copy is spread over the whole kernel), and this
// unit's piece is cut again between the epilogue warps (`wi` of `nw`).  The
// warp copies its part with plain 16-byte loads (lane l takes vectors l,
// l + 32, ...; four per lane in flight) and writes each vector to every
// rank's buffer, each warp access covering 512 contiguous bytes.  Shared
// memory and the bulk-copy engine, which feed the mainloop, are not used.
__device__ __forceinline__ void gather_slice_warp(const KParams& p, int r, int mt, int nt, int tile_m, int wi, int nw,
                                                  int lane) {
    const int rows = min(tile_m, p.m - mt * tile_m);
    const long long vpr = p.k / 8;   // 16-byte vectors per row
    const long long total = rows * vpr;
    const long long Q = static_cast<long long>(p.R) * p.n_tiles;
    const long long qi = static_cast<long long>(r) * p.n_tiles + nt;
    const long long u0 = total * qi / Q, u1 = total * (qi + 1) / Q;
    const long long a = u0 + (u1 - u0) * wi / nw, b = u0 + (u1 - u0) * (wi + 1) / nw;
    const long long gbase = static_cast<long long>(mt) * tile_m * vpr;       // tile's first vector
    const long long shard_vecs = static_cast<long long>(p.rows_per_rank) * vpr;
    for (long long v0 = a; v0 < b; v0 += 32 * 4) {
        uint4 d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long v = v0 + u * 32 + lane;
            d[u] = make_uint4(0u, 0u, 0u, 0u);
            if (v < b) {
                const long long gv = gbase + v;
                const long long sh = gv / shard_vecs;   // the shard holding this row
                d[u] = __ldg(reinterpret_cast<const uint4*>(p.gsrc[sh] + (gv - sh * shard_vecs) * 8));
            }
        }
        for (int dd = 0; dd < p.R; ++dd) {
            uint16_t* dst = p.gdst[dd];
            if (dst == nullptr) continue;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const long long v = v0 + u * 32 + lane;
                if (v < b) *reinterpret_cast<uint4*>(dst + (gbase + v) * 8) = d[u];
            }
        }
    }
}

// Rank split, end of a part: one epilogue warp has written its 32-row slab of
// the part to the scratch.  Count the part; true for the warp whose part
// completes the slab, which then adds the parts and stores the outputs.  No
// warp waits for another: the last to arrive does the work, and the fences
// make every counted part's writes visible to its reads.
__device__ __forceinline__ bool split_last(const KParams& p, int ksplit, int tile_id, uint32_t rank, int q, int lane,
                                           int npair) {
    __threadfence();
    __syncwarp();
    unsigned* cnt = p.part_cnt + (static_cast<long long>(tile_id) * npair + rank) * NUM_EPI_WARPS + q;
    unsigned prev = 0;
    if (lane == 0) prev = atomicAdd(cnt, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const bool last = (prev == static_cast<unsigned>(ksplit - 1));
    if (last) __threadfence();
    return last;
}

// ------------------------------------------------------------ the kernel ---

// Shared-memory rings.  AR/RS/AG: one ring of SA stages holding an A and a B
// tile each (TMA fills both, the MMA frees both).  w8A16: three rings — A
// tiles (TMA -> MMA), raw int8 W tiles (TMA -> dequant warps) and fp16 B
// tiles (dequant warps -> MMA) — so TMA can run SR k-blocks ahead while the
// dequantisation and the MMA work on earlier ones.  With PAIR each CTA holds
// half of the B columns, which halves B and raw stage sizes.
template <int OP, bool PAIR>
struct Cfg {
    static constexpr bool W8 = (OP == OP_W8);
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;        // rows per work unit
    static constexpr int BN_CTA = PAIR ? BN / 2 : BN;        // B columns held by one CTA
    static constexpr int B_BYTES = BN_CTA * BK * 2;          // fp16/bf16 B stage
    static constexpr int RAW_BYTES = BN_CTA * BK;            // int8 W stage
    // w8A16 raw and B rings have an even depth: with XFORM_GROUPS = 2 groups
    // taking alternate k-blocks, each stage then belongs to one group, so a
    // stage's barrier phases are always consumed in order by one waiter.
    static constexpr int SA = W8 ? (PAIR ? 6 : 4) : (PAIR ? 6 : 4);   // A (+B) stages
    static constexpr int SB = W8 ? (PAIR ? 4 : 2) : SA;      // B stages (shared with A except for w8A16)
    static constexpr int SR = W8 ? 4 : 0;                    // raw int8 stages
    static_assert(!W8 || (SB % XFORM_GROUPS == 0 && SR % XFORM_GROUPS == 0), "rings must split between groups");
    static constexpr int WARPS = 2 + NUM_EPI_WARPS + (W8 ? NUM_XFORM_WARPS : 0);
    static constexpr int THREADS = WARPS * 32;
    // Epilogue staging buffers per warp: two (a sub-tile's stores drain while the
    // next is written) except for w8A16, which trades the second for ring depth.
    static constexpr int EPI_NBUF = W8 ? 1 : 2;
    static constexpr int EPI_BYTES = NUM_EPI_WARPS * EPI_NBUF * EPI_BUF_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM = 1024 + SA * A_STAGE_BYTES + (W8 ? SB * B_BYTES : SA * B_BYTES) + SR * RAW_BYTES +
                                EPI_BYTES + BAR_BYTES;
};

template <int OP, bool BF16, bool PAIR>
__global__ void __launch_bounds__(Cfg<OP, PAIR>::THREADS, 1) coc_fused_kernel(const __grid_constant__ KParams p) {
    using C = Cfg<OP, PAIR>;
    constexpr int S = C::SA;
    constexpr bool W8 = C::W8;
    constexpr int TILE_M = C::TILE_M;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint8_t* a_st = smem;                                        // SA x 16 KiB
    uint8_t* b_st = a_st + C::SA * A_STAGE_BYTES;                // (W8 ? SB : SA) x B_BYTES
    uint8_t* raw_st = b_st + (W8 ? C::SB : C::SA) * C::B_BYTES;  // SR x RAW_BYTES (w8A16)
    uint8_t* epi = raw_st + C::SR * C::RAW_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_BYTES);
    uint64_t* full = bars;             // [SA] A (+B) stage landed (the leader's counts both CTAs' bytes)
    uint64_t* empty = full + C::SA;    // [SA] A (+B) stage consumed by the MMA
    uint64_t* bfull = empty + C::SA;   // [SB] w8A16: fp16 B stage written by the dequant warps
    uint64_t* bempty = bfull + C::SB;  // [SB] w8A16: fp16 B stage consumed by the MMA
    uint64_t* rfull = bempty + C::SB;  // [SR] w8A16: raw int8 tile landed
    uint64_t* rempty = rfull + C::SR;  // [SR] w8A16: raw int8 tile read by the dequant warps
    uint64_t* accf = rempty + C::SR;   // [2]  accumulator ready for the epilogue
    uint64_t* acce = accf + 2;         // [2]  accumulator drained by the epilogue (leader: both CTAs)
    uint64_t* never = acce + 2;        // [1]  nothing arrives here (fault-injection test)
    uint64_t* drain = never + 1;       // [1]  MMA drain before TMEM release
    uint64_t* red_ready = drain + 1;   // [1]  rank split in a cluster: every part-CTA pushed its slices here
    uint64_t* ring_free = red_ready + 1;   // [1]  rank split in a cluster: every part-CTA's MMAs are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring_free + 1);
    uint32_t* abort_word = tmem_slot + 1;
    // w8A16 pair: 16-byte landing slots for the peer's per-stage "B half ready" copies
    uint8_t* sig_slots = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(abort_word + 1) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Ctl ctl{abort_word, p.status};
    const uint32_t rank = PAIR ? cluster_rank() : 0u;       // 0 = leader
    const int first_unit = PAIR ? static_cast<int>(cluster_id()) : static_cast<int>(blockIdx.x);
    const int unit_step = PAIR ? static_cast<int>(cluster_count()) : static_cast<int>(gridDim.x);
    constexpr int NPAIR = PAIR ? 2 : 1;

    // the operand maps' descriptors start loading at once, in parallel
    if (warp == 0 && lane < p.num_kshards && lane < COC_MAX_RANKS) {
        prefetch_tmap(&p.tm_a[lane]);
        prefetch_tmap(&p.tm_b[lane]);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::SA; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < C::SB; ++s) {
            mbar_init(smem_u32(&bfull[s]), 1);   // the (leader's) dequant group; the peer's copy adds tx bytes
            mbar_init(smem_u32(&bempty[s]), 1);
        }
        for (int s = 0; s < C::SR; ++s) {
            mbar_init(smem_u32(&rfull[s]), 1);
            mbar_init(smem_u32(&rempty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), NPAIR * NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(never), 1);
        mbar_init(smem_u32(drain), 1);
        // rank split in a cluster: one arrival per part-CTA and epilogue warp
        // holding output rows of this CTA's row tile (one unit per CTA; the
        // cluster's CTAs share the tile)
        int active_warps = NUM_EPI_WARPS;
        if (p.split_cluster && p.ksplit > 1) {
            int r_, mt_, nt_;
            decode_unit<OP>(p, static_cast<int>(blockIdx.x) / p.ksplit, r_, mt_, nt_);
            active_warps = min(NUM_EPI_WARPS, (min(p.m - mt_ * BM, BM) + 31) / 32);
        }
        mbar_init(smem_u32(red_ready), p.split_cluster ? p.ksplit * active_warps : 1);
        mbar_init(smem_u32(ring_free), p.split_cluster ? p.ksplit : 1);
        *abort_word = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        // two 128-lane x 256-column fp32 accumulators = all 512 columns
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), 2 * BN);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), 2 * BN);
            tmem_relinquish();
        }
    }
    // split in a cluster (single-CTA tiles): the cluster's barriers must all
    // exist before any part-CTA arrives remotely
    const bool csplit = !PAIR && (OP == OP_AR || OP == OP_RS) && p.split_cluster && p.ksplit > 1;
    // Single-CTA tiles: the producer warp (whose lane 0 initialised the
    // barriers) needs nothing the others set up, so it only arrives and
    // starts its loads while TMEM is allocated; it waits for the cluster
    // barrier at the end, before the teardown.  CTA pairs: the peer's loads
    // complete on the leader's barriers, so everyone waits.
    constexpr uint32_t kSetupBar = 3;   // named barrier (1 and 2: the dequant groups' votes)
    const bool early_producer = !PAIR && warp == 0;
    tc_fence_before();
    if (early_producer) __syncwarp();   // lane 0's barrier initialisation is visible to the warp
    if (PAIR) {
        cluster_sync();   // both CTAs' barriers exist before any cross-CTA traffic
    } else if (csplit) {
        cluster_arrive();   // the cluster's barriers exist before any part-CTA arrives remotely
        if (!early_producer) cluster_wait();
    } else if (early_producer) {
        named_arrive(kSetupBar, C::THREADS);
    } else {
        named_sync(kSetupBar, C::THREADS);
    }
    tc_fence_after();
    // Everything above touches only this CTA's shared and tensor memory and
    // the kernel parameters, so with a programmatic launch it overlaps the
    // previous kernel in the stream; global memory is touched only after it
    // has completed.  Every CTA of this grid is resident at once, so the next
    // kernel may then start on the SMs this one leaves free.
    grid_dependency_wait();
    grid_dependents_launch();
    const uint32_t tmem_base = early_producer ? 0u : *tmem_slot;
    // clock probe: block 0 measures the SM cycles and nanoseconds it spends
    const bool probe = p.clock_slot >= 0 && blockIdx.x == 0 && threadIdx.x == 0;
    uint64_t probe_clk = 0, probe_ns = 0;
    if (probe) {
        probe_clk = clock64();
        probe_ns = globaltimer();
    }
    const int total_kb = p.num_kshards * p.kblocks;
    // split by rank: a unit is part u % ksplit of tile u / ksplit and sums
    // R / ksplit shards (AllReduce / ReduceScatter only)
    const int ksplit = ((OP == OP_AR || OP == OP_RS) && p.ksplit > 1) ? p.ksplit : 1;
    const int unit_kb = total_kb / ksplit;   // k-blocks one unit accumulates
    // work units: fixed by the host, except for the grouped GEMM whose expert
    // group sizes the routing kernel wrote to device memory
    int n_units = p.units;
    if constexpr (OP == OP_GMM) n_units = gmm_units(p, TILE_M);
    auto decode = [&](int u, int& r, int& mt, int& nt) {
        if constexpr (OP == OP_GMM) gmm_decode(p, u, TILE_M, r, mt, nt);
        else decode_unit<OP>(p, ksplit > 1 ? u / ksplit : u, r, mt, nt);
    };

    if (warp == 0) {
        // ================================================= TMA producer ===
        uint32_t stage = 0, phase = 0, rstage = 0, rphase = 0;
        uint32_t filled = 0, fill_parity = 0;     // per-stage bit masks of the last fill (A ring)
        uint32_t rfilled = 0, rfill_parity = 0;   // same for the raw int8 ring
        // bytes the leader's full barrier receives per stage (both CTAs' loads)
        constexpr uint32_t kFullBytes = NPAIR * (A_STAGE_BYTES + (W8 ? 0 : C::B_BYTES));
        const uint64_t pol_a = make_l2_policy(p.a_hint), pol_b = make_l2_policy(p.b_hint);
        bool ok = true;
        int ks_lo = 0, ks_hi = p.num_kshards;   // the unit's shards (all but with the rank split)
        // One unit's k-loop.  issue_a / issue_b put the unit's A and B boxes of
        // one k-block into a stage; they are chosen once per unit (below), so
        // the loop that runs per k-block has no layout branches: measured,
        // deciding the AllGather A-box layout inside this loop cost ~13% on the
        // LLaMA2-70B AG layer.
        auto unit_loop = [&](int col_base, auto&& issue_a, auto&& issue_b) {
            for (int ks = ks_lo; ok && ks < ks_hi; ++ks) {
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    ok = warp_wait(smem_u32(&empty[stage]), phase ^ 1u, ctl, 0x100u + stage);
                    if (!ok) break;
                    const int kc = kb * BK;
                    if (lane == 0) {
                        const uint32_t fb_local = smem_u32(&full[stage]);
                        const uint32_t fb = PAIR ? map_to_rank(fb_local, 0) : fb_local;
                        if (rank == 0) mbar_expect_tx(fb_local, kFullBytes);
                        auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, uint64_t pol) {
                            if constexpr (PAIR) tma_load_2d_pair(dst, map, c0, c1, fb, pol);
                            else tma_load_2d_hint(dst, map, c0, c1, fb, pol);
                        };
                        issue_a(load, smem_u32(a_st + stage * A_STAGE_BYTES), ks, kc);
                        if constexpr (!W8) issue_b(load, smem_u32(b_st + stage * C::B_BYTES), ks, kc);
                        filled |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    }
                    __syncwarp();
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                    if constexpr (W8) {
                        // this CTA's raw int8 W columns into its own ring
                        ok = warp_wait(smem_u32(&rempty[rstage]), rphase ^ 1u, ctl, 0x140u + rstage);
                        if (!ok) break;
                        if (lane == 0) {
                            const uint32_t rb = smem_u32(&rfull[rstage]);
                            mbar_expect_tx(rb, C::RAW_BYTES);
                            tma_load_2d_hint(smem_u32(raw_st + rstage * C::RAW_BYTES), &p.tm_b[ks], col_base, kc, rb,
                                             pol_b);
                            rfilled |= 1u << rstage;
                            rfill_parity = (rfill_parity & ~(1u << rstage)) | (rphase << rstage);
                        }
                        __syncwarp();
                        if (++rstage == C::SR) { rstage = 0; rphase ^= 1u; }
                    }
                }
            }
        };
        for (int u = first_unit; ok && u < n_units; u += unit_step) {
            int r, mt, nt;
            decode(u, r, mt, nt);
            if (ksplit > 1) {
                const int per = p.num_kshards / ksplit;
                ks_lo = (u % ksplit) * per;
                ks_hi = ks_lo + per;
            }
            const int row_base = mt * TILE_M + static_cast<int>(rank) * BM;   // this CTA's first A row
            const int col_base = nt * BN + static_cast<int>(rank) * C::BN_CTA;  // this CTA's first B column
            // A: one 128-row box (AllGather: from the shard holding the rows,
            // which then hold the whole tile; rows past the end read beyond the
            // last shard and are zero-filled), ...
            int a_shard = 0, a_row = row_base;
            if constexpr (OP == OP_AG) {
                a_shard = min(row_base / p.rows_per_rank, p.R - 1);
                a_row = row_base - a_shard * p.rows_per_rank;
            }
            // (the unit's map is resolved here: kernel parameters are re-read after
            // every asm with a memory clobber, so nothing is hoisted out of the loop)
            const CUtensorMap* amap_unit = (OP == OP_AG)    ? &p.tm_a[a_shard]
                                           : (OP == OP_GMM) ? &p.tm_a[r / p.gmm_eloc]
                                                            : &p.tm_a[0];
            auto a_single = [&](auto& load, uint32_t dst, int ks, int kc) {
                load(dst, (OP == OP_AG || OP == OP_GMM) ? amap_unit : &p.tm_a[ks], kc, a_row, pol_a);
            };
            // ... several boxes when a shard holds fewer rows than a tile, ...
            auto a_multi = [&](auto& load, uint32_t dst, int, int kc) {
                for (int rb = 0; rb < BM; rb += p.a_box_rows) {
                    const int g = row_base + rb;
                    int sh = g / p.rows_per_rank;
                    if (sh > p.R - 1) sh = p.R - 1;
                    load(dst + rb * 128, &p.tm_a[sh], kc, g - sh * p.rows_per_rank, pol_a);
                }
            };
            // ... or, for the weight gradient, A = dY_r^T read from rank r's dY
            // (tokens x rows) as two 64-row blocks of 64 tokens (MN-major, like B).
            auto a_mn = [&](auto& load, uint32_t dst, int, int kc) {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j) load(dst + j * (64 * BK * 2), &p.tm_a[r], row_base + j * 64, kc, pol_a);
            };
            // B: W stored k x n, read as 64-column MN-major boxes, or W stored
            // n x k, one box of this CTA's B rows (n) x 64 k laid out like A.
            // (grouped GEMM: one map over the stacked expert weights, expert r's
            // rows starting at r * k)
            const CUtensorMap* bmaps = &p.tm_b[(OP == OP_AG) ? r : 0];
            const int b_k0 = (OP == OP_GMM) ? r * p.k : 0;
            auto b_mn = [&](auto& load, uint32_t dst, int ks, int kc) {
                const CUtensorMap* bm = (OP == OP_AG || OP == OP_GMM) ? bmaps : &p.tm_b[ks];
#pragma unroll
                for (int j = 0; j < C::BN_CTA / 64; ++j)
                    load(dst + j * (64 * BK * 2), bm, col_base + j * 64, b_k0 + kc, pol_b);
            };
            auto b_kmaj = [&](auto& load, uint32_t dst, int ks, int kc) {
                load(dst, (OP == OP_AG) ? bmaps : &p.tm_b[ks], kc, col_base, pol_b);
            };
            auto with_b = [&](auto&& issue_a) {
                if constexpr (W8) unit_loop(col_base, issue_a, b_mn);   // B comes from the dequant warps
                else if (OP != OP_GMM && p.b_kmajor) unit_loop(col_base, issue_a, b_kmaj);
                else unit_loop(col_base, issue_a, b_mn);
            };
            if constexpr (OP == OP_AG) {
                if (p.a_mnmajor) with_b(a_mn);
                else if (p.a_box_rows == BM) with_b(a_single);
                else with_b(a_multi);
            } else {
                with_b(a_single);
            }
        }
        if (!ok && lane == 0) {
            // leave no TMA load in flight into shared memory
            if (rank == 0) {
                for (int s = 0; s < C::SA; ++s)
                    if (filled & (1u << s)) drain_wait(smem_u32(&full[s]), (fill_parity >> s) & 1u, kDrainNs);
            } else {
                // the peer's loads complete on the leader's barriers: give them time
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {
                }
            }
            for (int s = 0; s < C::SR; ++s)
                if (rfilled & (1u << s)) drain_wait(smem_u32(&rfull[s]), (rfill_parity >> s) & 1u, kDrainNs);
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer ===
        // (with PAIR only the leader issues; the peer's warp 1 just owns its TMEM)
        if (rank == 0) {
            // B K-major (W stored n x k) clears the "B transposed" bit; an MN-major A
            // (the weight-gradient pass) sets the "A transposed" bit
            const uint32_t idesc =
                (make_idesc(BF16, TILE_M, BN) & (p.b_kmajor ? ~(1u << 16) : ~0u)) | (p.a_mnmajor ? (1u << 15) : 0u);
            const uint32_t a_lbo = p.a_mnmajor ? 64u * BK * 2u : 16u;
            const uint64_t a_step = p.a_mnmajor ? 128u : 2u;
            const uint32_t b_lbo = p.b_kmajor ? 16u : 64u * BK * 2u;
            const uint64_t b_step = p.b_kmajor ? 2u : 128u;   // 16-element k step, in 16-byte units
            uint32_t stage = 0, phase = 0, bstage = 0, bphase = 0;
            int acc_i = 0;
            bool ok = true;
            for (int u = first_unit; ok && u < n_units; u += unit_step) {
                const int buf = acc_i & 1;
                const uint32_t aph = (acc_i >> 1) & 1;
                ok = warp_wait<PAIR>(smem_u32(&acce[buf]), aph ^ 1u, ctl, 0x200u + buf);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int i = 0; i < unit_kb; ++i) {
                    ok = warp_wait<PAIR>(smem_u32(&full[stage]), phase, ctl, 0x210u + stage);
                    if (W8 && ok) ok = warp_wait<PAIR>(smem_u32(&bfull[bstage]), bphase, ctl, 0x220u + bstage);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t ad = make_sdesc(smem_u32(a_st + stage * A_STAGE_BYTES), a_lbo, 1024);
                        const uint64_t bd = make_sdesc(smem_u32(b_st + (W8 ? bstage : stage) * C::B_BYTES), b_lbo, 1024);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            // K-major operand: +32 bytes per 16-element k step inside the
                            // 128-byte swizzle row; MN-major operand: +2 eight-row groups (2 KiB)
                            const uint64_t a_k = ad + static_cast<uint64_t>(kk) * a_step;
                            const uint64_t b_k = bd + static_cast<uint64_t>(kk) * b_step;
                            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                            if constexpr (PAIR) tc_mma_f16_pair(d_tmem, a_k, b_k, idesc, acc);
                            else tc_mma_f16(d_tmem, a_k, b_k, idesc, acc);
                        }
                        if constexpr (PAIR) {
                            tc_commit_pair_both(smem_u32(&empty[stage]));
                            if (W8) tc_commit_pair_both(smem_u32(&bempty[bstage]));
                        } else {
                            tc_commit(smem_u32(&empty[stage]));
                            if (W8) tc_commit(smem_u32(&bempty[bstage]));
                        }
                    }
                    __syncwarp();
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                    if (W8 && ++bstage == C::SB) { bstage = 0; bphase ^= 1u; }
                }
                if (!ok) break;
                if (lane == 0) {
                    if constexpr (PAIR) tc_commit_pair_both(smem_u32(&accf[buf]));
                    else tc_commit(smem_u32(&accf[buf]));
                }
                __syncwarp();
                ++acc_i;
            }
            // every issued MMA must finish before TMEM is released
            if (lane == 0) {
                if constexpr (PAIR) tc_commit_pair_local(smem_u32(drain));
                else tc_commit(smem_u32(drain));
                drain_wait(smem_u32(drain), 0, kDrainNs);
            }
            __syncwarp();
        }
    } else if (warp < 2 + NUM_EPI_WARPS) {
        // ================================================= epilogue ===
        const int q = warp & 3;                 // TMEM lane quadrant this warp may read
        uint8_t* my_epi = epi + (warp - 2) * C::EPI_NBUF * EPI_BUF_BYTES;
        const uint32_t acce_base = PAIR ? map_to_rank(smem_u32(acce), 0) : smem_u32(acce);
        int acc_i = 0, sb_i = 0;
        bool ok = true;
        if (p.inject_timeout) ok = warp_wait(smem_u32(never), 0, ctl, 0x300u);
        for (int u = first_unit; ok && u < n_units; u += unit_step) {
            int r, mt, nt;
            decode(u, r, mt, nt);
            const int buf = acc_i & 1;
            const uint32_t aph = (acc_i >> 1) & 1;
            ok = warp_wait<PAIR>(smem_u32(&accf[buf]), aph, ctl, 0x310u + buf);
            if (!ok) break;
            tc_fence_after();
            const int row0 = mt * TILE_M + static_cast<int>(rank) * BM + 32 * q;
            if (csplit) {
                // this CTA's MMAs are done, so its operand ring is idle: tell every
                // part-CTA of the cluster, and push only once all rings are idle
                if (q == 0 && lane == 0)
                    for (int j = 0; j < ksplit; ++j) mbar_arrive_cluster(map_to_rank(smem_u32(ring_free), j));
                if (row0 < p.m) {
                    ok = warp_wait<true>(smem_u32(ring_free), 0, ctl, 0x320u);
                    if (!ok) break;
                }
            }
            const int tile_id = mt * p.n_tiles + nt;
            const int part_s = (ksplit > 1) ? u % ksplit : 0;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * BN;
            // this warp's 32-row slab of part sp of the tile (rank split scratch)
            auto part_slab = [&](int sp) {
                return p.part + (((static_cast<long long>(tile_id) * ksplit + sp) * NPAIR + rank) * NUM_EPI_WARPS + q) *
                                    (32LL * BN);
            };
            // Round one 32-row x 64-column sub-tile (fp32 bits, lane = row) and
            // store it: staged once in swizzled shared memory, then the
            // operator's stores.
            auto emit = [&](int sub, const uint32_t (&va)[32], const uint32_t (&vb)[32]) {
                const int col = nt * BN + sub * EPI_COLS;
                uint8_t* sbuf = my_epi + (sb_i % C::EPI_NBUF) * EPI_BUF_BYTES;
                ++sb_i;
                // the stores that last read this buffer are done
                if (lane == 0) {
                    if constexpr (C::EPI_NBUF == 2) bulk_wait_read<1>();
                    else bulk_wait_read<0>();
                }
                __syncwarp();
                uint8_t* rowp = sbuf + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t* v = (j < 4) ? (va + 8 * j) : (vb + 8 * (j - 4));
                    uint4 w4;
                    w4.x = pack2<BF16>(v[0], v[1]);
                    w4.y = pack2<BF16>(v[2], v[3]);
                    w4.z = pack2<BF16>(v[4], v[5]);
                    w4.w = pack2<BF16>(v[6], v[7]);
                    *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) = w4;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t src = smem_u32(sbuf);
                    if constexpr (OP == OP_RS) {
                        for (int rb = 0; rb < 32; rb += p.store_rows) {
                            const int g = row0 + rb;
                            if (g >= p.m) break;
                            const int dst = g / p.rows_per_rank;
                            tma_store_2d(&p.tm_out[dst], src + rb * 128, col, g - dst * p.rows_per_rank);
                        }
                    } else if constexpr (OP == OP_AG) {
                        tma_store_2d(&p.tm_out[r], src, col, row0);
                    } else if constexpr (OP == OP_GMM) {
                        if (p.gmm_srcmap == nullptr) tma_store_2d(&p.tm_out[r / p.gmm_eloc], src, col, row0);
                    } else {
                        if (!p.replica_stores)
                            for (int o = 0; o < p.n_out; ++o) tma_store_2d(&p.tm_out[o], src, col, row0);
                    }
                    bulk_commit();
                }
                if constexpr (OP == OP_GMM) {
                    if (p.gmm_srcmap != nullptr) {
                        // MoE combine (the all-to-all back): each row of the sub-tile goes
                        // to its token's row on the source rank.  Coalesced read-back as
                        // for the AllReduce copies (lane l: chunk l % 8 of rows l / 8 + 4i).
                        const int ch = lane & 7;
                        const int c = col + ch * 8;
                        const int32_t* smap = p.gmm_srcmap + static_cast<long long>(r / p.gmm_eloc) * p.rows_per_rank;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = (lane >> 3) + 4 * i;
                            const uint4 v = *reinterpret_cast<const uint4*>(sbuf + rr * 128 + ((ch ^ (rr & 7)) << 4));
                            const int g = row0 + rr;
                            const int tok = (g < p.m) ? __ldg(smap + g) : -1;
                            if (tok >= 0 && c < p.n) {
                                const int sr = tok / p.gmm_T;
                                *reinterpret_cast<uint4*>(p.outp[sr] + static_cast<long long>(tok - sr * p.gmm_T) * p.n + c) = v;
                            }
                        }
                    }
                }
                if constexpr (OP == OP_AR || OP == OP_W8) {
                    if (p.replica_stores) {
                        // The R copies of this AllReduce sub-tile: read it back once in
                        // coalesced order (lane l: 16-byte chunk l % 8 of rows l / 8 + 4i)
                        // and write it to every rank's output with plain global stores,
                        // each warp store covering four whole 128-byte row segments.  This
                        // keeps the R-fold output off the TMA unit that feeds the mainloop
                        // (measured: R TMA stores of each staged sub-tile cost more).
                        const int ch = lane & 7;
                        uint4 v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = (lane >> 3) + 4 * i;
                            v[i] = *reinterpret_cast<const uint4*>(sbuf + rr * 128 + ((ch ^ (rr & 7)) << 4));
                        }
                        const int c = col + ch * 8;   // n % 8 == 0: a chunk is wholly inside or outside
                        if (c < p.n) {
                            for (int o = 0; o < p.n_out; ++o) {
                                uint16_t* base = p.outp[o] + c;
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int g = row0 + (lane >> 3) + 4 * i;
                                    if (g < p.m) *reinterpret_cast<uint4*>(base + static_cast<long long>(g) * p.n) = v[i];
                                }
                            }
                        }
                    }
                }
            };
            for (int sub = 0; sub < BN / EPI_COLS; ++sub) {
                uint32_t va[32], vb[32];
                if (unit_kb > 0) {
                    tmem_ld_32cols(t_row + sub * EPI_COLS, va);
                    tmem_ld_32cols(t_row + sub * EPI_COLS + 32, vb);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) { va[i] = 0u; vb[i] = 0u; }
                }
                if (sub == BN / EPI_COLS - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t ab = acce_base + buf * static_cast<uint32_t>(sizeof(uint64_t));
                        if constexpr (PAIR) mbar_arrive_cluster(ab);
                        else mbar_arrive(ab);
                    }
                }
                if (csplit) {
                    // rank split in a cluster: the sub-tile's 64 columns belong to part-CTA
                    // `owner`; push this part's fp32 sums straight into the owner's
                    // reception area (its operand ring, idle once ring_free completed):
                    // slot [part][q][row = lane] of (BN / ksplit) columns, 16-byte chunk
                    // c of a row at chunk c ^ (row & 7)
                    if (row0 < p.m) {
                        const int nsub = (BN / EPI_COLS) / ksplit;
                        const uint32_t owner = static_cast<uint32_t>(sub / nsub);
                        const uint32_t row_bytes = static_cast<uint32_t>(BN * 4 / ksplit);
                        const uint32_t rb = smem_u32(a_st) +
                                            ((static_cast<uint32_t>(part_s) * NUM_EPI_WARPS + q) * 32 + lane) * row_bytes;
                        const uint32_t rb_owner = map_to_rank(rb, owner);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint32_t* v = (j < 8) ? (va + 4 * j) : (vb + 4 * (j - 8));
                            const uint32_t cidx = static_cast<uint32_t>((sub % nsub) * 16 + j);
                            asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};"
                                         ::"r"(rb_owner + ((cidx ^ (lane & 7)) << 4)),
                                         "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                                         : "memory");
                        }
                    }
                    continue;
                }
                if (row0 >= p.m || nt * BN + sub * EPI_COLS >= p.n) continue;   // sub-tile outside the output
                if (ksplit > 1) {
                    // rank split: this part's fp32 sums into the slab's scratch, laid
                    // out so that a warp access is 512 contiguous bytes
                    float* dst = part_slab(part_s) + static_cast<long long>(sub) * (16 * 32 * 4) + lane * 4;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t* v = (j < 8) ? (va + 4 * j) : (vb + 4 * (j - 8));
                        *reinterpret_cast<uint4*>(dst + j * (32 * 4)) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                    continue;
                }
                emit(sub, va, vb);
                __syncwarp();
            }
            if (csplit && row0 < p.m) {
                // every part of this warp's rows is in this CTA's ring once each
                // part-CTA's active warps pushed their slices and arrived here
                __syncwarp();
                if (lane == 0)
                    for (int j = 0; j < ksplit; ++j) mbar_arrive_cluster(map_to_rank(smem_u32(red_ready), j));
                ok = warp_wait<true>(smem_u32(red_ready), 0, ctl, 0x330u);
                if (!ok) break;
                // this CTA (part `me`) adds, for its columns, the ksplit parts in part
                // order (part 0 taken as is), from its own shared memory
                const uint32_t me = cluster_rank();
                const int nsub = (BN / EPI_COLS) / ksplit;
                const uint32_t row_bytes = static_cast<uint32_t>(BN * 4 / ksplit);
                for (int s = 0; s < nsub; ++s) {
                    const int sub = static_cast<int>(me) * nsub + s;
                    if (nt * BN + sub * EPI_COLS >= p.n) break;
                    uint32_t va[32], vb[32];
                    for (int sp = 0; sp < ksplit; ++sp) {
                        // part sp's 64 columns of this row, pushed into this CTA's ring
                        const uint32_t rb = smem_u32(a_st) +
                                            ((static_cast<uint32_t>(sp) * NUM_EPI_WARPS + q) * 32 + lane) * row_bytes;
                        uint4 v[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint32_t cidx = static_cast<uint32_t>(s * 16 + j);
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(v[j].x), "=r"(v[j].y), "=r"(v[j].z), "=r"(v[j].w)
                                         : "r"(rb + ((cidx ^ (lane & 7)) << 4))
                                         : "memory");
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            uint32_t* d = (j < 8) ? (va + 4 * j) : (vb + 4 * (j - 8));
                            if (sp == 0) {
                                d[0] = v[j].x; d[1] = v[j].y; d[2] = v[j].z; d[3] = v[j].w;
                            } else {
                                d[0] = __float_as_uint(__uint_as_float(d[0]) + __uint_as_float(v[j].x));
                                d[1] = __float_as_uint(__uint_as_float(d[1]) + __uint_as_float(v[j].y));
                                d[2] = __float_as_uint(__uint_as_float(d[2]) + __uint_as_float(v[j].z));
                                d[3] = __float_as_uint(__uint_as_float(d[3]) + __uint_as_float(v[j].w));
                            }
                        }
                    }
                    emit(sub, va, vb);
                    __syncwarp();
                }
            }
            if (!csplit && ksplit > 1 && row0 < p.m && split_last(p, ksplit, tile_id, rank, q, lane, NPAIR)) {
                // the last part of this slab to arrive: add the parts in part order
                // (part 0 taken as is), then round and store as an unsplit tile
                for (int sub = 0; sub < BN / EPI_COLS; ++sub) {
                    if (nt * BN + sub * EPI_COLS >= p.n) break;
                    uint32_t va[32], vb[32];
                    const float* src = part_slab(0) + static_cast<long long>(sub) * (16 * 32 * 4) + lane * 4;
                    const long long pstride = 32LL * BN * NUM_EPI_WARPS * NPAIR;   // between parts
                    for (int sp = 0; sp < ksplit; ++sp, src += pstride) {
                        float4 v[16];   // one part's 64 columns: all loads in flight together
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __ldcg(reinterpret_cast<const float4*>(src + j * (32 * 4)));
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            uint32_t* d = (j < 8) ? (va + 4 * j) : (vb + 4 * (j - 8));
                            if (sp == 0) {
                                d[0] = __float_as_uint(v[j].x); d[1] = __float_as_uint(v[j].y);
                                d[2] = __float_as_uint(v[j].z); d[3] = __float_as_uint(v[j].w);
                            } else {
                                d[0] = __float_as_uint(__uint_as_float(d[0]) + v[j].x);
                                d[1] = __float_as_uint(__uint_as_float(d[1]) + v[j].y);
                                d[2] = __float_as_uint(__uint_as_float(d[2]) + v[j].z);
                                d[3] = __float_as_uint(__uint_as_float(d[3]) + v[j].w);
                            }
                        }
                    }
                    emit(sub, va, vb);
                    __syncwarp();
                }
            }
            ++acc_i;
            if constexpr (OP == OP_AG) {
                if (p.has_gather)
                    gather_slice_warp(p, r, mt, nt, TILE_M, static_cast<int>(rank) * NUM_EPI_WARPS + (warp - 2),
                                      NPAIR * NUM_EPI_WARPS, lane);
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if constexpr (W8) {
        // ================================================= w8A16 dequant ===
        // Two groups of dequant warps take alternate k-blocks, so two
        // k-blocks are in conversion at once.  In a group, thread tt owns 8
        // consecutive columns (cc) of this CTA's B columns and the k-block
        // rows kr0, kr0 + R_STEP, ...
        constexpr int GT = XFORM_GROUP_WARPS * 32;                  // threads per group
        constexpr int CHUNKS = C::BN_CTA / 8;                       // 8-column chunks per row
        constexpr int R_STEP = GT / CHUNKS;                         // rows covered per pass
        constexpr int ROWS = BK / R_STEP;
        const int xw = warp - 2 - NUM_EPI_WARPS;                     // 0 .. NUM_XFORM_WARPS-1
        const int group = xw / XFORM_GROUP_WARPS;
        const int tt = (xw % XFORM_GROUP_WARPS) * 32 + lane;
        const int cc = tt % CHUNKS;
        const int kr0 = tt / CHUNKS;
        const int blk = cc >> 3, c16 = cc & 7;
        const uint32_t bfull_base = PAIR ? map_to_rank(smem_u32(bfull), 0) : smem_u32(bfull);
        const W8Layout w8l{p.gran, p.group, p.n};
        uint32_t cnt = 0;   // global k-block counter (all units, ranks, k-blocks in order)
        bool ok = true;
        for (int u = first_unit; ok && u < n_units; u += unit_step) {
            int r, mt, nt;
            decode(u, r, mt, nt);
            const int j0 = nt * BN + static_cast<int>(rank) * C::BN_CTA + cc * 8;   // first global column
            for (int ks = 0; ok && ks < p.num_kshards; ++ks) {
                const uint16_t* sc = p.scale[ks];
                const int8_t* zp = p.has_zero ? p.zero[ks] : nullptr;
                // per-tensor / per-channel constants do not depend on the k-block:
                // load them once per rank; per-group ones per k-block below
                Dq<BF16> dq;
                if (p.gran != COC_SCALE_GROUP) dq.load(w8l, sc, zp, 0, j0);
                for (int kb = 0; kb < p.kblocks; ++kb, ++cnt) {
                    if (static_cast<int>(cnt % XFORM_GROUPS) != group) continue;
                    const uint32_t rstage = cnt % C::SR, rphase = (cnt / C::SR) & 1u;
                    const uint32_t bstage = cnt % C::SB, bphase = (cnt / C::SB) & 1u;
                    if (p.gran == COC_SCALE_GROUP) dq.load(w8l, sc, zp, kb * BK, j0);
                    bool ok_k = warp_wait(smem_u32(&rfull[rstage]), rphase, ctl, 0x400u + rstage);
                    if (ok_k) ok_k = warp_wait<PAIR>(smem_u32(&bempty[bstage]), bphase ^ 1u, ctl, 0x410u + bstage);
                    if (ok_k) {
                        const uint8_t* raw = raw_st + rstage * C::RAW_BYTES;
                        uint8_t* bst = b_st + bstage * C::B_BYTES + blk * (64 * BK * 2);
                        // all loads first, then convert and store (independent work per row)
                        uint2 q8[ROWS];
#pragma unroll
                        for (int i = 0; i < ROWS; ++i)
                            q8[i] = *reinterpret_cast<const uint2*>(raw + (kr0 + R_STEP * i) * C::BN_CTA + cc * 8);
#pragma unroll
                        for (int i = 0; i < ROWS; ++i) {
                            const int kk = kr0 + R_STEP * i;
                            const uint4 o = dq.convert(q8[i]);
                            // MN-major 128-byte-swizzled B layout: 64-column blocks of
                            // 64 rows x 128 bytes, 16-byte chunks XOR-ed with row % 8
                            *reinterpret_cast<uint4*>(bst + kk * 128 + ((c16 ^ (kk & 7)) << 4)) = o;
                        }
                        fence_proxy_async_smem();
                    }
                    // The group's warps agree (barrier with OR-reduction) on whether every
                    // warp converted this stage; on any failure they all leave together,
                    // so no warp is left waiting at a named barrier.
                    const uint32_t fail = (!ok_k || *reinterpret_cast<volatile uint32_t*>(abort_word) != 0u) ? 1u : 0u;
                    uint32_t any_fail;
                    asm volatile(
                        "{\n\t.reg .pred pf, pa;\n\t"
                        "setp.ne.u32 pf, %1, 0;\n\t"
                        "bar.red.or.pred pa, %2, %3, pf;\n\t"
                        "selp.u32 %0, 1, 0, pa;\n\t}"
                        : "=r"(any_fail)
                        : "r"(fail), "r"(1 + group), "n"(GT)
                        : "memory");
                    if (any_fail) { ok = false; break; }
                    if (tt == 0) {
                        mbar_arrive(smem_u32(&rempty[rstage]));
                        const uint32_t bf = bfull_base + bstage * static_cast<uint32_t>(sizeof(uint64_t));
                        if constexpr (PAIR) {
                            if (rank == 0) {
                                mbar_expect_tx(smem_u32(&bfull[bstage]), 16);   // arrive + the peer's 16 bytes
                            } else {
                                // async-proxy signal: ordered after this group's fenced B writes
                                const uint32_t slot = map_to_rank(smem_u32(sig_slots + 16 * bstage), 0);
                                bulk_copy_s2s_signal(slot, smem_u32(b_st + bstage * C::B_BYTES), 16, bf);
                            }
                        } else {
                            mbar_arrive(bf);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    if constexpr (PAIR) {
        // After an abort the peer may still have loads or signal copies in
        // flight toward the leader's shared memory: give them time to land
        // before either CTA can exit.
        if (*reinterpret_cast<volatile uint32_t*>(abort_word) != 0u) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 200000ull) {
            }
        }
        cluster_sync();   // the leader's MMAs (which write both TMEMs) and all cross-CTA traffic are done
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc_pair(tmem_base, 2 * BN);
        }
    } else {
        // split in a cluster: no CTA may leave while the others read its shared memory
        if (csplit) {
            if (early_producer) cluster_wait();   // the setup phase this warp only arrived at
            cluster_sync();
        } else {
            __syncthreads();
        }
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, 2 * BN);
        }
    }
    if (probe) {
        unsigned long long* slot =
            reinterpret_cast<unsigned long long*>(p.status + STATUS_WORDS) + 2 * p.clock_slot;
        atomicAdd(slot, static_cast<unsigned long long>(clock64() - probe_clk));
        atomicAdd(slot + 1, static_cast<unsigned long long>(globaltimer() - probe_ns));
    }
}

// The dynamic shared-memory limit of a kernel instance is raised once per
// device (first launch there), not on every call: the call path then makes
// only capture-safe API calls, so the operators can be recorded into CUDA
// graphs after one eager call on the device.
constexpr int kMaxDevices = 64;

template <int OP, bool BF16, bool PAIR>
cudaError_t launch_t(const KParams& p, int grid, cudaStream_t stream, int cluster = 1) {
    using C = Cfg<OP, PAIR>;
    auto kern = coc_fused_kernel<OP, BF16, PAIR>;
    static std::atomic<unsigned char> smem_set[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !smem_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) smem_set[dev].store(1, std::memory_order_release);
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (PAIR || cluster > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = PAIR ? 2 : cluster;
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

template <int OP, bool BF16>
int max_split_clusters_t(int cluster) {
    using C = Cfg<OP, false>;
    auto kern = coc_fused_kernel<OP, BF16, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

template <int OP, bool BF16>
int max_pairs_t() {
    using C = Cfg<OP, true>;
    auto kern = coc_fused_kernel<OP, BF16, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace

cudaError_t launch(int op, bool bf16, bool pair, const KParams& p, int grid, cudaStream_t stream) {
#define COC_LAUNCH(OPV, B16)                                                                       \
    return pair ? launch_t<OPV, B16, true>(p, grid, stream) : launch_t<OPV, B16, false>(p, grid, stream)
    switch (op) {
        case OP_AR: if (bf16) { COC_LAUNCH(OP_AR, true); } else { COC_LAUNCH(OP_AR, false); }
        case OP_RS: if (bf16) { COC_LAUNCH(OP_RS, true); } else { COC_LAUNCH(OP_RS, false); }
        case OP_AG: if (bf16) { COC_LAUNCH(OP_AG, true); } else { COC_LAUNCH(OP_AG, false); }
        case OP_W8: if (bf16) { COC_LAUNCH(OP_W8, true); } else { COC_LAUNCH(OP_W8, false); }
        case OP_GMM: if (bf16) { COC_LAUNCH(OP_GMM, true); } else { COC_LAUNCH(OP_GMM, false); }
        default: return cudaErrorInvalidValue;
    }
#undef COC_LAUNCH
}

cudaError_t launch_split(int op, bool bf16, const KParams& p, int grid, int cluster, cudaStream_t stream) {
    switch (op) {
        case OP_AR: return bf16 ? launch_t<OP_AR, true, false>(p, grid, stream, cluster)
                                : launch_t<OP_AR, false, false>(p, grid, stream, cluster);
        case OP_RS: return bf16 ? launch_t<OP_RS, true, false>(p, grid, stream, cluster)
                                : launch_t<OP_RS, false, false>(p, grid, stream, cluster);
        default: return cudaErrorInvalidValue;
    }
}

int max_split_clusters(int op, bool bf16, int cluster) {
    switch (op) {
        case OP_AR: return bf16 ? max_split_clusters_t<OP_AR, true>(cluster) : max_split_clusters_t<OP_AR, false>(cluster);
        case OP_RS: return bf16 ? max_split_clusters_t<OP_RS, true>(cluster) : max_split_clusters_t<OP_RS, false>(cluster);
        default: return 0;
    }
}

int max_pairs(int op, bool bf16) {
    switch (op) {
        case OP_AR: return bf16 ? max_pairs_t<OP_AR, true>() : max_pairs_t<OP_AR, false>();
        case OP_RS: return bf16 ? max_pairs_t<OP_RS, true>() : max_pairs_t<OP_RS, false>();
        case OP_AG: return bf16 ? max_pairs_t<OP_AG, true>() : max_pairs_t<OP_AG, false>();
        case OP_W8: return bf16 ? max_pairs_t<OP_W8, true>() : max_pairs_t<OP_W8, false>();
        case OP_GMM: return bf16 ? max_pairs_t<OP_GMM, true>() : max_pairs_t<OP_GMM, false>();
        default: return 0;
    }
}

static_assert(Cfg<OP_AR, false>::SMEM <= 232448 && Cfg<OP_W8, false>::SMEM <= 232448 &&
                  Cfg<OP_AR, true>::SMEM <= 232448 && Cfg<OP_W8, true>::SMEM <= 232448,
              "shared memory above 227 KiB");

}  // namespace coc
