// w8A16 MATMUL_ALL_REDUCE in one launch, the dequantised weight held in
// tensor memory (CoC page, 融合算子实现, last bullet: the pseudo-quantised
// fp16 MATMUL_ALL_REDUCE with per-tensor, per-channel and per-group scales).
//
// The contraction is taken transposed, Y^T = Wd^T X^T, so that the weight is
// the MMA's A operand, which tcgen05.mma can read from tensor memory: the
// int8 tile goes TMA -> shared memory -> registers (one transposing
// ldmatrix per 16 x 16 block) -> dequantisation in registers ->
// tcgen05.st into a TMEM ring, and the 16-bit weight never touches shared
// memory.  X is the B operand, TMA-loaded K-major as in the other kernels.
//
// CTA pairs (a cluster of two CTAs on neighbouring SMs, tcgen05 cta_group::2),
// persistent.  A work unit is 256 weight columns (the MMA's M: 128 per CTA,
// its TMEM lanes) by NR activation rows (its N, NR = 32 .. 256 chosen from
// m: NR / 2 rows of X in each CTA's shared memory), summed over all R shards
// (rank 0..R-1, k ascending) into one fp32 accumulator per CTA, rounded once
// and written to all R rank outputs.  The even CTA ("leader") issues the
// MMAs for both; the peer's X loads complete on the leader's barrier, the
// peer's dequant warps report their TMEM stages to the leader's barrier, and
// the leader's commits release both CTAs' stages.
//
// Warp roles (each CTA):
//   warp 0       TMA producer of X (this CTA's NR / 2 rows per k-block)
//   warp 1       TMEM owner; in the leader, the MMA issuer (A from TMEM)
//   warps 2-5    epilogue: each drains its 32-lane quadrant of the
//                accumulator (32 weight columns x NR rows) into its own
//                staging area, transposed to row-major, releases the
//                accumulator, then writes the R output copies
//   warps 6-13   dequantisation, two groups of four (one warp per TMEM lane
//                quadrant) taking alternate k-blocks
//   warp 14      TMA producer of the raw int8 weight (this CTA's 128
//                columns), running ahead of X on its own ring
//
// Every mbarrier wait is bounded (COC_WAIT_NS); a wait that runs out sets the
// CTA abort flag and the device status word, every role leaves its loop,
// issued copies and MMAs are drained, TMEM is freed and the kernel returns.
#include <atomic>

#include "coc_dequant.cuh"
#include "coc_internal.h"
#include "coc_ptx.cuh"

namespace coc {
namespace {

constexpr int TS_CTA_COLS = TS_UNIT_COLS / 2;          // weight columns per CTA (TMEM lanes): 128
constexpr int TS_SX = 6;                               // X stages: up to 128 rows x 64 k x 2 bytes
constexpr int TS_SW = 8;                               // int8 weight stages: 64 k x 128 columns
constexpr int TS_SA = 8;                               // dequantised A stages in TMEM, 32 columns each
constexpr int TS_GROUPS = 2;                           // dequant groups taking alternate k-blocks
constexpr int TS_WARPS = 2 + NUM_EPI_WARPS + 4 * TS_GROUPS + 1;
constexpr int TS_THREADS = TS_WARPS * 32;
constexpr int TS_WPROD_WARP = TS_WARPS - 1;            // the int8 producer
constexpr int TS_X_BYTES = (TS_MAX_ROWS / 2) * BK * 2; // 16 KiB (fewer bytes used for smaller NR)
constexpr int TS_W_BYTES = TS_CTA_COLS * BK;           // 8 KiB
constexpr int TS_ROW_BYTES = 32 * 2;                   // staging row: one warp's 32 columns
constexpr int TS_STAGE_BYTES = TS_MAX_ROWS * TS_ROW_BYTES;   // 16 KiB per epilogue warp
constexpr int TS_EPI_BYTES = NUM_EPI_WARPS * TS_STAGE_BYTES;
constexpr int TS_BAR_BYTES = 1024;                    // barriers, TMEM slot, abort word, signal slots
constexpr int TS_SMEM = 1024 + TS_SX * TS_X_BYTES + TS_SW * TS_W_BYTES + TS_EPI_BYTES + TS_BAR_BYTES;
constexpr uint32_t TS_A_COL0 = TS_MAX_ROWS;            // accumulator: columns [0, NR); A stage a: 256 + 32 a
static_assert(TS_CTA_COLS == 128, "the warp roles assume 128 weight columns per CTA");
static_assert(TS_SMEM <= 232448, "shared memory above 227 KiB");
static_assert(TS_A_COL0 + 32 * TS_SA <= 512, "TMEM: accumulator + A ring above 512 columns");
static_assert(TS_SW % TS_GROUPS == 0 && TS_SA % TS_GROUPS == 0, "each ring stage must belong to one dequant group");

// tcgen05.mma kind::f16 over a CTA pair, A in tensor memory (each CTA's
// half in its own TMEM at the same address), B from shared memory (each CTA's
// half of the N rows at the same offset).
__device__ __forceinline__ void tc_mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 x 16 bytes of shared memory (16 rows of 16 bytes, one address per row
// from lanes 0-15), transposed: thread t receives column t / 4 (r0) and
// column t / 4 + 8 (r1), four consecutive rows 4 (t % 4) .. 4 (t % 4) + 3
// in each, lowest row in the lowest byte.
__device__ __forceinline__ void ldsm_16x16_trans_b8(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// 16 TMEM lanes x 32 columns: repeat j covers columns 8 j .. 8 j + 7; thread t
// writes v[4j], v[4j+1] to lane t / 4 columns 8j + 2 (t % 4) and + 1, v[4j+2],
// v[4j+3] to lane t / 4 + 8 at the same columns.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Dequantisation constants of one weight column j, and the conversion of four
// int8 values of that column (consecutive k, lowest in the lowest byte) to two
// words of two 16-bit values: Wd = rne((q - z) * s), the same operations as
// coc_dequant.cuh's Dq (so the same bits): the bias trick of Kim et al. 2022
// gives q - z exactly, one multiply rounds once.  Columns past n get s = 0.
template <bool BF16>
struct DqCol;

template <>
struct DqCol<false> {
    __half2 s2, c2;
    __device__ __forceinline__ void load(const W8Layout& L, const uint16_t* sc, const int8_t* zp, int row, int j) {
        uint16_t sv = 0;
        int z = 0;
        if (L.gran == COC_SCALE_TENSOR) {
            sv = sc[0];
            z = zp ? zp[0] : 0;
        } else if (j < L.n) {
            const long long o = w8_table_row(L, row) + j;
            sv = __ldg(sc + o);
            z = zp ? static_cast<int>(__ldg(zp + o)) : 0;
        }
        const uint32_t w = static_cast<uint32_t>(sv) | (static_cast<uint32_t>(sv) << 16);
        s2 = *reinterpret_cast<const __half2*>(&w);
        c2 = __floats2half2_rn(static_cast<float>(1152 + z), static_cast<float>(1152 + z));
    }
    __device__ __forceinline__ void convert(uint32_t q4, uint32_t& lo, uint32_t& hi) const {
        const uint32_t u = q4 ^ 0x80808080u;
        const uint32_t a = prmt(u, 0x64646464u, 0x4140u);   // binary16 1024 + u0, 1024 + u1
        const uint32_t b = prmt(u, 0x64646464u, 0x4342u);   // 1024 + u2, 1024 + u3
        const __half2 d0 = __hmul2_rn(__hsub2(*reinterpret_cast<const __half2*>(&a), c2), s2);
        const __half2 d1 = __hmul2_rn(__hsub2(*reinterpret_cast<const __half2*>(&b), c2), s2);
        lo = *reinterpret_cast<const uint32_t*>(&d0);
        hi = *reinterpret_cast<const uint32_t*>(&d1);
    }
};

template <>
struct DqCol<true> {
    float s, c;
    __device__ __forceinline__ void load(const W8Layout& L, const uint16_t* sc, const int8_t* zp, int row, int j) {
        uint16_t sv = 0;
        int z = 0;
        if (L.gran == COC_SCALE_TENSOR) {
            sv = sc[0];
            z = zp ? zp[0] : 0;
        } else if (j < L.n) {
            const long long o = w8_table_row(L, row) + j;
            sv = __ldg(sc + o);
            z = zp ? static_cast<int>(__ldg(zp + o)) : 0;
        }
        s = __uint_as_float(static_cast<uint32_t>(sv) << 16);
        c = 8388736.0f + static_cast<float>(z);   // 2^23 + 128 + z, exact
    }
    __device__ __forceinline__ void convert(uint32_t q4, uint32_t& lo, uint32_t& hi) const {
        const uint32_t u = q4 ^ 0x80808080u;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(__fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7650u + e)), c), s);
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2], v[3]);
        lo = *reinterpret_cast<const uint32_t*>(&b0);
        hi = *reinterpret_cast<const uint32_t*>(&b1);
    }
};

template <bool BF16>
__device__ __forceinline__ uint16_t round16(uint32_t fbits) {
    const float f = __uint_as_float(fbits);
    if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    else return __half_as_ushort(__float2half_rn(f));
}

// Staging of one epilogue warp: 256 rows of its 32 columns (64 bytes), the
// 16-byte chunk c of row r stored at chunk c ^ ((r >> 1) & 3) so that eight
// consecutive rows read by one warp hit distinct banks.
__device__ __forceinline__ uint32_t stage_off(int row, int chunk) {
    return static_cast<uint32_t>(row * TS_ROW_BYTES + ((chunk ^ ((row >> 1) & 3)) << 4));
}

template <bool BF16>
__global__ void __launch_bounds__(TS_THREADS, 1) coc_w8_ts_kernel(const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* x_st = smem;                                   // TS_SX x 16 KiB
    uint8_t* w_st = x_st + TS_SX * TS_X_BYTES;              // TS_SW x 8 KiB
    uint8_t* epi = w_st + TS_SW * TS_W_BYTES;               // 4 x 16 KiB
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + TS_EPI_BYTES);
    uint64_t* xfull = bars;                 // [SX] X stage landed (leader's: both CTAs' bytes)
    uint64_t* xempty = xfull + TS_SX;       // [SX] X stage consumed (the leader's multicast commit)
    uint64_t* wfull = xempty + TS_SX;       // [SW] int8 stage landed (local)
    uint64_t* wempty = wfull + TS_SW;       // [SW] int8 stage read by this CTA's dequant group
    uint64_t* afull = wempty + TS_SW;       // [SA] leader's: both CTAs' TMEM A stages written
    uint64_t* aempty = afull + TS_SA;       // [SA] TMEM A stage consumed (the leader's multicast commit)
    uint64_t* accf = aempty + TS_SA;        // accumulator ready (multicast commit)
    uint64_t* acce = accf + 1;              // leader's: both CTAs' accumulators drained (8 epilogue warps)
    uint64_t* never = acce + 1;             // nothing arrives here (fault-injection test)
    uint64_t* drain = never + 1;            // MMA drain before TMEM release
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    uint32_t* abort_word = tmem_slot + 1;
    // 16-byte landing slots (one per A stage) for the peer's "A stage written" signals
    uint8_t* sig_slots = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(abort_word + 1) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Ctl ctl{abort_word, p.status};
    const uint32_t rank = cluster_rank();   // 0 = leader
    const int first_unit = static_cast<int>(cluster_id());
    const int unit_step = static_cast<int>(cluster_count());
    const int NR = p.unit_rows;             // activation rows per unit (MMA N)
    const int half_rows = NR / 2;           // rows of X held by this CTA
    const uint32_t x_bytes = static_cast<uint32_t>(half_rows) * BK * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TS_SX; ++s) {
            mbar_init(smem_u32(&xfull[s]), 1);
            mbar_init(smem_u32(&xempty[s]), 1);
        }
        for (int s = 0; s < TS_SW; ++s) {
            mbar_init(smem_u32(&wfull[s]), 1);
            mbar_init(smem_u32(&wempty[s]), 1);
        }
        for (int s = 0; s < TS_SA; ++s) {
            mbar_init(smem_u32(&afull[s]), 1);   // the leader group's arrival; the peer adds 16 tx bytes
            mbar_init(smem_u32(&aempty[s]), 1);
        }
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(acce), 2 * NUM_EPI_WARPS);
        mbar_init(smem_u32(never), 1);
        mbar_init(smem_u32(drain), 1);
        *abort_word = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const bool probe = p.clock_slot >= 0 && blockIdx.x == 0 && threadIdx.x == 0;
    uint64_t probe_clk = 0, probe_ns = 0;
    if (probe) {
        probe_clk = clock64();
        probe_ns = globaltimer();
    }
    const int unit_kb = p.num_kshards * p.kblocks;   // k-blocks per unit (all shards)

    if (warp == 0) {
        // ================================================= X producer ===
        if (lane == 0)
            for (int i = 0; i < p.num_kshards && i < COC_MAX_RANKS; ++i) prefetch_tmap(&p.tm_a[i]);
        const uint64_t pol_a = make_l2_policy(p.a_hint);
        uint32_t filled = 0, par = 0;   // per-stage masks of the last fill (leader's drain after an abort)
        uint32_t c = 0;                 // k-block counter over all units
        bool ok = true;
        for (int u = first_unit; ok && u < p.units; u += unit_step) {
            int r, mt, nt;
            decode_unit<OP_AR>(p, u, r, mt, nt);
            const int row0 = mt * NR + static_cast<int>(rank) * half_rows;
            for (int ks = 0; ok && ks < p.num_kshards; ++ks) {
                for (int kb = 0; kb < p.kblocks; ++kb, ++c) {
                    const uint32_t s = c % TS_SX, ph = (c / TS_SX) & 1u;
                    ok = warp_wait<true>(smem_u32(&xempty[s]), ph ^ 1u, ctl, 0x500u + s);
                    if (!ok) break;
                    if (lane == 0) {
                        const uint32_t fb_local = smem_u32(&xfull[s]);
                        if (rank == 0) mbar_expect_tx(fb_local, 2 * x_bytes);
                        tma_load_2d_pair(smem_u32(x_st + s * TS_X_BYTES), &p.tm_a[ks], kb * BK, row0,
                                         map_to_rank(fb_local, 0), pol_a);
                        filled |= 1u << s;
                        par = (par & ~(1u << s)) | (ph << s);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok && lane == 0) {
            if (rank == 0) {
                for (int s = 0; s < TS_SX; ++s)
                    if (filled & (1u << s)) drain_wait(smem_u32(&xfull[s]), (par >> s) & 1u, kDrainNs);
            } else {
                const uint64_t t0 = globaltimer();   // the peer's loads complete on the leader's barriers
                while (globaltimer() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == TS_WPROD_WARP) {
        // ================================================= int8 producer ===
        if (lane == 0)
            for (int i = 0; i < p.num_kshards && i < COC_MAX_RANKS; ++i) prefetch_tmap(&p.tm_b[i]);
        const uint64_t pol_b = make_l2_policy(p.b_hint);
        uint32_t filled = 0, par = 0;
        uint32_t c = 0;
        bool ok = true;
        for (int u = first_unit; ok && u < p.units; u += unit_step) {
            int r, mt, nt;
            decode_unit<OP_AR>(p, u, r, mt, nt);
            const int col0 = nt * TS_UNIT_COLS + static_cast<int>(rank) * TS_CTA_COLS;
            for (int ks = 0; ok && ks < p.num_kshards; ++ks) {
                for (int kb = 0; kb < p.kblocks; ++kb, ++c) {
                    const uint32_t s = c % TS_SW, ph = (c / TS_SW) & 1u;
                    ok = warp_wait(smem_u32(&wempty[s]), ph ^ 1u, ctl, 0x510u + s);
                    if (!ok) break;
                    if (lane == 0) {
                        const uint32_t fb = smem_u32(&wfull[s]);
                        mbar_expect_tx(fb, TS_W_BYTES);
                        tma_load_2d_hint(smem_u32(w_st + s * TS_W_BYTES), &p.tm_b[ks], col0, kb * BK, fb, pol_b);
                        filled |= 1u << s;
                        par = (par & ~(1u << s)) | (ph << s);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok && lane == 0)
            for (int s = 0; s < TS_SW; ++s)
                if (filled & (1u << s)) drain_wait(smem_u32(&wfull[s]), (par >> s) & 1u, kDrainNs);
    } else if (warp == 1) {
        // ================================================= MMA issuer (leader) ===
        // A (the dequantised weight, 256 columns x 16 k over the pair) from
        // TMEM, B (X, NR rows x 16 k over the pair) K-major from shared
        // memory: both operands K-major.
        if (rank == 0) {
            const uint32_t idesc = make_idesc(BF16, TS_UNIT_COLS, NR) & ~(1u << 16);
            uint32_t c = 0;
            int acc_i = 0;
            bool ok = true;
            for (int u = first_unit; ok && u < p.units; u += unit_step, ++acc_i) {
                ok = warp_wait<true>(smem_u32(acce), (acc_i & 1) ^ 1u, ctl, 0x600u);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < unit_kb; ++i, ++c) {
                    const uint32_t xs = c % TS_SX, as = c % TS_SA;
                    ok = warp_wait<true>(smem_u32(&xfull[xs]), (c / TS_SX) & 1u, ctl, 0x610u + xs);
                    if (ok) ok = warp_wait<true>(smem_u32(&afull[as]), (c / TS_SA) & 1u, ctl, 0x620u + as);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t bd = make_sdesc(smem_u32(x_st + xs * TS_X_BYTES), 16, 1024);
                        const uint32_t at = tmem_base + TS_A_COL0 + as * 32;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            tc_mma_f16_ts_pair(tmem_base, at + kk * 8, bd + static_cast<uint64_t>(kk) * 2, idesc,
                                               (i > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_pair_both(smem_u32(&xempty[xs]));
                        tc_commit_pair_both(smem_u32(&aempty[as]));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) tc_commit_pair_both(smem_u32(accf));
                __syncwarp();
            }
            if (lane == 0) {
                tc_commit_pair_local(smem_u32(drain));
                drain_wait(smem_u32(drain), 0, kDrainNs);
            }
            __syncwarp();
        }
    } else if (warp < 2 + NUM_EPI_WARPS) {
        // ================================================= epilogue ===
        const int q = warp & 3;   // TMEM lane quadrant: weight columns 32 q .. 32 q + 31 of this CTA's 128
        uint8_t* stg = epi + (warp - 2) * TS_STAGE_BYTES;
        const uint32_t stg_s = smem_u32(stg);
        const uint32_t acce_leader = map_to_rank(smem_u32(acce), 0);
        int acc_i = 0;
        bool ok = true;
        if (p.inject_timeout) ok = warp_wait(smem_u32(never), 0, ctl, 0x700u);
        for (int u = first_unit; ok && u < p.units; u += unit_step, ++acc_i) {
            int r, mt, nt;
            decode_unit<OP_AR>(p, u, r, mt, nt);
            ok = warp_wait<true>(smem_u32(accf), acc_i & 1, ctl, 0x710u);
            if (!ok) break;
            tc_fence_after();
            // drain: thread `lane` holds weight column 32 q + lane; 32 rows per load
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll 1
            for (int ch = 0; ch < NR / 32; ++ch) {
                uint32_t v[32];
                if (unit_kb > 0) {
                    tmem_ld_32cols(t_row + ch * 32, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int row = ch * 32 + i;
                    const uint32_t a = stg_s + stage_off(row, lane >> 3) + (lane & 7) * 2;
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(round16<BF16>(v[i])) : "memory");
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader);   // the MMA may overwrite the accumulator now
            // the R copies: this warp's 32 columns of the unit's rows, 64 bytes per row
            const int c0 = nt * TS_UNIT_COLS + static_cast<int>(rank) * TS_CTA_COLS + 32 * q;
            if (c0 < p.n) {
                const int ch = lane & 3;         // 16-byte chunk of the row (8 columns)
                const int c = c0 + ch * 8;       // n % 16 == 0: a chunk is wholly inside or outside
#pragma unroll 1
                for (int rb = 0; rb < NR; rb += 64) {
                    uint4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = rb + (lane >> 2) + 8 * i;
                        v[i] = row < NR ? *reinterpret_cast<const uint4*>(stg + stage_off(row, ch))
                                        : make_uint4(0u, 0u, 0u, 0u);
                    }
                    if (c < p.n) {
                        for (int o = 0; o < p.n_out; ++o) {
                            uint16_t* base = p.outp[o] + c;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int row = rb + (lane >> 2) + 8 * i;
                                const long long g = static_cast<long long>(mt) * NR + row;
                                if (row < NR && g < p.m) *reinterpret_cast<uint4*>(base + g * p.n) = v[i];
                            }
                        }
                    }
                }
            }
            __syncwarp();
        }
    } else {
        // ================================================= dequantisation ===
        // Warp (group g, quadrant qd) converts, for every k-block of its group,
        // this CTA's weight columns 32 qd .. 32 qd + 31 of the unit (the TMEM
        // lanes of its quadrant) and writes them to the k-block's TMEM A
        // stage.  Thread t owns columns 32 qd + {t/4, t/4 + 8, t/4 + 16,
        // t/4 + 24}.  The group's k-blocks of a unit are li = g, g + 2, ...
        // (rank li / kblocks).
        const int xw = warp - 2 - NUM_EPI_WARPS;
        const int group = xw >> 2;
        const int qd = warp & 3;
        const int gcol = lane >> 2;
        const W8Layout L{p.gran, p.group, p.n};
        const uint32_t afull_leader = map_to_rank(smem_u32(afull), 0);
        uint32_t c = 0;   // k-block counter over all units (same sequence as the producers and MMA)
        bool ok = true;
        for (int u = first_unit; ok && u < p.units; u += unit_step) {
            int r, mt, nt;
            decode_unit<OP_AR>(p, u, r, mt, nt);
            const int jbase = nt * TS_UNIT_COLS + static_cast<int>(rank) * TS_CTA_COLS + 32 * qd + gcol;
            // constants of this group's k-block `li` of the unit (rank li / kblocks)
            auto load_consts = [&](DqCol<BF16> (&d)[4], int li) {
                const int ks = li / p.kblocks, kb = li - ks * p.kblocks;
                const uint16_t* sc = p.scale[ks];
                const int8_t* zp = p.has_zero ? p.zero[ks] : nullptr;
#pragma unroll
                for (int e = 0; e < 4; ++e) d[e].load(L, sc, zp, kb * BK, jbase + 8 * e);
            };
            // one k-block of this group: `cur` holds its constants, `nxt` receives
            // those of the group's next k-block, loading while this one converts
            auto step = [&](const DqCol<BF16> (&cur)[4], DqCol<BF16> (&nxt)[4], int li) -> bool {
                if (li + TS_GROUPS < unit_kb) load_consts(nxt, li + TS_GROUPS);
                const uint32_t cc = c + static_cast<uint32_t>(li);
                const uint32_t ws = cc % TS_SW, as = cc % TS_SA;
                bool ok_k = warp_wait(smem_u32(&wfull[ws]), (cc / TS_SW) & 1u, ctl, 0x800u + ws);
                if (ok_k) ok_k = warp_wait<true>(smem_u32(&aempty[as]), ((cc / TS_SA) & 1u) ^ 1u, ctl, 0x810u + as);
                if (ok_k) {
                    tc_fence_after();
                    const uint32_t wsb = smem_u32(w_st + ws * TS_W_BYTES);
                    // all eight 16 x 16 blocks of this warp's 32 columns x 64 k first ...
                    uint32_t q8[2][4][2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int chunk = 2 * qd + h;   // 16-byte chunk of the 128-byte int8 row
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int k = 16 * j + (lane & 15);
                            ldsm_16x16_trans_b8(wsb + k * 128 + ((chunk ^ (k & 7)) << 4), q8[h][j][0], q8[h][j][1]);
                        }
                    }
                    // ... then convert and write them to the k-block's TMEM A stage
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            cur[2 * h].convert(q8[h][j][0], o[4 * j], o[4 * j + 1]);
                            cur[2 * h + 1].convert(q8[h][j][1], o[4 * j + 2], o[4 * j + 3]);
                        }
                        tmem_st_16x256b_x4(
                            tmem_base + (static_cast<uint32_t>(32 * qd + 16 * h) << 16) + TS_A_COL0 + as * 32, o);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                // The group's four warps agree (barrier with OR-reduction) that each
                // wrote its quadrant; on any failure they all leave together, so no
                // warp is left waiting at the named barrier.  One thread then
                // signals: in the leader a local arrive, in the peer a 16-byte
                // shared-to-shared bulk copy completing on the leader's barrier
                // (an async-proxy signal issued after the TMEM stores completed,
                // instead of a cluster-scope release per k-block).
                const uint32_t fail = (!ok_k || *reinterpret_cast<volatile uint32_t*>(abort_word) != 0u) ? 1u : 0u;
                uint32_t any_fail;
                asm volatile(
                    "{\n\t.reg .pred pf, pa;\n\t"
                    "setp.ne.u32 pf, %1, 0;\n\t"
                    "bar.red.or.pred pa, %2, %3, pf;\n\t"
                    "selp.u32 %0, 1, 0, pa;\n\t}"
                    : "=r"(any_fail)
                    : "r"(fail), "r"(1 + group), "n"(128)
                    : "memory");
                if (any_fail) return false;
                if (qd == 0 && lane == 0) {
                    const uint32_t af = afull_leader + as * static_cast<uint32_t>(sizeof(uint64_t));
                    if (rank == 0) mbar_expect_tx(smem_u32(&afull[as]), 16);   // arrive + the peer's 16 bytes
                    else bulk_copy_s2s_signal(map_to_rank(smem_u32(sig_slots + 16 * as), 0),
                                              smem_u32(sig_slots + 16 * as), 16, af);
                    mbar_arrive(smem_u32(&wempty[ws]));
                }
                return true;
            };
            int li = (static_cast<int>(c % TS_GROUPS) == group) ? 0 : 1;   // this group's first k-block
            DqCol<BF16> ca[4], cb[4];
            if (li < unit_kb) load_consts(ca, li);
            for (; ok && li < unit_kb; li += 2 * TS_GROUPS) {
                ok = step(ca, cb, li);
                if (ok && li + TS_GROUPS < unit_kb) ok = step(cb, ca, li + TS_GROUPS);
            }
            c += static_cast<uint32_t>(unit_kb);
        }
    }

    tc_fence_before();
    // After an abort the peer may still have loads in flight toward the
    // leader's barriers: give them time to land before either CTA can exit.
    if (*reinterpret_cast<volatile uint32_t*>(abort_word) != 0u) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) {
        }
    }
    cluster_sync();   // the leader's MMAs (which read and write both CTAs' TMEM) and all cross-CTA traffic are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
    if (probe) {
        unsigned long long* slot = reinterpret_cast<unsigned long long*>(p.status + STATUS_WORDS) + 2 * p.clock_slot;
        atomicAdd(slot, static_cast<unsigned long long>(clock64() - probe_clk));
        atomicAdd(slot + 1, static_cast<unsigned long long>(globaltimer() - probe_ns));
    }
}

constexpr int kMaxDevices = 64;

template <bool BF16>
cudaError_t ensure_smem(int dev) {
    static std::atomic<unsigned char> smem_set[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && smem_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(coc_w8_ts_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, TS_SMEM);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) smem_set[dev].store(1, std::memory_order_release);
    return e;
}

cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(TS_THREADS, 1, 1);
    cfg.dynamicSmemBytes = TS_SMEM;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <bool BF16>
cudaError_t launch_ts_t(const KParams& p, int grid, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = ensure_smem<BF16>(dev)) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(grid, stream, attr);
    return cudaLaunchKernelEx(&cfg, coc_w8_ts_kernel<BF16>, p);
}

template <bool BF16>
int max_pairs_t() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || ensure_smem<BF16>(dev) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, coc_w8_ts_kernel<BF16>, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace

cudaError_t launch_w8_ts(const KParams& p, bool bf16, int grid, cudaStream_t stream) {
    return bf16 ? launch_ts_t<true>(p, grid, stream) : launch_ts_t<false>(p, grid, stream);
}

int w8_ts_max_pairs(bool bf16) { return bf16 ? max_pairs_t<true>() : max_pairs_t<false>(); }

}  // namespace coc
