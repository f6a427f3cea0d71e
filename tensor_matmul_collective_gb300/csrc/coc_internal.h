// Internal interface between the host API (coc_api.cu) and the persistent
// kernel (coc_kernel.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>            // CUtensorMap (types only; the driver is reached
                             // through cudaGetDriverEntryPointByVersion)
#include <cuda_runtime_api.h>
#include <stdint.h>

#include "../../include/coc.h"

namespace coc {

// ---- tile geometry (one CTA, one tcgen05 MMA of 128 x 256 per k-step) ----
constexpr int BM = 128;         // tile rows   (TMEM lanes)
constexpr int BN = 256;         // tile cols   (TMEM fp32 columns per accumulator)
constexpr int BK = 64;          // k per stage (one 128-byte swizzle row of 16-bit data)
constexpr int UMMA_K = 16;      // k per tcgen05.mma kind::f16
constexpr int EPI_COLS = 64;    // epilogue sub-tile width (one 128-byte swizzle row)
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_XFORM_WARPS = 8;   // w8A16 dequant warps (2 per SM sub-partition)
constexpr int XFORM_GROUPS = 2;      // dequant warp groups taking alternate k-blocks
constexpr int XFORM_GROUP_WARPS = NUM_XFORM_WARPS / XFORM_GROUPS;

constexpr int A_STAGE_BYTES = BM * BK * 2;        // 16 KiB
constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;  // 4 KiB per warp per buffer

enum OpKind : int { OP_AR = 0, OP_RS = 1, OP_AG = 2, OP_W8 = 3, OP_GMM = 4 };
constexpr int NUM_OPS = 5;

// Device status words (per device, zero when healthy).
enum : unsigned { DEV_ERR_TIMEOUT = 1u, DEV_ERR_BAD_INDEX = 2u };
constexpr int STATUS_WORDS = 8;   // [0] error bits, [1] first "where" code, [2] block
// After the status words, CLOCK_SLOTS clock-probe slots of two uint64 each
// (SM cycles, ns) accumulated by block 0 of every fused-kernel launch made
// while coc_debug_clock_probe selects that slot: the clock the kernels
// actually ran at is cycles / ns.
constexpr int CLOCK_SLOTS = 8;
constexpr int STATUS_BLOCK_WORDS = STATUS_WORDS + 4 * CLOCK_SLOTS;

struct KParams {
    CUtensorMap tm_a[COC_MAX_RANKS];    // A operand (X shards), K-major, 128B swizzle
    CUtensorMap tm_b[COC_MAX_RANKS];    // B operand (W shards), MN-major, 128B swizzle (int8: no swizzle)
    CUtensorMap tm_out[COC_MAX_RANKS];  // outputs, 128B swizzle, box 64 x store_rows

    const uint16_t* gsrc[COC_MAX_RANKS];  // AG-V2: X shards (gather source)
    uint16_t* gdst[COC_MAX_RANKS];        // AG-V2: gathered outputs (NULL = skip)
    const uint16_t* scale[COC_MAX_RANKS]; // w8A16 scales (rank views, activation type)
    const int8_t* zero[COC_MAX_RANKS];    // w8A16 zero points (rank views; has_zero)
    uint16_t* outp[COC_MAX_RANKS];        // AllReduce outputs (m x n) written by plain stores (replica_stores)
    unsigned* status;                     // STATUS_WORDS device words

    int R;             // ranks
    int n_out;         // output maps written by an AR tile (R, or 1 for the plain GEMM)
    int m;             // output rows (AG: gathered rows R * m_shard)
    int n;             // output columns per buffer (AG: n_shard)
    int k;             // contraction length per shard (AG: full k)
    int num_kshards;   // shards summed per tile (AR/RS/W8: R; AG: 1)
    int kblocks;       // ceil(k / BK)
    int m_tiles, n_tiles;
    int units;         // work units (tiles; AG: R * tiles)
    int chunk_mt;      // m-tiles per chunk for chunk-major order; 0 = row order
    int group_mt;      // m-tiles per L2 group inside a chunk (divides chunk_mt); 0 = whole chunk
    int rows_per_rank; // RS: m/R; AG: m_shard
    int a_box_rows;    // AG: rows per A TMA box (divides m_shard and BM)
    int store_rows;    // rows per output TMA store box (divides 32)
    int gran;          // w8A16 scale granularity
    int group;         // w8A16 group size (rows of K)
    int inject_timeout;
    int clock_slot;    // clock-probe slot this launch accumulates into; -1: none
    int unit_rows;     // w8A16 tensor-memory kernel: activation rows per unit (32, 64, 128 or 256)
    int has_gather;    // AG-V2
    int a_hint, b_hint;  // L2 policy of A / B loads: 0 evict_normal, 1 evict_first, 2 evict_last
    int b_kmajor;      // W stored n x k (K-major B operand) instead of k x n
    int a_mnmajor;     // weight gradient: A = dY_r^T read MN-major from rank r's dY (AG path only)
    int has_zero;      // w8A16: zero points given
    const int32_t* gmm_counts;   // grouped GEMM: rows per expert (device, written by the routing kernel)
    const int32_t* gmm_offsets;  // grouped GEMM: first row of each expert's group (multiple of 256)
    int gmm_E, gmm_eloc;         // grouped GEMM: experts, experts per rank
    const int32_t* gmm_srcmap;   // combine: per destination rank (stride rows_per_rank) the source
                                 // token r * gmm_T + t of each dispatched row, -1 for padding; NULL: no combine
    int gmm_T;                   // combine: tokens per rank
    int replica_stores; // AllReduce: write the n_out outputs with plain stores (outp) instead of TMA
    // Split by rank (AllReduce / ReduceScatter with few output tiles): each
    // tile's contraction is cut into ksplit unit-sized parts of R / ksplit
    // shards each; a part's fp32 sum goes to part, and per epilogue-warp row
    // slab the last part to arrive (part_cnt) adds the ksplit parts in order
    // 0..ksplit-1 and writes the outputs.  ksplit <= 1: off.
    int ksplit;
    float* part;          // tiles x ksplit x TILE_M x BN fp32
    unsigned* part_cnt;   // tiles x (CTAs per tile) x NUM_EPI_WARPS arrival counters, zero at launch
    // Rank split through distributed shared memory (single-CTA tiles, ksplit 2
    // or 4, one unit per CTA): the ksplit part-CTAs of a tile are one cluster;
    // each drains its fp32 part into its own shared memory, and CTA j adds
    // all parts (in part order) of columns [j BN / ksplit, (j+1) BN / ksplit)
    // read from the cluster's shared memory.  part / part_cnt are unused.
    int split_cluster;
    // Column-slab kernel (decode-sized m): 64-column groups per slab (1 or
    // 2), operand stages, k-blocks per stage (1, 2 or 4, dividing kblocks),
    // and whether the A (and n x k B) maps are 3-D (k in block, row, k-block)
    // so that one box holds a stage; a_box_rows is then the rows of X per
    // k-block.
    int slab_boxes;
    int slab_stages;
    int slab_kps;
    int slab_a3d;
    // CTAs per slab (1, 2 or 4, one cluster): part j sums the j-th of
    // slab_split contiguous ranges of the contraction's stages and finalises
    // the j-th of slab_split column ranges, adding the parts in part order.
    int slab_split;
};

// Argument checks of coc_matmul_all_reduce and the per-thread error text
// (coc_api.cu), reused by the allocation-free entry point (coc_noalloc.cu).
coc_status_t validate_all_reduce_args(int R, int64_t m, int64_t n, int64_t k_shard, const void* const* x,
                                      const void* const* w, void* const* out, coc_dtype_t dt, int chunks,
                                      int deterministic);
coc_status_t report_error(coc_status_t st, const char* msg);
// coc_debug_inject_timeout's flag, for kernels launched outside coc_api.cu.
int inject_timeout_enabled();
// Allocation-free entry point (coc_noalloc.cu): read and clear its static
// status block on the current device (all zero if it never ran there), and
// forget the per-device set-up (coc_shutdown, so a later call after a device
// reset looks the block's address up again).
coc_status_t noalloc_take_status(unsigned (&words)[STATUS_WORDS]);
void noalloc_forget_devices();

// w8A16 streaming pre-pass (coc_w8_prepass.cu): dequantise every rank's int8
// weight once, Wd = rne((q - z) * s) in the activation type, into a 16-bit
// k x n buffer per rank (same conversion code as the fused kernel).
struct W8PrepassArgs {
    const int8_t* q[COC_MAX_RANKS];        // k x n int8 per rank
    const uint16_t* scale[COC_MAX_RANKS];  // scale views (activation type)
    const int8_t* zero[COC_MAX_RANKS];     // zero-point views, NULL = symmetric
    uint16_t* out[COC_MAX_RANKS];          // k x n fp16/bf16 per rank
    int R, k, n, gran, group;
};
cudaError_t launch_w8_prepass(const W8PrepassArgs& a, bool bf16, int sm_count, cudaStream_t stream);

// w8A16 AllReduce with the dequantised weight in tensor memory
// (coc_w8_ts.cu), run by CTA pairs: a unit is TS_UNIT_COLS weight columns
// (TS_UNIT_COLS / 2 per CTA) x p.unit_rows activation rows (half per CTA).
// p as for the fused kernel's w8A16 operator, with n_tiles counting
// TS_UNIT_COLS-column tiles, m_tiles unit_rows-row tiles, the X maps boxed
// BK x unit_rows / 2 (128-byte swizzle), the int8 weight maps boxed
// TS_UNIT_COLS / 2 x BK (128-byte swizzle), and the R outputs in outp.
// grid = 2 x min(units, w8_ts_max_pairs()).
constexpr int TS_UNIT_COLS = 256;
constexpr int TS_MAX_ROWS = 256;
cudaError_t launch_w8_ts(const KParams& p, bool bf16, int grid, cudaStream_t stream);
int w8_ts_max_pairs(bool bf16);

// MoE dispatch (coc_moe.cu): the routing kernel counts each rank's tokens per
// expert and gives every token its row in its expert's (256-row aligned)
// group on the destination rank; the permute kernel copies the token rows
// there (the all-to-all).  Tokens with an expert id outside [0, E) are not
// dispatched and set DEV_ERR_BAD_INDEX.
constexpr int MOE_GROUP_ALIGN = 256;
constexpr int MOE_MAX_EXPERTS = 256;
struct MoeRouteArgs {
    const int32_t* idx[COC_MAX_RANKS];   // T expert ids per rank
    int32_t* dest;                        // R x T: destination row (-1: not dispatched)
    int32_t* srcmap;                      // R x cap: source token of each dispatched row (NULL: not kept)
    int cap;
    int32_t* counts;                      // E
    int32_t* offsets;                     // E
    unsigned* status;
    int R, T, E, eloc;
};
struct MoePermuteArgs {
    const uint16_t* x[COC_MAX_RANKS];     // tokens x h per rank
    uint16_t* xd[COC_MAX_RANKS];          // cap x h per destination rank
    const int32_t* idx[COC_MAX_RANKS];    // T routing entries per rank (entry i: token i / k, slot i % k)
    const int32_t* dest;
    int R, T, h, E, eloc, k;
};
// Top-k combine: out[r][t] = rne(sum_j gates[r][t*k+j] * y[q_j][dest_j]) in fp32, slots in order.
struct MoeCombineArgs {
    const uint16_t* y[COC_MAX_RANKS];     // cap x f expert outputs per destination rank
    const int32_t* idx[COC_MAX_RANKS];    // tokens*k entries per rank
    const float* gates[COC_MAX_RANKS];    // tokens*k per rank
    const int32_t* dest;                  // R x tokens*k
    uint16_t* out[COC_MAX_RANKS];         // tokens x f per rank
    int R, tokens, k, f, E, eloc;
};
cudaError_t launch_moe_route(const MoeRouteArgs& a, cudaStream_t stream);
cudaError_t launch_moe_permute(const MoePermuteArgs& a, int sm_count, cudaStream_t stream);
cudaError_t launch_moe_combine(const MoeCombineArgs& a, bool bf16, int sm_count, cudaStream_t stream);

// Host-side launch helpers implemented in coc_kernel.cu.  `pair` selects the
// 2-SM variant (a cluster of two CTAs per 256-row tile; grid = 2 x pairs);
// otherwise one CTA per 128-row tile.
cudaError_t launch(int op, bool bf16, bool pair, const KParams& p, int grid, cudaStream_t stream);
// Single-CTA kernel launched in clusters of `cluster` CTAs (the rank split
// through distributed shared memory, p.split_cluster), and the number of such
// clusters that can be co-resident.
cudaError_t launch_split(int op, bool bf16, const KParams& p, int grid, int cluster, cudaStream_t stream);

// Column-slab kernel (coc_slab.cu), AllReduce, ReduceScatter and AllGather at
// decode-sized m: one unit per slab of 64 x slab_boxes output columns, all m
// rows (m <= 128), the whole contraction in one CTA.  Launched with grid =
// min(units, SMs), slab_smem_bytes of dynamic shared memory.  128-byte
// swizzle everywhere.  A maps: BK x a_box_rows boxes (2-D), or dims (BK, m,
// kblocks) with boxes (BK, a_box_rows, slab_kps) (3-D, slab_a3d).  B maps,
// k x n storage: 64 x (slab_kps BK) boxes; n x k storage (b_kmajor): BK x
// 64 slab_boxes boxes (2-D) or dims (BK, n, kblocks) with boxes (BK, 64
// slab_boxes, slab_kps) (3-D, slab_a3d).  outp holds the n_out outputs
// (AllReduce) or the R rank outputs (ReduceScatter, AllGather).  AllGather
// (op OP_AG): num_kshards 1, n = n_shard, n_tiles slabs per rank output and
// units R n_tiles, tm_a[0] over the gathered X (m = R m_shard rows, written
// by launch_ag_gather first), tm_b[r] over rank r's W; V2 (has_gather): the
// kernel copies that X (gsrc[0]) into every non-NULL gdst.  With slab_split > 1
// the grid is slab_split x the slabs run at once, in clusters of
// slab_split CTAs.
// w8A16 (AllReduce, w8 true): the B maps are the int8 weights, boxed 64
// slab_boxes x (slab_kps BK) without swizzle; scale / zero / gran / group as
// for the persistent kernel; the kernel dequantises into kSlabW8BStages
// 16-bit B stages.
constexpr int kSlabMaxStages = 32;
constexpr int kSlabW8BStages = 2;
constexpr int kSlabSmemCap = 227 * 1024;                                // dynamic shared memory per CTA
// Programmatic dependent launches (the persistent and column-slab kernels
// start their set-up while the previous kernel in the stream finishes and
// wait for it before touching global memory); COC_PDL=0: plain stream order.
bool pdl_launch();
int slab_stages(int a_rows, int boxes, int kps, int split, bool w8);    // most stages that fit (at least 2)
int slab_smem_bytes(int stages, int a_rows, int boxes, int kps, int split, bool w8);
cudaError_t launch_slab(int op, bool bf16, bool w8, const KParams& p, int grid, cudaStream_t stream);
int slab_max_clusters(bool bf16, bool w8, int split, int smem);         // clusters of `split` resident at once
// AllGather ahead of the column-slab kernel: dst (m x k) = the R shards
// src[i] (m_shard x k each) stacked in rank order; shard_vecs = m_shard k / 8
// (k % 8 == 0).
struct AgGatherParams {
    const uint16_t* src[COC_MAX_RANKS];
    uint16_t* dst;
    int R;
    long long shard_vecs;
};
cudaError_t launch_ag_gather(const AgGatherParams& g, int sm_count, cudaStream_t stream);
int max_split_clusters(int op, bool bf16, int cluster);
// Co-resident CTA pairs the 2-SM variant can have on the current device.
int max_pairs(int op, bool bf16);

}  // namespace coc
