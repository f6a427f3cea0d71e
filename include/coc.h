/*
 * coc.h — fused tensor-parallel matmul + collective operators for GB300 (sm_103a).
 *
 * The operators are those of the MindSpeed developer guide page on
 * compute-communication parallelism (CoC), section 融合算子实现
 * ("fused-operator implementation"):
 *
 *   MATMUL_ALL_REDUCE (and its deterministic form)      coc_matmul_all_reduce
 *   MATMUL_REDUCE_SCATTER (and its deterministic form)  coc_matmul_reduce_scatter
 *   ALL_GATHER_MATMUL                                   coc_all_gather_matmul
 *   ALL_GATHER_MATMUL_V2 (also returns the gather)      coc_all_gather_matmul_v2
 *   w8A16 pseudo-quantised MATMUL_ALL_REDUCE, fp16,
 *     per tensor / per channel / per group scales       coc_matmul_all_reduce_w8a16
 *     + zero point, bf16 activations (extension)         coc_matmul_all_reduce_w8a16_ex
 *
 * and the expert-parallel form of the blog's MC2 section (extension):
 *   MoE token dispatch + expert GroupedMatMul           coc_moe_dispatch_grouped_matmul
 *     + the combine (all-to-all back)                   coc_moe_dispatch_grouped_matmul_combine
 *     top-k routing with the gated combine              coc_moe_topk_grouped_matmul_combine
 *
 * The same page's section 问题分析 ("problem analysis") places them in the
 * Megatron ColumnParallelLinear / RowParallelLinear layers: the matmul is
 * followed by AllReduce without sequence parallelism, by AllGather or
 * ReduceScatter with it.
 *
 * One GPU, R emulated ranks.  Each tensor-parallel rank is a separate set of
 * caller-owned device buffers ("shards"), so every collective is carried out
 * inside one persistent CUDA kernel: AllReduce becomes a cross-shard
 * reduction in the tensor-core accumulator whose result is stored to all R
 * rank outputs, ReduceScatter routes each row block to its owning rank, and
 * AllGather routes each operand tile from the shard that holds its rows.
 *
 * Chunking.  Following the page's CoC idea (section 解决思路: split compute
 * and communication into smaller sub-tasks and pipeline them; the left
 * matmul operand is split along m into 2/4/8 parts and m must be a multiple
 * of the split count), `chunks` in {1, 2, 4, 8} cuts the output rows into C
 * equal chunks and sets the order in which the kernel issues its output
 * tiles: every tile of chunk c before any tile of chunk c+1.  When a chunk
 * boundary falls inside a tile (m / C not a multiple of the tile height:
 * 128 rows up to m = 128, 256 rows above), the tiles are issued in plain row
 * order instead, which keeps the chunk order at tile granularity (a tile
 * that straddles two chunks is issued with the earlier one).  chunks = 1
 * means no chunking.  The overlap of communication with compute does not
 * depend on `chunks`: the accumulator is double-buffered in tensor memory,
 * so every tile's reduce/scatter/gather epilogue runs while the next tile's
 * mainloop runs.  The result never depends on `chunks`.
 *
 * Deterministic mode (same section, which lists a deterministic form of the
 * AllReduce and of the ReduceScatter operator).  Every call is
 * bitwise reproducible for identical inputs on the same GPU and library
 * build, across runs and across chunk counts: each output element is
 * accumulated in fp32 in the fixed order rank 0..R-1, k ascending, and
 * rounded once (round-to-nearest-even) to the output type.  No call combines
 * partial sums with atomics or in arrival order; the splits of the
 * contraction at decode-sized m (the column-slab split and the rank split,
 * below) depend on the shape and the GPU only and add their parts in a
 * fixed order.
 * There is no faster non-deterministic schedule, so `deterministic` is
 * accepted and has no effect: deterministic = 0 gives the same bits.
 *
 * Conventions for every entry point:
 *   - All matrices are row-major and densely packed, in device memory the
 *     caller owns (allocated through PyTorch or cudaMalloc).  Base pointers
 *     must be 16-byte aligned and every row must span a multiple of 16 bytes
 *     (TMA requirement), see the per-call alignment notes.
 *   - Array-of-pointer arguments (`x`, `w`, `out`, ...) are HOST arrays of R
 *     device pointers, read before the call returns.
 *   - Library-owned device memory.  The first call on a device allocates a
 *     small status buffer (a few words).  Calls that need scratch (the fp32
 *     parts of a rank-split AllReduce / ReduceScatter, the MoE routing
 *     tables, the w8A16 pre-pass's dequantised weight, the stacked X of an
 *     AllGather that keeps no gathered copy) take it from a
 *     workspace the library keeps per stream: allocated by the first such
 *     call on the stream and grown only when a later call needs more (the
 *     growing call waits for the earlier users of the old buffer first), so
 *     repeated calls of the same shapes make no allocating call at all
 *     (coc_debug_alloc_count counts them).  One call takes at most 4 GiB of
 *     scratch (COC_ERR_SHAPE beyond).  Calls captured into a CUDA graph take
 *     their scratch as stream-ordered allocations from a device pool, which
 *     become memory nodes of the graph, so graph replays allocate nothing
 *     either.  coc_shutdown() frees all of it.  Calls on different streams
 *     use different workspaces and may overlap freely.
 *     coc_matmul_all_reduce_noalloc takes none of this memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Outputs must not alias inputs or each other.
 *   - Argument errors are detected on the host before any CUDA call and are
 *     returned as status codes; nothing is thrown across the ABI and no
 *     output is touched when a call is rejected.
 *   - A launch failure returns COC_ERR_CUDA.  Every wait inside the kernel is
 *     bounded (about one second); a wait that runs out stops the kernel
 *     cleanly and records COC_ERR_TIMEOUT in the status buffer, which
 *     coc_sync_status() reports.  Results of a call that timed out are
 *     undefined.  The bound is the build-time constant COC_WAIT_NS (ns);
 *     raise it where the GPU is time-sliced between processes, since a
 *     pause of the kernel counts against it.
 *   - The first call on a device creates the library's per-device state
 *     (status block, kernel attributes), and the first call on a stream
 *     that needs scratch sizes that stream's workspace (synchronising CUDA
 *     calls).  After them, calls make no synchronising CUDA call and can be
 *     captured into CUDA graphs.
 *   - Environment variables that force a schedule (tuning and tests only;
 *     every value gives correct results): COC_PAIR=0|1 (single-CTA or 2-SM
 *     tiles), COC_W8_PATH=fused|prepass|ts|slab (w8A16 dequantisation in the
 *     GEMM kernel's shared memory, in a pre-pass, in tensor memory, or the
 *     column-slab kernel), COC_KSPLIT=<n> (rank-split part count, rounded
 *     down to a power of two dividing R), COC_SPLIT_PATH=scratch (rank split
 *     through global memory), COC_SLAB=0|1 (column-slab kernel off / for
 *     every m <= 128; AllGather: gathered m) with COC_SLAB_BOXES=1|2
 *     (w8A16 also 4),
 *     COC_SLAB_SPLIT=1|2|4 and COC_SLAB_KPS=1|2|4 (its slab width in
 *     64-column groups, CTAs per slab, k-blocks per stage; 256-column slabs
 *     take one k-block per stage), COC_PDL=0 (the kernels launched in
 *     plain stream order instead of as programmatic dependent launches,
 *     which run their set-up while the previous kernel in the stream
 *     finishes).  Forcing one can change the last bit of
 *     results (a different summation grouping).
 */
#ifndef COC_H_
#define COC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define COC_MAX_RANKS 8

typedef enum {
    COC_OK = 0,
    COC_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, R or chunks not in {1,2,4,8} */
    COC_ERR_SHAPE = 2,         /* sizes that do not fit together or exceed the limits */
    COC_ERR_ALIGN = 3,         /* base pointer or row pitch not 16-byte aligned */
    COC_ERR_UNSUPPORTED = 4,   /* device is not sm_103 / feature not built */
    COC_ERR_CUDA = 5,          /* a CUDA runtime call or the kernel launch failed */
    COC_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out (see coc_sync_status) */
} coc_status_t;

typedef enum { COC_FP16 = 0, COC_BF16 = 1 } coc_dtype_t;

typedef enum {
    COC_SCALE_TENSOR = 0,      /* one scale for the whole weight */
    COC_SCALE_CHANNEL = 1,     /* one scale per output column j */
    COC_SCALE_GROUP = 2        /* one scale per (group of group_size rows of K, column j) */
} coc_scale_t;

/* Fused operator selector for coc_fused_matmul. */
typedef enum {
    COC_OP_ALL_REDUCE = 0,      /* MATMUL_ALL_REDUCE */
    COC_OP_REDUCE_SCATTER = 1,  /* MATMUL_REDUCE_SCATTER */
    COC_OP_ALL_GATHER = 2,      /* ALL_GATHER_MATMUL */
    COC_OP_ALL_GATHER_V2 = 3,   /* ALL_GATHER_MATMUL_V2 */
    COC_OP_WEIGHT_GRAD = 4      /* per-rank weight gradient dW_r = dY_r^T X_r (no collective) */
} coc_op_t;

/* Storage of each weight shard. */
typedef enum {
    COC_W_KN = 0,   /* k x n row-major (inner x cols): the layout of the named entry points */
    COC_W_NK = 1    /* n x k row-major (cols x inner): Megatron's [out_features, in_features] */
} coc_wlayout_t;

/* Opaque CUDA stream handle; identical to cudaStream_t / CUstream. */
typedef struct CUstream_st* coc_stream_t;

/*
 * MATMUL_ALL_REDUCE — row-parallel linear followed by AllReduce
 * (CoC page, 融合算子实现, first bullet; 问题分析 for the layer).
 *
 *   Y = sum_{r=0}^{R-1} X_r @ W_r          (fp32 accumulation)
 *   out[r] = round_rne(Y)  for every r     (all R copies bit-identical)
 *
 * R        ranks, in {1, 2, 4, 8}
 * m, n     output rows / columns; k_shard = contraction length held by each rank
 *          (the full contraction is K = R * k_shard)
 * x[r]     m x k_shard,   dtype `dt`, row pitch k_shard elements
 * w[r]     k_shard x n,   dtype `dt`, row pitch n elements
 * out[r]   m x n,         dtype `dt`, row pitch n elements
 * chunks   in {1, 2, 4, 8}; m % chunks == 0 (COC_ERR_SHAPE otherwise)
 * Alignment: k_shard % 8 == 0 and n % 8 == 0 (16-byte rows), pointers 16-byte
 * aligned.  m, n, k_shard in [0, 2^31); m == 0 or n == 0 is a no-op and
 * k_shard == 0 writes zeros.
 *
 * Decode-sized m (this call, coc_matmul_reduce_scatter, coc_matmul,
 * coc_fused_matmul's AllReduce / ReduceScatter, and the w8A16 AllReduce):
 * for m <= 128 a column-slab kernel streams the weights over all SMs in
 * slabs of 128 output columns (all m rows; w8A16 also 64 or 256), each
 * summed over the whole contraction by one CTA (the same bits as one
 * accumulator) or, while the slabs fill at most half of the SMs, by a
 * cluster of 2 or 4 CTAs that each sum a fixed contiguous range of it and
 * add the ranges in order.
 *
 * Rank split (the same operators except w8A16, with COC_SLAB=0): for m <= 128 with at most
 * half as many 128 x 256 output tiles as the GPU has SMs,
 * each tile's R shards are cut into ksplit parts (the largest power of two
 * dividing R that keeps tiles x ksplit within one wave), each a work unit of
 * its own, and the parts' fp32 sums are added in part order 0..ksplit-1
 * before the one rounding.  (Not for w8A16 or the no-alloc call.)
 * ksplit depends on the shape and the GPU only, so results stay bitwise
 * reproducible across calls and chunk counts; they can differ in the last
 * bit from the same sums taken in one accumulator.
 */
coc_status_t coc_matmul_all_reduce(int R, int64_t m, int64_t n, int64_t k_shard,
                                   const void* const* x, const void* const* w,
                                   void* const* out, coc_dtype_t dt,
                                   int chunks, int deterministic, coc_stream_t stream);

/*
 * MATMUL_REDUCE_SCATTER — row-parallel linear followed by ReduceScatter along
 * the rows (sequence parallelism) (CoC page, 融合算子实现, second bullet).
 *
 *   Y = sum_r X_r @ W_r;   out[r] = round_rne(Y[r*m/R : (r+1)*m/R, :])
 *
 * Rank r always owns the contiguous row block [r*m/R, (r+1)*m/R), whatever
 * `chunks` is.  Arguments as coc_matmul_all_reduce, except
 * out[r]   (m/R) x n.
 * Shape:   m % R == 0, (m/R) % 8 == 0, m % chunks == 0.
 */
coc_status_t coc_matmul_reduce_scatter(int R, int64_t m, int64_t n, int64_t k_shard,
                                       const void* const* x, const void* const* w,
                                       void* const* out, coc_dtype_t dt,
                                       int chunks, int deterministic, coc_stream_t stream);

/*
 * ALL_GATHER_MATMUL — AllGather of the sequence-parallel input followed by a
 * column-parallel linear (CoC page, 融合算子实现, third bullet).
 *
 *   Xg = [X_0; X_1; ...; X_{R-1}]   (rows stacked in rank order, R*m_shard x k)
 *   out[r] = round_rne(Xg @ W_r)
 *
 * x[r]     m_shard x k,          row pitch k
 * w[r]     k x n_shard,          row pitch n_shard
 * out[r]   (R*m_shard) x n_shard, row pitch n_shard
 * Shape:   m_shard % 8 == 0, (R*m_shard) % chunks == 0; chunks split the
 *          gathered rows.  k % 8 == 0, n_shard % 8 == 0.
 * `deterministic` is accepted; there is no cross-rank sum, so results are
 * always reproducible.
 * Where m_shard is not a multiple of 128, Xg is first stacked by a copy
 * kernel (into the first non-NULL gathered output for V2, else into the
 * call's scratch, which the persistent kernel then reads as one operand).
 * Decode-sized m (R*m_shard <= 128, this call, the V2 call and
 * coc_fused_matmul's AllGather forms): the column-slab kernel takes one unit
 * per 128-column slab of one rank's output, after a copy kernel has stacked
 * Xg once (into the first non-NULL gathered output for V2, else into the
 * call's scratch: the stream's workspace, or a stream-ordered allocation
 * while the stream is being captured).  Each slab is one accumulator over k
 * (the persistent kernel's bits) or, in clusters of 2 or 4 CTAs, fixed
 * contiguous k ranges added in order.
 */
coc_status_t coc_all_gather_matmul(int R, int64_t m_shard, int64_t n_shard, int64_t k,
                                   const void* const* x, const void* const* w,
                                   void* const* out, coc_dtype_t dt,
                                   int chunks, int deterministic, coc_stream_t stream);

/*
 * ALL_GATHER_MATMUL_V2 — as coc_all_gather_matmul, and the AllGather
 * intermediate is also returned (CoC page, 融合算子实现, third bullet: the V2
 * form hands the gathered input back to the caller as well).
 *
 * gathered[r]  (R*m_shard) x k, row pitch k: receives a bit-exact copy of Xg.
 *              Entries may be NULL to skip that rank's copy; `gathered`
 *              itself must not be NULL.
 * Shape:   as coc_all_gather_matmul, and n_shard > 0.
 */
coc_status_t coc_all_gather_matmul_v2(int R, int64_t m_shard, int64_t n_shard, int64_t k,
                                      const void* const* x, const void* const* w,
                                      void* const* out, void* const* gathered,
                                      coc_dtype_t dt, int chunks, int deterministic,
                                      coc_stream_t stream);

/*
 * w8A16 MATMUL_ALL_REDUCE — fp16 activations, int8 weights dequantised in the
 * kernel (CoC page, 融合算子实现, last bullet: fake-quantised int8 weights
 * with fp16 activations, scaled per tensor, per channel or per group).
 *
 *   Wd_r[t, j] = fp16_rne( float(Wq_r[t, j]) * s_r(t, j) )   (exact product, one rounding)
 *   Y = sum_r X_r @ Wd_r;  out[r] = fp16_rne(Y) for every r
 *
 * x[r]      m x k_shard fp16
 * w[r]      k_shard x n int8 (symmetric; no zero point)
 * scale[r]  fp16 scales as seen by rank r:
 *             COC_SCALE_TENSOR:  1 value
 *             COC_SCALE_CHANNEL: n values, s(t, j) = scale[r][j]
 *             COC_SCALE_GROUP:   (k_shard/group_size) x n, row-major,
 *                                s(t, j) = scale[r][(t / group_size) * n + j]
 *                                (rank r's rows of the full (K/group_size) x n table)
 * group_size  used for COC_SCALE_GROUP only: a multiple of 64 dividing k_shard.
 * out[r]    m x n fp16
 * Alignment: k_shard % 8 == 0, n % 16 == 0 (16-byte int8 rows).
 */
coc_status_t coc_matmul_all_reduce_w8a16(int R, int64_t m, int64_t n, int64_t k_shard,
                                         const void* const* x, const void* const* w,
                                         const void* const* scale, coc_scale_t gran,
                                         int64_t group_size, void* const* out,
                                         int chunks, int deterministic, coc_stream_t stream);

/*
 * w8A16 MATMUL_ALL_REDUCE with the two extensions the page does not spell
 * out (its 融合算子实现 section names only the symmetric fp16 form): an int8
 * zero point (asymmetric quantisation) and bf16 activations.
 *
 *   Wd_r[t, j] = rne_dt( (Wq_r[t, j] - z_r(t, j)) * s_r(t, j) )   (exact, one rounding)
 *   Y = sum_r X_r @ Wd_r;  out[r] = rne_dt(Y) for every r
 *
 * dt        COC_FP16 or COC_BF16: the type of x, scale and out.
 * zero      NULL (symmetric, z = 0) or one int8 zero-point view per rank,
 *           laid out and indexed exactly like scale[r] (1 value, n values,
 *           or (k_shard/group_size) x n).  q - z lies in [-255, 255].
 * Other arguments as coc_matmul_all_reduce_w8a16, whose call equals this one
 * with zero = NULL and dt = COC_FP16.
 * Alignment: per-channel / per-group scale[r] and zero[r] 16-byte aligned;
 * per-tensor: scale 2-byte aligned, zero unconstrained.
 * Errors: COC_ERR_INVALID_ARG (NULL entries, unknown dt or granularity),
 * COC_ERR_SHAPE, COC_ERR_ALIGN as coc_matmul_all_reduce_w8a16.
 */
coc_status_t coc_matmul_all_reduce_w8a16_ex(int R, int64_t m, int64_t n, int64_t k_shard,
                                            const void* const* x, const void* const* w,
                                            const void* const* scale, const void* const* zero,
                                            coc_scale_t gran, int64_t group_size, void* const* out,
                                            coc_dtype_t dt, int chunks, int deterministic,
                                            coc_stream_t stream);

/*
 * MoE expert-parallel dispatch fused with the experts' GroupedMatMul (the
 * "EP MC2" form named in the MindSpeed-LLM overlap blog, section 第二层MC2:
 * the token all-to-all fused with the expert GroupedMatMul).  Reading of the
 * blog (it gives no formula): R expert-parallel ranks, E = R * experts_per_rank
 * experts with expert e held by rank q = e / experts_per_rank, top-1 routing.
 *
 *   Dispatch (the all-to-all): rank q receives every token routed to one of
 *   its experts, grouped by expert (ascending), inside an expert by source
 *   rank (ascending), inside a source rank by token index (ascending).
 *   Expert e's group occupies rows offsets[e] .. offsets[e] + counts[e] - 1
 *   of xd[q] and y[q]; offsets are multiples of 256 (the rows between groups
 *   are unspecified).
 *   GroupedMatMul: y[q][row] = xd[q][row] @ W_e  (fp32 accumulate, RNE to dt).
 *
 * x[r]        tokens x h, rank r's tokens (dt)
 * idx[r]      tokens int32 expert ids in [0, E); others are not dispatched
 *             and coc_sync_status then reports COC_ERR_INVALID_ARG
 * w           E x h x f, the experts' weights stacked (expert e's h x f block
 *             at e * h * f elements), dt
 * xd[q], y[q] capacity x h and capacity x f, written (the dispatched tokens,
 *             a bit-exact copy, and the expert outputs)
 * counts, offsets  E int32 each, written by the device
 * capacity    rows of xd[q] / y[q]; at least coc_moe_capacity(R, tokens,
 *             experts_per_rank)
 * Shape: h a positive multiple of 64; f * 2 % 16 == 0; E <= 256.
 * Alignment: x, xd, y, w 16-byte aligned; idx, counts, offsets 4-byte.
 * Ownership: all buffers are the caller's device memory; a routing table of
 * R x tokens int32 lives in the stream's workspace (see the conventions
 * above) for the duration of the call.  Runs on `stream` (three kernels:
 * routing, token copy, grouped GEMM); no host synchronisation once the
 * workspace is sized.
 */
coc_status_t coc_moe_dispatch_grouped_matmul(int R, int64_t tokens, int64_t h, int64_t f, int experts_per_rank,
                                             const void* const* x, const int32_t* const* idx, const void* w,
                                             void* const* xd, void* const* y, int64_t capacity,
                                             int32_t* counts, int32_t* offsets, coc_dtype_t dt,
                                             coc_stream_t stream);

/*
 * The same dispatch and GroupedMatMul followed by the combine, the all-to-all
 * back: each expert output row is written to its token's row on the source
 * rank instead of to the dispatched layout,
 *
 *   y_tok[r][t] = x[r][t] @ W_{idx[r][t]}      (top-1 routing: one expert per token)
 *
 * y_tok[r]  tokens x f (dt), rank r's tokens in their own order; rows of
 *           tokens with an out-of-range expert id are not written.
 * Other arguments as coc_moe_dispatch_grouped_matmul (xd still receives the
 * dispatched tokens).  The routing table grows by R x capacity int32 (the
 * source token of each dispatched row), in the same workspace.
 */
coc_status_t coc_moe_dispatch_grouped_matmul_combine(int R, int64_t tokens, int64_t h, int64_t f, int experts_per_rank,
                                                     const void* const* x, const int32_t* const* idx, const void* w,
                                                     void* const* xd, void* const* y_tok, int64_t capacity,
                                                     int32_t* counts, int32_t* offsets, coc_dtype_t dt,
                                                     coc_stream_t stream);

/*
 * Top-k routing: every token has k expert ids idx[r][t*k + j] (j < k) and k
 * fp32 gates gates[r][t*k + j].  Each (token, slot) entry is dispatched as
 * its own row (inside an expert ordered by source rank, token, slot), the
 * GroupedMatMul writes the dispatched layout y[q] (as
 * coc_moe_dispatch_grouped_matmul), and the combine then forms
 *
 *   y_tok[r][t] = rne( sum_{j < k} gates[r][t*k+j] * y[e_j's rank][row of (t, j)] )
 *
 * in fp32, slots in order (deterministic).  capacity must be at least
 * coc_moe_capacity(R, tokens * k, experts_per_rank); k in [1, 8]; gates 4-byte
 * aligned.  Entries with an out-of-range id contribute nothing (and
 * coc_sync_status reports COC_ERR_INVALID_ARG).  Four kernels on `stream`.
 */
coc_status_t coc_moe_topk_grouped_matmul_combine(int R, int64_t tokens, int k, int64_t h, int64_t f,
                                                 int experts_per_rank, const void* const* x,
                                                 const int32_t* const* idx, const float* const* gates, const void* w,
                                                 void* const* xd, void* const* y, void* const* y_tok,
                                                 int64_t capacity, int32_t* counts, int32_t* offsets,
                                                 coc_dtype_t dt, coc_stream_t stream);

/* Rows xd[q] / y[q] need for coc_moe_dispatch_grouped_matmul: R * tokens plus
 * 255 rows of padding per expert of a rank, rounded up to 256; -1 on bad
 * arguments.  Host only. */
int64_t coc_moe_capacity(int R, int64_t tokens, int experts_per_rank);

/*
 * Any of the four bf16/fp16 fused operators with a choice of weight layout.
 * The operators are those above (CoC page, 融合算子实现); the layouts are
 * those of the Megatron layers the page's 问题分析 section names: a linear
 * layer keeps its weight as [out_features, in_features] (COC_W_NK), so its
 * forward pass is X @ W^T, while its backward (data-gradient) pass multiplies
 * by W itself — which, read as a k x n matrix, is the COC_W_KN layout.  Both
 * layouts therefore cover the forward and the backward pairings:
 *
 *   RowParallelLinear forward:  AR / RS of X_r @ W_r^T        (COC_W_NK)
 *   ColumnParallelLinear fwd:   AllGather(X) @ W_r^T           (COC_W_NK)
 *   RowParallel backward, SP:   AllGather(dY) @ W_r            (COC_W_KN)
 *   ColumnParallel backward SP: ReduceScatter(dY_r @ W_r)      (COC_W_KN)
 *
 * The weight-gradient pass completes the pairings: dW_r = dY_r^T X_r, with
 * X_r the layer input as rank r holds it after the forward pass — for a
 * ColumnParallel layer with SP, the gathered input ALL_GATHER_MATMUL_V2
 * returned (the reason V2 returns it), for a RowParallel layer its own X_r.
 *
 * op       COC_OP_ALL_REDUCE / _REDUCE_SCATTER: (rows, cols, inner) =
 *          (m, n, k_shard), x[r] m x k_shard, out[r] m x n (AR) or
 *          (m/R) x n (RS).  COC_OP_ALL_GATHER / _V2: (rows, cols, inner) =
 *          (m_shard, n_shard, k), x[r] m_shard x k, out[r] (R*m_shard) x n_shard.
 * w[r]     COC_W_KN: inner x cols row-major; COC_W_NK: cols x inner row-major.
 *          COC_OP_WEIGHT_GRAD: (rows, cols, inner) = (out_features, in_features,
 *          tokens); x[r] = dY_r, inner x rows; w[r] = X_r, inner x cols
 *          (COC_W_KN only); out[r] = dW_r, rows x cols ([out, in], Megatron's
 *          weight layout).  rows % 8 == 0, cols % 8 == 0, rows % chunks == 0.
 * gathered used by COC_OP_ALL_GATHER_V2 only (as in coc_all_gather_matmul_v2).
 * Results, constraints, alignment and errors are those of the named entry
 * point of the same operator; with COC_W_KN the call is identical to it.
 * With COC_W_NK the products and their accumulation order are the same, so
 * the result is bit-identical to the COC_W_KN call on the transposed weights.
 */
coc_status_t coc_fused_matmul(coc_op_t op, int R, int64_t rows, int64_t cols, int64_t inner,
                              const void* const* x, const void* const* w, coc_wlayout_t layout,
                              void* const* out, void* const* gathered, coc_dtype_t dt,
                              int chunks, int deterministic, coc_stream_t stream);

/*
 * Plain sharded contraction with a single output: out = round_rne(sum_r X_r @ W_r).
 * The same kernel as coc_matmul_all_reduce with a plain one-buffer epilogue;
 * it is the denominator of the fused-overhead measurement (the pages have no
 * counterpart of their own).  Arguments as coc_matmul_all_reduce, `out` a
 * single m x n buffer.
 */
coc_status_t coc_matmul(int R, int64_t m, int64_t n, int64_t k_shard,
                        const void* const* x, const void* const* w, void* out,
                        coc_dtype_t dt, coc_stream_t stream);

/*
 * Allocation-free MATMUL_ALL_REDUCE.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory where
 * they call the operator — runtimes that pre-carve all device memory into
 * their own pools, latency-critical paths where cudaMalloc's implicit
 * synchronisation is not acceptable, processes whose allocations must all go
 * through a custom allocator.
 *
 * Same arguments, results and checks as coc_matmul_all_reduce.  The library
 * makes no cudaMalloc/cudaFree or other allocating call here (it never takes
 * the rank split, whose fp32 parts would need a workspace).  The kernel's
 * only scratch (its 32-byte status block) lives in a fixed 256-byte
 * __device__ array that every GPU loading the library holds until the
 * process exits; this scratch does not grow with m, n or k, and a need
 * beyond 256 bytes would be rejected with COC_ERR_SHAPE.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress) with the device current and clears it; make
 *     that first call before any stream capture.
 *   - Every call shares the array.  Kernels only ever set bits in it (a
 *     bounded wait that runs out records COC_ERR_TIMEOUT there), so calls
 *     whose kernels overlap on the GPU (different streams) may both record a
 *     timeout, and the report cannot tell which of them it came from.
 *   - coc_sync_status() reads this block too (without allocating) and clears
 *     it when it reports a timeout; until then the timeout stays recorded,
 *     whatever calls follow.
 *   - coc_shutdown() forgets the looked-up address; call it before a
 *     cudaDeviceReset if calls continue afterwards.
 */
coc_status_t coc_matmul_all_reduce_noalloc(int R, int64_t m, int64_t n, int64_t k_shard,
                                           const void* const* x, const void* const* w,
                                           void* const* out, coc_dtype_t dt,
                                           int chunks, int deterministic, coc_stream_t stream);

/*
 * Waits for `stream`, then returns and clears the device-side status of
 * this library on the current device (the status buffer of the allocating
 * entry points and the static block of coc_matmul_all_reduce_noalloc):
 * COC_ERR_TIMEOUT if a kernel's bounded wait ran out since the last check,
 * COC_ERR_INVALID_ARG if a MoE dispatch met an expert id out of range,
 * COC_ERR_CUDA if the stream reports an error, COC_OK otherwise.  It creates
 * no library state and allocates nothing.
 */
coc_status_t coc_sync_status(coc_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* coc_status_string(coc_status_t status);

/* Details of the most recent error on this thread (static per-thread buffer). */
const char* coc_last_error(void);

/* Library ABI version: (major << 16) | minor. */
int coc_version(void);

/*
 * Test hook: while `enable` is non-zero, kernels launched afterwards make
 * their epilogue wait on a barrier nothing arrives at, so the bounded waits
 * run out and the kernel stops with COC_ERR_TIMEOUT.  For fault-handling
 * tests only.
 */
coc_status_t coc_debug_inject_timeout(int enable);

/*
 * Test and audit hook: the number of device allocations (cudaMalloc, and
 * stream-ordered allocations of captured calls) the library has made in
 * this process.  Steady-state calls of unchanged shapes on a stream leave it
 * unchanged.
 */
int64_t coc_debug_alloc_count(void);

/*
 * Measurement hook: while `slot` (0..7) is selected, block 0 of every fused
 * kernel launched afterwards adds the SM clock cycles and the nanoseconds
 * (%globaltimer) it ran for to that slot of the device status buffer; -1
 * stops it.  coc_debug_clock_read waits for the device, returns a slot's two
 * sums and clears them: cycles / ns is the SM clock the kernels actually ran
 * at, which a clock sampled through NVML does not show on a power-capped GPU.
 * (The allocation-free entry point never records.)
 */
coc_status_t coc_debug_clock_probe(int slot);
coc_status_t coc_debug_clock_read(int slot, int64_t* cycles, int64_t* ns);

/* Frees the per-device status buffers, the per-stream workspaces and the
 * graph-capture pool; forgets the allocation-free entry point's set-up.
 * Further calls re-create what they need. */
coc_status_t coc_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* COC_H_ */
