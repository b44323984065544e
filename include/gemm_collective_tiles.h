/*
 * gemm_collective_tiles.h -- C ABI of the GB300 (sm_103a) fused GEMM + collective library.
 *
 * One persistent kernel per call interleaves dense GEMM tiles (tcgen05 tensor
 * cores, TMA-fed shared-memory pipeline, fp32 accumulators in tensor memory)
 * with collective-communication tiles (vectorised copy / reduce) that are
 * linked to the GEMM tiles by release/acquire ready-flags.
 *
 * The W ranks of the collective are emulated on one GPU as W regions of a
 * symmetric heap: region r starts at heap->base + r * heap->rank_stride, and a
 * tensor that "lives on every rank" sits at the same byte offset in every
 * region (the heap_bases address translation of the iris symmetric heap,
 * iris docs "Fused Communication and Compute Operations", atomic_sub:
 * heap_bases holds each rank's heap base and a pointer moves between ranks by
 * its offset).  Collective results are reproduced bit for bit on the device.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Matrices are row-major ("NN"): A is M x K with K contiguous, B is K x N
 *    with N contiguous, outputs are rows x N with N contiguous.  Element type
 *    of A, B, bias and 16-bit outputs: IRIS_F16 or IRIS_BF16 (A and B always
 *    share one type).  Accumulation is fp32.
 *  - Tensor arguments named off_* are BYTE OFFSETS into a heap region (the
 *    same offset in every region that holds the tensor).  Every offset must be
 *    16-byte aligned and every row must be a multiple of 16 bytes (the tensor
 *    memory accelerator's rule), i.e. K, N, K/W, N/W as the op requires must be
 *    multiples of 8 elements.  M may be anything (ragged row tails are masked).
 *    IRIS_NO_BIAS as off_bias means "no bias".
 *  - Ownership: the caller owns the heap, the workspace and the stream.  The
 *    library allocates no device memory per call; it keeps only a per-process
 *    cache of kernel attributes.
 *  - Asynchrony: every op enqueues one kernel on `stream` and returns.  The
 *    iris ops' async_op=False (a barrier at the end) is the caller
 *    synchronising the stream; iris_b200_query_status() does that and reports
 *    device-side failures.
 *  - Workspace: `workspace` is caller-allocated device memory of at least
 *    iris_b200_workspace_size() bytes, ZERO-FILLED ONCE before its first use.
 *    It holds the queue counters, the launch epoch, a status word, the
 *    ready-flags and (reduce ops) the fp32 partial products.  It may be reused
 *    by any later call on the same stream without clearing (flags carry the
 *    launch epoch).  Two calls that share a workspace must not overlap in time.
 *  - Config: NULL or a zero-filled struct selects the defaults field by field.
 *  - Return value: IRIS_OK (0) or a negative IRIS_E* code; nothing is launched
 *    when an error is returned.  There is no silent fallback path.
 */
#ifndef GEMM_COLLECTIVE_TILES_H
#define GEMM_COLLECTIVE_TILES_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define IRIS_API __attribute__((visibility("default")))
#else
#define IRIS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define IRIS_OK 0
#define IRIS_EINVAL (-1)      /* null pointer, bad size, world size, divisibility, config value */
#define IRIS_EALIGN (-2)      /* offset or row pitch not a multiple of 16 bytes */
#define IRIS_ENOWS (-3)       /* workspace missing or smaller than iris_b200_workspace_size() */
#define IRIS_ECUDA (-4)       /* CUDA runtime / driver error (launch, attribute, tensor map) */
#define IRIS_ETIMEOUT (-5)    /* a bounded device wait gave up (reported by query_status) */
#define IRIS_EUNSUPPORTED (-6) /* valid request the library does not implement */

#define IRIS_NO_BIAS ((size_t)-1)
#define IRIS_MAX_WORLD 16

typedef enum { IRIS_F16 = 0, IRIS_BF16 = 1, IRIS_F32 = 2 } iris_dtype;

typedef enum {
    IRIS_COLL_ALL_GATHER = 0,
    IRIS_COLL_ALL_REDUCE = 1,
    IRIS_COLL_REDUCE_SCATTER = 2,
    IRIS_COLL_ALL_TO_ALL = 3,
    IRIS_COLL_BROADCAST = 4
} iris_coll;

typedef enum {
    IRIS_OP_ALL_GATHER_MATMUL = 0,
    IRIS_OP_MATMUL_REDUCE_SCATTER = 1,
    IRIS_OP_MATMUL_ALL_GATHER = 2,
    IRIS_OP_MATMUL_ALL_REDUCE = 3,
    IRIS_OP_CONCURRENT = 4
} iris_op;

/* Tuning knobs (the iris FusedConfig / concurrent gemm_wgs).  0 = default. */
typedef struct {
    int tile_m;            /* GEMM tile rows: 256 = one tile per pair of SMs (a
                              2-CTA cluster sharing the tensor-core instruction;
                              the default wherever it applies: tile_n 256, the
                              chained reduce schedule, a launch with a GEMM), or
                              128 = one tile per SM (tile_n 128, the other reduce
                              schedules and collective-only launches always use
                              it).  With pairs, a CTA split (gemm_ctas) is taken
                              per pair: the pair whose even CTA is below gemm_ctas
                              prefers the GEMM queue. */
    int tile_n;            /* GEMM tile columns: 128 or 256 (default 256) */
    int tile_k;            /* K block: 64 (only value); a pipeline stage holds one
                              K block, or two in the three-stage CTA-pair
                              pipeline (see stages) */
    int group_m;           /* GROUP_M tile swizzle width in 128-row M blocks
                              (default 32; 16 in the concurrent mode and for
                              the reduce ops when a rank's A exceeds 64 MB) */
    int gemm_ctas;         /* CTAs whose first choice is the GEMM queue; the rest
                              prefer the comm queue and every CTA spills to the
                              other queue when its own runs dry.  0 = op default
                              (concurrent: 65% of the grid; the dependent ops: all
                              CTAs); -1 = balanced (every CTA draws from both queues
                              so that both finish together). */
    int stages;            /* CTA-pair tiles: shared-memory pipeline (192 KB either
                              way).  0 = by K: 3 stages of two 64-deep K blocks
                              (one A and one B TMA box per stage), or, when
                              K > 98304 and the operands stream from DRAM, 6
                              stages of one K block (more, smaller loads in
                              flight), in every mode, the concurrent one with
                              a collective included; 3 or 6 choose.  Other values, or a nonzero value
                              with one-CTA tiles: IRIS_EINVAL. */
    int comm_block;        /* concurrent mode: elements per comm tile (default 131072) */
    int replicate_outputs; /* 1: also write the W-1 identical copies of replicated
                              outputs into the other heap regions */
    int bias_on_m;         /* 1: bias has one entry per output row (length M) */
    int grid;              /* persistent CTAs (default: one per SM).  A dependent
                              op with fewer work items (GEMM tiles, gathers,
                              reduce parts) than CTAs (pairs) launches one CTA
                              (pair) per item instead. */
    unsigned long long wait_ns; /* limit of every device-side wait (default 2e9 ns) */
    int debug_skip_flag;   /* test hook: 0 = off; k > 0 makes the kernel never
                              release ready-flag k-1, so the tile waiting on it
                              runs into its bounded wait (IRIS_ETIMEOUT from
                              query_status).  Never set it in production. */
    unsigned long long trace_buf; /* optional device buffer (as an address) for a
                              per-CTA timeline: 4 streams per CTA (scheduler, MMA,
                              TMA, workers) of trace_cap (event, ns) u64 pairs,
                              pair 0 holding the count; the scheduler stream also
                              records each CTA's kernel entry and the end of
                              its teardown; 0 = off */
    int trace_cap;         /* pairs per stream (>= 2 when trace_buf is set) */
    int reduce_mode;       /* matmul_reduce_scatter / matmul_all_reduce reduce schedule:
                              0 = auto (3 when every rank's output slice is whole
                                  32-column chunks, else 2);
                              1 = comm queue: reduce tiles claimed like GEMM tiles,
                                  waiting on per-partial ready-flags (the gemm_ctas
                                  split applies);
                              2 = distributed parts: each output tile's rows split in
                                  W parts that idle worker warps claim once all W
                                  partials are in (epoch-tagged tile counters);
                              3 = chained: rank s adds its partial to the running fp32
                                  sum of ranks 0..s-1 in its GEMM epilogue and hands the
                                  tile on; the last rank writes the rounded output
                                  (a per-tile ring reduction; workspace holds one M x N
                                  fp32 sum instead of W partials) */
    int root;              /* concurrent broadcast: source rank (default 0) */
    int rank_inner;        /* reduce ops: 1 = order GEMM tiles with the rank index
                              fastest; 0 (default) = rank by rank inside each GROUP_M
                              group, so one rank's operands share the L2 at a time */
    int coll_ring;         /* concurrent collectives: shared-memory buffers per
                              worker warp (1 to 4; 0 = default 2).  With more
                              than one, a warp's next loads are in flight
                              while it sums and stores a sub-chunk; with one,
                              each load is a whole 48 KB buffer and the four
                              worker warps overlap each other instead. */
    int coll_l2_hint;      /* concurrent collectives: L2 policy of their bulk
                              copies.  0 = default (none), 1 = evict first (the
                              streamed collective data does not push the
                              concurrent GEMM's operands out of the L2),
                              2 = none. */
    int coll_path;         /* concurrent collectives: how their data moves.
                              0 = default (3 where it applies, else 1);
                              1 = TMA bulk loads into the CTA's pipeline
                                  stages (lent by the GEMM for the tile) and
                                  TMA bulk stores;
                              2 = as 1, but the results are stored from the
                                  worker threads' registers;
                              3 = all-reduce and reduce-scatter with count and
                                  comm_block multiples of 256: one 3-D TMA box
                                  brings the same rows of all W sources (fewer,
                                  larger requests); IRIS_EINVAL elsewhere. */
    int gather_parts;      /* all_gather_matmul: gather items per (128-row block,
                              shard) copy, each a row part of the block
                              (1..16; 0 = default 1).  More parts spread a
                              shard's copies over more CTAs at the cost of
                              more claims and synchronisation per byte. */
    int startup_gather;    /* all_gather_matmul: who copies the gathers a CTA
                              pair claims before its first GEMM tile.  1 = the
                              worker threads, 16-byte copies through
                              registers; 2 = the TMA producer, with TMA boxes
                              through its still idle pipeline stages (whole
                              128-row blocks: needs gather_parts 1, else the
                              workers copy); 0 = default: 2 for M <= 16384
                              when a work item's K (a split-K chunk's, or
                              all of K) is at most 32768, else 1. */
    int gemm_l2_hint;      /* L2 policy of the GEMM operand loads of CTA-pair
                              tiles: 0 = default (evict last), 1 = evict last
                              (the operands keep their place in the L2 against
                              the outputs, partial sums and collective data
                              streaming through it), 2 = none. */
    int out_l2_hint;       /* L2 policy of the final 16-bit output stores:
                              0 = default (none), 1 = evict first (outputs are
                              not read again), 2 = none. */
    int sum_l2_hint;       /* reduce ops, chained schedule: L2 policy of the
                              fp32 running-sum stores and reduce-adds.  0 =
                              default (none), 1 = evict first, 2 = evict last,
                              3 = none. */
    int k_split;           /* the fused ops on CTA pairs (N % 32 == 0; the
                              reduce ops with the chained reduce): K chunks per
                              output tile (of each rank).  Chunk j of a tile is
                              a GEMM item of its own; all partials are summed
                              in (rank, chunk) order through an fp32 running
                              sum in the workspace (all_gather_matmul and
                              matmul_all_gather: M x N fp32 more, counted by
                              iris_b200_workspace_size) before the one rounding
                              to 16 bits.  0 = default: chunks of about 16384
                              K when K > 32768 (shorter tiles keep the tiles
                              running at once on nearby K, where they share
                              their operand blocks in L2), else none; 1 = none;
                              n = n chunks. */
    int coll_out_stage;    /* concurrent all-reduce and reduce-scatter: where a
                              worker warp sums a sub-chunk of its W sources
                              before storing it.  Staged: into its own 4 KB
                              staging halves (when a sub-chunk fits, e.g. the
                              3 KB of W = 8 with the default ring), so the
                              load buffer is refilled right after the sum and
                              all coll_ring loads stay in flight.  In place:
                              in the load buffer, refilled once the stores
                              have read it.  0 = default (staged for
                              all-reduce, whose stores go to all W regions; in
                              place for reduce-scatter), 1 = in place,
                              2 = staged. */
} iris_b200_config;

/* Symmetric heap: W regions of rank_stride bytes starting at base (device memory). */
typedef struct {
    void* base;
    size_t rank_stride;    /* multiple of 16 bytes */
    int world;             /* W, 1..IRIS_MAX_WORLD */
} iris_b200_heap;

/*
 * Workspace bytes needed by `op` for this problem (M, N, K in the op's own
 * convention as below; for IRIS_OP_CONCURRENT pass the GEMM's M, N, K).
 * Writes *bytes.  Errors: IRIS_EINVAL for a null `bytes` or bad sizes.
 */
IRIS_API int iris_b200_workspace_size(iris_op op, int64_t M, int64_t N, int64_t K, int world,
                             iris_dtype dtype, const iris_b200_config* cfg, size_t* bytes);

/*
 * all_gather_matmul  -- iris docs "Fused Communication and Compute
 * Operations", all_gather_matmul: output = all_gather(A_sharded) @ B + bias,
 * A_sharded (M, K_local), B (K, N) with K = K_local * world_size.
 *
 *   off_A        region r holds rank r's shard A_r: M x (K/W), 16-bit.
 *   off_B        region 0 holds B: K x N (shared by every rank).
 *   off_bias     region 0 holds bias: N (or M with bias_on_m) entries, or IRIS_NO_BIAS.
 *   off_out      region 0 receives out = gathered @ B + bias: M x N, 16-bit
 *                (with replicate_outputs, every region receives the same bits).
 *   off_gathered region 0 receives the gathered A: M x K, shard s in columns
 *                [s*K/W, (s+1)*K/W) -- bit-exact copies of the shards.
 * Comm tiles copy each shard's row block into the gathered buffer, a row part
 * at a time (cfg->gather_parts parts per 128-row block), and count themselves into a
 * per-(shard, row block) ready counter (epoch-tagged, release); GEMM tiles
 * acquire the counters of the shards they consume just before loading them.
 * Requires K % W == 0, (K/W) % 8 == 0, N % 8 == 0.
 */
IRIS_API int iris_b200_all_gather_matmul(const iris_b200_heap* heap, size_t off_A, size_t off_B,
                                size_t off_bias, size_t off_out, size_t off_gathered,
                                int64_t M, int64_t N, int64_t K, iris_dtype dtype,
                                const iris_b200_config* cfg, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * matmul_reduce_scatter -- iris docs, matmul_reduce_scatter: output =
 * reduce_scatter(A @ B + bias) along N; output (M, N_local), N_local = N / W.
 *
 *   off_A    region r holds A_r: M x K.       off_B  region r holds B_r: K x N.
 *   off_bias region r holds rank r's bias (N entries, or M with bias_on_m);
 *            every rank adds its own bias to its partial, so the sum holds W biases.
 *   off_out  region r receives out_r: M x N_local, 16-bit:
 *            out_r = RNE16( sum_{s=0..W-1} (A_s @ B_s + bias_s)[:, r*N_local:(r+1)*N_local] )
 *            with the partials kept in fp32 (in the workspace) and summed in
 *            rank order 0..W-1.
 * Requires N % W == 0, (N/W) % 8 == 0, K % 8 == 0.
 */
IRIS_API int iris_b200_matmul_reduce_scatter(const iris_b200_heap* heap, size_t off_A, size_t off_B,
                                    size_t off_bias, size_t off_out, int64_t M, int64_t N,
                                    int64_t K, iris_dtype dtype, const iris_b200_config* cfg,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * matmul_all_gather -- iris docs, matmul_all_gather: output = all_gather(A @ B
 * + bias) along M; A (M_local, K) per rank, output (M_local * W, N).
 *
 *   M        the GATHERED row count (M_local = M / W).
 *   off_A    region r holds A_r: (M/W) x K.   off_B  region 0 holds B: K x N (shared).
 *   off_bias region 0: N entries (or M/W with bias_on_m, the same on every rank).
 *   off_out  region 0 receives out: M x N, rows [r*M/W, (r+1)*M/W) = RNE16(A_r @ B + bias)
 *            (with replicate_outputs, every region receives the same bits).
 * Requires M % W == 0, K % 8 == 0, N % 8 == 0.
 */
IRIS_API int iris_b200_matmul_all_gather(const iris_b200_heap* heap, size_t off_A, size_t off_B,
                                size_t off_bias, size_t off_out, int64_t M, int64_t N,
                                int64_t K, iris_dtype dtype, const iris_b200_config* cfg,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * matmul_all_reduce -- iris docs, matmul_all_reduce: output = all_reduce(A @ B + bias).
 *
 *   off_A, off_B, off_bias  per region as for matmul_reduce_scatter.
 *   off_out  region 0 receives out: M x N = RNE16(rank-order fp32 sum of the
 *            W partials); with replicate_outputs every region receives it.
 * Requires K % 8 == 0, N % 8 == 0.
 */
IRIS_API int iris_b200_matmul_all_reduce(const iris_b200_heap* heap, size_t off_A, size_t off_B,
                                size_t off_bias, size_t off_out, int64_t M, int64_t N,
                                int64_t K, iris_dtype dtype, const iris_b200_config* cfg,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * concurrent_gemm_collective -- ROCm/iris PR #544 "Add iris.concurrent":
 * an independent GEMM runs concurrently with a collective in one persistent
 * kernel with a GEMM queue and a comm queue; cfg->gemm_ctas is the explicit
 * CTA split (the pages' gemm_wgs).
 *
 *   A, B, C    plain device pointers: C (M x N, gemm_dtype) = RNE16(A @ B), no bias.
 *              M, N or K may be 0 (K = 0 writes zeros); M = 0 or N = 0 runs the
 *              collective alone.
 *   coll       the collective over the W heap regions, elements of coll_dtype:
 *     IRIS_COLL_ALL_REDUCE     (IRIS_F32)  out_r[i] = sum_{s=0..W-1} in_s[i] (fp32,
 *                              rank order) for every r; `count` elements per rank;
 *                              off_out == off_in runs it in place.
 *     IRIS_COLL_REDUCE_SCATTER (IRIS_F32)  out_r[i] = (sum_s in_s)[r*count/W + i];
 *                              count % (4W) == 0.
 *     IRIS_COLL_ALL_GATHER     (any type)  out_r[s*count + i] = in_s[i] for every r.
 *     IRIS_COLL_ALL_TO_ALL     (any type)  each buffer is W chunks of count/W elements:
 *                              out_r[s*count/W + i] = in_s[r*count/W + i]; count % W == 0.
 *     IRIS_COLL_BROADCAST      (any type)  out_r[i] = in_root[i] for every r (cfg->root).
 *   count      elements per rank's input (0 runs the GEMM alone); count *
 *              element size must be a multiple of 16 bytes.
 */
IRIS_API int iris_b200_concurrent_gemm_collective(const void* A, const void* B, void* C, int64_t M,
                                         int64_t N, int64_t K, iris_dtype gemm_dtype,
                                         iris_coll coll, const iris_b200_heap* heap,
                                         size_t off_in, size_t off_out, int64_t count,
                                         iris_dtype coll_dtype, const iris_b200_config* cfg,
                                         void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/*
 * Two-stream concurrent mode -- ROCm/iris PR #544 (mode="concurrent": the
 * GEMM and the collective as separate persistent kernels on different
 * streams).  Same operands and semantics as iris_b200_concurrent_gemm_collective;
 * the GEMM kernel runs on cfg->gemm_ctas CTAs (default half of cfg->grid or of
 * the SMs) on `gemm_stream`, the collective kernel on the remaining CTAs on
 * `comm_stream`.  Each kernel holds one CTA per SM, so the two run side by
 * side on disjoint SMs.  Each launch needs its own workspace (of
 * iris_b200_workspace_size(IRIS_OP_CONCURRENT, ...) bytes); the caller orders
 * later work after both streams.
 */
IRIS_API int iris_b200_concurrent_two_stream(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                             int64_t K, iris_dtype gemm_dtype, iris_coll coll,
                                             const iris_b200_heap* heap, size_t off_in, size_t off_out,
                                             int64_t count, iris_dtype coll_dtype, const iris_b200_config* cfg,
                                             void* gemm_workspace, size_t gemm_workspace_bytes,
                                             void* comm_workspace, size_t comm_workspace_bytes,
                                             cudaStream_t gemm_stream, cudaStream_t comm_stream);

/*
 * SM partition for the two-stream mode -- ROCm/iris PR #544 (mode
 * "concurrent": the GEMM and the collective as separate persistent kernels
 * with an explicit split of the compute units).  Creates two CUDA green
 * contexts on the current device with disjoint SM sets -- the first with at
 * least `gemm_sms` SMs (rounded up to the device's partition granularity), the
 * second with the rest -- and a non-blocking stream in each.  Kernels launched
 * into *gemm_stream run only on the first set and those in *comm_stream only
 * on the second, so iris_b200_concurrent_two_stream given these streams (with
 * cfg->gemm_ctas = *gemm_sms_out and cfg->grid = *gemm_sms_out + *comm_sms_out)
 * runs its two kernels on disjoint SMs by construction rather than by
 * occupancy.  The library owns the contexts and streams, one partition per
 * device: a new call replaces the device's previous partition, and
 * iris_b200_sm_partition_release destroys it; the caller must have finished
 * its work on the old streams first.  Returns IRIS_EINVAL for gemm_sms outside
 * [1, #SMs), IRIS_EUNSUPPORTED when the driver offers no green contexts,
 * IRIS_ECUDA otherwise.
 */
IRIS_API int iris_b200_sm_partition_streams(int gemm_sms, cudaStream_t* gemm_stream, cudaStream_t* comm_stream,
                                            int* gemm_sms_out, int* comm_sms_out);
IRIS_API int iris_b200_sm_partition_release(void);

/*
 * all_gather_matmul without a caller-provided workspace.  This entry point
 * has no counterpart on the pages; it exists for callers that cannot
 * allocate device memory themselves and still want the fused op -- e.g. a
 * custom allocator's own bootstrap (the allocator is not usable yet), a host
 * framework that owns every device allocation and hands out no scratch, or a
 * latency-critical path that must not call cudaMalloc (which can synchronise
 * the device).  The caller passes the heap (inputs and outputs) exactly
 * as for iris_b200_all_gather_matmul.  The queue counters, launch epoch,
 * status word and ready-flags live instead in a fixed static device array of
 * IRIS_NOALLOC_SCRATCH_BYTES bytes inside this library (every GPU that loads
 * the library holds it until the process exits).
 *   - Limit: W * ceil(M / 128) ready counters (8 bytes each, one per
 *     128-row block and shard) must fit, i.e. W * ceil(M/128) <=
 *     IRIS_NOALLOC_MAX_FLAGS; larger problems return IRIS_ENOWS and launch
 *     nothing.
 *   - `stream` must belong to the current device: the array used is the
 *     current device's copy.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, which allocates nothing; no address is cached,
 *     so a device reset cannot leave a stale one), zeroes the part of it this
 *     problem uses -- the 256-byte header and W * ceil(M / 128) counters -- with
 *     one cudaMemsetAsync on `stream`, and launches the kernel.  No call
 *     allocates or frees memory.  The first call on a device may load the
 *     library's GPU code (lazy module loading), so make it before any stream
 *     capture.
 *   - All calls share the one array, which keeps the last call's contents:
 *     calls whose kernels overlap on the GPU (different streams, or several
 *     host threads) race and must not be made.
 *   - A bounded device wait that gives up is recorded in the array and
 *     cleared by the next call; it is not reported to the caller (use the
 *     workspace entry point and iris_b200_query_status when that is needed).
 */
#define IRIS_NOALLOC_MAX_FLAGS 16384
#define IRIS_NOALLOC_SCRATCH_BYTES (256 + 8 * IRIS_NOALLOC_MAX_FLAGS)
IRIS_API int iris_b200_all_gather_matmul_noalloc(const iris_b200_heap* heap, size_t off_A,
                                                 size_t off_B, size_t off_bias, size_t off_out,
                                                 size_t off_gathered, int64_t M, int64_t N,
                                                 int64_t K, iris_dtype dtype,
                                                 const iris_b200_config* cfg, cudaStream_t stream);

/*
 * Synchronises `stream`, reads the workspace status word written by the last
 * kernels that used `workspace`, clears it, and returns IRIS_OK or
 * IRIS_ETIMEOUT (a bounded device wait gave up; the kernel then stopped early,
 * released its resources and left its outputs incomplete).  *device_status
 * (may be NULL) receives the raw status; *where / *index (may be NULL) tell
 * which wait gave up (see the kernel source) and on which flag.
 */
IRIS_API int iris_b200_query_status(void* workspace, cudaStream_t stream, int* device_status,
                           int* where, int* index);

/* Human-readable text of an IRIS_* code (static storage). */
IRIS_API const char* iris_b200_strerror(int code);

/* Number of SMs of the current device (the default persistent grid). */
IRIS_API int iris_b200_num_sms(int* n);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_COLLECTIVE_TILES_H */
