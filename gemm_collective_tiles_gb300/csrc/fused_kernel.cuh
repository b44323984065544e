// Persistent work-stealing kernel that interleaves dense GEMM tiles with
// collective-communication tiles (ROCm/iris PR #544 "Add iris.concurrent":
// one persistent kernel with a GEMM queue and a comm queue, GROUP_M tile
// swizzle, explicit GEMM/comm CTA split; iris docs "Fused Communication and
// Compute Operations" for the four dependent ops).
//
// CTA layout (224 threads, one CTA per SM):
//   warp 0      scheduler (lane 0): claims work items from the two global
//               queues with atomics and publishes them into a small
//               shared-memory item ring, ahead of the warps that run them.
//   warp 1      tensor-memory owner; lane 0 issues tcgen05.mma (128 x BN x 16
//               steps, fp32 accumulators in TMEM, double-buffered).
//   warp 2      TMA producer (lane 0): for GEMM items streams the A/B K-blocks
//               into a STAGES-deep shared-memory pipeline.
//   warps 3..6  workers, one per tensor-memory lane quadrant: GEMM epilogue
//               (tcgen05.ld -> +bias -> fp16/bf16 or
//               fp32 partial -> global) and comm tiles (128-bit vector copy /
//               rank-order fp32 reduce), so the comm tiles of one SM run
//               while its tensor cores work on the next GEMM tile.
// CTA pairs (template CG = 2, launched as clusters of two): a GEMM item is a
// 256 x BN tile.  The even CTA's scheduler publishes every item into both
// CTAs' rings and its MMA thread issues tcgen05.mma.cta_group::2 (M = 256)
// for both; each CTA's TMA producer loads its 128 rows of A and BN/2 columns
// of B, counted on the even CTA's full barrier; each CTA's workers drain
// their own 128 accumulator rows and release them on the even CTA's
// acc_empty barrier.  Comm items (all_gather_matmul gathers) run in both
// CTAs, each on its own 128 rows.
// Every wait is bounded (globaltimer); a wait that gives up records the
// failure in the workspace status word, sets the launch's abort epoch, and
// every role drains its in-flight async work and leaves.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gct {

enum : int { OP_AG_MM = 0, OP_MM_RS = 1, OP_MM_AG = 2, OP_MM_AR = 3, OP_CONC = 4 };
enum : int { COLL_AG = 0, COLL_AR = 1, COLL_RS = 2, COLL_A2A = 3, COLL_BC = 4 };

constexpr int BM = 128;           // tile rows (tcgen05 M for cta_group::1)
constexpr int BK = 64;            // K per block: 64 x 16-bit = one 128-byte swizzle row
// K blocks per pipeline stage: the three-stage CTA-pair pipeline takes two
// (one A box and one B box of 128 K rows per stage and CTA); the six-stage
// one (operands streaming from DRAM: more, smaller stages in flight) and
// one-CTA tiles take one
__host__ __device__ constexpr int k_per_stage(int cg, int stages) { return (cg == 2 && stages <= 3) ? 2 : 1; }
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int NUM_WORKER_WARPS = 4;  // one per tensor-memory lane quadrant (or a multiple of 4)
constexpr int FIRST_WORKER_WARP = 3;   // warps 0..2: scheduler, MMA issuer, TMA producer
constexpr int NUM_THREADS = 32 * (FIRST_WORKER_WARP + NUM_WORKER_WARPS);
constexpr int RING = 8;           // work-item ring depth
// all_gather_matmul: look-ahead gather blocks claimed per GEMM item (times
// the gather parts per block)
constexpr int GATHER_AHEAD = 2;
constexpr uint32_t ITEM_END = 0xFFFFFFFFu;
constexpr uint32_t ITEM_COMM = 0x80000000u;
constexpr int DEV_TIMEOUT = 1;

// where-codes recorded when a bounded wait gives up
enum : int {
    WAIT_ITEM_EMPTY = 1,
    WAIT_ITEM_FULL_MMA = 2,
    WAIT_ITEM_FULL_WORKER = 3,
    WAIT_SMEM_EMPTY = 4,
    WAIT_SMEM_FULL = 5,
    WAIT_ACC_EMPTY = 6,
    WAIT_ACC_FULL = 7,
    WAIT_FLAG_GATHER = 8,
    WAIT_FLAG_PARTIAL = 9,
    WAIT_WORKER_SYNC = 10,
    WAIT_TEARDOWN_TMA = 11,
    WAIT_TEARDOWN_MMA = 12,
    WAIT_ITEM_FULL_TMA = 13,
    WAIT_REDUCE_PARTS = 14,
    WAIT_CHAIN = 15,
    WAIT_CHAIN_LOAD = 16,
    WAIT_LEASE = 17,
    WAIT_LEASE_DONE = 18,
    WAIT_COLL_LOAD = 19,
    WAIT_DRAIN = 20,
    WAIT_GATHER_TMA = 21,
};

// First 256 bytes of the workspace.
struct WsHeader {
    uint32_t epoch;        // epoch of the last completed launch
    uint32_t gemm_ctr;     // GEMM queue head (reset to 0 by the last CTA)
    uint32_t comm_ctr;     // comm queue head
    uint32_t done_ctr;     // CTAs finished in this launch
    int status;            // sticky first device error (0 = none)
    uint32_t abort_epoch;  // == current epoch while the launch is aborting
    int err_where;
    int err_index;
    uint32_t part_ctr;     // next reduce part to claim (distributed reduce schedule)
    uint32_t pad[55];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

struct Params {
    CUtensorMap tmA;  // 3-D {k, row, rank}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmB;  // 3-D {n, k, rank},   box {64, 64, 1},  128-byte swizzle
    CUtensorMap tmC;  // 4-D {n, row, row block, region} output, box {32, 32, 1, 1}:
                      // fp32 partials (128-byte swizzle) or 16-bit outputs (64-byte swizzle)
    CUtensorMap tmS;  // chained reduce: the fp32 running-sum tile buffer, box {32, 32, 1, 1}
    CUtensorMap tmBc; // B as 64-column chunks: 4-D {64, k, n / 64, rank}, box {64, 64 KS, BN / CG / 64, 1}
                      // (one load per stage fills a CTA's B columns; set when N % 64 == 0)
    CUtensorMap tmAc; // A as 64-column K chunks: 4-D {64, row, k / 64, rank}, box {64, 128, KS, 1}
                      // (CTA pairs: one load per stage; set when K % 64 == 0)
    CUtensorMap tmGs; // all_gather_matmul start-up gathers: the shards, 3-D {K_l, M, W}, box {gather_box, 128, 1}
    CUtensorMap tmGd; // ... and the gathered buffer, 3-D {K, M, 1}, box {gather_box, 128, 1} (no swizzle)
    CUtensorMap tmX;  // concurrent all-reduce / reduce-scatter input (coll_path 3): 3-D fp32
                      // {256, count / 256, W} (1 KB rows; regions rank_stride apart), box {256, R, W}
    int b_chunked;    // tmBc is valid
    int a_chunked;    // tmAc is valid
    int op, W, bf16, coll;
    int M;            // rows of one GEMM (M_local for matmul_all_gather)
    int N, K;
    int m_blocks, mb_per_rank, n_blocks, k_blocks, group_m, n_tiles;
    uint32_t n_gemm, n_comm;
    uint32_t n_parts;    // reduce ops, distributed parts schedule: output tiles x W row parts
    uint32_t g_split;    // first GEMM item that is a column half of a split tail tile (n_gemm: none)
    int gemm_ctas;    // CTAs preferring GEMM; < 0 = balanced
    uint32_t lookahead;  // all_gather_matmul: GEMM items ahead whose gathers are claimed early
    uint32_t first_wave; // GEMM items of the first wave (one per CTA or CTA pair)
    char* heap;
    unsigned long long rank_stride;
    unsigned long long off_A, off_out, off_bias, off_gathered, off_in, off_cout;
    int has_bias, bias_on_m, replicate;
    int K_local, N_local;
    WsHeader* ws;
    uint32_t* flags;
    float* partials;
    unsigned long long partial_elems;  // per rank: M * N
    void* C;                           // concurrent GEMM output
    long long count;                   // concurrent collective elements per rank
    int comm_block;                    // concurrent elements per comm tile
    int root;                          // broadcast root rank
    int elem_bytes;
    unsigned long long wait_ns;
    uint32_t debug_skip;               // flag index + 1 that is never released (0 = none)
    int reduce_mode;                   // reduce ops: 1 = comm queue, 2 = distributed parts, 3 = chained
    int coll_ring;                     // concurrent collectives: buffers per worker warp (2..4)
    int coll_evict_first;              // concurrent collectives: bulk copies with an L2 evict-first policy
    int coll_path;                     // concurrent collectives: 1 TMA, 2 TMA loads + register stores,
                                       // 3 one 3-D TMA box per sub-chunk for all W sources
    int coll_box_rows;                 // coll_path 3: 1 KB rows per source in one box (R)
    int coll_out_stage;                // summing collectives: 0 staged for all-reduce, 1 in place, 2 staged
    int gather_parts;                  // all_gather_matmul: gather items (row parts) per (row block, shard)
    int gemm_evict_last;               // CTA-pair operand loads carry an L2 evict-last policy
    int out_evict_first;               // final 16-bit output stores carry an L2 evict-first policy
    int split;                         // split-K: K chunks per (rank's) output tile (0 / 1: none)
    int kb_chunk;                      // ... K blocks per chunk (a whole number of stages)
    unsigned long long* chain;         // ... chained-reduce tile counters (after the gather counters)
    int sum_l2_policy;                 // chained reduce running-sum stores / reduce-adds: 0 none,
                                       // 1 evict first, 2 evict last
    int startup_gather;                // all_gather_matmul: the TMA producer copies the gathers claimed
                                       // before its CTA's first GEMM item (TMA boxes through its idle stages)
    int gather_box;                    // ... columns per box
    int rank_inner;                    // reduce ops: 1 = rank index fastest in the GEMM item order
    unsigned long long* trace;         // optional per-CTA event trace (nullptr = off)
    int trace_cap;                     // events per (CTA, role)
};

// Optional timeline: each CTA owns 4 role streams (scheduler, MMA, TMA,
// workers) of trace_cap (event, globaltimer ns) pairs; slot 0 of a stream
// holds its event count.
enum : int { TR_SCHED = 0, TR_MMA = 1, TR_TMA = 2, TR_WORK = 3 };
// EV_KERNEL_BEGIN / EV_KERNEL_END (scheduler stream, thread 0 of every CTA):
// entry into the kernel and the end of its teardown
enum : unsigned long long { EV_CLAIM = 1, EV_BEGIN = 2, EV_END = 3, EV_READY = 4, EV_KERNEL_BEGIN = 5,
                            EV_KERNEL_END = 6 };
struct Tracer {
    unsigned long long* buf = nullptr;
    int cap = 0, n = 0;
    __device__ void init(const Params& p, int role) {
        if (p.trace && p.trace_cap > 1) {
            buf = p.trace + (static_cast<size_t>(blockIdx.x) * 4 + role) * p.trace_cap * 2;
            cap = p.trace_cap;
            n = 1;
        }
    }
    __device__ __forceinline__ void rec(unsigned long long ev, uint32_t item) {
        if (buf && n < cap) {
            buf[2 * n] = (ev << 56) | item;
            buf[2 * n + 1] = global_timer_ns();
            ++n;
        }
    }
    __device__ void finish() {
        if (buf) {
            buf[0] = static_cast<unsigned long long>(n - 1);
            buf[1] = 0;
        }
    }
};

struct Ctl {
    WsHeader* ws;
    uint32_t epoch;
    unsigned long long limit;
    int half;  // CTA-pair kernels: this CTA's rank in the pair (0 issues the MMAs); else 0
};

__device__ __forceinline__ bool launch_aborted(const Ctl& c) {
    return *reinterpret_cast<volatile uint32_t*>(&c.ws->abort_epoch) == c.epoch;
}

__device__ __noinline__ void raise_timeout(const Ctl& c, int where, int index) {
    if (atomicCAS(&c.ws->status, 0, DEV_TIMEOUT) == 0) {
        c.ws->err_where = where;
        c.ws->err_index = index;
    }
    __threadfence();
    atomicExch(&c.ws->abort_epoch, c.epoch);
}

// Epoch-tagged arrival counter (high 32 bits: launch epoch, low 32: count):
// returns this arrival's count within the current launch (1 = first).  A
// counter left by an earlier (or aborted) launch is restarted, so no per-launch
// reset is needed.  Lock-free: each failed CAS means another arrival succeeded.
__device__ __forceinline__ uint32_t arrive_count(unsigned long long* ctr, uint32_t epoch) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
    while (true) {
        const unsigned long long want = (static_cast<uint32_t>(cur >> 32) == epoch)
                                            ? cur + 1
                                            : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
        const unsigned long long prev = atomicCAS(ctr, cur, want);
        if (prev == cur) return static_cast<uint32_t>(want);
        cur = prev;
    }
}

// A gather copy counts itself into its (block, shard) ready counter.  With one
// copy per counter (gather_parts 1, the default) the counter is complete at
// the first arrival, so the copy publishes (epoch, 1) with one release store
// instead of a read and a compare-and-swap: two L2 round trips fewer on the
// path from the copy to the GEMM tiles that wait for it.
__device__ __forceinline__ void arrive_gather(const Params& p, unsigned long long* ctr, uint32_t epoch) {
    if (p.gather_parts == 1)
        st_release_gpu_u64(ctr, (static_cast<unsigned long long>(epoch) << 32) | 1ull);
    else
        arrive_count(ctr, epoch);
}

// Bounded wait on an mbarrier phase. false = gave up (timeout or abort).
// `cluster`: the barrier receives release-arrivals from the peer CTA of a
// pair, so the wait acquires at cluster scope.
__device__ __forceinline__ bool try_bar(uint64_t* bar, uint32_t parity, bool cluster) {
    return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}
__device__ __forceinline__ bool wait_bar(const Ctl& c, uint64_t* bar, uint32_t parity, int where,
                                         bool cluster = false) {
    if (try_bar(bar, parity, cluster)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_bar(bar, parity, cluster)) return true;
        if ((i & 15) == 0) {
            if (launch_aborted(c)) return false;
            if (global_timer_ns() - t0 > c.limit) {
                raise_timeout(c, where, -1);
                return false;
            }
        }
    }
}

// Bounded wait for a ready-flag to hold this launch's epoch (acquire).
__device__ __forceinline__ bool wait_flag(const Ctl& c, const uint32_t* flag, int where, int index) {
    if (ld_acquire_gpu(flag) == c.epoch) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (ld_acquire_gpu(flag) == c.epoch) return true;
        if ((i & 7) == 0) {
            if (launch_aborted(c)) return false;
            if (global_timer_ns() - t0 > c.limit) {
                raise_timeout(c, where, index);
                return false;
            }
        }
    }
}

// Bounded wait for a 64-bit counter to hold `want` (acquire).
__device__ __forceinline__ bool wait_count(const Ctl& c, const unsigned long long* ctr, unsigned long long want,
                                           int where, int index) {
    if (ld_acquire_gpu_u64(ctr) == want) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (ld_acquire_gpu_u64(ctr) == want) return true;
        if ((i & 7) == 0) {
            if (launch_aborted(c)) return false;
            if (global_timer_ns() - t0 > c.limit) {
                raise_timeout(c, where, index);
                return false;
            }
        }
    }
}

// Teardown wait: same as wait_bar but ignores the abort flag (the async work
// it waits for always completes); still bounded.
__device__ __forceinline__ bool drain_bar(const Ctl& c, uint64_t* bar, uint32_t parity, int where) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > c.limit) {
            raise_timeout(c, where, -1);
            return false;
        }
    }
    return true;
}

// Split-K (every fused op): each output tile's K range is cut into p.split
// chunks of p.kb_chunk K blocks; chunk j of a tile (of a rank) is a GEMM item
// of its own, and the partials are summed through the chained reduce, in
// (rank, chunk) order for the reduce ops and in chunk order otherwise, so the
// tiles running at once stay short and share their operand blocks in L2.
__device__ __forceinline__ bool split_k(const Params& p) { return p.split > 1; }
__device__ __forceinline__ bool reduce_op_of(const Params& p) { return p.op == OP_MM_RS || p.op == OP_MM_AR; }
// the links of a tile's reduce chain: W ranks (reduce ops) x the K chunks
__device__ __forceinline__ int chain_ranks(const Params& p) {
    return (reduce_op_of(p) ? p.W : 1) * max(1, p.split);
}

// GROUP_M swizzle: linear output-tile id -> (m block, n block).  Tiles run
// over groups of group_m m-blocks; inside a group the m index moves fastest so
// consecutive tiles share B columns and neighbouring A rows in L2.
__device__ __forceinline__ void swizzle_tile(const Params& p, uint32_t t, int& mb, int& nb) {
    const uint32_t group_size = static_cast<uint32_t>(p.group_m) * p.n_blocks;
    const uint32_t group = t / group_size;
    const int first_m = static_cast<int>(group) * p.group_m;
    const int gsz = min(p.m_blocks - first_m, p.group_m);
    const uint32_t local = t - group * group_size;
    mb = first_m + static_cast<int>(local % gsz);
    nb = static_cast<int>(local / gsz);
}

// The GEMM item -> (rank, m block, n block, output tile).
// Reduce ops run W GEMMs over the same output tiles.  By default the items of
// one GROUP_M swizzle group are ordered rank by rank (all of rank 0's tiles of
// the group, then rank 1's, ...), so the L2 holds one rank's A rows and B at a
// time; with rank_inner the rank index moves fastest instead.
struct GemmCoord {
    int rank, mb, nb;
    int chunk;  // split-K: the item's K chunk (0 when not split)
    int link;   // chained reduce: the item's place in its tile's chain, rank * split + chunk
    uint32_t tile;
    int hn;  // -1: the whole tile; 0 / 1: column half of a split tail tile
};
// GEMM items from g_split on are the column halves of the last tiles (the
// launch's final, partly empty wave split in two, so it takes half a tile's
// time): item g_split + 2i + h is half h of tile g_split + i.
__device__ __forceinline__ uint32_t tile_item(const Params& p, uint32_t g, int& hn) {
    if (g < p.g_split) {
        hn = -1;
        return g;
    }
    hn = static_cast<int>((g - p.g_split) & 1u);
    return p.g_split + ((g - p.g_split) >> 1);
}
__device__ __forceinline__ uint32_t group_tiles(const Params& p) {
    return static_cast<uint32_t>(p.group_m) * p.n_blocks;
}
__device__ __forceinline__ GemmCoord decode_gemm(const Params& p, uint32_t item) {
    GemmCoord gc;
    const uint32_t g = tile_item(p, item, gc.hn);
    if (p.op == OP_MM_RS || p.op == OP_MM_AR || split_k(p)) {
        const uint32_t R = static_cast<uint32_t>(chain_ranks(p));
        int link;
        if (p.rank_inner) {
            gc.tile = g / R;
            link = static_cast<int>(g % R);
        } else {
            const uint32_t T = group_tiles(p);
            const uint32_t sg = g / (T * R);
            const uint32_t Tsg = min(T, static_cast<uint32_t>(p.n_tiles) - sg * T);
            const uint32_t local = g - sg * T * R;
            link = static_cast<int>(local / Tsg);
            gc.tile = sg * T + (local - static_cast<uint32_t>(link) * Tsg);
        }
        const int S = max(1, p.split);
        gc.link = link;
        gc.chunk = link % S;
        gc.rank = reduce_op_of(p) ? link / S : 0;  // matmul_all_gather: set from the m-block below
    } else {
        gc.tile = g;
        gc.rank = 0;
        gc.chunk = 0;
        gc.link = 0;
    }
    swizzle_tile(p, gc.tile, gc.mb, gc.nb);
    if (p.op == OP_MM_AG) gc.rank = gc.mb / p.mb_per_rank;
    return gc;
}
// Inverse for the reduce ops: the GEMM item of (output tile t, rank s).
__device__ __forceinline__ uint32_t gemm_index(const Params& p, uint32_t t, int s) {
    if (p.rank_inner) return t * p.W + s;
    const uint32_t T = group_tiles(p);
    const uint32_t sg = t / T;
    const uint32_t Tsg = min(T, static_cast<uint32_t>(p.n_tiles) - sg * T);
    return sg * T * p.W + static_cast<uint32_t>(s) * Tsg + (t - sg * T);
}

// This CTA's block of BM rows inside GEMM item gc: an item's m-block spans CG
// such blocks, one per CTA of a pair.  matmul_all_gather counts blocks inside
// the item's rank; the other ops count them over all M rows.
template <int CG>
__device__ __forceinline__ int own_block(const Params& p, const GemmCoord& gc, int half) {
    const int mb = (p.op == OP_MM_AG) ? gc.mb % p.mb_per_rank : gc.mb;
    return mb * CG + half;
}

// all_gather_matmul gather items are numbered swizzle group by swizzle group
// (the groups of group_m m-blocks the GEMM order walks through) and, inside a
// group, shard-major, the p.gather_parts row parts of one (m-block, shard)
// consecutive: item = (first_m * W + s * gsz + (mb - first_m)) * parts + part.
// Parts let the copies of one shard spread over many CTAs, so the shards of
// a block land in order while its first tiles already run.
// Every m-block's shard 0 comes before any shard 1, so with the gathers
// spread over all CTAs the first K-blocks of the group's tiles arrive first.
struct GatherCoord {
    int mb, s, part;
};
__device__ __forceinline__ GatherCoord decode_gather(const Params& p, uint32_t c) {
    const uint32_t blk = c / static_cast<uint32_t>(p.gather_parts);  // (m-block, shard) copy
    const uint32_t per_group = static_cast<uint32_t>(p.group_m) * p.W;
    const int first_m = static_cast<int>(blk / per_group) * p.group_m;
    const int gsz = min(p.m_blocks - first_m, p.group_m);
    const int local = static_cast<int>(blk - static_cast<uint32_t>(first_m) * p.W);
    GatherCoord gc;
    gc.s = local / gsz;
    gc.mb = first_m + (local - gc.s * gsz);
    gc.part = static_cast<int>(c % static_cast<uint32_t>(p.gather_parts));
    return gc;
}

// Number of gather items that must be claimed before GEMM item x may be
// published: every item of the groups before x's, and in x's group the items
// up to shard W-1 of x's m-block (all its parts).  Inside a group the GEMM
// order first visits its m-blocks in order, so the need grows by one block
// per item there and stays at the whole group afterwards (monotonic in x).
__device__ __forceinline__ uint32_t gather_need(const Params& p, uint32_t x) {
    if (p.op == OP_AG_MM && split_k(p)) {
        // x is an item: chunk j of a tile of swizzle group sg; the chunk needs
        // the shards up to the one holding its last K block, and in the
        // group's shard-major numbering the gathers of earlier shards of
        // every m-block come first
        const uint32_t T = group_tiles(p), R = static_cast<uint32_t>(p.split);
        const uint32_t sg = x / (T * R);
        const uint32_t Tsg = min(T, static_cast<uint32_t>(p.n_tiles) - sg * T);
        const uint32_t local = x - sg * T * R;
        const int j = static_cast<int>(local / Tsg);
        const int t_local = static_cast<int>(local - static_cast<uint32_t>(j) * Tsg);
        const int first_m = static_cast<int>(sg) * p.group_m;
        const int gsz = min(p.m_blocks - first_m, p.group_m);
        const int kb_end = min(p.k_blocks, (j + 1) * p.kb_chunk);
        const int s_hi = min(p.W - 1, (kb_end * BK - 1) / p.K_local);
        return static_cast<uint32_t>(p.gather_parts) *
               (static_cast<uint32_t>(first_m) * p.W + static_cast<uint32_t>(s_hi * gsz + min(t_local, gsz - 1) + 1));
    }
    const uint32_t group_size = static_cast<uint32_t>(p.group_m) * p.n_blocks;
    const uint32_t group = x / group_size;
    const int first_m = static_cast<int>(group) * p.group_m;
    const int gsz = min(p.m_blocks - first_m, p.group_m);
    const int local = static_cast<int>(x - group * group_size);
    return static_cast<uint32_t>(p.gather_parts) * (static_cast<uint32_t>(first_m) * p.W +
                           static_cast<uint32_t>((p.W - 1) * gsz + min(local, gsz - 1) + 1));
}

// all_gather_matmul ready counters: one epoch-tagged 64-bit arrival counter
// per (128-row block, shard), complete when all its parts are in
__device__ __forceinline__ unsigned long long* gather_ctr(const Params& p, int fi) {
    return reinterpret_cast<unsigned long long*>(p.flags) + fi;
}
__device__ __forceinline__ unsigned long long gather_done(const Params& p, uint32_t epoch) {
    return (static_cast<unsigned long long>(epoch) << 32) | static_cast<uint32_t>(p.gather_parts);
}

__device__ __forceinline__ float bits16_to_float(uint32_t b, int bf16) {
    if (bf16) return __uint_as_float(b << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}
__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ============================================================ shared state
// CG = 2: the CTA pair computes a (2 BM) x BN tile; this CTA holds BM rows of
// A and BN / 2 columns of B per stage.
constexpr int SBARS = 4;  // per worker warp: running-sum loads (2) or collective buffers (1 to 4)
constexpr int MAX_COLL_RING = SBARS;

template <int BN, int STAGES, int CG>
struct Smem {
    static constexpr int KS = k_per_stage(CG, STAGES);  // K blocks per stage
    static constexpr uint32_t A_BYTES = BM * BK * KS * 2;  // KS chunks of 128 rows x 64 K, 16 KB apart
    static constexpr uint32_t B_BYTES = (BN / CG) * BK * KS * 2;  // 64-column chunks of 64 KS K rows
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TILES_BYTES = STAGES * STAGE_BYTES;
    static constexpr uint32_t STAGE_OUT_BYTES = 2 * 32 * 32 * 4;  // per worker warp: 2 x (32 rows x 32 fp32)
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * RING + 2 + SBARS * NUM_WORKER_WARPS + 3;
    static constexpr int READY_BITS = 4096;  // all_gather_matmul: m-blocks whose gathers this CTA has seen complete
    static constexpr uint32_t BYTES = 1024 /*align slack*/ + TILES_BYTES +
                                      NUM_WORKER_WARPS * STAGE_OUT_BYTES + NUM_BARS * 8 + (RING + 4) * 4 +
                                      READY_BITS / 8;
    uint8_t* tiles;
    uint8_t* stage_out;
    uint64_t *full, *empty, *acc_full, *acc_empty, *item_full, *item_empty, *wbar, *final_bar;
    uint64_t* sbar;  // per worker warp: SBARS barriers for running-sum / collective chunk loads
    uint64_t* lease;       // TMA producer -> workers: pipeline stages lent for a collective tile
    uint64_t* lease_done;  // workers -> TMA producer: stages returned
    uint64_t* gbar;        // TMA producer: its start-up gather loads
    volatile uint32_t* ring;
    uint32_t* tmem_slot;
    uint32_t* epoch_slot;
    uint32_t* ready_bits;

    __device__ void carve(uint8_t* raw) {
        uintptr_t a = reinterpret_cast<uintptr_t>(raw);
        a = (a + 1023) & ~static_cast<uintptr_t>(1023);
        tiles = reinterpret_cast<uint8_t*>(a);
        stage_out = tiles + TILES_BYTES;  // 1024-aligned: TILES_BYTES is a multiple of 1024
        uint64_t* b = reinterpret_cast<uint64_t*>(stage_out + NUM_WORKER_WARPS * STAGE_OUT_BYTES);
        full = b;
        empty = full + STAGES;
        acc_full = empty + STAGES;
        acc_empty = acc_full + 2;
        item_full = acc_empty + 2;
        item_empty = item_full + RING;
        wbar = item_empty + RING;
        final_bar = wbar + 1;
        sbar = final_bar + 1;
        lease = sbar + SBARS * NUM_WORKER_WARPS;
        lease_done = lease + 1;
        gbar = lease_done + 1;
        uint32_t* u = reinterpret_cast<uint32_t*>(gbar + 1);
        ring = u;
        tmem_slot = u + RING;
        epoch_slot = u + RING + 1;
        ready_bits = u + RING + 4;

    }
    __device__ uint8_t* a_tile(uint32_t s) const { return tiles + s * STAGE_BYTES; }
    __device__ uint8_t* b_tile(uint32_t s) const { return tiles + s * STAGE_BYTES + A_BYTES; }
};

// ============================================================ scheduler
// Claims work items from the two global queues and publishes them, in claim
// order, into the CTA's item ring.  An item is published only after every item
// it depends on has been claimed (by this or another CTA), so the ring order of
// every CTA is a topological order of the dependency graph and no CTA can wait
// on work that nobody will run.
template <int BN, int STAGES, int CG>
__device__ void run_scheduler(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, Tracer& tr) {
    uint32_t ring_n = 0;
    bool gemm_dry = (p.n_gemm == 0), comm_dry = (p.n_comm == 0);
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);
    const bool prefer_gemm = p.gemm_ctas < 0 || static_cast<int>(blockIdx.x) < p.gemm_ctas;

    // CTA pairs: the even CTA's scheduler feeds both CTAs' rings (the odd
    // CTA's consumers release slots on the even CTA's item_empty barriers)
    auto publish = [&](uint32_t item) -> bool {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        if (!wait_bar(ctl, &sm.item_empty[slot], (use & 1) ^ 1, WAIT_ITEM_EMPTY, CG == 2)) return false;
        sm.ring[slot] = item;
        if (CG == 2) {
            st_shared_cluster_u32(mapa_shared(const_cast<uint32_t*>(&sm.ring[slot]), 1), item);
            mbar_arrive_cluster(mapa_shared(&sm.item_full[slot], 1));
        }
        mbar_arrive(&sm.item_full[slot]);
        ++ring_n;
        tr.rec(EV_CLAIM, item);
        return true;
    };

    // all_gather_matmul start-up: before its first GEMM item every scheduler
    // claims an even share of the gathers the first wave of GEMM items needs,
    // so those copies run on all SMs at once instead of on the few CTAs whose
    // first items would otherwise have to claim them (gathers depend on
    // nothing, so claiming them first is always safe)
    bool first_gemm = true;
    auto take_first_share = [&]() -> bool {
        const uint32_t first_need = gather_need(p, min(p.first_wave, p.n_gemm) - 1);
        const uint32_t nsched = gridDim.x / CG;
        const uint32_t share = (first_need + nsched - 1) / nsched;
        for (uint32_t i = 0; i < share && !comm_dry; ++i) {
            if (ld_relaxed_gpu(&p.ws->comm_ctr) >= first_need) break;
            const uint32_t c = atomicAdd(&p.ws->comm_ctr, 1u);
            if (c >= p.n_comm) {
                comm_dry = true;
                break;
            }
            if (!publish(ITEM_COMM | c)) return false;
        }
        return true;
    };

    // Take one GEMM item (after claiming the gather items it depends on).
    auto take_gemm = [&](bool& got) -> bool {
        got = false;
        if (gemm_dry) return true;
        if (p.op == OP_AG_MM && first_gemm) {
            first_gemm = false;
            if (!take_first_share()) return false;
        }
        const uint32_t g = atomicAdd(&p.ws->gemm_ctr, 1u);
        if (g >= p.n_gemm) {
            gemm_dry = true;
            return true;
        }
        if (p.op == OP_AG_MM) {
            // gathers g itself needs are claimed before g (mandatory); gathers
            // for items up to `lookahead` (one swizzle group) ahead are claimed
            // at most GATHER_AHEAD per GEMM item, so the next group's gathers
            // spread over many CTAs and run in the background of the current
            // group's tiles instead of in a burst at the group boundary
            int hn_unused;
            const uint32_t need = gather_need(p, tile_item(p, g, hn_unused));
            const uint32_t need_ahead = gather_need(p, tile_item(p, min(g + p.lookahead, p.n_gemm - 1), hn_unused));
            int ahead = 0;
            while (!comm_dry) {
                const uint32_t head = ld_relaxed_gpu(&p.ws->comm_ctr);
                if (head >= need && (head >= need_ahead || ahead >= GATHER_AHEAD * p.gather_parts)) break;
                const uint32_t c = atomicAdd(&p.ws->comm_ctr, 1u);
                if (c >= p.n_comm) {
                    comm_dry = true;
                    break;
                }
                if (c >= need) ++ahead;
                if (!publish(ITEM_COMM | c)) return false;
            }
        }
        if (!publish(g)) return false;
        got = true;
        return true;
    };

    // Take one comm item.  Reduce ops: claim the GEMM items it depends on
    // first (help), or -- with only_if_ready -- take it only when all its
    // partials are already flagged (never blocks).
    auto take_comm = [&](bool& got, bool only_if_ready) -> bool {
        got = false;
        if (comm_dry) return true;
        if (reduce_op && only_if_ready) {
            const uint32_t c = ld_relaxed_gpu(&p.ws->comm_ctr);
            if (c >= p.n_comm) return true;
            if (ld_relaxed_gpu(&p.ws->gemm_ctr) < gemm_index(p, c, p.W - 1) + 1) return true;
            for (int s = 0; s < p.W; ++s)
                if (ld_relaxed_gpu(&p.flags[gemm_index(p, c, s)]) != ctl.epoch) return true;
            if (atomicCAS(&p.ws->comm_ctr, c, c + 1) != c) return true;
            if (!publish(ITEM_COMM | c)) return false;
            got = true;
            return true;
        }
        const uint32_t c = atomicAdd(&p.ws->comm_ctr, 1u);
        if (c >= p.n_comm) {
            comm_dry = true;
            return true;
        }
        if (reduce_op) {
            const uint32_t need = gemm_index(p, c, p.W - 1) + 1;
            while (!gemm_dry && ld_relaxed_gpu(&p.ws->gemm_ctr) < need) {
                const uint32_t g = atomicAdd(&p.ws->gemm_ctr, 1u);
                if (g >= p.n_gemm) {
                    gemm_dry = true;
                    break;
                }
                if (!publish(g)) return false;
            }
        }
        if (!publish(ITEM_COMM | c)) return false;
        got = true;
        return true;
    };

    bool ok = true;
    while (ok && !(gemm_dry && comm_dry)) {
        bool gemm_first = prefer_gemm;
        if (p.gemm_ctas < 0 && !comm_dry && !gemm_dry && !reduce_op && p.op != OP_AG_MM) {
            // balanced: keep the two queues' fractional progress equal
            const unsigned long long gc = min(ld_relaxed_gpu(&p.ws->gemm_ctr), p.n_gemm);
            const unsigned long long cc = min(ld_relaxed_gpu(&p.ws->comm_ctr), p.n_comm);
            gemm_first = gc * p.n_comm <= cc * p.n_gemm;
        }
        bool got = false;
        if (reduce_op && gemm_first && !gemm_dry) {
            ok = take_comm(got, true);
            if (!ok) break;
        }
        if (gemm_first) {
            ok = take_gemm(got);
            if (ok && !got) ok = take_comm(got, false);
        } else {
            ok = take_comm(got, false);
            if (ok && !got) ok = take_gemm(got);
        }
    }
    if (ok) publish(ITEM_END);
}

// A consumer is done with ring slot `slot` (CTA pairs: the even CTA's
// item_empty barrier counts the consumers of both CTAs).
template <int BN, int STAGES, int CG>
__device__ __forceinline__ void release_item(Smem<BN, STAGES, CG>& sm, uint32_t slot) {
    if (CG == 2)
        mbar_arrive_cluster(mapa_shared(&sm.item_empty[slot], 0));
    else
        mbar_arrive(&sm.item_empty[slot]);
}

// all_gather_matmul start-up gather, run by the TMA producer (startup_gather):
// the gathers a CTA pair claims before its first GEMM item arrive while its
// pipeline stages are still idle, so the producer copies this CTA's 128 rows
// of (m-block, shard) with TMA boxes of gather_box columns (up to 64 KB each)
// through the stages -- as many boxes in flight as the stages hold -- instead
// of leaving them to the worker threads' 16-byte copies.  Then the stores
// complete, the proxy fence orders them before the release, and the copy
// counts itself into the block's ready counter.
template <int BN, int STAGES, int CG>
__device__ bool tma_gather(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t c,
                           uint32_t& gphase) {
    const GatherCoord gq = decode_gather(p, c);
    const int mb = gq.mb * CG + ctl.half, s = gq.s;
    if (mb * BM >= p.M) return true;  // below the last row: nothing to copy, no consumer
    const uint32_t box_bytes = static_cast<uint32_t>(p.gather_box) * 2u * BM;
    const int slots = static_cast<int>(Smem<BN, STAGES, CG>::TILES_BYTES / box_bytes);
    const int nbox = p.K_local / p.gather_box;
    bool ok = true;
    for (int j0 = 0; j0 < nbox && ok; j0 += slots) {
        const int nb = min(slots, nbox - j0);
        // rows past M read as zeros and are not stored
        mbar_arrive_expect_tx(sm.gbar, box_bytes * static_cast<uint32_t>(nb));
        for (int j = 0; j < nb; ++j)
            tma_load_3d(sm.tiles + j * box_bytes, &p.tmGs, (j0 + j) * p.gather_box, mb * BM, s, sm.gbar);
        ok = wait_bar(ctl, sm.gbar, gphase, WAIT_GATHER_TMA);
        if (!ok) drain_bar(ctl, sm.gbar, gphase, WAIT_GATHER_TMA);  // the loads land before the stages are reused
        gphase ^= 1u;
        if (!ok) break;
        for (int j = 0; j < nb; ++j)
            tma_store_3d(&p.tmGd, sm.tiles + j * box_bytes, s * p.K_local + (j0 + j) * p.gather_box, mb * BM, 0);
        bulk_commit();
        bulk_wait_read_all();  // the next boxes (or the GEMM's loads) may overwrite the stages
    }
    bulk_wait_all();
    if (!ok) return false;
    fence_proxy_async_global();
    if (p.gather_parts != 1) __threadfence();  // the release store of one copy per counter orders the rest
    const uint32_t fi = static_cast<uint32_t>(mb * p.W + s);
    if (p.debug_skip != fi + 1) arrive_gather(p, gather_ctr(p, static_cast<int>(fi)), ctl.epoch);
    return true;
}

// ============================================================ TMA producer
// Follows the item ring; for every GEMM item streams its K-blocks of A and B
// into the STAGES-deep shared-memory pipeline (acquiring the gather flags of
// all_gather_matmul shards just before their first K-block).
template <int BN, int STAGES, int CG>
__device__ void run_tma(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm) {
    Tracer tr;
    tr.init(p, TR_TMA);
    uint32_t stage = 0, phase = 0, ring_n = 0;
    uint32_t issued_phase[STAGES];
    uint32_t used_mask = 0;
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);
    const uint64_t pol = p.gemm_evict_last ? l2_policy_evict_last() : 0ull;

    auto load_gemm = [&](uint32_t g) -> bool {
        const GemmCoord gc = decode_gemm(p, g);
        const int blk = own_block<CG>(p, gc, ctl.half);
        const int a_row = blk * BM;
        const int a_rank = (p.op == OP_MM_AG || reduce_op) ? gc.rank : 0;
        const int b_rank = reduce_op ? gc.rank : 0;
        int acquired = 0;  // all_gather_matmul: shards whose flags are held
        if (p.op == OP_AG_MM && a_row >= p.M) {
            acquired = p.W;  // this CTA's half of a pair tile lies below the last row: no gathers
        } else if (p.op == OP_AG_MM) {
            // an m-block seen complete before needs no flag traffic; else check
            // all W shard flags at once and take the per-shard waits below
            // only for the shards still missing
            const bool cacheable = gc.mb < Smem<BN, STAGES, CG>::READY_BITS;
            if (cacheable && (sm.ready_bits[gc.mb >> 5] >> (gc.mb & 31) & 1u)) {
                acquired = p.W;
            } else {
                // W relaxed loads in flight at once (acquire loads would run one
                // after another), then one acquire fence if all were complete
                uint32_t seen = 0;
                for (int s = 0; s < p.W; ++s)
                    seen += ld_relaxed_gpu_u64(gather_ctr(p, blk * p.W + s)) == gather_done(p, ctl.epoch) ? 1u : 0u;
                if (seen == static_cast<uint32_t>(p.W)) {
                    fence_acq_rel_gpu();
                    acquired = p.W;
                    fence_proxy_async_global();
                    if (cacheable) sm.ready_bits[gc.mb >> 5] |= 1u << (gc.mb & 31);
                }
            }
        }
        constexpr int KS = Smem<BN, STAGES, CG>::KS;
        // split-K: this item's chunk of the K blocks
        const int kb_lo = split_k(p) ? gc.chunk * p.kb_chunk : 0;
        const int kb_hi = split_k(p) ? min(p.k_blocks, kb_lo + p.kb_chunk) : p.k_blocks;
        for (int kb = kb_lo; kb < kb_hi; kb += KS) {
            if (!wait_bar(ctl, &sm.empty[stage], phase ^ 1, WAIT_SMEM_EMPTY)) return false;
            // B first: it depends on no gather, so its loads are in flight
            // while this stage's A shards may still be on their way
            constexpr uint32_t HALF_BYTES = Smem<BN, STAGES, CG>::A_BYTES + Smem<BN, STAGES, CG>::B_BYTES / 2;
            const bool hn = gc.hn >= 0;
            const uint32_t fb = CG == 2 ? mapa_shared(&sm.full[stage], 0) : 0u;
            if (CG == 1) {
                mbar_arrive_expect_tx(&sm.full[stage], Smem<BN, STAGES, CG>::STAGE_BYTES);
                if (p.b_chunked) {
                    tma_load_4d(sm.b_tile(stage), &p.tmBc, 0, kb * BK, gc.nb * (BN / 64), b_rank, &sm.full[stage]);
                } else {
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_3d(sm.b_tile(stage) + c * (64 * BK * 2), &p.tmB, gc.nb * BN + c * 64,
                                    kb * BK, b_rank, &sm.full[stage]);
                }
            } else {
                // both CTAs' boxes count on the even CTA's full barrier, which
                // expects the pair's bytes (the odd CTA's may land first: the
                // transaction count may dip below zero inside a phase).  A
                // column half (N = BN / 2) loads one 64-column box per CTA.
                if (ctl.half == 0)
                    mbar_arrive_expect_tx(&sm.full[stage], (hn ? HALF_BYTES : Smem<BN, STAGES, CG>::STAGE_BYTES) * CG);
                // B: 64-column chunks of KS x 64 K rows, 64 KS x 128 B apart
                const int bcol = gc.nb * BN + (hn ? gc.hn * (BN / 2) + ctl.half * (BN / 4) : ctl.half * (BN / CG));
                if (p.b_chunked && !hn) {
                    // the CTA's BN / CG columns as one box of 64-column chunks
                    if (p.gemm_evict_last)
                        tma_load_4d_pair_hint(sm.b_tile(stage), &p.tmBc, 0, kb * BK, bcol / 64, b_rank, fb, pol);
                    else
                        tma_load_4d_pair(sm.b_tile(stage), &p.tmBc, 0, kb * BK, bcol / 64, b_rank, fb);
                } else {
                    const int nbox = hn ? BN / 4 / 64 : BN / CG / 64;
                    for (int c = 0; c < nbox; ++c) {
                        if (p.gemm_evict_last)
                            tma_load_3d_pair_hint(sm.b_tile(stage) + c * (64 * BK * KS * 2), &p.tmB, bcol + c * 64,
                                                  kb * BK, b_rank, fb, pol);
                        else
                            tma_load_3d_pair(sm.b_tile(stage) + c * (64 * BK * KS * 2), &p.tmB, bcol + c * 64, kb * BK,
                                             b_rank, fb);
                    }
                }
            }
            // all_gather_matmul: the shards this stage's A rows come from
            bool flags_ok = true;
            if (p.op == OP_AG_MM && acquired < p.W) {
                const int s_hi = min(p.W - 1, ((kb + KS) * BK - 1) / p.K_local);
                if (s_hi >= acquired) {
                    for (int s = acquired; s <= s_hi && flags_ok; ++s) {
                        const int fi = blk * p.W + s;
                        flags_ok = wait_count(ctl, gather_ctr(p, fi), gather_done(p, ctl.epoch), WAIT_FLAG_GATHER, fi);
                    }
                    if (flags_ok) {
                        acquired = s_hi + 1;
                        fence_proxy_async_global();
                        if (acquired == p.W && gc.mb < Smem<BN, STAGES, CG>::READY_BITS)
                            sm.ready_bits[gc.mb >> 5] |= 1u << (gc.mb & 31);
                    }
                }
            }
            // A (issued even when a wait gave up, so that the stage's
            // transaction completes before the CTA stops; the launch is
            // aborting then and its results are discarded)
            if (CG == 1) {
                tma_load_3d(sm.a_tile(stage), &p.tmA, kb * BK, a_row, a_rank, &sm.full[stage]);
            } else if (p.a_chunked) {
                // the stage's KS K-chunks of this CTA's 128 rows, 16 KB apart
                if (p.gemm_evict_last) tma_load_4d_pair_hint(sm.a_tile(stage), &p.tmAc, 0, a_row, kb, a_rank, fb, pol);
                else tma_load_4d_pair(sm.a_tile(stage), &p.tmAc, 0, a_row, kb, a_rank, fb);
            } else {
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    if (p.gemm_evict_last)
                        tma_load_3d_pair_hint(sm.a_tile(stage) + j * (BM * BK * 2), &p.tmA, (kb + j) * BK, a_row,
                                              a_rank, fb, pol);
                    else
                        tma_load_3d_pair(sm.a_tile(stage) + j * (BM * BK * 2), &p.tmA, (kb + j) * BK, a_row, a_rank,
                                         fb);
                }
            }
            issued_phase[stage] = phase;
            used_mask |= 1u << stage;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
            if (!flags_ok) return false;
        }
        return true;
    };

    uint32_t leases = 0;
    bool seen_gemm = false;  // a GEMM item has passed (start-up gathers are the comm items before it)
    uint32_t gphase = 0;
    while (true) {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        if (!wait_bar(ctl, &sm.item_full[slot], use & 1, WAIT_ITEM_FULL_TMA, CG == 2)) break;
        const uint32_t item = sm.ring[slot];
        release_item(sm, slot);
        ++ring_n;
        if (item == ITEM_END) break;
        if (item & ITEM_COMM) {
            if (p.op == OP_AG_MM && p.startup_gather && !seen_gemm) {
                if (!tma_gather(p, ctl, sm, item & ~ITEM_COMM, gphase)) break;
                continue;
            }
            if (p.op != OP_CONC) continue;
            // lend the pipeline stages to the workers for this collective
            // tile: every load issued so far must have been consumed first
            bool ok = true;
            for (int s = 0; s < STAGES && ok; ++s)
                if (used_mask & (1u << s)) ok = wait_bar(ctl, &sm.empty[s], issued_phase[s], WAIT_DRAIN);
            if (!ok) break;
            mbar_arrive(sm.lease);
            if (!wait_bar(ctl, sm.lease_done, leases & 1, WAIT_LEASE_DONE)) break;
            ++leases;
            continue;
        }
        seen_gemm = true;
        tr.rec(EV_BEGIN, item);
        if (!load_gemm(item)) break;
        tr.rec(EV_END, item);
    }
    tr.finish();
    // drain: every TMA load issued into a stage has landed before the CTA
    // exits.  The odd CTA of a pair cannot wait on the even CTA's full
    // barrier; it waits until the MMA has consumed its last fill of each stage.
    for (int s = 0; s < STAGES; ++s)
        if (used_mask & (1u << s))
            drain_bar(ctl, ctl.half ? &sm.empty[s] : &sm.full[s], issued_phase[s], WAIT_TEARDOWN_TMA);
}

// ============================================================ MMA issuer
template <int BN, int STAGES, int CG>
__device__ void run_mma(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t tmem) {
    // CTA pairs: one instruction covers the pair's (2 BM) x BN tile (x BN/2
    // for the column half of a split tail tile)
    constexpr uint32_t IDESC_F16 = make_idesc(0, BM * CG, BN);
    constexpr uint32_t IDESC_BF16 = make_idesc(1, BM * CG, BN);
    constexpr uint32_t IDESC_F16_H = make_idesc(0, BM * CG, BN / 2);
    constexpr uint32_t IDESC_BF16_H = make_idesc(1, BM * CG, BN / 2);
    Tracer tr;
    tr.init(p, TR_MMA);
    uint32_t stage = 0, phase = 0, ring_n = 0, acc_i = 0;
    while (true) {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        if (!wait_bar(ctl, &sm.item_full[slot], use & 1, WAIT_ITEM_FULL_MMA)) break;
        const uint32_t item = sm.ring[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++ring_n;
        if (item == ITEM_END) break;
        if (item & ITEM_COMM) continue;
        const uint32_t buf = acc_i & 1, ause = acc_i >> 1;
        int hn;
        tile_item(p, item, hn);
        const uint32_t idesc = hn >= 0 ? (p.bf16 ? IDESC_BF16_H : IDESC_F16_H) : (p.bf16 ? IDESC_BF16 : IDESC_F16);
        // CTA pairs: the workers of both CTAs release the accumulator here
        if (!wait_bar(ctl, &sm.acc_empty[buf], (ause & 1) ^ 1, WAIT_ACC_EMPTY, CG == 2)) break;
        tc_fence_after();
        tr.rec(EV_BEGIN, item);
        const uint32_t d = tmem + buf * BN;
        bool ok = true;
        constexpr int KS = Smem<BN, STAGES, CG>::KS;
        // split-K: this item's chunk of the K blocks (the producer's range)
        int kb_lo = 0, kb_hi = p.k_blocks;
        if (split_k(p)) {
            kb_lo = decode_gemm(p, item).chunk * p.kb_chunk;
            kb_hi = min(p.k_blocks, kb_lo + p.kb_chunk);
        }
        for (int kb = kb_lo; kb < kb_hi; kb += KS) {
            if (!wait_bar(ctl, &sm.full[stage], phase, WAIT_SMEM_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // A: K-major, 128-byte swizzle, 8-row core groups 1024 B apart;
            //    K-chunk j of the stage 16 KB further.
            // B: MN-major, 128-byte swizzle: 64-column chunks 64 KS x 128 B
            //    apart (leading offset), 8-row K groups 1024 B apart (stride
            //    offset); K-chunk j starts 64 rows (8 KB) further.
            const uint32_t a_addr = smem_u32(sm.a_tile(stage));
            const uint64_t bdesc = smem_desc(smem_u32(sm.b_tile(stage)), 64 * BK * KS * 2, 1024);
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                if (kb + j >= kb_hi) break;  // K tail: the chunk past K holds zeros
                const uint64_t adesc = smem_desc(a_addr + j * (BM * BK * 2), 16, 1024);
#pragma unroll
                for (int k = 0; k < BK / UMMA_K; ++k) {
                    // advance A by 16 columns (32 B inside the swizzled row) and
                    // B by 16 rows (2 KB); descriptors hold addresses >> 4
                    umma_f16<CG>(d, adesc + static_cast<uint64_t>(k * 2),
                                 bdesc + static_cast<uint64_t>((j * (BK / UMMA_K) + k) * 128), idesc,
                                 ((kb - kb_lo) | j | k) != 0 ? 1u : 0u);
                }
            }
            // the stage is free again in both CTAs of a pair
            if (CG == 2)
                umma_commit_pair_both(&sm.empty[stage]);
            else
                umma_commit<1>(&sm.empty[stage]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok) break;
        if (CG == 2)
            umma_commit_pair_both(&sm.acc_full[buf]);
        else
            umma_commit<1>(&sm.acc_full[buf]);
        tr.rec(EV_END, item);
        ++acc_i;
    }
    tr.finish();
    // drain: every MMA issued by this thread has completed
    umma_commit<CG>(sm.final_bar);
    drain_bar(ctl, sm.final_bar, 0, WAIT_TEARDOWN_MMA);
}

// ============================================================ workers
struct WorkerCtx {
    int w;      // worker warp index
    int lane;
    int q;      // TMEM lane quarter of this warp (warp id % 4)
    int h;      // column slice of the accumulator this warp drains
    uint32_t wphase;
    uint32_t sphase;  // parity bits of this warp's two running-sum load barriers
};

template <int BN, int STAGES, int CG>
__device__ __noinline__ void reduce_body(const Params& p, uint32_t c, WorkerCtx& wc);

// Distributed reduce (reduce ops, reduce_mode 2).  Output tile t is cut into W
// row parts (part s = rows [s*rows/W, (s+1)*rows/W)); part i = t*W + s sits in
// one global queue.  A worker warp with nothing else to do takes the next part
// (fetch-and-add), and reduces its rows one at a time once tile t's arrival
// counter shows all W partials; until then it keeps doing its own GEMM work.
// No warp ever waits on work that another warp holds, and the reduce spreads
// over every SM with idle workers.
struct PartState {
    uint32_t cur;   // claimed part, or NO_PART
    int row;        // next row of it
    bool ready;     // its tile has all W partials
};
constexpr uint32_t NO_PART = 0xFFFFFFFFu;

// Output row r (inside tile mb, nb) of the rank-order reduce: the loads of
// up to SC ranks are issued before their adds.
template <int BN>
__device__ __forceinline__ void reduce_row(const Params& p, int mb, int nb, int r, int rows, WorkerCtx& wc) {
    constexpr int CPL = BN / 4 / 32;
    constexpr int SC = 4;
    constexpr int RU = 1;
    const int cols = min(BN, p.N - nb * BN);
    const size_t pe = p.partial_elems;
    const float* src0 = p.partials + static_cast<size_t>(mb * BM + r) * p.N + nb * BN;
    float4 acc[RU][CPL];
    for (int s0 = 0; s0 < p.W; s0 += SC) {
        float4 v[SC][RU][CPL];
#pragma unroll
        for (int ds = 0; ds < SC; ++ds)
#pragma unroll
            for (int u = 0; u < RU; ++u)
#pragma unroll
                for (int k = 0; k < CPL; ++k)
                    if (s0 + ds < p.W && r + u * NUM_WORKER_WARPS < rows && (wc.lane + 32 * k) * 4 < cols)
                        v[ds][u][k] = __ldcg(reinterpret_cast<const float4*>(
                                                 src0 + static_cast<size_t>(s0 + ds) * pe +
                                                 static_cast<size_t>(u * NUM_WORKER_WARPS) * p.N) +
                                             wc.lane + 32 * k);
#pragma unroll
        for (int ds = 0; ds < SC; ++ds)
#pragma unroll
            for (int u = 0; u < RU; ++u)
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    if (s0 + ds == 0) {
                        acc[u][k] = v[0][u][k];
                    } else if (s0 + ds < p.W) {
                        acc[u][k].x = acc[u][k].x + v[ds][u][k].x;
                        acc[u][k].y = acc[u][k].y + v[ds][u][k].y;
                        acc[u][k].z = acc[u][k].z + v[ds][u][k].z;
                        acc[u][k].w = acc[u][k].w + v[ds][u][k].w;
                    }
                }
    }
    const int nreg = (p.op == OP_MM_AR && p.replicate) ? p.W : 1;
#pragma unroll
    for (int u = 0; u < RU; ++u) {
        const int rr_row = r + u * NUM_WORKER_WARPS;
        if (rr_row >= rows) continue;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int c4 = wc.lane + 32 * k;
            if (c4 * 4 >= cols) continue;
            const int j = nb * BN + c4 * 4;
            size_t off;
            if (p.op == OP_MM_RS) {
                const int rr = j / p.N_local;
                off = static_cast<size_t>(rr) * p.rank_stride + p.off_out +
                      (static_cast<size_t>(mb * BM + rr_row) * p.N_local + (j - rr * p.N_local)) * 2;
            } else {
                off = p.off_out + (static_cast<size_t>(mb * BM + rr_row) * p.N + j) * 2;
            }
            uint2 o;
            o.x = pack2(acc[u][k].x, acc[u][k].y, p.bf16);
            o.y = pack2(acc[u][k].z, acc[u][k].w, p.bf16);
            for (int rg = 0; rg < nreg; ++rg)
                *reinterpret_cast<uint2*>(p.heap + static_cast<size_t>(rg) * p.rank_stride + off) = o;
        }
    }
}

__device__ __forceinline__ bool tile_ready(const Params& p, uint32_t epoch, uint32_t t) {
    const unsigned long long v =
        *reinterpret_cast<volatile unsigned long long*>(reinterpret_cast<unsigned long long*>(p.flags) + t);
    return v == ((static_cast<unsigned long long>(epoch) << 32) | static_cast<uint32_t>(p.W));
}

// One row of reduce work for this warp: continue the claimed part, or claim
// the head part if its tile is complete.  false = nothing to do right now.
template <int BN>
__device__ __noinline__ bool part_step(const Params& p, uint32_t epoch, PartState& ps, WorkerCtx& wc) {
    if (p.n_parts == 0) return false;
    if (ps.cur == NO_PART) {
        uint32_t got = NO_PART;
        if (wc.lane == 0 && ld_relaxed_gpu(&p.ws->part_ctr) < p.n_parts) {
            const uint32_t i = atomicAdd(&p.ws->part_ctr, 1u);
            if (i < p.n_parts) got = i;
        }
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (got == NO_PART) return false;
        ps.cur = got;
        ps.row = 0;
        ps.ready = false;
    }
    if (!ps.ready) {
        int rdy = 0;
        if (wc.lane == 0) rdy = tile_ready(p, epoch, ps.cur / p.W) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, rdy, 0)) return false;
        __threadfence();  // acquire side of the arrival-counter protocol
        ps.ready = true;
    }
    const uint32_t t = ps.cur / p.W;
    const int part = static_cast<int>(ps.cur % p.W);
    int mb, nb;
    swizzle_tile(p, t, mb, nb);
    const int rows = min(BM, p.M - mb * BM);
    const int lo = part * rows / p.W, hi = (part + 1) * rows / p.W;
    if (lo + ps.row < hi) reduce_row<BN>(p, mb, nb, lo + ps.row, hi, wc);
    ps.row += 1;
    if (lo + ps.row >= hi) ps.cur = NO_PART;
    return true;
}

// true once every part has been claimed and this warp holds none
__device__ __forceinline__ bool parts_done(const Params& p, const PartState& ps) {
    return ps.cur == NO_PART && ld_relaxed_gpu(&p.ws->part_ctr) >= p.n_parts;
}

// Bounded wait on an mbarrier phase that does reduce rows while the phase is
// not complete (warp-uniform: lane 0 polls).
template <int BN>
__device__ bool wait_bar_working(const Params& p, const Ctl& c, uint64_t* bar, uint32_t parity, int where,
                                 PartState& ps, WorkerCtx& wc, bool cluster = false) {
    uint64_t t0 = 0;
    bool timing = false;
    for (uint32_t i = 0;; ++i) {
        int ready = 0;
        if (wc.lane == 0) ready = try_bar(bar, parity, cluster) ? 1 : 0;
        if (__shfl_sync(0xFFFFFFFFu, ready, 0)) return true;
        if (part_step<BN>(p, c.epoch, ps, wc)) {
            timing = false;  // progress: restart the idle clock
            continue;
        }
        if (!timing) {
            t0 = global_timer_ns();
            timing = true;
        }
        if ((i & 15) == 0) {
            if (launch_aborted(c)) return false;
            if (global_timer_ns() - t0 > c.limit) {
                if (wc.lane == 0) raise_timeout(c, where, -1);
                return false;
            }
        }
    }
}

// barrier over the worker warps built on an mbarrier (bounded, abortable)
template <int BN, int STAGES, int CG>
__device__ __forceinline__ bool worker_sync(const Ctl& ctl, Smem<BN, STAGES, CG>& sm, WorkerCtx& wc) {
    __syncwarp();
    bool ok = true;
    if (wc.lane == 0) {
        mbar_arrive(sm.wbar);
        ok = wait_bar(ctl, sm.wbar, wc.wphase, WAIT_WORKER_SYNC);
    }
    wc.wphase ^= 1;
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// This warp has read its accumulator slice (CTA pairs: the even CTA's
// acc_empty barrier counts the worker warps of both CTAs).
template <int BN, int STAGES, int CG>
__device__ __forceinline__ void release_acc(Smem<BN, STAGES, CG>& sm, uint32_t buf) {
    if (CG == 2)
        mbar_arrive_cluster(mapa_shared(&sm.acc_empty[buf], 0));
    else
        mbar_arrive(&sm.acc_empty[buf]);
}

// GEMM epilogue of one tile: TMEM -> registers -> (+bias) -> global.
template <int BN, int STAGES, int CG>
__device__ bool epilogue(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t tmem,
                         uint32_t g, uint32_t acc_i, WorkerCtx& wc, Tracer& tr, PartState& ps) {
    const uint32_t buf = acc_i & 1, ause = acc_i >> 1;
    const GemmCoord gc = decode_gemm(p, g);
    const int blk = own_block<CG>(p, gc, ctl.half);
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);
    constexpr int COLS = BN * 4 / NUM_WORKER_WARPS;  // accumulator columns this warp drains
    // a column half of a split tail tile drains BN/2 columns, offset by coff;
    // CTA pairs: nothing to store when this CTA's half lies below the last row
    // (the accumulator is still released after acc_full, in step with the pair)
    const int coff = gc.hn >= 0 ? gc.hn * (BN / 2) : 0;
    const int colbase = gc.nb * BN + coff + wc.h * COLS;
    const int cols_end = (CG == 2 && blk * BM >= p.M) ? 0 : (gc.hn >= 0 ? COLS / 2 : COLS);
    const char* bias_base = nullptr;
    if (p.has_bias) {
        const int bias_region = reduce_op ? gc.rank : 0;
        bias_base = p.heap + static_cast<size_t>(bias_region) * p.rank_stride + p.off_bias;
    }
    // per-column bias of the warp's columns, fetched while the MMAs still run:
    // lane l holds the 8 values of columns colbase + 8l .. 8l + 7
    uint4 bias8 = make_uint4(0u, 0u, 0u, 0u);
    if (p.has_bias && !p.bias_on_m && wc.lane * 8 < cols_end && colbase + wc.lane * 8 < p.N)
        bias8 = *reinterpret_cast<const uint4*>(bias_base + static_cast<size_t>(colbase + wc.lane * 8) * 2);

    if (!wait_bar_working<BN>(p, ctl, &sm.acc_full[buf], ause & 1, WAIT_ACC_FULL, ps, wc)) return false;
    tc_fence_after();
    tr.rec(EV_READY, g);

    const int r_in_tile = wc.q * 32 + wc.lane;
    // output row of this thread and whether it exists
    int row;        // row inside the op's output (or partial)
    int bias_row;   // index into a per-row bias
    bool row_ok;
    if (p.op == OP_MM_AG) {
        const int lrow = blk * BM + r_in_tile;
        row_ok = lrow < p.M;
        row = gc.rank * p.M + lrow;
        bias_row = lrow;
    } else {
        row = blk * BM + r_in_tile;
        row_ok = row < p.M;
        bias_row = row;
    }
    (void)row;
    float row_bias = 0.f;
    if (p.has_bias && p.bias_on_m && row_ok)
        row_bias = bits16_to_float(reinterpret_cast<const uint16_t*>(bias_base)[bias_row], p.bf16);

    const uint32_t tbase = tmem + (static_cast<uint32_t>(wc.q * 32) << 16) + buf * BN + wc.h * COLS;
    // Each 32 x 32 chunk (the warp's 32 rows, one per lane) goes registers ->
    // swizzled shared-memory staging -> TMA tensor store, so global memory
    // sees whole 128-byte lines instead of 16-byte pieces of 32 rows.  The
    // warp's 8 KB staging area rotates over 4 buffers (16-bit chunks, 2 KB)
    // or 2 (fp32 chunks, 4 KB), so a chunk waits only for the store issued
    // that many chunks earlier.
    uint8_t* stg_base = sm.stage_out + wc.w * Smem<BN, STAGES, CG>::STAGE_OUT_BYTES;
    const uint32_t chunk_bytes = reduce_op ? 32 * 32 * 4 : 32 * 32 * 2;
    const uint32_t nbuf = Smem<BN, STAGES, CG>::STAGE_OUT_BYTES / chunk_bytes;
    // TMA coordinates of the warp's 32-row slab
    const int c_row = blk * BM + wc.q * 32;
    int c_blk, c_reg_lo = 0, c_reg_hi = 1;
    if (reduce_op) {
        c_blk = gc.rank;
    } else if (p.op == OP_MM_AG) {
        c_blk = gc.rank;
        if (p.replicate) c_reg_hi = p.W;
    } else {
        c_blk = 0;
        if (p.replicate && p.op == OP_AG_MM) c_reg_hi = p.W;
    }
    // final 16-bit outputs are not read again: evict first (fp32 partials are)
    const bool out_hint = p.out_evict_first && !reduce_op;
    const uint64_t opol = out_hint ? l2_policy_evict_first() : 0ull;
    uint32_t ci = 0;
#pragma unroll 1
    for (int cc = 0; cc < cols_end; cc += 32, ++ci) {
        uint32_t r[32];
        if (p.k_blocks > 0) {
            tmem_ld_32x32b_x32(tbase + cc, r);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        const int col0 = colbase + cc;
        if (col0 >= p.N) continue;  // whole chunk right of the matrix (warp-uniform; so are all later ones)
        uint8_t* stg = stg_base + (ci % nbuf) * chunk_bytes;
        // the store issued nbuf chunks ago (from this buffer) must have read it
        if (wc.lane == 0) {
            if (reduce_op) bulk_wait_read<1>();
            else bulk_wait_read<3>();
        }
        __syncwarp();
#pragma unroll
        for (int v = 0; v < 4; ++v) {  // 8 columns at a time: +bias, then into the staging row
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(r[v * 8 + i]);
            if (p.has_bias) {
                if (p.bias_on_m) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = x[i] + row_bias;
                } else {
                    const int src = (cc >> 3) + v;  // the lane holding columns col0 + 8v ..
                    const uint32_t bw[4] = {__shfl_sync(0xFFFFFFFFu, bias8.x, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.y, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.z, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.w, src)};
                    if (col0 + v * 8 < p.N) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            x[2 * i] = x[2 * i] + bits16_to_float(bw[i] & 0xFFFFu, p.bf16);
                            x[2 * i + 1] = x[2 * i + 1] + bits16_to_float(bw[i] >> 16, p.bf16);
                        }
                    }
                }
            }
            if (reduce_op) {
                // fp32 row = 8 chunks of 16 B; chunk index XOR (row % 8) (128-byte swizzle)
                const int c0 = 2 * v, c1 = 2 * v + 1;
                *reinterpret_cast<float4*>(stg + wc.lane * 128 + ((c0 ^ (wc.lane & 7)) << 4)) =
                    make_float4(x[0], x[1], x[2], x[3]);
                *reinterpret_cast<float4*>(stg + wc.lane * 128 + ((c1 ^ (wc.lane & 7)) << 4)) =
                    make_float4(x[4], x[5], x[6], x[7]);
            } else {
                // 16-bit row = 4 chunks of 16 B; chunk index XOR ((row / 2) % 4) (64-byte swizzle)
                uint4 o;
                o.x = pack2(x[0], x[1], p.bf16);
                o.y = pack2(x[2], x[3], p.bf16);
                o.z = pack2(x[4], x[5], p.bf16);
                o.w = pack2(x[6], x[7], p.bf16);
                *reinterpret_cast<uint4*>(stg + wc.lane * 64 + ((v ^ ((wc.lane >> 1) & 3)) << 4)) = o;
            }
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (wc.lane == 0) {
            if (out_hint) {
                for (int rg = c_reg_lo; rg < c_reg_hi; ++rg) tma_store_4d_hint(&p.tmC, stg, col0, c_row, c_blk, rg, opol);
            } else {
                for (int rg = c_reg_lo; rg < c_reg_hi; ++rg) tma_store_4d(&p.tmC, stg, col0, c_row, c_blk, rg);
            }
            bulk_commit();
        }
    }
    tc_fence_before();
    __syncwarp();
    if (wc.lane == 0) release_acc(sm, buf);

    if (reduce_op) {
        // publish this rank's partial tile: all worker warps' stores complete and
        // visible to generic-proxy readers, then the flag / arrival
        if (wc.lane == 0) {
            bulk_wait_all();
            fence_proxy_async_global();
        }
        __syncwarp();
        __threadfence();
        if (!worker_sync(ctl, sm, wc)) return false;
        if (p.reduce_mode == 2) {
            // count this partial in; the tile's reduce parts become claimable
            // once all W are in
            if (wc.w == 0 && wc.lane == 0 && p.debug_skip != g + 1) {
                __threadfence();
                arrive_count(reinterpret_cast<unsigned long long*>(p.flags) + gc.tile, ctl.epoch);
            }
        } else if (wc.w == 0 && wc.lane == 0 && p.debug_skip != g + 1) {
            st_release_gpu(&p.flags[g], ctl.epoch);
        }
    }
    return true;
}

// Chained reduce epilogue (reduce ops, reduce_mode 3): rank s of output tile t
// waits until ranks 0..s-1 have folded their partials into the fp32 running
// sum S[t] (tile counter = s), then folds in its own partial P_s = acc + bias_s,
// so S = ((P_0 + P_1) + P_2) + ... in rank order: rank 0 stores P_0, a middle
// rank adds P_s into S[t] with a TMA reduce-add (the add happens at the L2, no
// read-back), and the last rank loads S[t] chunk by chunk, adds P_{W-1} and
// rounds to the 16-bit output.  Every rank but the last then advances the
// counter.  This is a ring reduce-scatter/all-reduce done per tile inside the
// GEMM epilogues; each wait is on a GEMM item with a smaller index, which was
// claimed earlier and never waits on this one.
template <int BN, int STAGES, int CG>
__device__ __noinline__ bool epilogue_chain(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t tmem, uint32_t g,
                               uint32_t acc_i, WorkerCtx& wc, Tracer& tr, PartState& ps, bool stages_idle) {
    const uint32_t buf = acc_i & 1, ause = acc_i >> 1;
    const GemmCoord gc = decode_gemm(p, g);
    const int blk = own_block<CG>(p, gc, ctl.half);
    constexpr int COLS = BN * 4 / NUM_WORKER_WARPS;
    constexpr int NCH = COLS / 32;
    const int c_row = blk * BM + wc.q * 32;
    // matmul_all_gather (split-K): the running sum holds every rank's rows
    // (block coordinate = the rank), and its tiles are counted per rank
    const int s_blk = p.op == OP_MM_AG ? gc.rank : 0;
    // (a valid block is below ceil(M_l / BM): blocks past the rank's rows
    // leave before the counter is touched)
    const int cblk = p.op == OP_MM_AG ? gc.rank * ((p.M + BM - 1) / BM) + blk : blk;
    // a column half of a split tail tile (only the last rank's tiles are split)
    const int colbase = gc.nb * BN + (gc.hn >= 0 ? gc.hn * (BN / 2) : 0) + wc.h * COLS;
    // number of 32-column chunks inside the matrix (N is a multiple of 32 here)
    const int nch = max(0, min(gc.hn >= 0 ? NCH / 2 : NCH, (p.N - colbase) / 32));
    const int R = chain_ranks(p);
    if (gc.link == R - 1 && gc.link > 0 && blk * BM < p.M && wc.lane == 0) {
        // the last rank will read this warp's running-sum rows: pull them into
        // L2 while the tile's MMAs still run
        for (int ci = 0; ci < nch; ++ci) tma_prefetch_l2_4d(&p.tmS, colbase + ci * 32, c_row, s_blk, 0);
    }
    const int s = gc.link;
    // the reduce ops add each rank's own bias, all_gather_matmul its one bias
    // (region 0); with split-K, with the rank's first chunk
    const bool add_bias = p.has_bias && gc.chunk == 0;
    const int bias_region = reduce_op_of(p) ? gc.rank : 0;
    const char* bias_base =
        add_bias ? p.heap + static_cast<size_t>(bias_region) * p.rank_stride + p.off_bias : nullptr;
    // per-column bias of the warp's columns, fetched while the MMAs still run:
    // lane l holds the 8 values of columns colbase + 8l .. 8l + 7
    uint4 bias8 = make_uint4(0u, 0u, 0u, 0u);
    if (add_bias && !p.bias_on_m && wc.lane < nch * 4)
        bias8 = *reinterpret_cast<const uint4*>(bias_base + static_cast<size_t>(colbase + wc.lane * 8) * 2);
    // this CTA's half of a pair tile may lie below the last row: no partial,
    // no sum, no counter
    const bool below = CG == 2 && blk * BM >= p.M;
    const bool last = (s == R - 1);
    const int row = blk * BM + wc.q * 32 + wc.lane;
    float row_bias = 0.f;
    if (add_bias && p.bias_on_m && row < p.M)
        row_bias = bits16_to_float(reinterpret_cast<const uint16_t*>(bias_base)[row], p.bf16);
    // one counter per BM-row block and column block
    unsigned long long* ctr = (reduce_op_of(p) ? reinterpret_cast<unsigned long long*>(p.flags) : p.chain) +
                              (cblk * p.n_blocks + gc.nb);
    const unsigned long long tag = static_cast<unsigned long long>(ctl.epoch) << 32;
    // the previous link's hand-off, checked while this tile's MMAs still run
    // (it waits on an item with a smaller index, never on this accumulator)
    if (s > 0 && !below) {
        int ok = 1;
        if (wc.lane == 0) ok = wait_count(ctl, ctr, tag | static_cast<uint32_t>(s), WAIT_CHAIN, static_cast<int>(g));
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
        if (wc.lane == 0) fence_proxy_async_global();  // S[t] was written by the TMA of another SM
    }
    if (!wait_bar_working<BN>(p, ctl, &sm.acc_full[buf], ause & 1, WAIT_ACC_FULL, ps, wc)) return false;
    tc_fence_after();
    tr.rec(EV_READY, g);
    if (below) {
        // release the accumulator in step with the pair
        tc_fence_before();
        __syncwarp();
        if (wc.lane == 0) release_acc(sm, buf);
        return true;
    }
    const uint32_t tbase = tmem + (static_cast<uint32_t>(wc.q * 32) << 16) + buf * BN + wc.h * COLS;
    uint8_t* stg_base = sm.stage_out + wc.w * Smem<BN, STAGES, CG>::STAGE_OUT_BYTES;
    uint64_t* lbar = sm.sbar + SBARS * wc.w;
    auto issue_load = [&](int ci) {
        // the staging half must be free: earlier stores have read it
        bulk_wait_read_all();
        mbar_arrive_expect_tx(&lbar[ci & 1], 32 * 32 * 4);
        tma_load_4d(stg_base + (ci & 1) * 4096, &p.tmS, colbase + ci * 32, c_row, s_blk, 0, &lbar[ci & 1]);
    };
    // only the last rank reads the running sum: the middle ranks add their
    // partial into it at the L2 (TMA reduce-add), in the same rank order
    const bool reads_sum = last && s > 0;
    const uint64_t spol = p.sum_l2_policy == 1   ? l2_policy_evict_first()
                          : p.sum_l2_policy == 2 ? l2_policy_evict_last()
                                                 : 0ull;
    // The CTA's last GEMM item (its pipeline stages idle once the accumulator
    // is full): the warp loads every chunk of its running-sum rows at once,
    // into its quarter of the stages, instead of one chunk ahead through its
    // staging buffer -- this epilogue is the one the launch cannot hide
    constexpr uint32_t STAGE_QUARTER = Smem<BN, STAGES, CG>::TILES_BYTES / NUM_WORKER_WARPS;
    static_assert(STAGE_QUARTER >= NCH * 4096u, "a warp's quarter of the stages holds all its running-sum chunks");
    const bool burst = reads_sum && stages_idle && nch > 0;
    uint8_t* const sbase = sm.tiles + wc.w * STAGE_QUARTER;
    if (burst && wc.lane == 0) {
        mbar_arrive_expect_tx(&lbar[0], static_cast<uint32_t>(nch) * 32 * 32 * 4);
        for (int ci = 0; ci < nch; ++ci)
            tma_load_4d(sbase + ci * 4096, &p.tmS, colbase + ci * 32, c_row, s_blk, 0, &lbar[0]);
    } else if (reads_sum && nch > 0 && wc.lane == 0) {
        issue_load(0);
    }
#pragma unroll 1
    for (int ci = 0; ci < nch; ++ci) {
        uint8_t* stg = burst ? sbase + ci * 4096 : stg_base + (ci & 1) * 4096;
        uint32_t r[32];
        if (p.k_blocks > 0) {
            tmem_ld_32x32b_x32(tbase + ci * 32, r);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        const int col0 = colbase + ci * 32;
        if (reads_sum && !burst && ci + 1 < nch && wc.lane == 0) issue_load(ci + 1);
        // P_s = acc + bias_s (fp32)
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
        if (add_bias) {
            if (p.bias_on_m) {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = x[i] + row_bias;
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int src = ci * 4 + v;  // the lane holding columns col0 + 8v ..
                    const uint32_t bw[4] = {__shfl_sync(0xFFFFFFFFu, bias8.x, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.y, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.z, src),
                                            __shfl_sync(0xFFFFFFFFu, bias8.w, src)};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[v * 8 + 2 * i] = x[v * 8 + 2 * i] + bits16_to_float(bw[i] & 0xFFFFu, p.bf16);
                        x[v * 8 + 2 * i + 1] = x[v * 8 + 2 * i + 1] + bits16_to_float(bw[i] >> 16, p.bf16);
                    }
                }
            }
        }
        if (reads_sum) {
            // S_new = S_old + P_s (S_old holds ranks 0..s-1 in order)
            if (!burst || ci == 0) {
                // one chunk's load, or (burst) all of them, on one barrier
                const int lb = burst ? 0 : (ci & 1);
                int ok = 1;
                if (wc.lane == 0) {
                    const uint32_t par = (wc.sphase >> lb) & 1u;
                    ok = wait_bar(ctl, &lbar[lb], par, WAIT_CHAIN_LOAD) ? 1 : 0;
                    // stopped: the burst's other chunks still land in the stages
                    if (!ok && burst) drain_bar(ctl, &lbar[lb], par, WAIT_CHAIN_LOAD);
                }
                wc.sphase ^= 1u << lb;
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 o = *reinterpret_cast<const float4*>(stg + wc.lane * 128 + ((c ^ (wc.lane & 7)) << 4));
                x[4 * c + 0] = o.x + x[4 * c + 0];
                x[4 * c + 1] = o.y + x[4 * c + 1];
                x[4 * c + 2] = o.z + x[4 * c + 2];
                x[4 * c + 3] = o.w + x[4 * c + 3];
            }
            __syncwarp();  // every lane has read its row before the buffer is rewritten
        } else {
            // the store issued two chunks ago (from this buffer) must have read it
            if (wc.lane == 0) bulk_wait_read<1>();
            __syncwarp();
        }
        if (!last) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(stg + wc.lane * 128 + ((c ^ (wc.lane & 7)) << 4)) =
                    make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack2(x[8 * v + 0], x[8 * v + 1], p.bf16);
                o.y = pack2(x[8 * v + 2], x[8 * v + 3], p.bf16);
                o.z = pack2(x[8 * v + 4], x[8 * v + 5], p.bf16);
                o.w = pack2(x[8 * v + 6], x[8 * v + 7], p.bf16);
                *reinterpret_cast<uint4*>(stg + wc.lane * 64 + ((v ^ ((wc.lane >> 1) & 3)) << 4)) = o;
            }
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (wc.lane == 0) {
            if (!last && s == 0) {
                if (p.sum_l2_policy) tma_store_4d_hint(&p.tmS, stg, col0, c_row, s_blk, 0, spol);
                else tma_store_4d(&p.tmS, stg, col0, c_row, s_blk, 0);
            } else if (!last) {
                if (p.sum_l2_policy) tma_reduce_add_4d_hint(&p.tmS, stg, col0, c_row, s_blk, 0, spol);  // S += P_s
                else tma_reduce_add_4d(&p.tmS, stg, col0, c_row, s_blk, 0);  // S += P_s
            } else if (p.op == OP_MM_RS) {
                const int rr = col0 / p.N_local;
                if (p.out_evict_first)
                    tma_store_4d_hint(&p.tmC, stg, col0 - rr * p.N_local, c_row, rr, 0, l2_policy_evict_first());
                else
                    tma_store_4d(&p.tmC, stg, col0 - rr * p.N_local, c_row, rr, 0);
            } else {
                // all-reduce / all_gather_matmul: row block 0; matmul_all_gather:
                // the rank's block of the gathered output
                const int nreg = p.replicate ? p.W : 1;
                for (int rg = 0; rg < nreg; ++rg) {
                    if (p.out_evict_first)
                        tma_store_4d_hint(&p.tmC, stg, col0, c_row, s_blk, rg, l2_policy_evict_first());
                    else
                        tma_store_4d(&p.tmC, stg, col0, c_row, s_blk, rg);
                }
            }
            bulk_commit();
        }
    }
    tc_fence_before();
    __syncwarp();
    if (wc.lane == 0) release_acc(sm, buf);
    if (!last) {
        // S[t] complete and visible, then hand the tile to rank s+1
        if (wc.lane == 0) {
            bulk_wait_all();
            fence_proxy_async_global();
        }
        __syncwarp();
        fence_acq_rel_gpu();  // release side: the barrier, then one release store
        if (!worker_sync(ctl, sm, wc)) return false;
        if (wc.w == 0 && wc.lane == 0 && p.debug_skip != g + 1)
            st_release_gpu_u64(ctr, tag | static_cast<uint32_t>(s + 1));
    }
    return true;
}

// all_gather_matmul gather tile: shard s rows of m-block mb -> gathered buffer.
template <int BN, int STAGES, int CG>
__device__ bool gather_tile(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t c,
                            WorkerCtx& wc) {
    // CTA pairs: both CTAs run the item, each copying (and flagging) its own
    // block of BM rows of the pair's m-block
    const GatherCoord gq = decode_gather(p, c);
    const int mb = gq.mb * CG + ctl.half, s = gq.s;
    if (mb * BM >= p.M) return true;  // below the last row: nothing to copy, no consumer
    const int block_rows = min(BM, p.M - mb * BM);
    // this item's row part of the block
    const int r_lo = gq.part * block_rows / p.gather_parts, r_hi = (gq.part + 1) * block_rows / p.gather_parts;
    const int rows = r_hi - r_lo;
    const int vpr = p.K_local / 8;  // 16-byte vectors per shard row
    const int Kv = p.K / 8;         // vectors per gathered row
    const uint4* src = reinterpret_cast<const uint4*>(p.heap + static_cast<size_t>(s) * p.rank_stride + p.off_A) +
                       (static_cast<size_t>(mb) * BM + r_lo) * vpr;
    uint4* dst = reinterpret_cast<uint4*>(p.heap + p.off_gathered) + (static_cast<size_t>(mb) * BM + r_lo) * Kv +
                 static_cast<size_t>(s) * vpr;
    // The shard block (rows x vpr vectors, contiguous) is copied as one flat
    // range: thread t takes vectors t, t + 128, ...; U loads per thread are in
    // flight before their stores (32 KB per CTA), whatever the row length.
    constexpr int U = 16;
    constexpr int NT = NUM_WORKER_WARPS * 32;
    const int tid = wc.w * 32 + wc.lane;
    const int total = rows * vpr;
    for (int base = 0; base < total; base += NT * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * NT + tid;
            if (i < total) v[u] = __ldcs(src + i);  // read once: evict-first
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * NT + tid;
            if (i < total) {
                const int r = i / vpr;
                // not re-read until its GEMM tiles run: evict-first
                __stcs(dst + static_cast<size_t>(r) * Kv + (i - r * vpr), v[u]);
            }
        }
    }
    fence_proxy_async_global();
    fence_acq_rel_gpu();  // release side: the barrier, then one arrival
    if (!worker_sync(ctl, sm, wc)) return false;
    // count this part in; the block's counter completes with the last part
    // (the test hook drops part 0's arrival of one block)
    const uint32_t fi = static_cast<uint32_t>(mb * p.W + s);
    if (wc.w == 0 && wc.lane == 0 && !(p.debug_skip == fi + 1 && gq.part == 0)) {
        // a release store orders the copies (each thread fenced its own before
        // the barrier); the compare-and-swap of row parts needs the fence
        if (p.gather_parts != 1) __threadfence();
        arrive_gather(p, gather_ctr(p, static_cast<int>(fi)), ctl.epoch);
    }
    return true;
}

// matmul_reduce_scatter / matmul_all_reduce comm tile: rank-order fp32 sum
// of the W partial tiles of output tile c, rounded and scattered.
template <int BN, int STAGES, int CG>
__device__ bool reduce_tile(const Params& p, const Ctl& ctl, uint32_t c, WorkerCtx& wc) {
    bool ok = true;
    if (wc.lane == 0) {
        for (int s = 0; s < p.W && ok; ++s) {
            const int fi = static_cast<int>(gemm_index(p, c, s));
            ok = wait_flag(ctl, &p.flags[fi], WAIT_FLAG_PARTIAL, fi);
        }
    }
    if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) return false;
    reduce_body<BN, STAGES, CG>(p, c, wc);
    return true;
}

// The reduce itself: warp w takes rows w, w+8, ... of output tile c; lane l
// takes the 16-byte column chunks l, l+32, ... of each row, so every load and
// store instruction of a warp covers 512 contiguous bytes.  SC ranks of a row
// are loaded together before their adds; partials are summed in rank order
// 0..W-1 in fp32.
template <int BN, int STAGES, int CG>
__device__ __noinline__ void reduce_body(const Params& p, uint32_t c, WorkerCtx& wc) {
    constexpr int CPL = BN / 4 / 32;  // float4 chunks per lane per row
    constexpr int SC = 4;             // ranks per load batch
    int mb, nb;
    swizzle_tile(p, c, mb, nb);
    const int rows = min(BM, p.M - mb * BM);
    const int cols = min(BN, p.N - nb * BN);
    const size_t pe = p.partial_elems;
    bool cok[CPL];
    int dcol[CPL];
    size_t dbase[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c4 = wc.lane + 32 * k;
        cok[k] = c4 * 4 < cols;
        const int j = nb * BN + c4 * 4;
        if (p.op == OP_MM_RS) {
            const int rr = cok[k] ? j / p.N_local : 0;
            dcol[k] = j - rr * p.N_local;
            dbase[k] = static_cast<size_t>(rr) * p.rank_stride + p.off_out;
        } else {
            dcol[k] = j;
            dbase[k] = p.off_out;
        }
    }
    const int ldo = (p.op == OP_MM_RS) ? p.N_local : p.N;
    const int nreg = (p.op == OP_MM_AR && p.replicate) ? p.W : 1;
    for (int r = wc.w; r < rows; r += NUM_WORKER_WARPS) {
        float4 acc[CPL];
        const float* src0 = p.partials + static_cast<size_t>(mb * BM + r) * p.N + nb * BN;
        for (int s0 = 0; s0 < p.W; s0 += SC) {
            float4 v[SC][CPL];
#pragma unroll
            for (int ds = 0; ds < SC; ++ds)
#pragma unroll
                for (int k = 0; k < CPL; ++k)
                    if (s0 + ds < p.W && cok[k])
                        v[ds][k] = __ldcg(reinterpret_cast<const float4*>(src0 + static_cast<size_t>(s0 + ds) * pe) +
                                          wc.lane + 32 * k);
#pragma unroll
            for (int ds = 0; ds < SC; ++ds)
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    if (s0 + ds == 0) {
                        acc[k] = v[0][k];
                    } else if (s0 + ds < p.W) {
                        acc[k].x = acc[k].x + v[ds][k].x;
                        acc[k].y = acc[k].y + v[ds][k].y;
                        acc[k].z = acc[k].z + v[ds][k].z;
                        acc[k].w = acc[k].w + v[ds][k].w;
                    }
                }
        }
        const size_t orow = static_cast<size_t>(mb * BM + r) * ldo;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            if (!cok[k]) continue;
            uint2 o;
            o.x = pack2(acc[k].x, acc[k].y, p.bf16);
            o.y = pack2(acc[k].z, acc[k].w, p.bf16);
            for (int rg = 0; rg < nreg; ++rg)
                *reinterpret_cast<uint2*>(p.heap + static_cast<size_t>(rg) * p.rank_stride + dbase[k] +
                                          (orow + dcol[k]) * 2) = o;
        }
    }
}

// Concurrent-mode collective item c: bytes [b0, b1) of a source range.
// Sources: src_n regions starting at src_lo, at src_base + (b - b0).
// Destinations: every region (dst_all), the owning rank's slice
// (reduce-scatter), or region dst_region, at dst_base + (b - b0).
struct CollRange {
    size_t b0, b1, src_base, dst_base;
    int src_lo, src_n, dst_region;
    bool dst_all;
};
__device__ __forceinline__ CollRange coll_range(const Params& p, uint32_t c) {
    const size_t esz = static_cast<size_t>(p.elem_bytes);
    const size_t bytes_per_rank = static_cast<size_t>(p.count) * esz;
    const size_t chunk = static_cast<size_t>(p.comm_block) * esz;
    size_t b0, b1, src_base, dst_base;
    int src_lo, src_n, dst_region = -1;
    bool dst_all = false;
    if (p.coll == COLL_AG) {
        const size_t chunks = (bytes_per_rank + chunk - 1) / chunk;
        const int s = static_cast<int>(c / chunks);
        b0 = (c - s * chunks) * chunk;
        b1 = min(bytes_per_rank, b0 + chunk);
        src_lo = s;
        src_n = 1;
        src_base = p.off_in + b0;
        dst_base = p.off_cout + static_cast<size_t>(s) * bytes_per_rank + b0;
        dst_all = true;
    } else if (p.coll == COLL_A2A) {
        // pair (r receives from s): rank s's slice r -> rank r's slot s
        const size_t sb = bytes_per_rank / p.W;
        const size_t chunks = (sb + chunk - 1) / chunk;
        const uint32_t pair = static_cast<uint32_t>(c / chunks);
        const int r = static_cast<int>(pair / p.W), s = static_cast<int>(pair % p.W);
        b0 = (c - pair * chunks) * chunk;
        b1 = min(sb, b0 + chunk);
        src_lo = s;
        src_n = 1;
        src_base = p.off_in + static_cast<size_t>(r) * sb + b0;
        dst_base = p.off_cout + static_cast<size_t>(s) * sb + b0;
        dst_region = r;
    } else if (p.coll == COLL_BC) {
        b0 = static_cast<size_t>(c) * chunk;
        b1 = min(bytes_per_rank, b0 + chunk);
        src_lo = p.root;
        src_n = 1;
        src_base = p.off_in + b0;
        dst_base = p.off_cout + b0;
        dst_all = true;
    } else {  // all-reduce, reduce-scatter: fp32 sum over all W sources
        b0 = static_cast<size_t>(c) * p.comm_block * 4;
        b1 = min(static_cast<size_t>(p.count) * 4, b0 + static_cast<size_t>(p.comm_block) * 4);
        src_lo = 0;
        src_n = p.W;
        src_base = p.off_in + b0;
        dst_base = p.off_cout + b0;
        dst_all = (p.coll == COLL_AR);
    }
    CollRange r;
    r.b0 = b0;
    r.b1 = b1;
    r.src_base = src_base;
    r.dst_base = dst_base;
    r.src_lo = src_lo;
    r.src_n = src_n;
    r.dst_region = dst_region;
    r.dst_all = dst_all;
    return r;
}

// Concurrent-mode collective tile through the TMA engine, run while the TMA
// producer lends the CTA's pipeline stages (STAGES x STAGE_BYTES bytes of
// shared memory) to the workers.  Worker warp w owns 1/4 of that space as a
// ring of p.coll_ring buffers; for each sub-chunk of its slice of tile c it
// bulk-loads the sources (all W ranks for all-reduce / reduce-scatter, rank s
// for all-gather) into the next buffer while earlier ones are summed in rank
// order (fp32) and bulk-stored to the destinations.  Staged (the default
// for all-reduce, whose stores go to every region), a sub-chunk that fits
// half of the warp's 8 KB staging buffer is summed into that half (the two
// halves alternate), so the load buffer takes its next load right after the
// sum and all coll_ring loads stay in flight; otherwise the sum stays in the
// load buffer, which is refilled once the stores have read it (coll_ring - 1
// loads in flight).  With p.coll_evict_first the copies
// carry an L2 evict-first policy, so the streamed collective data does not
// push the concurrent GEMM's operands out of the L2.
template <int BN, int STAGES, int CG>
__device__ bool coll_tile_tma(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t c, WorkerCtx& wc) {
    constexpr uint32_t AREA = STAGES * Smem<BN, STAGES, CG>::STAGE_BYTES / NUM_WORKER_WARPS;
    const int nb = p.coll_ring;
    const uint32_t BUF = (AREA / static_cast<uint32_t>(nb)) & ~15u;
    uint8_t* area = sm.tiles + wc.w * AREA;
    uint64_t* bar = sm.sbar + SBARS * wc.w;
    const CollRange cr = coll_range(p, c);
    const size_t b0 = cr.b0, b1 = cr.b1, src_base = cr.src_base, dst_base = cr.dst_base;
    const int src_lo = cr.src_lo, src_n = cr.src_n, dst_region = cr.dst_region;
    const bool dst_all = cr.dst_all;
    // the warp's contiguous slice (16-byte granules) of [b0, b1), as offsets
    // from b0; a CTA pair runs the item together, one slice per worker warp
    // of either CTA
    // coll_path 3 loads whole 1 KB rows of all W sources with one box: the
    // slice and the sub-chunks are then counted in rows
    const bool box = p.coll_path == 3;
    const size_t gran = box ? 1024 : 16;
    const size_t g_tot = (b1 - b0) / gran;
    const size_t ww = static_cast<size_t>(ctl.half * NUM_WORKER_WARPS + wc.w), nww = CG * NUM_WORKER_WARPS;
    const size_t g_lo = g_tot * ww / nww, g_hi = g_tot * (ww + 1) / nww;
    const uint32_t sub = box ? static_cast<uint32_t>(p.coll_box_rows) * 1024u
                             : (BUF / src_n) & ~15u;  // bytes per source per sub-chunk
    const size_t s_lo = g_lo * gran, s_hi = g_hi * gran;
    const int nsub = static_cast<int>((s_hi - s_lo + sub - 1) / sub);
    const size_t cw_bytes = static_cast<size_t>(p.count / p.W) * 4;  // reduce-scatter slice per rank
    const bool hint = p.coll_evict_first != 0;
    const uint64_t pol = hint ? l2_policy_evict_first() : 0ull;
    auto store = [&](void* g, const void* s, uint32_t n) {
        if (hint) bulk_store_hint(g, s, n, pol);
        else bulk_store(g, s, n);
    };
    // lane 0: bulk-store n bytes at byte offset o of the slice from smem `from`
    // to every destination of the collective, as one bulk group
    auto store_out = [&](const uint8_t* from, size_t o, uint32_t n) {
        if (p.coll == COLL_RS) {
            // the item may cross a rank boundary: split the store there
            size_t done = 0;
            while (done < n) {
                const size_t e = b0 + o + done;  // byte index into the summed vector
                const int rr = static_cast<int>(e / cw_bytes);
                const size_t piece = min(static_cast<size_t>(n) - done, (rr + 1) * cw_bytes - e);
                store(p.heap + static_cast<size_t>(rr) * p.rank_stride + p.off_cout + (e - rr * cw_bytes),
                      from + done, static_cast<uint32_t>(piece));
                done += piece;
            }
        } else if (dst_all) {
            for (int r = 0; r < p.W; ++r) store(p.heap + static_cast<size_t>(r) * p.rank_stride + dst_base + o, from, n);
        } else {
            store(p.heap + static_cast<size_t>(dst_region) * p.rank_stride + dst_base + o, from, n);
        }
        bulk_commit();
    };
    constexpr uint32_t OUT_HALF = Smem<BN, STAGES, CG>::STAGE_OUT_BYTES / 2;
    const bool staged = src_n > 1 && p.coll_path != 2 && sub <= OUT_HALF &&
                        (p.coll_out_stage == 2 || (p.coll_out_stage == 0 && p.coll == COLL_AR));
    uint8_t* const outb = sm.stage_out + wc.w * Smem<BN, STAGES, CG>::STAGE_OUT_BYTES;
    // load sub-chunk i into buffer i % nb (whose earlier store has read it)
    auto issue = [&](int i) {
        const size_t o = s_lo + static_cast<size_t>(i) * sub;
        const uint32_t n = static_cast<uint32_t>(min(static_cast<size_t>(sub), s_hi - o));
        uint8_t* buf = area + (i % nb) * BUF;
        if (box) {
            // rows [(b0 + o) / 1 KB, + R) of every region in one box (rows
            // past the tensor read as zeros; rows past this warp's slice
            // are loaded but not used)
            mbar_arrive_expect_tx(&bar[i % nb], sub * src_n);
            if (hint) tma_load_3d_hint(buf, &p.tmX, 0, static_cast<int>((b0 + o) / 1024), 0, &bar[i % nb], pol);
            else tma_load_3d(buf, &p.tmX, 0, static_cast<int>((b0 + o) / 1024), 0, &bar[i % nb]);
            return;
        }
        mbar_arrive_expect_tx(&bar[i % nb], n * src_n);
        for (int r = 0; r < src_n; ++r) {
            const char* src = p.heap + static_cast<size_t>(src_lo + r) * p.rank_stride + src_base + o;
            if (hint) bulk_load_hint(buf + r * sub, src, n, &bar[i % nb], pol);
            else bulk_load(buf + r * sub, src, n, &bar[i % nb]);
        }
    };
    int issued = 0;  // lane 0: sub-chunks whose loads were issued
    if (wc.lane == 0) {
        // staged: an earlier epilogue's stores may still read the staging buffer
        if (staged) bulk_wait_read_all();
        for (; issued < min(staged ? nb : nb - 1, nsub); ++issued) issue(issued);
    }
    int i = 0;
    bool ok = true;
    for (; i < nsub; ++i) {
        int got = 1;
        if (wc.lane == 0) {
            // in place: keep nb - 1 loads in flight; the next one goes into
            // the buffer of sub-chunk i - 1, whose stores (the newest group)
            // must have read it
            if (!staged && issued < nsub) {
                bulk_wait_read_all();
                issue(issued);
                ++issued;
            }
            got = wait_bar(ctl, &bar[i % nb], (wc.sphase >> (i % nb)) & 1u, WAIT_COLL_LOAD) ? 1 : 0;
        }
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
            ok = false;
            break;
        }
        wc.sphase ^= 1u << (i % nb);
        const size_t o = s_lo + static_cast<size_t>(i) * sub;
        const uint32_t n = static_cast<uint32_t>(min(static_cast<size_t>(sub), s_hi - o));
        uint8_t* buf = area + (i % nb) * BUF;
        if (p.coll_path == 2) {
            // every lane stores its 16-byte granules straight from registers
            // (consecutive lanes, consecutive granules: 512 B per warp store)
            for (uint32_t q = wc.lane; q < n / 16; q += 32) {
                uint4 v = *reinterpret_cast<const uint4*>(buf + q * 16);
                if (src_n > 1) {
                    // rank-order fp32 sum
                    float4 a = *reinterpret_cast<const float4*>(&v);
                    for (int r = 1; r < src_n; ++r) {
                        const float4 u = *reinterpret_cast<const float4*>(buf + r * sub + q * 16);
                        a.x = a.x + u.x;
                        a.y = a.y + u.y;
                        a.z = a.z + u.z;
                        a.w = a.w + u.w;
                    }
                    v = *reinterpret_cast<const uint4*>(&a);
                }
                const size_t og = o + static_cast<size_t>(q) * 16;  // byte offset from the item start
                if (p.coll == COLL_RS) {
                    const size_t e = b0 + og;
                    const int rr = static_cast<int>(e / cw_bytes);
                    *reinterpret_cast<uint4*>(p.heap + static_cast<size_t>(rr) * p.rank_stride + p.off_cout +
                                              (e - rr * cw_bytes)) = v;
                } else if (dst_all) {
                    for (int r = 0; r < p.W; ++r)
                        *reinterpret_cast<uint4*>(p.heap + static_cast<size_t>(r) * p.rank_stride + dst_base + og) = v;
                } else {
                    *reinterpret_cast<uint4*>(p.heap + static_cast<size_t>(dst_region) * p.rank_stride + dst_base +
                                              og) = v;
                }
            }
            __syncwarp();  // the buffer is free for the next load once every lane has read it
            continue;
        }
        if (staged) {
            // this staging half was last stored from two sub-chunks ago: its
            // group (every group but the newest) has finished reading it
            if (wc.lane == 0) bulk_wait_read<1>();
            __syncwarp();
            uint8_t* ob = outb + (i & 1) * OUT_HALF;
            for (uint32_t q = wc.lane; q < n / 16; q += 32) {
                float4 a = *reinterpret_cast<const float4*>(buf + q * 16);
                for (int r = 1; r < src_n; ++r) {
                    const float4 v = *reinterpret_cast<const float4*>(buf + r * sub + q * 16);
                    a.x = a.x + v.x;
                    a.y = a.y + v.y;
                    a.z = a.z + v.z;
                    a.w = a.w + v.w;
                }
                *reinterpret_cast<float4*>(ob + q * 16) = a;
            }
            // the sums are visible to the stores, and the lanes' reads of the
            // load buffer are ordered before the load that refills it
            fence_proxy_async_shared();
            __syncwarp();
            if (wc.lane == 0) {
                store_out(ob, o, n);
                if (issued < nsub) {
                    issue(issued);  // into buffer i % nb, just summed
                    ++issued;
                }
            }
            __syncwarp();
            continue;
        }
        if (src_n > 1) {
            // rank-order fp32 sum into the rank-0 slot
            for (uint32_t q = wc.lane; q < n / 16; q += 32) {
                float4 a = *reinterpret_cast<const float4*>(buf + q * 16);
                for (int r = 1; r < src_n; ++r) {
                    const float4 v = *reinterpret_cast<const float4*>(buf + r * sub + q * 16);
                    a.x = a.x + v.x;
                    a.y = a.y + v.y;
                    a.z = a.z + v.z;
                    a.w = a.w + v.w;
                }
                *reinterpret_cast<float4*>(buf + q * 16) = a;
            }
            fence_proxy_async_shared();
        }
        __syncwarp();
        if (wc.lane == 0) store_out(buf, o, n);
        __syncwarp();
    }
    if (!ok && wc.lane == 0) {
        // stopped early: the loads still in flight land in the leased stages,
        // so wait (bounded) for each before the stages can be returned
        for (int j = i; j < issued; ++j) {
            drain_bar(ctl, &bar[j % nb], (wc.sphase >> (j % nb)) & 1u, WAIT_COLL_LOAD);
            wc.sphase ^= 1u << (j % nb);
        }
    }
    // the stages go back to the TMA producer once every store has read them
    if (wc.lane == 0) bulk_wait_read_all();
    __syncwarp();
    return ok;
}

template <int BN, int STAGES, int CG>
__device__ void run_workers(const Params& p, const Ctl& ctl, Smem<BN, STAGES, CG>& sm, uint32_t tmem,
                            int warp, int lane) {
    WorkerCtx wc;
    wc.w = warp - FIRST_WORKER_WARP;
    wc.lane = lane;
    wc.q = warp & 3;
    wc.h = (warp - FIRST_WORKER_WARP) >> 2;
    Tracer tr;
    if (wc.w == 0 && lane == 0) tr.init(p, TR_WORK);
    wc.wphase = 0;
    wc.sphase = 0;
    uint32_t leases = 0;
    PartState ps;
    ps.cur = NO_PART;
    ps.row = 0;
    ps.ready = false;
    uint32_t ring_n = 0, acc_i = 0;
    bool ok = true;
    bool seen_gemm = false;  // as the TMA producer tracks it
    while (true) {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        ok = wait_bar_working<BN>(p, ctl, &sm.item_full[slot], use & 1, WAIT_ITEM_FULL_WORKER, ps, wc, CG == 2);
        if (!ok) break;
        // lane 0 did the acquire; it reads the slot and hands the item on
        uint32_t item = 0;
        if (lane == 0) item = sm.ring[slot];
        item = __shfl_sync(0xFFFFFFFFu, item, 0);
        if (lane == 0) release_item(sm, slot);
        ++ring_n;
        if (item == ITEM_END) break;
        tr.rec(EV_BEGIN, item);
        if (item & ITEM_COMM) {
            const uint32_t c = item & ~ITEM_COMM;
            if (p.op == OP_AG_MM && p.startup_gather && !seen_gemm) {
                // a start-up gather: the TMA producer copies it
            } else if (p.op == OP_AG_MM) {
                ok = gather_tile(p, ctl, sm, c, wc);
            } else if (p.op == OP_CONC) {
                int got = 1;
                if (lane == 0) got = wait_bar(ctl, sm.lease, leases & 1, WAIT_LEASE) ? 1 : 0;
                ++leases;
                ok = __shfl_sync(0xFFFFFFFFu, got, 0) != 0 && coll_tile_tma<BN, STAGES, CG>(p, ctl, sm, c, wc);
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.lease_done);
            } else {
                ok = reduce_tile<BN, STAGES, CG>(p, ctl, c, wc);
            }
        } else {
            seen_gemm = true;
            if (split_k(p) || (p.reduce_mode == 3 && (p.op == OP_MM_RS || p.op == OP_MM_AR)))
            {
                // the next ring entry already published as the end marker: this
                // is the CTA's last GEMM item, so its stages fall idle once the
                // accumulator is full (no further loads are issued)
                int idle = 0;
                if (lane == 0) {
                    const uint32_t nslot = ring_n % RING, nuse = ring_n / RING;
                    idle = try_bar(&sm.item_full[nslot], nuse & 1, CG == 2) && sm.ring[nslot] == ITEM_END;
                }
                idle = __shfl_sync(0xFFFFFFFFu, idle, 0);
                ok = epilogue_chain(p, ctl, sm, tmem, item, acc_i, wc, tr, ps, idle != 0);
            }
            else
                ok = epilogue(p, ctl, sm, tmem, item, acc_i, wc, tr, ps);
            ++acc_i;
        }
        tr.rec(EV_END, item);
        if (!ok) break;
    }
    // help with the reduce parts left: their tiles' GEMM items are all
    // claimed and run without waiting on parts, so they complete (bounded)
    if (ok && p.n_parts > 0) {
        uint64_t t0 = 0;
        bool timing = false;
        for (uint32_t i = 0; !parts_done(p, ps); ++i) {
            if (part_step<BN>(p, ctl.epoch, ps, wc)) {
                timing = false;
                continue;
            }
            if (!timing) {
                t0 = global_timer_ns();
                timing = true;
            }
            __nanosleep(128);
            if ((i & 15) == 0) {
                if (launch_aborted(ctl)) break;
                if (global_timer_ns() - t0 > ctl.limit) {
                    if (lane == 0) raise_timeout(ctl, WAIT_REDUCE_PARTS, -1);
                    break;
                }
            }
        }
    }
    tr.rec(EV_END, 0x7FFFFFFEu);  // workers done (after the reduce parts)
    tr.finish();
    // the staging buffer must outlive every store that reads it
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

// ============================================================ kernel
template <int BN, int STAGES, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1) fused_gemm_coll_kernel(const __grid_constant__ Params p) {
    constexpr int TMEM_COLS = 2 * BN;
    extern __shared__ uint8_t smem_raw[];
    Smem<BN, STAGES, CG> sm;
    sm.carve(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // CTA pairs (cluster of 2): the even CTA runs the scheduler and issues the
    // MMAs for both; each CTA loads its halves of A and B and drains its own
    // half of the accumulator
    const int half = (CG == 2) ? static_cast<int>(cluster_ctarank()) : 0;
    Tracer ktr;  // thread 0: the scheduler stream (kernel entry, claims, teardown end)
    if (threadIdx.x == 0) {
        ktr.init(p, TR_SCHED);
        ktr.rec(EV_KERNEL_BEGIN, blockIdx.x);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], CG * NUM_WORKER_WARPS);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(&sm.item_full[i], 1);
            // MMA + TMA + workers (pairs: plus the odd CTA's TMA + workers)
            mbar_init(&sm.item_empty[i], 2 + NUM_WORKER_WARPS + (CG == 2 ? 1 + NUM_WORKER_WARPS : 0));
        }
        mbar_init(sm.wbar, NUM_WORKER_WARPS);
        mbar_init(sm.final_bar, 1);
        for (int i = 0; i < SBARS * NUM_WORKER_WARPS; ++i) mbar_init(&sm.sbar[i], 1);
        mbar_init(sm.lease, 1);
        mbar_init(sm.lease_done, NUM_WORKER_WARPS);
        mbar_init(sm.gbar, 1);
        for (int i = 0; i < Smem<BN, STAGES, CG>::READY_BITS / 32; ++i) sm.ready_bits[i] = 0u;
        fence_mbar_init();
        uint32_t e = *reinterpret_cast<volatile uint32_t*>(&p.ws->epoch) + 1u;
        if (e == 0u) e = 1u;
        *sm.epoch_slot = e;
        if (p.n_gemm > 0 && p.k_blocks > 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
            if (p.b_chunked) tma_prefetch_desc(&p.tmBc);
            if (p.a_chunked) tma_prefetch_desc(&p.tmAc);
        }
        if (p.n_gemm > 0) tma_prefetch_desc(&p.tmC);
        if (p.n_comm > 0 && p.coll_path == 3) tma_prefetch_desc(&p.tmX);
        if (p.n_gemm > 0 && p.reduce_mode == 3) tma_prefetch_desc(&p.tmS);
    }
    if (warp == 1) tmem_alloc<TMEM_COLS, CG>(sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    // pairs: both CTAs' barriers are initialised before either signals the other's
    if (CG == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;
    const Ctl ctl{p.ws, *sm.epoch_slot, p.wait_ns, half};

    if (warp == 0) {
        if (lane == 0 && half == 0) run_scheduler<BN, STAGES, CG>(p, ctl, sm, ktr);
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0) run_tma<BN, STAGES, CG>(p, ctl, sm);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && half == 0) run_mma<BN, STAGES, CG>(p, ctl, sm, tmem);
        __syncwarp();
    } else {
        run_workers<BN, STAGES, CG>(p, ctl, sm, tmem, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    // pairs: neither CTA leaves (or frees tensor memory) while the other may
    // still signal its barriers or read the accumulators the MMAs wrote
    if (CG == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<TMEM_COLS, CG>(tmem);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(&p.ws->done_ctr, 1u);
        if (done == gridDim.x - 1) {
            // last CTA of the launch (every other CTA has counted itself out
            // and touches the header no more): publish the epoch and reset
            // the queues for the next launch on this workspace.  The epoch
            // and the three counters after it are one 16-byte store; the next
            // launch sees them after the kernel boundary.
            p.ws->part_ctr = 0u;
            *reinterpret_cast<uint4*>(p.ws) = make_uint4(ctl.epoch, 0u, 0u, 0u);
        }
        ktr.rec(EV_KERNEL_END, blockIdx.x);
        ktr.finish();
    }
}

}  // namespace gct
