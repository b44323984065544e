// Host side of the C ABI declared in include/gemm_collective_tiles.h:
// argument checks, workspace layout, TMA tensor maps, and the launch of the
// persistent fused kernel (fused_kernel.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_collective_tiles.h"
#include "fused_kernel.cuh"

using namespace gct;

namespace {

constexpr int BN_WIDE = 256, STAGES_WIDE = 4;
constexpr int BN_NARROW = 128, STAGES_NARROW = 6;
// CTA pairs (tile_m 256): 256 x 256 tiles over two SMs; each SM stages
// 128 x 64 of A and 64 x 128 of B (32 KB) per K-block.  Three stages of two
// K-blocks (one A and one B box per stage: half the TMA instructions and
// barrier hand-offs), or six stages of one K-block when the operands stream
// from DRAM (long K), where more, smaller stages keep more bytes in flight.
constexpr int STAGES_PAIR = 3;
constexpr int STAGES_PAIR_STREAM = 6;
constexpr int64_t STREAM_K = 98304;  // K above which the six-stage pipeline is the default
// all_gather_matmul split-K by default above 2 x SPLIT_K_CHUNK, in chunks of
// about SPLIT_K_CHUNK K: the tiles running at once then stay short enough to
// share their operand blocks in L2, as at K = 16384 (measured, 8 x 16384-row
// or 8192-row shapes: +9 % at K = 49152, +1-15 % at 65536, +27-49 % at 131072
// and 262144; at K <= 32768 a split loses or gains nothing; chunks of 8192 or
// 32768 lose to 16384 at every long K tried)
constexpr int64_t SPLIT_K_CHUNK = 16384;
constexpr size_t WS_HEADER = 256;
constexpr unsigned long long DEFAULT_WAIT_NS = 2000000000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

// IRIS_B200_DEBUG=1 in the environment prints the failing step of an
// IRIS_ECUDA return to stderr.
bool debug_on() {
    static const bool on = [] {
        const char* e = std::getenv("IRIS_B200_DEBUG");
        return e && e[0] && e[0] != '0';
    }();
    return on;
}
int cuda_fail(const char* what, int code) {
    if (debug_on()) std::fprintf(stderr, "[iris_b200] %s failed: %d\n", what, code);
    return IRIS_ECUDA;
}
bool g_attr_done[64] = {false};

EncodeTiledFn encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

template <int BN, int STAGES, int CG>
constexpr size_t smem_bytes() {
    return Smem<BN, STAGES, CG>::BYTES;
}

// Every kernel variant lends the same pipeline bytes to a collective tile.
constexpr uint32_t LEASE_BYTES = Smem<BN_WIDE, STAGES_PAIR, 2>::TILES_BYTES;
static_assert(Smem<BN_WIDE, STAGES_PAIR_STREAM, 2>::TILES_BYTES == LEASE_BYTES &&
                  Smem<BN_WIDE, STAGES_WIDE, 1>::TILES_BYTES == LEASE_BYTES &&
                  Smem<BN_NARROW, STAGES_NARROW, 1>::TILES_BYTES == LEASE_BYTES,
              "collective tiles assume one lease size for every kernel variant");

int g_pair_clusters[64] = {0};  // co-resident CTA pairs of the pair kernel, per device

cudaLaunchConfig_t pair_launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr,
                                      size_t smem = smem_bytes<BN_WIDE, STAGES_PAIR, 2>()) {
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    lc.gridDim = dim3(grid, 1, 1);
    lc.blockDim = dim3(NUM_THREADS, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = 2;
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return lc;
}

int ensure_attrs(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= 64) return IRIS_ECUDA;
    if (g_attr_done[dev]) return IRIS_OK;
    cudaError_t e = cudaFuncSetAttribute(fused_gemm_coll_kernel<BN_WIDE, STAGES_WIDE, 1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<BN_WIDE, STAGES_WIDE, 1>()));
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (tile_n 256)", static_cast<int>(e));
    e = cudaFuncSetAttribute(fused_gemm_coll_kernel<BN_NARROW, STAGES_NARROW, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<BN_NARROW, STAGES_NARROW, 1>()));
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (tile_n 128)", static_cast<int>(e));
    e = cudaFuncSetAttribute(fused_gemm_coll_kernel<BN_WIDE, STAGES_PAIR, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<BN_WIDE, STAGES_PAIR, 2>()));
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (tile_m 256)", static_cast<int>(e));
    e = cudaFuncSetAttribute(fused_gemm_coll_kernel<BN_WIDE, STAGES_PAIR_STREAM, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<BN_WIDE, STAGES_PAIR_STREAM, 2>()));
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (tile_m 256, 6 stages)", static_cast<int>(e));
    // how many CTA pairs fit at once (one CTA per SM; a pair needs two SMs of
    // one GPC): the persistent pair grid is twice that
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IRIS_ECUDA;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t lc = pair_launch_config(sms - (sms & 1), 0, &attr);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, fused_gemm_coll_kernel<BN_WIDE, STAGES_PAIR, 2>, &lc);
    if (e != cudaSuccess || clusters < 1) return cuda_fail("cudaOccupancyMaxActiveClusters", static_cast<int>(e));
    g_pair_clusters[dev] = clusters;
    g_attr_done[dev] = true;
    return IRIS_OK;
}

// co-resident CTA pairs on the current device (0 on error)
int pair_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || ensure_attrs(dev) != IRIS_OK) return 0;
    return g_pair_clusters[dev];
}

int num_sms_current(int* n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IRIS_ECUDA;
    if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IRIS_ECUDA;
    return IRIS_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Resolved configuration.
struct Cfg {
    int tile_m;   // requested: 0 = per op default, 128, 256 (CTA pairs)
    int cg;       // resolved: 1 = one CTA per tile, 2 = CTA pairs
    int tile_n, group_m, gemm_ctas, comm_block, replicate, bias_on_m, grid;
    unsigned long long wait_ns;
    uint32_t debug_skip;
    int root;
    unsigned long long* trace;
    int trace_cap;
    int reduce_mode;  // resolved by the reduce ops (resolve_reduce_mode)
    int rank_inner;
    int stages;       // CTA pairs: requested 0 / 3 / 6, resolved by resolve_stages; one-CTA tiles: 0
    int coll_ring;    // concurrent collectives: buffers per worker warp
    int coll_evict_first;
    int coll_path;       // concurrent collectives: 1 TMA, 2 TMA loads + register stores, 3 one box of all sources
    int gather_parts;    // all_gather_matmul: gather items per (row block, shard)
    int startup_gather;  // all_gather_matmul: 0 = by M, 1 = worker copies, 2 = the TMA producer copies start-up gathers
    int gemm_evict_last; // CTA-pair operand loads with an L2 evict-last policy
    int out_evict_first; // final 16-bit output stores with an L2 evict-first policy
    int sum_l2_policy;   // chained reduce running sum: 0 none, 1 evict first, 2 evict last
    int k_split;         // all_gather_matmul: requested K chunks per tile (0 auto, 1 none)
    int coll_out_stage;  // summing collectives: 0 default (staged for all-reduce), 1 in place, 2 staged
};

int resolve_cfg(const iris_b200_config* c, iris_op op, int64_t N, Cfg& out) {
    iris_b200_config z;
    std::memset(&z, 0, sizeof(z));
    if (!c) c = &z;
    if (c->tile_m != 0 && c->tile_m != BM && c->tile_m != 2 * BM) return IRIS_EINVAL;
    if (c->tile_m == 2 * BM && c->tile_n != 0 && c->tile_n != 256) return IRIS_EINVAL;
    out.tile_m = c->tile_m;
    out.cg = 1;
    if (c->tile_k != 0 && c->tile_k != BK) return IRIS_EINVAL;
    if (c->stages != 0 && c->stages != STAGES_PAIR && c->stages != STAGES_PAIR_STREAM) return IRIS_EINVAL;
    out.stages = c->stages;
    if (c->tile_n != 0 && c->tile_n != 128 && c->tile_n != 256) return IRIS_EINVAL;
    out.tile_n = c->tile_n ? c->tile_n : (N <= 128 ? 128 : 256);
    if (c->group_m < 0) return IRIS_EINVAL;
    // 32 m-blocks per swizzle group (measured best on the reduce ops, where it
    // also keeps one rank's operands in L2 per group phase and spaces a
    // tile's W ranks several waves apart, and on all_gather_matmul); 16 for
    // the concurrent mode, whose GEMM shares the L2 with a streaming
    // collective (8192^3 beside an 8 x 64Mi all-reduce: 1.144 against 1.180 ms)
    out.group_m = c->group_m ? c->group_m : (op == IRIS_OP_CONCURRENT ? 16 : 32);
    // concurrent mode: 128Ki elements per collective item.  Beside an 8192^3
    // bf16 GEMM, W=8 fp32, 131072 against 65536: all-reduce 1.150 against
    // 1.175 ms, reduce-scatter 0.960 / 0.989, all-gather (8Mi) 0.993 / 1.012,
    // all-to-all 1.204 / 1.301, broadcast 0.998 / 1.019 (fewer stage leases
    // per byte); 262144 leaves too few items to balance (all-reduce 1.31 ms)
    out.comm_block = c->comm_block ? c->comm_block : 131072;
    if (out.comm_block < 0 || out.comm_block % 8 != 0) return IRIS_EINVAL;
    out.replicate = c->replicate_outputs ? 1 : 0;
    out.bias_on_m = c->bias_on_m ? 1 : 0;
    int sms = 0;
    if (num_sms_current(&sms) != IRIS_OK) return IRIS_ECUDA;
    if (c->grid < 0 || c->grid > sms) return IRIS_EINVAL;
    out.grid = c->grid ? c->grid : sms;
    if (c->gemm_ctas < -1 || c->gemm_ctas > out.grid) return IRIS_EINVAL;
    if (c->gemm_ctas != 0)
        out.gemm_ctas = c->gemm_ctas;
    else  // concurrent: 65% of the CTAs prefer the GEMM; others: all.  Beside an 8192^3
          // bf16 GEMM, W=8 fp32, 128Ki-element items, ms at 99 / 106 / 114 GEMM CTAs:
          // all-reduce 1.140 / 1.152 / 1.176, reduce-scatter 0.928 / 0.947 / 0.952,
          // all-to-all 1.193 / 1.198 / 1.205, all-gather (8Mi) 0.991 / 0.985 / 0.965,
          // broadcast 0.998 / 0.990 / 0.970 (with 64Ki-element items 106 was best)
        out.gemm_ctas = (op == IRIS_OP_CONCURRENT) ? std::max(1, (out.grid * 65 + 50) / 100) : out.grid;
    out.wait_ns = c->wait_ns ? c->wait_ns : DEFAULT_WAIT_NS;
    if (c->debug_skip_flag < 0) return IRIS_EINVAL;
    out.debug_skip = static_cast<uint32_t>(c->debug_skip_flag);
    if (c->root < 0 || c->root >= IRIS_MAX_WORLD) return IRIS_EINVAL;
    out.root = c->root;
    if (c->trace_buf && (c->trace_cap < 2 || (c->trace_buf & 7))) return IRIS_EINVAL;
    out.trace = reinterpret_cast<unsigned long long*>(c->trace_buf);
    out.trace_cap = c->trace_buf ? c->trace_cap : 0;
    if (c->reduce_mode < 0 || c->reduce_mode > 3) return IRIS_EINVAL;
    out.reduce_mode = c->reduce_mode;
    out.rank_inner = c->rank_inner ? 1 : 0;
    if (c->coll_ring != 0 && (c->coll_ring < 1 || c->coll_ring > MAX_COLL_RING)) return IRIS_EINVAL;
    out.coll_ring = c->coll_ring ? c->coll_ring : 2;
    if (c->coll_l2_hint < 0 || c->coll_l2_hint > 2) return IRIS_EINVAL;
    out.coll_evict_first = c->coll_l2_hint == 1 ? 1 : 0;
    if (c->gather_parts < 0 || c->gather_parts > 16) return IRIS_EINVAL;
    // one gather item per (128-row block, shard) copy: splitting it in row
    // parts measured slower on every shape tried (more claims contending on
    // the comm queue counter and more per-item synchronisation)
    out.gather_parts = c->gather_parts ? c->gather_parts : 1;
    // CTA-pair operand loads evict last by default: they then keep their
    // place in the L2 against the outputs, partial sums and collective data
    // streaming through it (measured 0.7-1.4 % faster on all four fused ops)
    if (c->gemm_l2_hint < 0 || c->gemm_l2_hint > 2) return IRIS_EINVAL;
    out.gemm_evict_last = c->gemm_l2_hint == 2 ? 0 : 1;
    if (c->sum_l2_hint < 0 || c->sum_l2_hint > 3) return IRIS_EINVAL;
    out.sum_l2_policy = c->sum_l2_hint == 1 ? 1 : c->sum_l2_hint == 2 ? 2 : 0;
    if (c->out_l2_hint < 0 || c->out_l2_hint > 2) return IRIS_EINVAL;
    out.out_evict_first = c->out_l2_hint == 1 ? 1 : 0;
    if (c->k_split < 0 || c->k_split > 4096) return IRIS_EINVAL;
    out.k_split = c->k_split;
    if (c->coll_out_stage < 0 || c->coll_out_stage > 2) return IRIS_EINVAL;
    out.coll_out_stage = c->coll_out_stage;
    if (c->startup_gather < 0 || c->startup_gather > 2) return IRIS_EINVAL;
    out.startup_gather = c->startup_gather;
    if (c->coll_path < 0 || c->coll_path > 3) return IRIS_EINVAL;
    out.coll_path = c->coll_path;  // 0: chosen per collective (resolve_coll_path)
    return IRIS_OK;
}

// Reduce schedule of matmul_reduce_scatter / matmul_all_reduce: 1 = comm
// queue, 2 = distributed parts, 3 = chained through the epilogues (needs every
// rank's output slice in whole 32-column chunks).  0 (auto) picks 3 when it
// applies, else 2.  Returns -1 for an invalid request.
int resolve_reduce_mode(const iris_b200_config* c, iris_op op, int64_t N, int W) {
    const int req = c ? c->reduce_mode : 0;
    const int64_t slice = (op == IRIS_OP_MATMUL_REDUCE_SCATTER && W > 0) ? N / W : N;
    const bool chain_ok = N % 32 == 0 && slice % 32 == 0;
    if (req == 0) return chain_ok ? 3 : 2;
    if (req == 1 || req == 2) return req;
    if (req == 3) return chain_ok ? 3 : -1;
    return -1;
}

// CTA pairs (tile_m 256) wherever they apply: 256-wide tiles, the chained
// schedule for the reduce ops, and a GEMM in the launch (a collective-only
// launch of the concurrent mode keeps one CTA per item).  The default is
// pairs; tile_m 128 keeps one CTA per tile.  The pair grid is every
// co-resident pair (at most grid / 2).
// CTA pairs: the pipeline by K unless the config chose one
void resolve_stages(Cfg& c, int64_t K) {
    if (c.cg != 2) {
        c.stages = 0;
        return;
    }
    if (c.stages == 0) c.stages = K > STREAM_K ? STAGES_PAIR_STREAM : STAGES_PAIR;
}

// all_gather_matmul split-K: the K chunks per output tile and the K blocks per
// chunk (a whole number of two-K-block stages), or {1, 0} for none.  It needs
// CTA pairs, the chained reduce's whole 32-column chunks (N % 32 == 0) and
// K > 0; by default it applies above 2 x SPLIT_K_CHUNK.
struct SplitK {
    int split, kb_chunk;
};
SplitK resolve_split(int k_split, bool pairs, int64_t M, int64_t N, int64_t K) {
    SplitK r{1, 0};
    if (!pairs || M <= 0 || K <= 0 || N % 32 != 0 || k_split == 1) return r;
    const int64_t want = k_split > 1 ? k_split : (K > 2 * SPLIT_K_CHUNK ? cdiv(K, SPLIT_K_CHUNK) : 1);
    if (want <= 1) return r;
    const int64_t kblocks = cdiv(K, BK);
    int64_t kbc = cdiv(kblocks, want);
    kbc += kbc & 1;
    const int64_t split = cdiv(kblocks, kbc);
    if (split <= 1) return r;
    r.split = static_cast<int>(split);
    r.kb_chunk = static_cast<int>(kbc);
    return r;
}

int resolve_pair(Cfg& c, iris_op op, bool has_gemm = true) {
    const bool reduce_op = op == IRIS_OP_MATMUL_REDUCE_SCATTER || op == IRIS_OP_MATMUL_ALL_REDUCE;
    const bool applies = has_gemm && c.tile_n == BN_WIDE && (!reduce_op || c.reduce_mode == 3);
    if (c.tile_m == 2 * BM && !applies && has_gemm) return IRIS_EINVAL;
    c.cg = (c.tile_m == BM || !applies) ? 1 : 2;
    if (c.cg == 1 && c.stages != 0 && has_gemm) return IRIS_EINVAL;  // the pipeline choice is the pairs'
    if (c.cg == 2) {
        const int pairs = std::min(pair_clusters(), c.grid / 2);
        if (pairs < 1) {
            if (c.tile_m == 2 * BM || c.stages != 0) return c.grid < 2 ? IRIS_EINVAL : IRIS_ECUDA;
            c.cg = 1;
            return IRIS_OK;
        }
        c.grid = 2 * pairs;
        c.gemm_ctas = std::min(c.gemm_ctas, c.grid);
    }
    return IRIS_OK;
}

// Sizes of the workspace pieces for one call.
struct WsLayout {
    size_t flags_off, n_flags, partial_off, partial_elems, total;
};

WsLayout ws_layout(iris_op op, int64_t M, int64_t N, int W, int tile_n, int reduce_mode, int split = 1) {
    WsLayout L{};
    L.flags_off = WS_HEADER;
    const int64_t mb = cdiv(M, BM), nb = cdiv(N, tile_n);
    const bool reduce_op = op == IRIS_OP_MATMUL_REDUCE_SCATTER || op == IRIS_OP_MATMUL_ALL_REDUCE;
    if (op == IRIS_OP_ALL_GATHER_MATMUL)
        // 8-byte ready counters per (128-row block, shard); split-K: then one
        // 8-byte chained-reduce counter per tile
        L.n_flags = 2 * static_cast<size_t>(W) * mb + (split > 1 ? 2 * static_cast<size_t>(mb) * nb : 0);
    else if (op == IRIS_OP_MATMUL_ALL_GATHER && split > 1)
        // split-K: one 8-byte chained-reduce counter per (rank, 128-row block, tile column)
        L.n_flags = 2 * static_cast<size_t>(W) * static_cast<size_t>(cdiv(M / std::max(W, 1), BM)) * nb;
    else if (reduce_op)
        L.n_flags = static_cast<size_t>(std::max(W, 2)) * mb * nb;  // also 8-byte tile counters
    L.partial_off = round_up(L.flags_off + L.n_flags * 4, 256);
    if (reduce_op || ((op == IRIS_OP_ALL_GATHER_MATMUL || op == IRIS_OP_MATMUL_ALL_GATHER) && split > 1))
        L.partial_elems = static_cast<size_t>(M) * N;
    // one fp32 running sum (chained) or one fp32 partial per rank
    const size_t copies = L.partial_elems ? ((reduce_mode == 3 || !reduce_op) ? 1 : W) : 0;
    L.total = round_up(L.partial_off + L.partial_elems * 4 * copies, 256);
    return L;
}

bool aligned16(size_t x) { return (x & 15) == 0; }

// tensor [off, off+bytes) inside a heap region, 16-byte aligned
int check_region(const iris_b200_heap* h, size_t off, size_t bytes) {
    if (!aligned16(off)) return IRIS_EALIGN;
    if (off > h->rank_stride || bytes > h->rank_stride - off) return IRIS_EINVAL;
    return IRIS_OK;
}

int check_heap(const iris_b200_heap* h) {
    if (!h || !h->base) return IRIS_EINVAL;
    if (h->world < 1 || h->world > IRIS_MAX_WORLD) return IRIS_EINVAL;
    if (!aligned16(h->rank_stride) || !aligned16(reinterpret_cast<uintptr_t>(h->base))) return IRIS_EALIGN;
    return IRIS_OK;
}

int make_map(CUtensorMap* m, const void* base, int bf16, uint64_t d0, uint64_t d1, uint64_t d2,
             uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1) {
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? IRIS_OK : cuda_fail("cuTensorMapEncodeTiled (operand)", static_cast<int>(r));
}

// B as 64-column chunks: 4-D {64, k, n / 64, region} (strides N * 2, 128,
// region), box {64, BK * KS, tile_n / cg / 64, 1}.  One load fills all of a
// CTA's B columns for a stage, chunk after chunk 64 KS x 128 B apart -- the
// layout the 3-D map's per-chunk loads produce.  Only when N % 64 == 0, so
// that no chunk runs past the end of a row; otherwise the 3-D map serves alone.
int make_b_chunk_map(Params& p, const Cfg& c, const void* base, int64_t N, int64_t K, uint64_t regions,
                     uint64_t region_stride) {
    p.b_chunked = 0;
    if (N % 64 != 0 || N <= 0 || K <= 0) return IRIS_OK;
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N / 64), regions};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(N) * 2, 128, region_stride};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(BK * k_per_stage(c.cg, c.stages)),
                         static_cast<cuuint32_t>(c.tile_n / c.cg / 64), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(&p.tmBc, p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                     const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail("cuTensorMapEncodeTiled (B chunks)", static_cast<int>(r));
    p.b_chunked = 1;
    return IRIS_OK;
}

// A as 64-column K chunks (CTA pairs, whose stages hold KS > 1 K blocks):
// 4-D {64, row, k / 64, region} (strides K * 2, 128, region), box {64, BM,
// KS, 1}: one load fills a stage's KS chunks of the CTA's 128 rows, 16 KB
// apart.  Only when K % 64 == 0, so that no chunk runs past the end of a row.
int make_a_chunk_map(Params& p, const Cfg& c, const void* base, int64_t rows, int64_t K, uint64_t regions,
                     uint64_t region_stride) {
    p.a_chunked = 0;
    const int ks = k_per_stage(c.cg, c.stages);
    if (ks == 1 || K % 64 != 0 || K <= 0 || rows <= 0) return IRIS_OK;
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 64), regions};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(K) * 2, 128, region_stride};
    cuuint32_t box[4] = {64, BM, static_cast<cuuint32_t>(ks), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(&p.tmAc, p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                     const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail("cuTensorMapEncodeTiled (A chunks)", static_cast<int>(r));
    p.a_chunked = 1;
    return IRIS_OK;
}

// all_gather_matmul start-up gathers by the TMA producer: the shards as 3-D
// {K_l, M, W} (regions rank_stride apart) and the gathered buffer as 3-D
// {K, M, 1}, both with an unswizzled box {gi, 128, 1}, gi the widest of 256,
// 128, ..., 8 columns dividing K_l.  A box lands in shared memory as 128 rows
// of gi columns and leaves the same way.
int make_gather_maps(Params& p, const iris_b200_heap* heap, size_t off_A, size_t off_gathered, int64_t M,
                     int64_t K, int64_t K_l) {
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    int gi = 256;
    while (K_l % gi != 0) gi /= 2;
    p.gather_box = gi;
    const CUtensorMapDataType dt = p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint32_t box[3] = {static_cast<cuuint32_t>(gi), BM, 1};
    cuuint32_t es[3] = {1, 1, 1};
    cuuint64_t sdims[3] = {static_cast<cuuint64_t>(K_l), static_cast<cuuint64_t>(M),
                           static_cast<cuuint64_t>(heap->world)};
    cuuint64_t sstrides[2] = {static_cast<cuuint64_t>(K_l) * 2, heap->rank_stride};
    CUresult r = enc(&p.tmGs, dt, 3, static_cast<char*>(heap->base) + off_A, sdims, sstrides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail("cuTensorMapEncodeTiled (gather source)", static_cast<int>(r));
    cuuint64_t ddims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M), 1};
    cuuint64_t dstrides[2] = {static_cast<cuuint64_t>(K) * 2, round_up(size_t(M) * K * 2, 16)};
    r = enc(&p.tmGd, dt, 3, static_cast<char*>(heap->base) + off_gathered, ddims, dstrides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? IRIS_OK : cuda_fail("cuTensorMapEncodeTiled (gather destination)", static_cast<int>(r));
}

// Concurrent all-reduce / reduce-scatter input for coll_path 3: 3-D fp32
// {256, count / 256, W} (1 KB rows, regions rank_stride apart), box {256, R,
// W}: one load brings R rows of every source.
int make_coll_map(Params& p, const void* base, int64_t count, int W, uint64_t region_stride, int R) {
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    cuuint64_t dims[3] = {256, static_cast<cuuint64_t>(count / 256), static_cast<cuuint64_t>(W)};
    cuuint64_t strides[2] = {1024, region_stride};
    cuuint32_t box[3] = {256, static_cast<cuuint32_t>(R), static_cast<cuuint32_t>(W)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(&p.tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? IRIS_OK : cuda_fail("cuTensorMapEncodeTiled (collective input)", static_cast<int>(r));
}

// Output map: 4-D {n, row, row block, region} with a 32 x 32 box, written by
// the epilogue's TMA stores.  fp32 (partials) use the 128-byte swizzle (one
// 128-byte staging row), 16-bit outputs the 64-byte swizzle.
int make_out_map(CUtensorMap* m, const void* base, int kind /*0 f16, 1 bf16, 2 f32*/, uint64_t n,
                 uint64_t rows, uint64_t blocks, uint64_t regions, uint64_t row_pitch, uint64_t block_pitch,
                 uint64_t region_pitch) {
    EncodeTiledFn enc = encoder();
    if (!enc) return IRIS_ECUDA;
    cuuint64_t dims[4] = {n, rows, blocks, regions};
    cuuint64_t strides[3] = {row_pitch, block_pitch, region_pitch};
    cuuint32_t box[4] = {32, 32, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = kind == 2   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : kind == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     kind == 2 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? IRIS_OK : cuda_fail("cuTensorMapEncodeTiled (output)", static_cast<int>(r));
}

void fill_geometry(Params& p, int64_t M_rows, int64_t N, int64_t K, int m_blocks, const Cfg& c) {
    p.M = static_cast<int>(M_rows);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.m_blocks = m_blocks;
    p.n_blocks = static_cast<int>(cdiv(N, c.tile_n));
    p.k_blocks = static_cast<int>(cdiv(K, BK));
    // CTA pairs: an m-block is 2 x 128 rows; group_m stays in 128-row units
    p.group_m = std::max(1, c.group_m / c.cg);
    p.n_tiles = p.m_blocks * p.n_blocks;
    p.gemm_ctas = c.gemm_ctas;
    p.first_wave = static_cast<uint32_t>(c.grid / c.cg);
    // all_gather_matmul claims a swizzle group's gathers while the group before
    // it runs (measured: long-K shapes lose ~20 % with a one-wave look-ahead)
    p.lookahead = static_cast<uint32_t>(p.group_m) * p.n_blocks;
    p.replicate = c.replicate;
    p.bias_on_m = c.bias_on_m;
    p.wait_ns = c.wait_ns;
    p.debug_skip = c.debug_skip;
    p.trace = c.trace;
    p.trace_cap = c.trace_cap;
    p.reduce_mode = c.reduce_mode;
    p.rank_inner = c.rank_inner;
    p.coll_ring = c.coll_ring;
    p.coll_evict_first = c.coll_evict_first;
    p.coll_path = c.coll_path;
    p.coll_out_stage = c.coll_out_stage;
    p.gemm_evict_last = c.gemm_evict_last;
    p.out_evict_first = c.out_evict_first;
    p.sum_l2_policy = c.sum_l2_policy;
}

int launch(Params& p, Cfg c, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IRIS_ECUDA;
    int rc = ensure_attrs(dev);
    if (rc != IRIS_OK) return rc;
    // A dependent op with fewer work items than CTAs (pairs) runs one CTA
    // (pair) per item: the idle ones would only add set-up, tensor-memory
    // allocation and queue polling (W=2 256^3 all_gather_matmul: 22.5 us per
    // step on 152 CTAs, 20.5 us on 4-76).  The concurrent mode keeps its
    // grid, whose split between the queues is the caller's.
    if (p.op != OP_CONC) {
        const uint64_t items = static_cast<uint64_t>(p.n_gemm) + p.n_comm + p.n_parts;
        const uint64_t need = std::max<uint64_t>(1, items) * static_cast<uint64_t>(c.cg);
        if (need < static_cast<uint64_t>(c.grid)) {
            c.grid = static_cast<int>(need);
            p.first_wave = static_cast<uint32_t>(c.grid / c.cg);
            p.gemm_ctas = std::min(p.gemm_ctas, c.grid);
        }
    }
    if (c.cg == 2) {
        cudaLaunchAttribute attr;
        const bool stream_k = c.stages == STAGES_PAIR_STREAM;
        const cudaLaunchConfig_t lc =
            pair_launch_config(c.grid, stream, &attr,
                               stream_k ? smem_bytes<BN_WIDE, STAGES_PAIR_STREAM, 2>() : smem_bytes<BN_WIDE, STAGES_PAIR, 2>());
        const cudaError_t e = stream_k ? cudaLaunchKernelEx(&lc, fused_gemm_coll_kernel<BN_WIDE, STAGES_PAIR_STREAM, 2>, p)
                                       : cudaLaunchKernelEx(&lc, fused_gemm_coll_kernel<BN_WIDE, STAGES_PAIR, 2>, p);
        if (e != cudaSuccess) return cuda_fail("kernel launch (CTA pairs)", static_cast<int>(e));
    } else if (c.tile_n == BN_WIDE) {
        fused_gemm_coll_kernel<BN_WIDE, STAGES_WIDE, 1>
            <<<c.grid, NUM_THREADS, smem_bytes<BN_WIDE, STAGES_WIDE, 1>(), stream>>>(p);
    } else {
        fused_gemm_coll_kernel<BN_NARROW, STAGES_NARROW, 1>
            <<<c.grid, NUM_THREADS, smem_bytes<BN_NARROW, STAGES_NARROW, 1>(), stream>>>(p);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? IRIS_OK : cuda_fail("kernel launch", static_cast<int>(e));
}

// The last wave of GEMM items is partly empty when the item count is not a
// multiple of the CTA pairs.  When at most half the pairs would get a tile in
// it, those tail tiles are split into column halves (N = BN / 2) so the wave
// takes half a tile's time.  Reduce ops split only the last rank's tiles (the
// chained reduce keeps one counter per whole tile), which in the rank-major
// order are the final items of the last swizzle group.
void tail_split(Params& p, const Cfg& c, bool reduce_op) {
    p.g_split = p.n_gemm;
    if (c.cg != 2 || p.n_gemm == 0 || c.tile_n != BN_WIDE) return;
    if (reduce_op && (c.reduce_mode != 3 || c.rank_inner)) return;
    const uint32_t pairs = static_cast<uint32_t>(c.grid / 2);
    const uint32_t T = p.n_gemm;
    const uint32_t tail = T % pairs;
    if (tail == 0 || 2 * tail > pairs) return;
    if (reduce_op) {
        const uint32_t Tg = static_cast<uint32_t>(p.group_m) * p.n_blocks;
        const uint32_t last_sg = (static_cast<uint32_t>(p.n_tiles) - 1) / Tg;
        const uint32_t Tsg = std::min(Tg, static_cast<uint32_t>(p.n_tiles) - last_sg * Tg);
        if (tail > Tsg) return;
    }
    p.g_split = T - tail;
    p.n_gemm = T + tail;
}

bool dims_ok(int64_t M, int64_t N, int64_t K) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    return M >= 0 && N >= 0 && K >= 0 && M <= lim && N <= lim && K <= lim;
}

int prepare_ws(Params& p, void* ws, size_t ws_bytes, iris_op op, int64_t M, int64_t N, int W,
               const Cfg& c) {
    const int split = ((op == IRIS_OP_ALL_GATHER_MATMUL || op == IRIS_OP_MATMUL_ALL_GATHER) && p.split > 1) ? p.split : 1;
    const WsLayout L = ws_layout(op, M, N, W, c.tile_n, c.reduce_mode, split);
    if (!ws || ws_bytes < L.total) return IRIS_ENOWS;
    if (!aligned16(reinterpret_cast<uintptr_t>(ws))) return IRIS_EALIGN;
    p.ws = reinterpret_cast<WsHeader*>(ws);
    p.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + L.flags_off);
    // split-K: the chained-reduce counters (all_gather_matmul: after the W x
    // m-block gather counters)
    p.chain = reinterpret_cast<unsigned long long*>(p.flags) +
              (op == IRIS_OP_ALL_GATHER_MATMUL ? static_cast<size_t>(W) * cdiv(M, BM) : 0);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + L.partial_off);
    p.partial_elems = L.partial_elems;
    return IRIS_OK;
}

}  // namespace

extern "C" {

const char* iris_b200_strerror(int code) {
    switch (code) {
        case IRIS_OK: return "ok";
        case IRIS_EINVAL: return "invalid argument";
        case IRIS_EALIGN: return "misaligned offset or row pitch (16-byte rule)";
        case IRIS_ENOWS: return "workspace missing or too small";
        case IRIS_ECUDA: return "CUDA error";
        case IRIS_ETIMEOUT: return "a bounded device wait gave up";
        case IRIS_EUNSUPPORTED: return "unsupported request";
        default: return "unknown error";
    }
}

int iris_b200_num_sms(int* n) {
    if (!n) return IRIS_EINVAL;
    return num_sms_current(n);
}

int iris_b200_workspace_size(iris_op op, int64_t M, int64_t N, int64_t K, int world, iris_dtype dtype,
                             const iris_b200_config* cfg, size_t* bytes) {
    if (!bytes || !dims_ok(M, N, K) || world < 1 || world > IRIS_MAX_WORLD) return IRIS_EINVAL;
    if (op < IRIS_OP_ALL_GATHER_MATMUL || op > IRIS_OP_CONCURRENT) return IRIS_EINVAL;
    (void)dtype;
    if (cfg && cfg->stages != 0 && cfg->stages != STAGES_PAIR && cfg->stages != STAGES_PAIR_STREAM) return IRIS_EINVAL;
    int tile_n = 256;
    if (cfg && cfg->tile_n) {
        if (cfg->tile_n != 128 && cfg->tile_n != 256) return IRIS_EINVAL;
        tile_n = cfg->tile_n;
    } else if (N <= 128) {
        tile_n = 128;
    }
    int64_t Mrows = M;
    if (op == IRIS_OP_MATMUL_ALL_GATHER) Mrows = 0;  // no flags or partials
    int mode = 0;
    if (op == IRIS_OP_MATMUL_REDUCE_SCATTER || op == IRIS_OP_MATMUL_ALL_REDUCE) {
        mode = resolve_reduce_mode(cfg, op, N, world);
        if (mode < 0) return IRIS_EINVAL;
    }
    int split = 1;
    if (op == IRIS_OP_ALL_GATHER_MATMUL || op == IRIS_OP_MATMUL_ALL_GATHER) {
        // sized for CTA pairs wherever the config allows them (a launch that
        // ends up on one-CTA tiles does not split and uses less)
        const int ks = cfg ? cfg->k_split : 0;
        if (ks < 0 || ks > 4096) return IRIS_EINVAL;
        const bool pairs = !(cfg && (cfg->tile_m == BM || (cfg->tile_n != 0 && cfg->tile_n != 256))) && N > 128;
        const int64_t rows = op == IRIS_OP_MATMUL_ALL_GATHER ? M / world : M;
        split = resolve_split(ks, pairs, rows, N, K).split;
        if (op == IRIS_OP_MATMUL_ALL_GATHER && split > 1) Mrows = M;  // counters and the running sum
    }
    *bytes = ws_layout(op, Mrows, N, world, tile_n, mode, split).total;
    return IRIS_OK;
}

int iris_b200_all_gather_matmul(const iris_b200_heap* heap, size_t off_A, size_t off_B, size_t off_bias,
                                size_t off_out, size_t off_gathered, int64_t M, int64_t N, int64_t K,
                                iris_dtype dtype, const iris_b200_config* cfg, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
    int rc = check_heap(heap);
    if (rc) return rc;
    if (!dims_ok(M, N, K) || (dtype != IRIS_F16 && dtype != IRIS_BF16)) return IRIS_EINVAL;
    const int W = heap->world;
    if (K % W != 0) return IRIS_EINVAL;
    const int64_t K_l = K / W;
    if (K_l % 8 != 0 || N % 8 != 0) return IRIS_EALIGN;
    Cfg c;
    if ((rc = resolve_cfg(cfg, IRIS_OP_ALL_GATHER_MATMUL, N, c))) return rc;
    if ((rc = resolve_pair(c, IRIS_OP_ALL_GATHER_MATMUL))) return rc;
    const SplitK sk = resolve_split(c.k_split, c.cg == 2, M, N, K);
    // the pipeline by the K one item runs
    resolve_stages(c, sk.split > 1 ? int64_t(sk.kb_chunk) * BK : K);
    if ((rc = check_region(heap, off_A, size_t(M) * K_l * 2))) return rc;
    if ((rc = check_region(heap, off_B, size_t(K) * N * 2))) return rc;
    if ((rc = check_region(heap, off_out, size_t(M) * N * 2))) return rc;
    if ((rc = check_region(heap, off_gathered, size_t(M) * K * 2))) return rc;
    const bool has_bias = off_bias != IRIS_NO_BIAS;
    if (has_bias && (rc = check_region(heap, off_bias, size_t(c.bias_on_m ? M : N) * 2))) return rc;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.op = OP_AG_MM;
    p.W = W;
    p.bf16 = dtype == IRIS_BF16;
    const int mblocks = static_cast<int>(cdiv(M, BM * c.cg));
    fill_geometry(p, M, N, K, mblocks, c);
    p.mb_per_rank = mblocks;
    p.K_local = static_cast<int>(K_l);
    p.heap = static_cast<char*>(heap->base);
    p.rank_stride = heap->rank_stride;
    p.off_A = off_A;
    p.off_out = off_out;
    p.off_gathered = off_gathered;
    p.off_bias = has_bias ? off_bias : 0;
    p.has_bias = has_bias;
    p.n_gemm = (M > 0 && N > 0) ? static_cast<uint32_t>(p.n_tiles) : 0u;
    if (sk.split > 1) {
        // chunk j of every tile is an item; the chunks' partials are summed
        // in chunk order by the chained reduce (one fp32 running sum)
        if (uint64_t(p.n_gemm) * sk.split >= 0x7FFFFFFFull) return IRIS_EINVAL;
        p.split = sk.split;
        p.kb_chunk = sk.kb_chunk;
        p.n_gemm *= static_cast<uint32_t>(sk.split);
        p.reduce_mode = 3;
        p.rank_inner = 0;
        // gathers claimed a whole swizzle group (all its chunks) ahead
        p.lookahead *= static_cast<uint32_t>(sk.split);
    }
    p.gather_parts = c.gather_parts;
    // the producer's start-up copies move whole 128-row blocks.  By default
    // the producer takes them up to 16384 rows when an item's K is at most
    // 32768 (split or not), where the first swizzle group's gathers hold
    // back a larger share of the launch (0.4-2.4 % faster over the PR #506
    // shapes of that size, about 1 us off a 256^3 launch); the workers take
    // them beyond 16384 rows (within 0.5 % either way there) and for unsplit
    // long K, where the producer's copies delay its own first tile
    const int64_t item_k = sk.split > 1 ? int64_t(sk.kb_chunk) * BK : K;
    const int startup = c.startup_gather ? c.startup_gather : (M <= 16384 && item_k <= 32768 ? 2 : 1);
    p.startup_gather = (startup == 2 && c.gather_parts == 1 && M > 0 && K_l > 0) ? 1 : 0;
    if (p.startup_gather && (rc = make_gather_maps(p, heap, off_A, off_gathered, M, K, K_l))) return rc;
    if (int64_t(mblocks) * W * c.gather_parts >= 0x7FFFFFFF) return IRIS_EINVAL;
    p.n_comm = static_cast<uint32_t>(mblocks) * W * c.gather_parts;
    if (sk.split > 1)
        p.g_split = p.n_gemm;  // no column-half tail items (the chain counts whole tiles)
    else
        tail_split(p, c, false);
    if ((rc = prepare_ws(p, workspace, workspace_bytes, IRIS_OP_ALL_GATHER_MATMUL, M, N, W, c))) return rc;
    if (p.n_gemm > 0 && K > 0) {
        char* g = p.heap + off_gathered;
        if ((rc = make_map(&p.tmA, g, p.bf16, K, M, 1, K * 2, round_up(size_t(M) * K * 2, 16), BK, BM))) return rc;
        if ((rc = make_a_chunk_map(p, c, g, M, K, 1, round_up(size_t(M) * K * 2, 16)))) return rc;
        if ((rc = make_map(&p.tmB, p.heap + off_B, p.bf16, N, K, 1, N * 2, round_up(size_t(K) * N * 2, 16), 64,
                           BK * k_per_stage(c.cg, c.stages))))
            return rc;
        if ((rc = make_b_chunk_map(p, c, p.heap + off_B, N, K, 1, round_up(size_t(K) * N * 2, 16)))) return rc;
    }
    if (p.n_gemm > 0 &&
        (rc = make_out_map(&p.tmC, p.heap + off_out, p.bf16, N, M, 1, W, N * 2, size_t(M) * N * 2, heap->rank_stride)))
        return rc;
    // split-K: the fp32 running sum of the chunks
    if (p.split > 1 &&
        (rc = make_out_map(&p.tmS, p.partials, 2, N, M, 1, 1, N * 4, size_t(M) * N * 4, size_t(M) * N * 4)))
        return rc;
    return launch(p, c, stream);
}

static int mm_reduce_common(iris_op op, const iris_b200_heap* heap, size_t off_A, size_t off_B,
                            size_t off_bias, size_t off_out, int64_t M, int64_t N, int64_t K,
                            iris_dtype dtype, const iris_b200_config* cfg, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    int rc = check_heap(heap);
    if (rc) return rc;
    if (!dims_ok(M, N, K) || (dtype != IRIS_F16 && dtype != IRIS_BF16)) return IRIS_EINVAL;
    const int W = heap->world;
    int64_t N_l = N;
    if (op == IRIS_OP_MATMUL_REDUCE_SCATTER) {
        if (N % W != 0) return IRIS_EINVAL;
        N_l = N / W;
    }
    if (K % 8 != 0 || N % 8 != 0 || N_l % 8 != 0) return IRIS_EALIGN;
    Cfg c;
    if ((rc = resolve_cfg(cfg, op, N, c))) return rc;
    // a rank's A larger than 64 MB: swizzle groups of 16 blocks, so a group's
    // A panels stay in L2 while its B streams (8192^3 W=8: 4.81 against
    // 4.86 ms; 4096^3 W=4 keeps 32)
    if ((!cfg || cfg->group_m == 0) && size_t(M) * size_t(K) * 2 > (size_t(64) << 20)) c.group_m = 16;
    c.reduce_mode = resolve_reduce_mode(cfg, op, N, W);
    if (c.reduce_mode < 0) return IRIS_EINVAL;
    if ((rc = resolve_pair(c, op))) return rc;
    // split-K rides on the chained reduce: the chain then runs over (rank, chunk)
    const SplitK sk = c.reduce_mode == 3 ? resolve_split(c.k_split, c.cg == 2, M, N, K) : SplitK{1, 0};
    resolve_stages(c, sk.split > 1 ? int64_t(sk.kb_chunk) * BK : K);
    if ((rc = check_region(heap, off_A, size_t(M) * K * 2))) return rc;
    if ((rc = check_region(heap, off_B, size_t(K) * N * 2))) return rc;
    if ((rc = check_region(heap, off_out, size_t(M) * N_l * 2))) return rc;
    const bool has_bias = off_bias != IRIS_NO_BIAS;
    if (has_bias && (rc = check_region(heap, off_bias, size_t(c.bias_on_m ? M : N) * 2))) return rc;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.op = (op == IRIS_OP_MATMUL_REDUCE_SCATTER) ? OP_MM_RS : OP_MM_AR;
    p.W = W;
    p.bf16 = dtype == IRIS_BF16;
    const int mblocks = static_cast<int>(cdiv(M, BM * c.cg));
    fill_geometry(p, M, N, K, mblocks, c);
    p.mb_per_rank = mblocks;
    p.N_local = static_cast<int>(N_l);
    p.heap = static_cast<char*>(heap->base);
    p.rank_stride = heap->rank_stride;
    p.off_A = off_A;
    p.off_out = off_out;
    p.off_bias = has_bias ? off_bias : 0;
    p.has_bias = has_bias;
    const uint64_t tiles = (M > 0 && N > 0) ? uint64_t(p.n_tiles) : 0;
    if (tiles * W * sk.split >= 0x7FFFFFFFull) return IRIS_EINVAL;
    p.n_gemm = static_cast<uint32_t>(tiles * W * sk.split);
    p.n_comm = c.reduce_mode == 1 ? static_cast<uint32_t>(tiles) : 0u;
    p.n_parts = c.reduce_mode == 2 ? static_cast<uint32_t>(tiles * W) : 0u;
    if (sk.split > 1) {
        p.split = sk.split;
        p.kb_chunk = sk.kb_chunk;
        p.rank_inner = 0;
        p.g_split = p.n_gemm;  // no column-half tail items
    } else {
        tail_split(p, c, true);
    }
    if ((rc = prepare_ws(p, workspace, workspace_bytes, op, M, N, W, c))) return rc;
    if (p.n_gemm > 0 && K > 0) {
        if ((rc = make_map(&p.tmA, p.heap + off_A, p.bf16, K, M, W, K * 2, heap->rank_stride, BK, BM))) return rc;
        if ((rc = make_a_chunk_map(p, c, p.heap + off_A, M, K, W, heap->rank_stride))) return rc;
        if ((rc = make_map(&p.tmB, p.heap + off_B, p.bf16, N, K, W, N * 2, heap->rank_stride, 64,
                           BK * k_per_stage(c.cg, c.stages))))
            return rc;
        if ((rc = make_b_chunk_map(p, c, p.heap + off_B, N, K, W, heap->rank_stride))) return rc;
    }
    if (p.n_gemm > 0) {
        if (c.reduce_mode == 3) {
            // running sum (fp32) and the 16-bit output written by the last rank
            if ((rc = make_out_map(&p.tmS, p.partials, 2, N, M, 1, 1, N * 4, size_t(M) * N * 4, size_t(M) * N * 4)))
                return rc;
            if (op == IRIS_OP_MATMUL_REDUCE_SCATTER)
                rc = make_out_map(&p.tmC, p.heap + off_out, p.bf16, N_l, M, W, 1, N_l * 2, heap->rank_stride,
                                  heap->rank_stride * W);
            else
                rc = make_out_map(&p.tmC, p.heap + off_out, p.bf16, N, M, 1, W, N * 2, size_t(M) * N * 2,
                                  heap->rank_stride);
            if (rc) return rc;
        } else if ((rc = make_out_map(&p.tmC, p.partials, 2, N, M, W, 1, N * 4, size_t(M) * N * 4,
                                      size_t(W) * M * N * 4))) {
            return rc;
        }
    }
    return launch(p, c, stream);
}

int iris_b200_matmul_reduce_scatter(const iris_b200_heap* heap, size_t off_A, size_t off_B, size_t off_bias,
                                    size_t off_out, int64_t M, int64_t N, int64_t K, iris_dtype dtype,
                                    const iris_b200_config* cfg, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    return mm_reduce_common(IRIS_OP_MATMUL_REDUCE_SCATTER, heap, off_A, off_B, off_bias, off_out, M, N, K,
                            dtype, cfg, workspace, workspace_bytes, stream);
}

int iris_b200_matmul_all_reduce(const iris_b200_heap* heap, size_t off_A, size_t off_B, size_t off_bias,
                                size_t off_out, int64_t M, int64_t N, int64_t K, iris_dtype dtype,
                                const iris_b200_config* cfg, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    return mm_reduce_common(IRIS_OP_MATMUL_ALL_REDUCE, heap, off_A, off_B, off_bias, off_out, M, N, K, dtype,
                            cfg, workspace, workspace_bytes, stream);
}

int iris_b200_matmul_all_gather(const iris_b200_heap* heap, size_t off_A, size_t off_B, size_t off_bias,
                                size_t off_out, int64_t M, int64_t N, int64_t K, iris_dtype dtype,
                                const iris_b200_config* cfg, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    int rc = check_heap(heap);
    if (rc) return rc;
    if (!dims_ok(M, N, K) || (dtype != IRIS_F16 && dtype != IRIS_BF16)) return IRIS_EINVAL;
    const int W = heap->world;
    if (M % W != 0) return IRIS_EINVAL;
    const int64_t M_l = M / W;
    if (K % 8 != 0 || N % 8 != 0) return IRIS_EALIGN;
    Cfg c;
    if ((rc = resolve_cfg(cfg, IRIS_OP_MATMUL_ALL_GATHER, N, c))) return rc;
    if ((rc = resolve_pair(c, IRIS_OP_MATMUL_ALL_GATHER))) return rc;
    const SplitK sk = resolve_split(c.k_split, c.cg == 2, M_l, N, K);
    resolve_stages(c, sk.split > 1 ? int64_t(sk.kb_chunk) * BK : K);
    if ((rc = check_region(heap, off_A, size_t(M_l) * K * 2))) return rc;
    if ((rc = check_region(heap, off_B, size_t(K) * N * 2))) return rc;
    if ((rc = check_region(heap, off_out, size_t(M) * N * 2))) return rc;
    const bool has_bias = off_bias != IRIS_NO_BIAS;
    if (has_bias && (rc = check_region(heap, off_bias, size_t(c.bias_on_m ? M_l : N) * 2))) return rc;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.op = OP_MM_AG;
    p.W = W;
    p.bf16 = dtype == IRIS_BF16;
    const int mbpr = static_cast<int>(cdiv(M_l, BM * c.cg));
    fill_geometry(p, M_l, N, K, mbpr * W, c);
    p.mb_per_rank = mbpr;
    p.heap = static_cast<char*>(heap->base);
    p.rank_stride = heap->rank_stride;
    p.off_A = off_A;
    p.off_out = off_out;
    p.off_bias = has_bias ? off_bias : 0;
    p.has_bias = has_bias;
    p.n_gemm = (M_l > 0 && N > 0) ? static_cast<uint32_t>(p.n_tiles) : 0u;
    p.n_comm = 0;
    if (sk.split > 1) {
        // chunk j of every tile is an item; the chunks' partials are summed in
        // chunk order by the chained reduce (a running sum of all W x M_l rows)
        if (uint64_t(p.n_gemm) * sk.split >= 0x7FFFFFFFull) return IRIS_EINVAL;
        p.split = sk.split;
        p.kb_chunk = sk.kb_chunk;
        p.n_gemm *= static_cast<uint32_t>(sk.split);
        p.reduce_mode = 3;
        p.rank_inner = 0;
        p.g_split = p.n_gemm;
    } else {
        tail_split(p, c, false);
    }
    if ((rc = prepare_ws(p, workspace, workspace_bytes, IRIS_OP_MATMUL_ALL_GATHER, p.split > 1 ? M : 0, N, W, c)))
        return rc;
    if (p.n_gemm > 0 && K > 0) {
        if ((rc = make_map(&p.tmA, p.heap + off_A, p.bf16, K, M_l, W, K * 2, heap->rank_stride, BK, BM))) return rc;
        if ((rc = make_a_chunk_map(p, c, p.heap + off_A, M_l, K, W, heap->rank_stride))) return rc;
        if ((rc = make_map(&p.tmB, p.heap + off_B, p.bf16, N, K, 1, N * 2, round_up(size_t(K) * N * 2, 16), 64,
                           BK * k_per_stage(c.cg, c.stages))))
            return rc;
        if ((rc = make_b_chunk_map(p, c, p.heap + off_B, N, K, 1, round_up(size_t(K) * N * 2, 16)))) return rc;
    }
    if (p.n_gemm > 0 && (rc = make_out_map(&p.tmC, p.heap + off_out, p.bf16, N, M_l, W, W, N * 2,
                                           size_t(M_l) * N * 2, heap->rank_stride)))
        return rc;
    // split-K: the fp32 running sum, one block of M_l rows per rank
    if (p.split > 1 && (rc = make_out_map(&p.tmS, p.partials, 2, N, M_l, W, 1, N * 4, size_t(M_l) * N * 4,
                                          size_t(M) * N * 4)))
        return rc;
    return launch(p, c, stream);
}

// part: 0 = GEMM and collective in one launch; 1 = the GEMM alone on `grid`
// CTAs; 2 = the collective alone on `grid` CTAs (two-stream mode).
static int concurrent_impl(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                           iris_dtype gemm_dtype, iris_coll coll, const iris_b200_heap* heap, size_t off_in,
                           size_t off_out, int64_t count, iris_dtype coll_dtype, const iris_b200_config* cfg,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream, int part, int grid) {
    if (!dims_ok(M, N, K) || count < 0) return IRIS_EINVAL;
    if (gemm_dtype != IRIS_F16 && gemm_dtype != IRIS_BF16) return IRIS_EINVAL;
    const bool has_gemm = M > 0 && N > 0;
    if (has_gemm) {
        if (!C || (K > 0 && (!A || !B))) return IRIS_EINVAL;
        if (K % 8 != 0 || N % 8 != 0) return IRIS_EALIGN;
        if (!aligned16(reinterpret_cast<uintptr_t>(A)) || !aligned16(reinterpret_cast<uintptr_t>(B)) ||
            !aligned16(reinterpret_cast<uintptr_t>(C)))
            return IRIS_EALIGN;
    }
    int rc;
    int W = 1;
    int esz = 4;
    if (count > 0) {
        if ((rc = check_heap(heap))) return rc;
        W = heap->world;
        if (coll < IRIS_COLL_ALL_GATHER || coll > IRIS_COLL_BROADCAST) return IRIS_EINVAL;
        const bool sums = (coll == IRIS_COLL_ALL_REDUCE || coll == IRIS_COLL_REDUCE_SCATTER);
        if (sums) {
            if (coll_dtype != IRIS_F32) return IRIS_EUNSUPPORTED;
        } else {
            // pure data movement: any element type, moved as bytes
            esz = (coll_dtype == IRIS_F32) ? 4 : (coll_dtype == IRIS_F16 || coll_dtype == IRIS_BF16) ? 2 : 0;
            if (!esz) return IRIS_EINVAL;
        }
        if ((count * esz) % 16 != 0) return IRIS_EALIGN;
        if (coll == IRIS_COLL_REDUCE_SCATTER && count % (4 * W) != 0) return IRIS_EALIGN;
        if (coll == IRIS_COLL_ALL_TO_ALL && (count % W != 0 || ((count / W) * esz) % 16 != 0)) return IRIS_EALIGN;
    }
    Cfg c;
    if ((rc = resolve_cfg(cfg, IRIS_OP_CONCURRENT, N, c))) return rc;
    if (part != 0) {
        c.grid = grid;
        c.gemm_ctas = part == 1 ? grid : 0;
    }
    const bool launch_gemm = has_gemm && part != 2;
    if ((rc = resolve_pair(c, IRIS_OP_CONCURRENT, launch_gemm))) return rc;
    resolve_stages(c, K);
    if (count > 0) {
        if (size_t(c.comm_block) * esz % 16 != 0) return IRIS_EALIGN;
        const size_t in_bytes = size_t(count) * esz;
        const size_t out_bytes = coll == IRIS_COLL_ALL_GATHER      ? in_bytes * W
                                 : coll == IRIS_COLL_REDUCE_SCATTER ? in_bytes / W
                                                                    : in_bytes;
        if (coll == IRIS_COLL_BROADCAST && c.root >= W) return IRIS_EINVAL;
        if ((rc = check_region(heap, off_in, in_bytes))) return rc;
        if ((rc = check_region(heap, off_out, out_bytes))) return rc;
        // an in-place collective must use the same offsets exactly; partial overlap is refused
        if (off_in != off_out && off_in < off_out + out_bytes && off_out < off_in + in_bytes) return IRIS_EINVAL;
        if (off_in == off_out && coll != IRIS_COLL_ALL_REDUCE) return IRIS_EINVAL;
    }

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.op = OP_CONC;
    p.W = W;
    p.bf16 = gemm_dtype == IRIS_BF16;
    p.coll = coll == IRIS_COLL_ALL_GATHER      ? COLL_AG
             : coll == IRIS_COLL_ALL_REDUCE    ? COLL_AR
             : coll == IRIS_COLL_REDUCE_SCATTER ? COLL_RS
             : coll == IRIS_COLL_ALL_TO_ALL    ? COLL_A2A
                                               : COLL_BC;
    p.root = c.root;
    const int mblocks = static_cast<int>(cdiv(M, BM * c.cg));
    fill_geometry(p, M, N, K, mblocks, c);
    p.mb_per_rank = mblocks;
    p.C = C;
    p.n_gemm = (has_gemm && part != 2) ? static_cast<uint32_t>(p.n_tiles) : 0u;
    tail_split(p, c, false);
    if (count > 0 && part != 1) {
        p.heap = static_cast<char*>(heap->base);
        p.rank_stride = heap->rank_stride;
        p.off_in = off_in;
        p.off_cout = off_out;
        p.count = count;
        p.comm_block = c.comm_block;
        p.elem_bytes = esz;
        const int64_t chunks = cdiv(count, c.comm_block);
        const int64_t items = coll == IRIS_COLL_ALL_GATHER  ? chunks * W
                              : coll == IRIS_COLL_ALL_TO_ALL ? int64_t(W) * W * cdiv(count / W, c.comm_block)
                                                              : chunks;
        if (items >= 0x7FFFFFFF) return IRIS_EINVAL;
        p.n_comm = static_cast<uint32_t>(items);
        // one 3-D box of all W sources per sub-chunk (path 3) applies to the
        // summing collectives over whole 1 KB rows when R rows of all W
        // sources fit one ring buffer; measured faster than one copy per
        // source (fewer, larger TMA requests), so it is their default
        const int area = static_cast<int>(LEASE_BYTES / NUM_WORKER_WARPS);  // leased bytes per worker warp
        const int R = area / c.coll_ring / (1024 * W);
        const bool box_ok = (coll == IRIS_COLL_ALL_REDUCE || coll == IRIS_COLL_REDUCE_SCATTER) && count % 256 == 0 &&
                            c.comm_block % 256 == 0 && R >= 1;
        if (c.coll_path == 3 && !box_ok) return IRIS_EINVAL;
        if (c.coll_path == 0) c.coll_path = box_ok ? 3 : 1;
        p.coll_path = c.coll_path;
        if (c.coll_path == 3) {
            p.coll_box_rows = std::min(R, 256);
            if ((rc = make_coll_map(p, p.heap + off_in, count, W, heap->rank_stride, p.coll_box_rows))) return rc;
        }
    }
    if ((rc = prepare_ws(p, workspace, workspace_bytes, IRIS_OP_CONCURRENT, 0, N, W, c))) return rc;
    if (p.n_gemm > 0 && K > 0) {
        if ((rc = make_map(&p.tmA, A, p.bf16, K, M, 1, K * 2, round_up(size_t(M) * K * 2, 16), BK, BM))) return rc;
        if ((rc = make_a_chunk_map(p, c, A, M, K, 1, round_up(size_t(M) * K * 2, 16)))) return rc;
        if ((rc = make_map(&p.tmB, B, p.bf16, N, K, 1, N * 2, round_up(size_t(K) * N * 2, 16), 64,
                           BK * k_per_stage(c.cg, c.stages))))
            return rc;
        if ((rc = make_b_chunk_map(p, c, B, N, K, 1, round_up(size_t(K) * N * 2, 16)))) return rc;
    }
    if (p.n_gemm > 0 && (rc = make_out_map(&p.tmC, C, p.bf16, N, M, 1, 1, N * 2, size_t(M) * N * 2,
                                           size_t(M) * N * 2)))
        return rc;
    return launch(p, c, stream);
}

int iris_b200_concurrent_gemm_collective(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                         iris_dtype gemm_dtype, iris_coll coll, const iris_b200_heap* heap,
                                         size_t off_in, size_t off_out, int64_t count, iris_dtype coll_dtype,
                                         const iris_b200_config* cfg, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
    return concurrent_impl(A, B, C, M, N, K, gemm_dtype, coll, heap, off_in, off_out, count, coll_dtype, cfg,
                           workspace, workspace_bytes, stream, 0, 0);
}

int iris_b200_concurrent_two_stream(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                    iris_dtype gemm_dtype, iris_coll coll, const iris_b200_heap* heap,
                                    size_t off_in, size_t off_out, int64_t count, iris_dtype coll_dtype,
                                    const iris_b200_config* cfg, void* gemm_workspace, size_t gemm_workspace_bytes,
                                    void* comm_workspace, size_t comm_workspace_bytes, cudaStream_t gemm_stream,
                                    cudaStream_t comm_stream) {
    int sms = 0;
    if (num_sms_current(&sms) != IRIS_OK) return IRIS_ECUDA;
    const int total = (cfg && cfg->grid) ? cfg->grid : sms;
    if (total < 2 || total > sms) return IRIS_EINVAL;
    int gemm_grid = (cfg && cfg->gemm_ctas > 0) ? cfg->gemm_ctas : total / 2;
    if (gemm_grid >= total) return IRIS_EINVAL;
    const bool has_gemm = M > 0 && N > 0, has_coll = count > 0;
    if (!has_gemm) gemm_grid = 0;
    if (!has_coll) gemm_grid = total;
    if (gemm_workspace == comm_workspace && has_gemm && has_coll) return IRIS_EINVAL;  // each launch owns its queues
    int rc = IRIS_OK;
    if (has_gemm) {
        rc = concurrent_impl(A, B, C, M, N, K, gemm_dtype, coll, heap, off_in, off_out, 0, coll_dtype, cfg,
                             gemm_workspace, gemm_workspace_bytes, gemm_stream, 1, gemm_grid);
        if (rc) return rc;
    }
    if (has_coll)
        rc = concurrent_impl(nullptr, nullptr, nullptr, 0, 0, 0, gemm_dtype, coll, heap, off_in, off_out, count,
                             coll_dtype, cfg, comm_workspace, comm_workspace_bytes, comm_stream, 2,
                             total - gemm_grid);
    return rc;
}

int iris_b200_query_status(void* workspace, cudaStream_t stream, int* device_status, int* where, int* index) {
    if (!workspace) return IRIS_EINVAL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return IRIS_ECUDA;
    WsHeader h;
    if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return IRIS_ECUDA;
    if (device_status) *device_status = h.status;
    if (where) *where = h.err_where;
    if (index) *index = h.err_index;
    if (h.status != 0) {
        const int zero[4] = {0, 0, 0, 0};
        // clear status, abort epoch, where, index (bytes 16..31 of the header)
        if (cudaMemcpy(static_cast<char*>(workspace) + 16, zero, sizeof(zero), cudaMemcpyHostToDevice) !=
            cudaSuccess)
            return IRIS_ECUDA;
        return IRIS_ETIMEOUT;
    }
    return IRIS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation variant of all_gather_matmul: the workspace (header + flags)
// is a static device array of this translation unit instead of caller memory.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[IRIS_NOALLOC_SCRATCH_BYTES];
}  // namespace

extern "C" int iris_b200_all_gather_matmul_noalloc(const iris_b200_heap* heap, size_t off_A, size_t off_B,
                                                   size_t off_bias, size_t off_out, size_t off_gathered,
                                                   int64_t M, int64_t N, int64_t K, iris_dtype dtype,
                                                   const iris_b200_config* cfg, cudaStream_t stream) {
    if (!heap || heap->world < 1 || heap->world > IRIS_MAX_WORLD || !dims_ok(M, N, K)) return IRIS_EINVAL;
    // M <= INT32_MAX here, so the flag count cannot overflow
    const int64_t flags = int64_t(heap->world) * cdiv(M, BM);
    if (flags > IRIS_NOALLOC_MAX_FLAGS) return IRIS_ENOWS;
    // The array's device address on the current device, looked up on every
    // call: a lookup allocates nothing, and an address cached across a device
    // reset (which reloads the module) could be stale.
    void* scratch = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || !scratch) return cuda_fail("cudaGetSymbolAddress (no-alloc scratch)", static_cast<int>(e));
    // Every call starts from zeroed state: the header (queue counters, epoch,
    // status) and the ready-flags this problem uses, so nothing left by an
    // earlier call -- finished or stopped by a bounded wait -- can match.
    const size_t used = WS_HEADER + size_t(flags) * 8;
    e = cudaMemsetAsync(scratch, 0, used, stream);
    if (e != cudaSuccess) return cuda_fail("cudaMemsetAsync (no-alloc scratch)", static_cast<int>(e));
    // no split-K here: the static scratch has no room for its running sum
    iris_b200_config local;
    if (cfg)
        local = *cfg;
    else
        std::memset(&local, 0, sizeof(local));
    local.k_split = 1;
    return iris_b200_all_gather_matmul(heap, off_A, off_B, off_bias, off_out, off_gathered, M, N, K, dtype, &local,
                                       scratch, IRIS_NOALLOC_SCRATCH_BYTES, stream);
}

// ---------------------------------------------------------------------------
// SM partition for the two-stream concurrent mode: two CUDA green contexts
// with disjoint SM sets and one stream in each.  Driver functions are looked
// up through the runtime (no link-time dependency on the driver library).
namespace {
typedef CUresult (*DeviceGetFn)(CUdevice*, int);
typedef CUresult (*DeviceGetDevResourceFn)(CUdevice, CUdevResource*, CUdevResourceType);
typedef CUresult (*SmSplitFn)(CUdevResource*, unsigned int*, const CUdevResource*, CUdevResource*, unsigned int,
                              unsigned int);
typedef CUresult (*GenerateDescFn)(CUdevResourceDesc*, CUdevResource*, unsigned int);
typedef CUresult (*GreenCtxCreateFn)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned int);
typedef CUresult (*GreenCtxStreamCreateFn)(CUstream*, CUgreenCtx, unsigned int, int);
typedef CUresult (*StreamDestroyFn)(CUstream);
typedef CUresult (*GreenCtxDestroyFn)(CUgreenCtx);

struct GreenApi {
    DeviceGetFn device_get = nullptr;
    DeviceGetDevResourceFn get_resource = nullptr;
    SmSplitFn split = nullptr;
    GenerateDescFn gen_desc = nullptr;
    GreenCtxCreateFn ctx_create = nullptr;
    GreenCtxStreamCreateFn stream_create = nullptr;
    StreamDestroyFn stream_destroy = nullptr;
    GreenCtxDestroyFn ctx_destroy = nullptr;
};

// the driver functions at the ABI of the toolkit this file is compiled with
// (the prototypes above come from its header)
template <typename F>
bool driver_fn(const char* name, F& out) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, CUDART_VERSION, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        if (debug_on()) std::fprintf(stderr, "[iris_b200] driver entry point %s unavailable\n", name);
        return false;
    }
    out = reinterpret_cast<F>(fn);
    return true;
}

bool green_api(GreenApi& a) {
    return driver_fn("cuDeviceGet", a.device_get) && driver_fn("cuDeviceGetDevResource", a.get_resource) &&
           driver_fn("cuDevSmResourceSplitByCount", a.split) && driver_fn("cuDevResourceGenerateDesc", a.gen_desc) &&
           driver_fn("cuGreenCtxCreate", a.ctx_create) && driver_fn("cuGreenCtxStreamCreate", a.stream_create) &&
           driver_fn("cuStreamDestroy", a.stream_destroy) && driver_fn("cuGreenCtxDestroy", a.ctx_destroy);
}

struct Partition {
    CUgreenCtx ctx[2] = {nullptr, nullptr};
    CUstream stream[2] = {nullptr, nullptr};
    int sms[2] = {0, 0};
};
Partition g_partition[64];
std::mutex g_partition_mu;

void partition_destroy(const GreenApi& a, Partition& pt) {
    for (int i = 0; i < 2; ++i) {
        if (pt.stream[i]) a.stream_destroy(pt.stream[i]);
        if (pt.ctx[i]) a.ctx_destroy(pt.ctx[i]);
        pt.stream[i] = nullptr;
        pt.ctx[i] = nullptr;
        pt.sms[i] = 0;
    }
}
}  // namespace

extern "C" int iris_b200_sm_partition_streams(int gemm_sms, cudaStream_t* gemm_stream, cudaStream_t* comm_stream,
                                              int* gemm_sms_out, int* comm_sms_out) {
    if (!gemm_stream || !comm_stream) return IRIS_EINVAL;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IRIS_ECUDA;
    if (num_sms_current(&sms) != IRIS_OK) return IRIS_ECUDA;
    if (gemm_sms < 1 || gemm_sms >= sms) return IRIS_EINVAL;
    GreenApi a;
    if (!green_api(a)) return IRIS_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_partition_mu);
    Partition& pt = g_partition[dev];
    partition_destroy(a, pt);  // a new call replaces this device's partition
    CUdevice cudev;
    if (a.device_get(&cudev, dev) != CUDA_SUCCESS) return cuda_fail("cuDeviceGet", 0);
    CUdevResource all, part, rest;
    std::memset(&part, 0, sizeof(part));
    std::memset(&rest, 0, sizeof(rest));
    CUresult r = a.get_resource(cudev, &all, CU_DEV_RESOURCE_TYPE_SM);
    if (r != CUDA_SUCCESS) return cuda_fail("cuDeviceGetDevResource", static_cast<int>(r));
    unsigned int groups = 1;
    r = a.split(&part, &groups, &all, &rest, 0, static_cast<unsigned int>(gemm_sms));
    if (r != CUDA_SUCCESS || groups != 1 || rest.sm.smCount == 0)
        return r != CUDA_SUCCESS ? cuda_fail("cuDevSmResourceSplitByCount", static_cast<int>(r)) : IRIS_EINVAL;
    CUdevResource* res[2] = {&part, &rest};
    for (int i = 0; i < 2; ++i) {
        CUdevResourceDesc desc;
        r = a.gen_desc(&desc, res[i], 1);
        if (r == CUDA_SUCCESS) r = a.ctx_create(&pt.ctx[i], desc, cudev, CU_GREEN_CTX_DEFAULT_STREAM);
        if (r == CUDA_SUCCESS) r = a.stream_create(&pt.stream[i], pt.ctx[i], CU_STREAM_NON_BLOCKING, 0);
        if (r != CUDA_SUCCESS) {
            partition_destroy(a, pt);
            return cuda_fail("green context", static_cast<int>(r));
        }
        pt.sms[i] = static_cast<int>(res[i]->sm.smCount);
    }
    *gemm_stream = reinterpret_cast<cudaStream_t>(pt.stream[0]);
    *comm_stream = reinterpret_cast<cudaStream_t>(pt.stream[1]);
    if (gemm_sms_out) *gemm_sms_out = pt.sms[0];
    if (comm_sms_out) *comm_sms_out = pt.sms[1];
    return IRIS_OK;
}

extern "C" int iris_b200_sm_partition_release(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IRIS_ECUDA;
    GreenApi a;
    if (!green_api(a)) return IRIS_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_partition_mu);
    partition_destroy(a, g_partition[dev]);
    return IRIS_OK;
}
