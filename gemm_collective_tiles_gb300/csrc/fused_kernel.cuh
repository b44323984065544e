// Persistent work-stealing kernel that interleaves dense GEMM tiles with
// collective-communication tiles (ROCm/iris PR #544 "Add iris.concurrent":
// one persistent kernel with a GEMM queue and a comm queue, GROUP_M tile
// swizzle, explicit GEMM/comm CTA split; iris docs "Fused Communication and
// Compute Operations" for the four dependent ops).
//
// CTA layout (352 threads, one CTA per SM):
//   warp 0      scheduler (lane 0): claims work items from the two global
//               queues with atomics and publishes them into a small
//               shared-memory item ring, ahead of the warps that run them.
//   warp 1      tensor-memory owner; lane 0 issues tcgen05.mma (128 x BN x 16
//               steps, fp32 accumulators in TMEM, double-buffered).
//   warp 2      TMA producer (lane 0): for GEMM items streams the A/B K-blocks
//               into a STAGES-deep shared-memory pipeline.
//   warps 3..10 workers: GEMM epilogue (tcgen05.ld -> +bias -> fp16/bf16 or
//               fp32 partial -> global) and comm tiles (128-bit vector copy /
//               rank-order fp32 reduce), so the comm tiles of one SM run
//               while its tensor cores work on the next GEMM tile.
// Every wait is bounded (globaltimer); a wait that gives up records the
// failure in the workspace status word, sets the launch's abort epoch, and
// every role drains its in-flight async work and leaves.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gct {

enum : int { OP_AG_MM = 0, OP_MM_RS = 1, OP_MM_AG = 2, OP_MM_AR = 3, OP_CONC = 4 };
enum : int { COLL_AG = 0, COLL_AR = 1, COLL_RS = 2 };

constexpr int BM = 128;           // tile rows (tcgen05 M for cta_group::1)
constexpr int BK = 64;            // K per stage: 64 x 16-bit = one 128-byte swizzle row
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int NUM_WORKER_WARPS = 8;
constexpr int FIRST_WORKER_WARP = 3;   // warps 0..2: scheduler, MMA issuer, TMA producer
constexpr int NUM_THREADS = 32 * (FIRST_WORKER_WARP + NUM_WORKER_WARPS);
constexpr int RING = 8;           // work-item ring depth
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
    uint32_t pad[56];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

struct Params {
    CUtensorMap tmA;  // 3-D {k, row, rank}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmB;  // 3-D {n, k, rank},   box {64, 64, 1},  128-byte swizzle
    int op, W, bf16, coll;
    int M;            // rows of one GEMM (M_local for matmul_all_gather)
    int N, K;
    int m_blocks, mb_per_rank, n_blocks, k_blocks, group_m, n_tiles;
    uint32_t n_gemm, n_comm;
    int gemm_ctas;    // CTAs preferring GEMM; < 0 = balanced
    uint32_t lookahead;
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
    int elem_bytes;
    unsigned long long wait_ns;
    uint32_t debug_skip;               // flag index + 1 that is never released (0 = none)
    int reduce_mode;                   // reduce ops: 0 = last arriving rank reduces, 1 = comm queue
    int rank_inner;                    // reduce ops: 1 = rank index fastest in the GEMM item order
    unsigned long long* trace;         // optional per-CTA event trace (nullptr = off)
    int trace_cap;                     // events per (CTA, role)
};

// Optional timeline: each CTA owns 4 role streams (scheduler, MMA, TMA,
// workers) of trace_cap (event, globaltimer ns) pairs; slot 0 of a stream
// holds its event count.
enum : int { TR_SCHED = 0, TR_MMA = 1, TR_TMA = 2, TR_WORK = 3 };
enum : unsigned long long { EV_CLAIM = 1, EV_BEGIN = 2, EV_END = 3, EV_READY = 4 };
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

// Bounded wait on an mbarrier phase. false = gave up (timeout or abort).
__device__ __forceinline__ bool wait_bar(const Ctl& c, uint64_t* bar, uint32_t parity, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
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
    uint32_t tile;
};
__device__ __forceinline__ uint32_t group_tiles(const Params& p) {
    return static_cast<uint32_t>(p.group_m) * p.n_blocks;
}
__device__ __forceinline__ GemmCoord decode_gemm(const Params& p, uint32_t g) {
    GemmCoord gc;
    if (p.op == OP_MM_RS || p.op == OP_MM_AR) {
        if (p.rank_inner) {
            gc.tile = g / p.W;
            gc.rank = static_cast<int>(g % p.W);
        } else {
            const uint32_t T = group_tiles(p);
            const uint32_t sg = g / (T * p.W);
            const uint32_t Tsg = min(T, static_cast<uint32_t>(p.n_tiles) - sg * T);
            const uint32_t local = g - sg * T * p.W;
            gc.rank = static_cast<int>(local / Tsg);
            gc.tile = sg * T + (local - static_cast<uint32_t>(gc.rank) * Tsg);
        }
    } else {
        gc.tile = g;
        gc.rank = 0;
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

// all_gather_matmul: number of gather items that must be claimed before GEMM
// item x may be published (all shards of every m-block of x's swizzle group).
__device__ __forceinline__ uint32_t gather_need(const Params& p, uint32_t x) {
    const uint32_t group_size = static_cast<uint32_t>(p.group_m) * p.n_blocks;
    const int first_m = static_cast<int>(x / group_size) * p.group_m;
    const int gsz = min(p.m_blocks - first_m, p.group_m);
    return static_cast<uint32_t>(first_m + gsz) * p.W;
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
template <int BN, int STAGES>
struct Smem {
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TILES_BYTES = STAGES * STAGE_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * RING + 2;
    static constexpr uint32_t BYTES = 1024 /*align slack*/ + TILES_BYTES + NUM_BARS * 8 +
                                      (RING + 4) * 4;
    uint8_t* tiles;
    uint64_t *full, *empty, *acc_full, *acc_empty, *item_full, *item_empty, *wbar, *final_bar;
    volatile uint32_t* ring;
    uint32_t* tmem_slot;
    uint32_t* epoch_slot;
    uint32_t* bcast;

    __device__ void carve(uint8_t* raw) {
        uintptr_t a = reinterpret_cast<uintptr_t>(raw);
        a = (a + 1023) & ~static_cast<uintptr_t>(1023);
        tiles = reinterpret_cast<uint8_t*>(a);
        uint64_t* b = reinterpret_cast<uint64_t*>(tiles + TILES_BYTES);
        full = b;
        empty = full + STAGES;
        acc_full = empty + STAGES;
        acc_empty = acc_full + 2;
        item_full = acc_empty + 2;
        item_empty = item_full + RING;
        wbar = item_empty + RING;
        final_bar = wbar + 1;
        uint32_t* u = reinterpret_cast<uint32_t*>(final_bar + 1);
        ring = u;
        tmem_slot = u + RING;
        epoch_slot = u + RING + 1;
        bcast = u + RING + 2;
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
template <int BN, int STAGES>
__device__ void run_scheduler(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm) {
    Tracer tr;
    tr.init(p, TR_SCHED);
    uint32_t ring_n = 0;
    bool gemm_dry = (p.n_gemm == 0), comm_dry = (p.n_comm == 0);
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);
    const bool prefer_gemm = p.gemm_ctas < 0 || static_cast<int>(blockIdx.x) < p.gemm_ctas;

    auto publish = [&](uint32_t item) -> bool {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        if (!wait_bar(ctl, &sm.item_empty[slot], (use & 1) ^ 1, WAIT_ITEM_EMPTY)) return false;
        sm.ring[slot] = item;
        mbar_arrive(&sm.item_full[slot]);
        ++ring_n;
        tr.rec(EV_CLAIM, item);
        return true;
    };

    // Take one GEMM item (after claiming the gather items it depends on).
    auto take_gemm = [&](bool& got) -> bool {
        got = false;
        if (gemm_dry) return true;
        const uint32_t g = atomicAdd(&p.ws->gemm_ctr, 1u);
        if (g >= p.n_gemm) {
            gemm_dry = true;
            return true;
        }
        if (p.op == OP_AG_MM) {
            const uint32_t la = min(g + p.lookahead, p.n_gemm - 1);
            const uint32_t need = gather_need(p, la);
            while (!comm_dry && ld_relaxed_gpu(&p.ws->comm_ctr) < need) {
                const uint32_t c = atomicAdd(&p.ws->comm_ctr, 1u);
                if (c >= p.n_comm) {
                    comm_dry = true;
                    break;
                }
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
    tr.finish();
}

// ============================================================ TMA producer
// Follows the item ring; for every GEMM item streams its K-blocks of A and B
// into the STAGES-deep shared-memory pipeline (acquiring the gather flags of
// all_gather_matmul shards just before their first K-block).
template <int BN, int STAGES>
__device__ void run_tma(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm) {
    Tracer tr;
    tr.init(p, TR_TMA);
    uint32_t stage = 0, phase = 0, ring_n = 0;
    uint32_t issued_phase[STAGES];
    uint32_t used_mask = 0;
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);

    auto load_gemm = [&](uint32_t g) -> bool {
        const GemmCoord gc = decode_gemm(p, g);
        int a_row, a_rank;
        if (p.op == OP_MM_AG) {
            a_row = (gc.mb % p.mb_per_rank) * BM;
            a_rank = gc.rank;
        } else {
            a_row = gc.mb * BM;
            a_rank = reduce_op ? gc.rank : 0;
        }
        const int b_rank = reduce_op ? gc.rank : 0;
        int acquired = 0;  // all_gather_matmul: shards whose flags are held
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (p.op == OP_AG_MM) {
                const int s_hi = min(p.W - 1, (kb * BK + BK - 1) / p.K_local);
                if (s_hi >= acquired) {
                    for (int s = acquired; s <= s_hi; ++s) {
                        const int fi = gc.mb * p.W + s;
                        if (!wait_flag(ctl, &p.flags[fi], WAIT_FLAG_GATHER, fi)) return false;
                    }
                    acquired = s_hi + 1;
                    fence_proxy_async_global();
                }
            }
            if (!wait_bar(ctl, &sm.empty[stage], phase ^ 1, WAIT_SMEM_EMPTY)) return false;
            mbar_arrive_expect_tx(&sm.full[stage], Smem<BN, STAGES>::STAGE_BYTES);
            tma_load_3d(sm.a_tile(stage), &p.tmA, kb * BK, a_row, a_rank, &sm.full[stage]);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
                tma_load_3d(sm.b_tile(stage) + c * (64 * BK * 2), &p.tmB, gc.nb * BN + c * 64,
                            kb * BK, b_rank, &sm.full[stage]);
            issued_phase[stage] = phase;
            used_mask |= 1u << stage;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        return true;
    };

    while (true) {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        if (!wait_bar(ctl, &sm.item_full[slot], use & 1, WAIT_ITEM_FULL_TMA)) break;
        const uint32_t item = sm.ring[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++ring_n;
        if (item == ITEM_END) break;
        if (item & ITEM_COMM) continue;
        tr.rec(EV_BEGIN, item);
        if (!load_gemm(item)) break;
        tr.rec(EV_END, item);
    }
    tr.finish();
    // drain: every TMA load issued into a stage has landed before the CTA exits
    for (int s = 0; s < STAGES; ++s)
        if (used_mask & (1u << s)) drain_bar(ctl, &sm.full[s], issued_phase[s], WAIT_TEARDOWN_TMA);
}

// ============================================================ MMA issuer
template <int BN, int STAGES>
__device__ void run_mma(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm, uint32_t tmem) {
    constexpr uint32_t IDESC_F16 = make_idesc(0, BM, BN);
    constexpr uint32_t IDESC_BF16 = make_idesc(1, BM, BN);
    const uint32_t idesc = p.bf16 ? IDESC_BF16 : IDESC_F16;
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
        if (!wait_bar(ctl, &sm.acc_empty[buf], (ause & 1) ^ 1, WAIT_ACC_EMPTY)) break;
        tc_fence_after();
        tr.rec(EV_BEGIN, item);
        const uint32_t d = tmem + buf * BN;
        bool ok = true;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_bar(ctl, &sm.full[stage], phase, WAIT_SMEM_FULL)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // A: K-major, 128-byte swizzle, 8-row core groups 1024 B apart.
            // B: MN-major, 128-byte swizzle: 64-column chunks 8 KB apart
            //    (leading offset), 8-row K groups 1024 B apart (stride offset).
            const uint64_t adesc = smem_desc(smem_u32(sm.a_tile(stage)), 16, 1024);
            const uint64_t bdesc = smem_desc(smem_u32(sm.b_tile(stage)), 64 * BK * 2, 1024);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
                // advance A by 16 columns (32 B inside the swizzled row) and
                // B by 16 rows (2 KB); descriptors hold addresses >> 4
                umma_f16(d, adesc + static_cast<uint64_t>(k * 2), bdesc + static_cast<uint64_t>(k * 128),
                         idesc, (kb | k) != 0 ? 1u : 0u);
            }
            umma_commit(&sm.empty[stage]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok) break;
        umma_commit(&sm.acc_full[buf]);
        tr.rec(EV_END, item);
        ++acc_i;
    }
    tr.finish();
    // drain: every MMA issued by this thread has completed
    umma_commit(sm.final_bar);
    drain_bar(ctl, sm.final_bar, 0, WAIT_TEARDOWN_MMA);
}

// ============================================================ workers
struct WorkerCtx {
    int w;      // worker warp 0..7
    int lane;
    int q;      // TMEM lane quarter of this warp (warp id % 4)
    int h;      // column half of the accumulator this warp drains
    uint32_t wphase;
};

template <int BN, int STAGES>
__device__ __noinline__ void reduce_body(const Params& p, uint32_t c, WorkerCtx& wc);

// barrier over the 8 worker warps built on an mbarrier (bounded, abortable)
template <int BN, int STAGES>
__device__ __forceinline__ bool worker_sync(const Ctl& ctl, Smem<BN, STAGES>& sm, WorkerCtx& wc) {
    __syncwarp();
    bool ok = true;
    if (wc.lane == 0) {
        mbar_arrive(sm.wbar);
        ok = wait_bar(ctl, sm.wbar, wc.wphase, WAIT_WORKER_SYNC);
    }
    wc.wphase ^= 1;
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// GEMM epilogue of one tile: TMEM -> registers -> (+bias) -> global.
template <int BN, int STAGES>
__device__ bool epilogue(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm, uint32_t tmem,
                         uint32_t g, uint32_t acc_i, WorkerCtx& wc, Tracer& tr) {
    const uint32_t buf = acc_i & 1, ause = acc_i >> 1;
    bool ok = true;
    if (wc.lane == 0) ok = wait_bar(ctl, &sm.acc_full[buf], ause & 1, WAIT_ACC_FULL);
    if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) return false;
    tc_fence_after();
    tr.rec(EV_READY, g);

    const GemmCoord gc = decode_gemm(p, g);
    const int r_in_tile = wc.q * 32 + wc.lane;
    const bool reduce_op = (p.op == OP_MM_RS || p.op == OP_MM_AR);
    // output row of this thread and whether it exists
    int row;        // row inside the op's output (or partial)
    int bias_row;   // index into a per-row bias
    bool row_ok;
    if (p.op == OP_MM_AG) {
        const int lrow = (gc.mb % p.mb_per_rank) * BM + r_in_tile;
        row_ok = lrow < p.M;
        row = gc.rank * p.M + lrow;
        bias_row = lrow;
    } else {
        row = gc.mb * BM + r_in_tile;
        row_ok = row < p.M;
        bias_row = row;
    }
    const char* bias_base = nullptr;
    if (p.has_bias) {
        const int bias_region = reduce_op ? gc.rank : 0;
        bias_base = p.heap + static_cast<size_t>(bias_region) * p.rank_stride + p.off_bias;
    }
    float row_bias = 0.f;
    if (p.has_bias && p.bias_on_m && row_ok)
        row_bias = bits16_to_float(reinterpret_cast<const uint16_t*>(bias_base)[bias_row], p.bf16);

    const uint32_t tbase = tmem + (static_cast<uint32_t>(wc.q * 32) << 16) + buf * BN + wc.h * (BN / 2);
#pragma unroll 1
    for (int cc = 0; cc < BN / 2; cc += 32) {
        uint32_t r[32];
        if (p.k_blocks > 0) {
            tmem_ld_32x32b_x32(tbase + cc, r);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        const int col0 = gc.nb * BN + wc.h * (BN / 2) + cc;
        if (!row_ok) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int col = col0 + v * 8;
            if (col >= p.N) break;
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(r[v * 8 + i]);
            if (p.has_bias) {
                if (p.bias_on_m) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = x[i] + row_bias;
                } else {
                    const uint4 bb = *reinterpret_cast<const uint4*>(bias_base + static_cast<size_t>(col) * 2);
                    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] = x[2 * i] + bits16_to_float(bw[i] & 0xFFFFu, p.bf16);
                        x[2 * i + 1] = x[2 * i + 1] + bits16_to_float(bw[i] >> 16, p.bf16);
                    }
                }
            }
            if (reduce_op) {
                float* dst = p.partials + static_cast<size_t>(gc.rank) * p.partial_elems +
                             static_cast<size_t>(row) * p.N + col;
                reinterpret_cast<float4*>(dst)[0] = make_float4(x[0], x[1], x[2], x[3]);
                reinterpret_cast<float4*>(dst)[1] = make_float4(x[4], x[5], x[6], x[7]);
            } else {
                uint4 o;
                o.x = pack2(x[0], x[1], p.bf16);
                o.y = pack2(x[2], x[3], p.bf16);
                o.z = pack2(x[4], x[5], p.bf16);
                o.w = pack2(x[6], x[7], p.bf16);
                if (p.op == OP_CONC) {
                    *reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.C) +
                                              (static_cast<size_t>(row) * p.N + col) * 2) = o;
                } else {
                    const size_t off = p.off_out + (static_cast<size_t>(row) * p.N + col) * 2;
                    const int nreg = p.replicate ? p.W : 1;
                    for (int rg = 0; rg < nreg; ++rg)
                        *reinterpret_cast<uint4*>(p.heap + static_cast<size_t>(rg) * p.rank_stride + off) = o;
                }
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (wc.lane == 0) mbar_arrive(&sm.acc_empty[buf]);

    if (reduce_op) {
        // publish this rank's partial tile: all 8 warps' stores, then the flag
        __threadfence();
        if (!worker_sync(ctl, sm, wc)) return false;
        if (p.reduce_mode == 0) {
            // the rank whose partial completes the tile reduces it now, while
            // the other partials are still in L2
            if (wc.w == 0 && wc.lane == 0) {
                uint32_t last = 0;
                if (p.debug_skip != g + 1)
                    last = arrive_count(reinterpret_cast<unsigned long long*>(p.flags) + gc.tile, ctl.epoch) ==
                           static_cast<uint32_t>(p.W);
                __threadfence();
                *sm.bcast = last;
            }
            if (!worker_sync(ctl, sm, wc)) return false;
            if (*reinterpret_cast<volatile uint32_t*>(sm.bcast)) {
                __threadfence();
                reduce_body<BN, STAGES>(p, gc.tile, wc);
            }
        } else if (wc.w == 0 && wc.lane == 0 && p.debug_skip != g + 1) {
            st_release_gpu(&p.flags[g], ctl.epoch);
        }
    }
    return true;
}

// all_gather_matmul gather tile: shard s rows of m-block mb -> gathered buffer.
template <int BN, int STAGES>
__device__ bool gather_tile(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm, uint32_t c,
                            WorkerCtx& wc) {
    const int mb = static_cast<int>(c / p.W), s = static_cast<int>(c % p.W);
    const int rows = min(BM, p.M - mb * BM);
    const int vpr = p.K_local / 8;  // 16-byte vectors per shard row
    const int Kv = p.K / 8;         // vectors per gathered row
    const uint4* src = reinterpret_cast<const uint4*>(p.heap + static_cast<size_t>(s) * p.rank_stride + p.off_A) +
                       static_cast<size_t>(mb) * BM * vpr;
    uint4* dst = reinterpret_cast<uint4*>(p.heap + p.off_gathered) + static_cast<size_t>(mb) * BM * Kv +
                 static_cast<size_t>(s) * vpr;
    // warp w copies rows w, w+8, ...; lanes walk the row's 16-byte vectors
    constexpr int RU = 2, CU = 4;
    for (int r0 = wc.w; r0 < rows; r0 += NUM_WORKER_WARPS * RU) {
        for (int v0 = wc.lane; v0 < vpr; v0 += 32 * CU) {
            uint4 v[RU][CU];
#pragma unroll
            for (int u = 0; u < RU; ++u)
#pragma unroll
                for (int k = 0; k < CU; ++k)
                    if (r0 + u * NUM_WORKER_WARPS < rows && v0 + 32 * k < vpr)
                        v[u][k] = src[static_cast<size_t>(r0 + u * NUM_WORKER_WARPS) * vpr + v0 + 32 * k];
#pragma unroll
            for (int u = 0; u < RU; ++u)
#pragma unroll
                for (int k = 0; k < CU; ++k)
                    if (r0 + u * NUM_WORKER_WARPS < rows && v0 + 32 * k < vpr)
                        dst[static_cast<size_t>(r0 + u * NUM_WORKER_WARPS) * Kv + v0 + 32 * k] = v[u][k];
        }
    }
    fence_proxy_async_global();
    __threadfence();
    if (!worker_sync(ctl, sm, wc)) return false;
    if (wc.w == 0 && wc.lane == 0 && p.debug_skip != c + 1) st_release_gpu(&p.flags[c], ctl.epoch);
    return true;
}

// matmul_reduce_scatter / matmul_all_reduce comm tile: rank-order fp32 sum
// of the W partial tiles of output tile c, rounded and scattered.
template <int BN, int STAGES>
__device__ bool reduce_tile(const Params& p, const Ctl& ctl, uint32_t c, WorkerCtx& wc) {
    bool ok = true;
    if (wc.lane == 0) {
        for (int s = 0; s < p.W && ok; ++s) {
            const int fi = static_cast<int>(gemm_index(p, c, s));
            ok = wait_flag(ctl, &p.flags[fi], WAIT_FLAG_PARTIAL, fi);
        }
    }
    if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) return false;
    reduce_body<BN, STAGES>(p, c, wc);
    return true;
}

// The reduce itself: warp w takes rows w, w+8, ... of output tile c; lane l
// takes the 16-byte column chunks l, l+32, ... of each row, so every load and
// store instruction of a warp covers 512 contiguous bytes.  SC ranks of a row
// are loaded together before their adds; partials are summed in rank order
// 0..W-1 in fp32.
template <int BN, int STAGES>
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

// concurrent-mode collective tile over the W heap regions
__device__ __noinline__ void coll_tile(const Params& p, uint32_t c, WorkerCtx& wc) {
    const int tid = wc.w * 32 + wc.lane;
    constexpr int NT = NUM_WORKER_WARPS * 32;
    if (p.coll == COLL_AG) {
        // item c = (source rank s, chunk k) of comm_block elements
        const long long bytes_per_rank = p.count * p.elem_bytes;
        const long long chunk_bytes = static_cast<long long>(p.comm_block) * p.elem_bytes;
        const long long chunks = (bytes_per_rank + chunk_bytes - 1) / chunk_bytes;
        const int s = static_cast<int>(c / chunks);
        const long long k = c - static_cast<long long>(s) * chunks;
        const long long b0 = k * chunk_bytes;
        const long long nv = (min(bytes_per_rank, b0 + chunk_bytes) - b0) / 16;
        const uint4* src = reinterpret_cast<const uint4*>(p.heap + static_cast<size_t>(s) * p.rank_stride + p.off_in + b0);
        const size_t dst_off = p.off_cout + static_cast<size_t>(s) * bytes_per_rank + b0;
        constexpr int U = 4;
        for (long long base = tid; base < nv; base += NT * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (base + u * NT < nv) v[u] = __ldcs(src + base + u * NT);
            for (int r = 0; r < p.W; ++r) {
                uint4* dst = reinterpret_cast<uint4*>(p.heap + static_cast<size_t>(r) * p.rank_stride + dst_off);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (base + u * NT < nv) dst[base + u * NT] = v[u];
            }
        }
        return;
    }
    // all-reduce / reduce-scatter: chunk c of the element index space
    const long long e0 = static_cast<long long>(c) * p.comm_block;
    const long long e1 = min(p.count, e0 + p.comm_block);
    const long long nv = (e1 - e0) / 4;
    const long long cw = p.count / p.W;  // reduce-scatter chunk per rank
    int rs_rank = 0;
    long long rs_bound = cw;             // first element past rs_rank's chunk
    if (p.coll == COLL_RS) {
        const long long first = e0 + static_cast<long long>(tid) * 4;
        rs_rank = static_cast<int>(first / cw);
        rs_bound = static_cast<long long>(rs_rank + 1) * cw;
    }
    constexpr int U = 2;
    for (long long base = tid; base < nv; base += NT * U) {
        float4 acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * NT < nv)
                acc[u] = __ldcs(reinterpret_cast<const float4*>(p.heap + p.off_in) + e0 / 4 + base + u * NT);
        for (int s = 1; s < p.W; ++s) {
            const float4* xs = reinterpret_cast<const float4*>(p.heap + static_cast<size_t>(s) * p.rank_stride + p.off_in);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (base + u * NT < nv) {
                    const float4 v = __ldcs(xs + e0 / 4 + base + u * NT);
                    acc[u].x = acc[u].x + v.x;
                    acc[u].y = acc[u].y + v.y;
                    acc[u].z = acc[u].z + v.z;
                    acc[u].w = acc[u].w + v.w;
                }
        }
        if (p.coll == COLL_AR) {
            for (int r = 0; r < p.W; ++r) {
                float4* dst = reinterpret_cast<float4*>(p.heap + static_cast<size_t>(r) * p.rank_stride + p.off_cout);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (base + u * NT < nv) dst[e0 / 4 + base + u * NT] = acc[u];
            }
        } else {
            // elements of one thread increase monotonically, so the owning
            // rank only ever moves forward: advance it by comparison
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (base + u * NT < nv) {
                    const long long e = e0 + (base + u * NT) * 4;
                    while (e >= rs_bound) {
                        ++rs_rank;
                        rs_bound += cw;
                    }
                    float4* dst = reinterpret_cast<float4*>(p.heap + static_cast<size_t>(rs_rank) * p.rank_stride +
                                                            p.off_cout);
                    dst[(e - (rs_bound - cw)) / 4] = acc[u];
                }
        }
    }
}

template <int BN, int STAGES>
__device__ void run_workers(const Params& p, const Ctl& ctl, Smem<BN, STAGES>& sm, uint32_t tmem,
                            int warp, int lane) {
    WorkerCtx wc;
    wc.w = warp - FIRST_WORKER_WARP;
    wc.lane = lane;
    wc.q = warp & 3;
    wc.h = (warp - FIRST_WORKER_WARP) >> 2;
    Tracer tr;
    if (wc.w == 0 && lane == 0) tr.init(p, TR_WORK);
    wc.wphase = 0;
    uint32_t ring_n = 0, acc_i = 0;
    while (true) {
        const uint32_t slot = ring_n % RING, use = ring_n / RING;
        bool ok = true;
        if (lane == 0) ok = wait_bar(ctl, &sm.item_full[slot], use & 1, WAIT_ITEM_FULL_WORKER);
        if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
        const uint32_t item = sm.ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
        ++ring_n;
        if (item == ITEM_END) break;
        tr.rec(EV_BEGIN, item);
        if (item & ITEM_COMM) {
            const uint32_t c = item & ~ITEM_COMM;
            if (p.op == OP_AG_MM) ok = gather_tile(p, ctl, sm, c, wc);
            else if (p.op == OP_CONC) coll_tile(p, c, wc);
            else ok = reduce_tile<BN, STAGES>(p, ctl, c, wc);
        } else {
            ok = epilogue(p, ctl, sm, tmem, item, acc_i, wc, tr);
            ++acc_i;
        }
        tr.rec(EV_END, item);
        if (!ok) break;
    }
    tr.finish();
}

// ============================================================ kernel
template <int BN, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1) fused_gemm_coll_kernel(const __grid_constant__ Params p) {
    constexpr int TMEM_COLS = 2 * BN;
    extern __shared__ uint8_t smem_raw[];
    Smem<BN, STAGES> sm;
    sm.carve(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], NUM_WORKER_WARPS);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(&sm.item_full[i], 1);
            mbar_init(&sm.item_empty[i], 2 + NUM_WORKER_WARPS);  // MMA + TMA + workers
        }
        mbar_init(sm.wbar, NUM_WORKER_WARPS);
        mbar_init(sm.final_bar, 1);
        fence_mbar_init();
        uint32_t e = *reinterpret_cast<volatile uint32_t*>(&p.ws->epoch) + 1u;
        if (e == 0u) e = 1u;
        *sm.epoch_slot = e;
        if (p.n_gemm > 0 && p.k_blocks > 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
        }
    }
    if (warp == 1) tmem_alloc<TMEM_COLS>(sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;
    const Ctl ctl{p.ws, *sm.epoch_slot, p.wait_ns};

    if (warp == 0) {
        if (lane == 0) run_scheduler<BN, STAGES>(p, ctl, sm);
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0) run_tma<BN, STAGES>(p, ctl, sm);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) run_mma<BN, STAGES>(p, ctl, sm, tmem);
        __syncwarp();
    } else {
        run_workers<BN, STAGES>(p, ctl, sm, tmem, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<TMEM_COLS>(tmem);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(&p.ws->done_ctr, 1u);
        if (done == gridDim.x - 1) {
            // last CTA of the launch: reset the queues for the next launch on
            // this workspace and publish the epoch
            atomicExch(&p.ws->gemm_ctr, 0u);
            atomicExch(&p.ws->comm_ctr, 0u);
            atomicExch(&p.ws->done_ctr, 0u);
            __threadfence();
            atomicExch(&p.ws->epoch, ctl.epoch);
        }
    }
}

}  // namespace gct
