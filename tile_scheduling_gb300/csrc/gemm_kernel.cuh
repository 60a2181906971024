// Persistent, warp-specialised bf16 GEMM for sm_103a: D = A * B^T.
//
// The mainloop is the Merge example of CUTLASS TS "Pipeline Groups"
// (Overview): gmem_ab -> smem_a, smem_b -> tmem_c -> gmem_d.  By default A and
// B share one "full" and one "empty" mbarrier per ring stage (the FusedMerge
// layout, 2 * S barriers: one producer thread arrives with the summed
// transaction bytes of both loads, the single MMA consumer waits and releases
// once).  The MG = 1 variants take the Merge layout instead: A and B have a
// producer and a full barrier each and share the empty barrier (3 * S).
//
// Warp roles (256, 384 or 640 threads, one CTA per SM):
//   warp 0      TMA producer: per k-block, acquire an empty stage, arm the
//               full barrier with A+B bytes, issue the two tile loads
//               (TS "Introduction", Load-A skeleton: compute_coords, acquire,
//               tma_load_a, commit).
//   warp 1      TMEM allocator and the single MMA-issuing thread: per k-block,
//               wait full, 4 x tcgen05.mma (K = 16 each), commit -> empty.
//               The first MMA of every work tile overwrites the accumulator
//               (TS "Resources", per-work-tile scale_d reset).
//   warp 2      Cluster Launch Control scheduler (CLC mode only): fetches the
//               next tile while the current one is computed ("Cluster Launch
//               Control", overlap loop; TS "Schedules", dynamic persistent
//               shape with a dedicated scheduler task).
//   warp 3      barrier initialisation, then idle, the Fork row-sum task or
//               (Merge) the TMA producer of B.
//   warps 4..   epilogue, 4, 8 or 16 warps: TMEM -> registers (tcgen05.ld, 32
//               columns per load) -> fp32 or bf16 -> swizzled shared staging ->
//               TMA store, one subtile after another (TS "Resources", subtile
//               epilogue: load_subtile / store at column coordc_n +
//               subtile_idx * 32, bracketed by tmem_c.wait() / release()).
//               With 8 (16), two (four) warps share each TMEM lane quarter
//               and take its subtiles in turn.
//
// Every role walks the same tile sequence and advances at the same tile
// boundary (TS "Schedules", Persistent Scheduling).  Static mode: worker w of
// W takes tiles w, w + W, ... ("Cluster Launch Control", static persistent
// scheduler).  CLC mode: the grid covers all tiles, block (cluster) i starts
// on tile i and then takes the coordinates of launches it cancels.
// Non-persistent mode: the grid covers all tiles and block (cluster) i
// computes tile i alone (TS "Schedules", Scheduling Shapes).
//
// A work unit's k-blocks are loaded upwards, or downwards in the units of odd
// waves (GemmParams::k_alt), so each wave starts on operand panels the wave
// before it left in L2.  The previous kernel in the stream is waited for
// before any global memory access, or, with inputs_ready, by the epilogue
// first and by every other role after its first unit (the dependent-launch
// barrier as a resource of its own: see the comment at the wait).
//
// Two accumulators of BN fp32 columns live in TMEM, so the epilogue of one
// tile overlaps the mainloop of the next.  With CG = 2 a CTA pair computes a
// 256 x BN tile with cta_group::2 MMAs issued by the even CTA: each CTA loads
// its own 128 rows of A and BN/2 rows of B, both CTAs' loads complete on the
// even CTA's full barrier, and commits arrive on both CTAs' barriers.
//
// Every mbarrier wait is bounded (%globaltimer): on expiry the kernel records
// the wait in the device status word, raises a CTA-local abort flag, lets
// every role leave its loop, waits (with its own limit) for copies and MMAs
// still in flight, frees TMEM and returns.
//
// A logging instantiation (LOG = 1; a test instrument) has every role record
// its barrier operations in program order (PLog), for comparison with the
// host-side model of these role loops; in the product instantiations every
// logging call compiles to nothing.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace ts {

constexpr int kRoleWarps = 4;       // producer, MMA issuer, CLC scheduler, Fork task or B producer
constexpr int kSmemLimit = 232448;  // 227 KB: largest opt-in dynamic shared memory per CTA
constexpr int kMaxClcDepth = 2;
// Lazy CLC requests: the producer signals that its unit is nearly loaded this
// many k-blocks before the end of the unit (some 4 us of MMA on the pair tile,
// plus the ring's lead), so the request for the worker's next unit is issued
// shortly before that unit is needed rather than when the current one begins.
constexpr int kLazyLeadKBlocks = 16;

// EW_ epilogue warps: 4 (one per TMEM lane quarter), 8 or 16 (two or four per
// quarter, splitting the columns).  More warps hide more of the epilogue's
// instruction latencies when the K loop is short and the epilogue bounds the
// tile.  Sixteen are built for 256-column tiles only (each warp then stores
// one 128-byte-wide subtile per tile with bf16 output) and without the split
// tail's reduction, which does not fit their 96 registers per thread.
// MG_ selects the ring's barrier layout ("Pipeline Groups"): 0 is FusedMerge
// (one producer thread loads A and B onto one full barrier per stage, 2 * S
// barriers); 1 is Merge (a producer for A on warp 0 and one for B on warp 3,
// each with its own full barrier per stage, sharing the empty barrier:
// 3 * S barriers).  LOG_ = 1 compiles in the protocol log (a test instrument:
// every role records its barrier operations; see PLog); the product variants
// have LOG_ = 0, where every logging call compiles to nothing.
template <int BN_, int CG_, int OUT_, int EW_, int MG_ = 0, int LOG_ = 0>
struct GemmCfg {
    static constexpr int BN = BN_, CG = CG_, OUT = OUT_;
    static constexpr int EPI_WARPS = EW_;
    static constexpr int MERGE = MG_;
    static constexpr bool LOG = LOG_ != 0;
    static constexpr int THREADS = 32 * (kRoleWarps + EPI_WARPS);
    static constexpr int BM = 128;              // accumulator rows per CTA = TMEM lanes
    static constexpr int TILE_M = BM * CG;      // output rows per worker
    static constexpr int BK = 64;               // bf16 per 128-byte swizzle row
    static constexpr int UMMA_K = 16;
    static constexpr int B_ROWS = BN / CG;      // rows of B loaded by each CTA
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TX_BYTES = STAGE_BYTES * CG;  // bytes landing on the even CTA's full barrier
    static constexpr int TX_A_BYTES = A_BYTES * CG;     // Merge: on the A full barrier
    static constexpr int TX_B_BYTES = B_BYTES * CG;     // Merge: on the B full barrier
    static constexpr int OUT_BYTES = OUT == OUT_F32 ? 4 : 2;
    static constexpr int SUB_COLS = 128 / OUT_BYTES;   // store subtile: 128 bytes of a row
    static constexpr int NUM_SUB = BN / SUB_COLS;
    static constexpr int EPI_BUF = 32 * 128;           // one warp: 32 rows x 128 bytes
    // staging buffers per epilogue warp: 32 KB in all with 4 or 8 warps, so
    // the ring keeps its depth (the warps of a quarter alternate); 64 KB with
    // 16, which costs the ring one stage (only short K loops use them)
    static constexpr int EPI_BUFS = EPI_WARPS == 4 ? 2 : 1;
    static constexpr bool SPLIT = EPI_WARPS != 16;  // the split tiles' reduction is compiled in
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUFS * EPI_BUF;
    static constexpr int TMEM_COLS = 2 * BN;           // two accumulators
    static constexpr int BAR_BYTES = 512;  // CLC responses, mbarriers, TMEM address, abort flag, next-unit slots
    static constexpr int STAGES = (kSmemLimit - 1024 - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    // Barrier arrival counts (one place: the kernel initialises its barriers
    // with these, and the host-side protocol checker models them).
    static constexpr int FULL_ARRIVALS = 1;   // the even CTA's producer of that barrier (arrive.expect_tx)
    static constexpr int EMPTY_ARRIVALS = 1;  // one tcgen05.commit per stage use
    static constexpr int TFULL_ARRIVALS = 1;  // one tcgen05.commit per accumulator use
    static constexpr int TEMPTY_ARRIVALS = EPI_WARPS * CG;  // every epilogue warp of the CTA pair
    static constexpr int ACCUMULATORS = 2;
    static constexpr int CLC_FULL_ARRIVALS = 1;  // this CTA's scheduler thread arms the slot
    static constexpr int CLC_RESPONSE_BYTES = 16;
    static constexpr int AUX_EMPTY_ARRIVALS = 1;  // the Fork row-sum task (lane 0 of warp 3)
    // Consumers of one CLC response: producer(s), MMA, the epilogue warps and the
    // scheduler in the even CTA; producer(s), epilogue warps and scheduler in the odd one.
    static constexpr int CLC_CONSUMERS = (3 + MERGE + EPI_WARPS) + (CG == 2 ? 2 + MERGE + EPI_WARPS : 0);
    // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
    // (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at
    // bits 17-22, M >> 4 at bits 24-28.
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                                      (uint32_t((BM * CG) >> 4) << 24);

    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N");
    static_assert(CG == 1 || CG == 2, "cluster size");
    static_assert(EPI_WARPS == 4 || EPI_WARPS == 8 || EPI_WARPS == 16, "epilogue warps");
    static_assert(MERGE == 0 || MERGE == 1, "barrier layout");
    static_assert(NUM_SUB % (EPI_WARPS / 4) == 0, "subtiles split evenly between a quarter's warps");
    static_assert(STAGES >= 2, "ring too shallow");
    static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static_assert(3 * STAGES * 8 + 6 * 8 + 2 * kMaxClcDepth * 8 + 16 * kMaxClcDepth + 8 + 4 * EPI_WARPS <= BAR_BYTES,
                  "barrier region");
};

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4 (unused for this layout)
//   bits 32-45 stride byte offset >> 4 bits 46-48 fixed 0b001
//   bits 49-51 base offset (0: atoms 1024-aligned)   bits 61-63 layout (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    return uint64_t((smem_addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void report_timeout(const GemmParams &p, int where) {
    const unsigned long long info = (static_cast<unsigned long long>(where) << 32) | blockIdx.x;
    if (atomicCAS(&p.status[0], 0ull, 1ull) == 0ull) atomicExch(&p.status[1], info);
    atomicAdd(&p.status[2], 1ull);
}

// Bounded phase wait.  honor_abort: give up as soon as another role aborted
// (role loops); drains pass false and rely on their own limit alone.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort_flag,
                                       bool honor_abort, const GemmParams &p, int where) {
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (honor_abort && *abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                report_timeout(p, where);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           const GemmParams &p, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, p.timeout_ns, abort_flag, true, p, where);
}

// Bounded wait for roles whose waits last about a tile and whose wake-up is not
// on the critical path (epilogue warps waiting for an accumulator, the CLC
// scheduler waiting for a free slot): it sleeps between polls, leaving the
// issue slots and shared-memory port of its SM sub-partition to the producer
// and the MMA issuer.  Measured: 0.5-1 % faster at 8192^3 than polling.
static __device__ __noinline__ bool wait_long_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                   const GemmParams &p, int where) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > p.timeout_ns) {
            report_timeout(p, where);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(500);
    }
}

__device__ __forceinline__ bool wait_long(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const GemmParams &p, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_long_slow(bar, parity, abort_flag, p, where);
}

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           const GemmParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, p.drain_ns, abort_flag, false, p, WAIT_DRAIN);
}

// Protocol log: the barrier operations of each role's thread, in program
// order, so that a host-side model of the role loops can be compared with what
// the kernel does.  Event word: op | family << 4 | index << 8 | parity << 16
// (for PL_UNIT: op | skip << 4 | k-blocks << 8).  Roles: 0 the (A) producer,
// 1 the MMA issuer, 2 the CLC scheduler, 3 warp 3 (Merge B producer or Fork
// task), 4 + j epilogue warp j (lane 0).  Per CTA and role the log holds a
// count (events recorded, which may exceed the capacity) and `cap` words.
enum PlogOp : int32_t {
    PL_WAIT = 1,    // mbarrier wait on (family, index) with the given parity
    PL_ARRIVE = 2,  // arrive (with expect-tx where the op arms transaction bytes)
    PL_TMA = 3,     // a TMA load completing on (family, index)
    PL_MMA = 4,     // the MMAs of one k-block, reading ring stage `index`
    PL_COMMIT = 5,  // tcgen05.commit arriving on (family, index)
    PL_CREQ = 6,    // a CLC request into response slot `index`
    PL_PDL = 7,     // the wait on the dependent-launch barrier
    PL_UNIT = 8,    // the producer begins a unit
    PL_TLOAD = 9,   // this warp's reads of accumulator `index` are complete
    PL_CREAD = 10,  // CLC response slot `index` read
    PL_SREAD = 11   // ring stage `index` read by the Fork task
};
enum PlogFamily : int32_t {
    PF_FULL = 0, PF_EMPTY = 1, PF_TFULL = 2, PF_TEMPTY = 3, PF_CLC_FULL = 4, PF_CLC_EMPTY = 5,
    PF_AUX = 6,  // the Fork task's empty barrier, or Merge's full barrier of B
    PF_BEGAN = 7, PF_MMA_DONE = 8, PF_NONE = 15
};
constexpr int kPlogRoles = kRoleWarps + 16;

template <bool ON>
struct PLog {
    int32_t *buf = nullptr;
    int32_t cap = 0, n = 0;
    __device__ __forceinline__ void open(const GemmParams &p, int role) {
        if constexpr (ON) {
            if (p.plog) {
                buf = p.plog + (static_cast<int64_t>(blockIdx.x) * kPlogRoles + role) * (p.plog_cap + 1);
                cap = p.plog_cap;
            }
        }
    }
    __device__ __forceinline__ void put(int32_t op, int32_t family, uint32_t index, uint32_t parity) {
        if constexpr (ON) {
            if (buf) {
                if (n < cap) buf[1 + n] = op | (family << 4) | static_cast<int32_t>(index << 8) |
                                          static_cast<int32_t>((parity & 1u) << 16);
                ++n;
            }
        }
    }
    __device__ __forceinline__ void unit(bool skip, int32_t nkb) {
        if constexpr (ON) {
            if (buf) {
                if (n < cap) buf[1 + n] = PL_UNIT | ((skip ? 1 : 0) << 4) | (nkb << 8);
                ++n;
            }
        }
    }
    __device__ __forceinline__ void close() {
        if constexpr (ON) {
            if (buf) buf[0] = n;
        }
    }
};

// Shared-memory map of one CTA.
template <class C>
struct Smem {
    uint32_t a, b, epi;        // tile ring and epilogue staging (shared addresses)
    uint32_t resp;             // CLC response slots, 16 bytes each
    uint32_t bars;             // mbarrier array
    uint32_t *tmem_slot;
    volatile int *abort_flag;
    int32_t *next_slot;        // per epilogue warp: its next work unit, taken early (lane 0 writes and reads)

    __device__ __forceinline__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return bars + 8u * (C::STAGES + s); }
    __device__ __forceinline__ uint32_t tfull(int a) const { return bars + 8u * (2 * C::STAGES + a); }
    __device__ __forceinline__ uint32_t tempty(int a) const { return bars + 8u * (2 * C::STAGES + 2 + a); }
    __device__ __forceinline__ uint32_t mma_done() const { return bars + 8u * (2 * C::STAGES + 4); }
    __device__ __forceinline__ uint32_t clc_full(int r) const { return bars + 8u * (2 * C::STAGES + 5 + r); }
    __device__ __forceinline__ uint32_t clc_empty(int r) const {
        return bars + 8u * (2 * C::STAGES + 5 + kMaxClcDepth + r);
    }
    // Fork: the second consumer of ring stage s (the row-sum task) releases it here.
    __device__ __forceinline__ uint32_t aux_empty(int s) const {
        return bars + 8u * (2 * C::STAGES + 5 + 2 * kMaxClcDepth + s);
    }
    // Merge: B's full barrier of stage s (full(s) then tracks A alone).  The
    // Fork consumer and Merge never run together, so they share the slots.
    __device__ __forceinline__ uint32_t full_b(int s) const { return aux_empty(s); }
    // The producer arrives here once per work unit, when at most
    // kLazyLeadKBlocks of the unit's k-blocks remain to be loaded (at once for a
    // shorter or empty unit): phase j completes when it reaches that point of its
    // j-th unit (lazy CLC requests wait on it).
    __device__ __forceinline__ uint32_t prod_began() const {
        return bars + 8u * (3 * C::STAGES + 5 + 2 * kMaxClcDepth);
    }
};

// One work unit: a whole output tile, or one K-range of a split tile.
struct Unit {
    int32_t tile;      // output tile id within its group (raster order)
    int32_t kb0, kb1;  // k-blocks [kb0, kb1)
    int32_t tail;      // index among the split tiles, or -1 for a whole tile
    int32_t part;      // K part of a split tile
    int32_t group;     // group of a grouped GEMM (0 otherwise)
    bool skip;         // the tile is skipped: no data work, only queue bookkeeping
};

__device__ __forceinline__ Unit decode_unit(int32_t u, const GemmParams &p) {
    Unit w;
    w.group = 0;
    if (p.groups > 0) {
        // dynamic domain: the k-block range comes from the group's offsets; the
        // groups are scheduled longest first (GemmParams::group_order)
        const int32_t slot = u / p.tiles_per_group;
        w.group = p.group_order[slot];
        w.tile = u - slot * p.tiles_per_group;
        w.kb0 = p.group_kb[w.group];
        w.kb1 = p.group_kb[w.group + 1];
        w.tail = -1;
        w.part = 0;
    } else if (u < p.split_tiles * p.parts) {
        // a K part of a split tile (those units come first)
        w.tail = u / p.parts;
        w.part = u - w.tail * p.parts;
        w.tile = w.tail;
        w.kb0 = static_cast<int32_t>(static_cast<int64_t>(w.part) * p.num_k_blocks / p.parts);
        w.kb1 = static_cast<int32_t>(static_cast<int64_t>(w.part + 1) * p.num_k_blocks / p.parts);
    } else {
        w.tile = u - p.split_tiles * (p.parts - 1);
        w.kb0 = 0;
        w.kb1 = p.num_k_blocks;
        w.tail = -1;
        w.part = 0;
    }
    // Skippable tiles (TS "Schedules", Skippable Tiles): every role still takes
    // and advances past the unit, but a skipped tile loads, multiplies and
    // stores nothing.
    w.skip = false;
    if (p.skip != nullptr) {
        int32_t mb, nb;
        raster(w.tile, p, mb, nb);
        w.skip = p.skip[w.group * p.tiles_per_group + mb * p.tiles_n + nb] != 0;
    }
    if (w.skip) w.kb1 = w.kb0;
    return w;
}

// Consume the next CLC response (one thread per consuming role).  Returns the
// next work unit, or -1 when the cancel failed (no pending launch left) or the
// kernel is aborting.
template <class C>
__device__ __forceinline__ int32_t clc_consume(const Smem<C> &sm, const GemmParams &p, uint32_t &idx,
                                               PLog<C::LOG> &lg) {
    const uint32_t depth = static_cast<uint32_t>(p.clc_depth);
    const uint32_t r = idx % depth;
    const uint32_t ph = (idx / depth) & 1u;
    ++idx;
    lg.put(PL_WAIT, PF_CLC_FULL, r, ph);
    if (!wait_phase(sm.clc_full(r), ph, sm.abort_flag, p, WAIT_CLC_FULL)) return -1;
    uint32_t x = 0;
    const bool ok = clc_query(sm.resp + 16u * r, x);
    lg.put(PL_CREAD, PF_CLC_FULL, r, 0);
    fence_proxy_async_smem();  // our generic read of the slot before the next async write into it
    lg.put(PL_ARRIVE, PF_CLC_EMPTY, r, 0);
    if constexpr (C::CG == 1)
        mbar_arrive(sm.clc_empty(r));
    else
        mbar_arrive_cluster(mapa(sm.clc_empty(r), 0));
    return ok ? static_cast<int32_t>(x / C::CG) : -1;
}

template <class C>
__device__ __forceinline__ int32_t next_unit(const Smem<C> &sm, const GemmParams &p, int32_t unit,
                                             uint32_t &clc_idx, PLog<C::LOG> &lg) {
    if (p.sched == SCHED_STATIC) {
        const int32_t u = unit + static_cast<int32_t>(gridDim.x / C::CG);
        return u < p.num_units ? u : -1;
    }
    if (p.sched == SCHED_NONPERSISTENT) return -1;  // one unit per CTA (cluster)
    return clc_consume(sm, p, clc_idx, lg);
}

template <int BN, int CG, int OUT, int EW, int MG, int LOG = 0>
__global__ void __launch_bounds__(32 * (kRoleWarps + EW), 1)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ GemmParams p) {
    using C = GemmCfg<BN, CG, OUT, EW, MG, LOG>;
    using Log = PLog<C::LOG>;
    constexpr int RAW = C::SUB_COLS;  // fp32 accumulator words per lane per store subtile
    extern __shared__ __align__(1024) uint8_t smem_raw[];

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    Smem<C> sm;
    sm.a = base;
    sm.b = sm.a + C::STAGES * C::A_BYTES;
    sm.epi = sm.b + C::STAGES * C::B_BYTES;
    sm.resp = sm.epi + C::EPI_BYTES;
    sm.bars = sm.resp + 16u * kMaxClcDepth;
    const uint32_t tail = sm.bars + 8u * (3 * C::STAGES + 6 + 2 * kMaxClcDepth);
    sm.tmem_slot = reinterpret_cast<uint32_t *>(gbase + (tail - base));
    sm.abort_flag = reinterpret_cast<volatile int *>(gbase + (tail - base) + 4);
    sm.next_slot = reinterpret_cast<int32_t *>(gbase + (tail - base) + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const int32_t worker = static_cast<int32_t>(blockIdx.x / CG);
    // Fork pipeline group (CUTLASS TS "Pipeline Groups", Fork): each ring stage
    // is filled once and read by two consumer tasks, the MMA issuer and the
    // row-sum task on warp 3; each releases the stage on its own empty barrier
    // and the producer refills it only after both.  One-CTA tiles only.
    const bool fork = !MG && CG == 1 && p.row_sums != nullptr;

    // ------------------------------------------------------------ prologue
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.tma_store) prefetch_tmap(&tmD);
    }
    if (warp == 3 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(sm.full(s), C::FULL_ARRIVALS);
            mbar_init(sm.empty(s), C::EMPTY_ARRIVALS);
        }
        for (int a = 0; a < C::ACCUMULATORS; ++a) {
            mbar_init(sm.tfull(a), C::TFULL_ARRIVALS);
            mbar_init(sm.tempty(a), C::TEMPTY_ARRIVALS);
        }
        mbar_init(sm.mma_done(), 1);
        for (int r = 0; r < kMaxClcDepth; ++r) {
            mbar_init(sm.clc_full(r), C::CLC_FULL_ARRIVALS);
            // with the Fork row-sum task, warp 3 consumes every response too (with
            // Merge, its B producer is counted in CLC_CONSUMERS)
            mbar_init(sm.clc_empty(r), C::CLC_CONSUMERS + (fork ? 1 : 0));
        }
        // Fork: the row-sum task's empty barriers; Merge: B's full barriers (one arrival each)
        for (int s = 0; s < C::STAGES; ++s) mbar_init(sm.aux_empty(s), MG ? C::FULL_ARRIVALS : C::AUX_EMPTY_ARRIVALS);
        mbar_init(sm.prod_began(), 1);
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(sm.tmem_slot), C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(sm.tmem_slot);
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: everything above touches only this CTA's shared memory, TMEM and
    // the kernel parameters, so it overlaps that kernel's tail.  The
    // dependent-launch barrier (the previous kernel's completion, its writes
    // visible) is a resource of its own (CUTLASS TS "Introduction", Core Terms:
    // a PDL barrier).  By default every role waits on it here, before any global
    // memory access.  With inputs_ready the caller states that A, B and the skip
    // mask were final before the previous kernel began: the epilogue, which
    // writes D (and the split partials, counters and trace), waits on it first;
    // every other role runs its first work unit ahead of it and waits on it
    // before its second (the producer before its first trace write, the Fork
    // task before its first row-sum store).  No wait of a role's first unit
    // depends on the epilogue (the ring drains into the first accumulator, the
    // first CLC response slots are free), so every bounded wait that could last
    // as long as the previous kernel starts after the barrier.  The first
    // units' loads and MMAs then overlap the previous kernel's tail.  The next
    // kernel is allowed to launch only after this barrier: it cannot occupy an
    // SM before this grid's CTA there has exited (a CTA takes all of an SM's
    // shared memory), and it waits on its own barrier in turn.
    if (!p.inputs_ready) {
        grid_dep_wait();
        grid_dep_launch();
    }
    // A role's wait on the barrier after its first unit (inputs_ready only).
    auto dep_wait_once = [&](bool &waited, Log &lg) {
        if (p.inputs_ready && !waited) {
            lg.put(PL_PDL, PF_NONE, 0, 0);
            grid_dep_wait();
            waited = true;
        }
    };

    const int32_t first_unit = worker < p.num_units ? worker : -1;

    // TMA producer loop of one thread: per k-block of the unit (upwards, or
    // downwards in the units of odd waves: GemmParams::k_alt), acquire the stage's
    // empty barrier (and the Fork consumer's), arm full_bar(stage) with `tx` bytes
    // (the even CTA), issue the A and/or B tile loads, which complete on the
    // even CTA's barrier.  FusedMerge: warp 0 loads both onto full(s).  Merge:
    // warp 0 loads A onto full(s) and warp 3 loads B onto full_b(s).
    auto produce = [&](const bool load_a, const bool load_b, const bool b_bar, const uint32_t tx) {
        auto full_bar = [&](uint32_t st) { return b_bar ? sm.full_b(st) : sm.full(st); };
        const int32_t full_fam = b_bar ? PF_AUX : PF_FULL;
        Log lg;
        lg.open(p, load_a ? 0 : 3);
        int32_t unit = first_unit;
        uint32_t clc_idx = 0, stage = 0, phase = 0, issued = 0;
        bool alive = true, waited = false;
        if (p.trace) dep_wait_once(waited, lg);  // the trace is written below
        while (unit >= 0 && alive) {
            const Unit w = decode_unit(unit, p);
            const int32_t nkb = w.kb1 - w.kb0;
            lg.unit(w.skip, nkb);
            // the load at which the unit counts as nearly loaded (lazy CLC requests wait for it)
            const int32_t near_end = nkb > kLazyLeadKBlocks ? nkb - kLazyLeadKBlocks : 0;
            const bool rev = p.k_alt && (fast_div(unit, p.div_wave) & 1);
            if (load_a && nkb <= 0) {
                lg.put(PL_ARRIVE, PF_BEGAN, 0, 0);
                mbar_arrive(sm.prod_began());
            }
            int32_t mb, nb;
            raster(w.tile, p, mb, nb);
            const int32_t a_row = mb * C::TILE_M + static_cast<int32_t>(rank) * C::BM;
            const int32_t b_row = nb * BN + static_cast<int32_t>(rank) * C::B_ROWS;
            if (p.trace && rank == 0 && load_a) p.trace[4 * unit + 2] = static_cast<long long>(globaltimer());
            for (int32_t i = 0; i < nkb; ++i) {
                const int32_t kb = rev ? w.kb1 - 1 - i : w.kb0 + i;
                if (load_a && i == near_end) {
                    lg.put(PL_ARRIVE, PF_BEGAN, 0, 0);
                    mbar_arrive(sm.prod_began());
                }
                lg.put(PL_WAIT, PF_EMPTY, stage, phase ^ 1u);
                if (!wait_phase(sm.empty(stage), phase ^ 1u, sm.abort_flag, p, WAIT_PRODUCER_EMPTY)) {
                    alive = false;
                    break;
                }
                if (fork) {
                    lg.put(PL_WAIT, PF_AUX, stage, phase ^ 1u);
                    if (!wait_phase(sm.aux_empty(stage), phase ^ 1u, sm.abort_flag, p, WAIT_PRODUCER_EMPTY)) {
                        alive = false;
                        break;
                    }
                }
                const uint32_t fb = full_bar(stage);
                if (rank == 0) {
                    lg.put(PL_ARRIVE, full_fam, stage, 0);
                    mbar_arrive_expect_tx(fb, tx);
                }
                const uint32_t da = sm.a + stage * C::A_BYTES;
                const uint32_t db = sm.b + stage * C::B_BYTES;
                if constexpr (CG == 1) {
                    if (load_a) tma_load_2d(da, &tmA, fb, kb * C::BK, a_row);
                    if (load_b) tma_load_2d(db, &tmB, fb, kb * C::BK, b_row);
                } else {
                    const uint32_t fb0 = mapa(fb, 0);
                    if (load_a) tma_load_2d_pair(da, &tmA, fb0, kb * C::BK, a_row);
                    if (load_b) tma_load_2d_pair(db, &tmB, fb0, kb * C::BK, b_row);
                }
                lg.put(PL_TMA, full_fam, stage, 0);  // this producer's loads of the stage
                ++issued;
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!alive) break;
            dep_wait_once(waited, lg);
            unit = next_unit(sm, p, unit, clc_idx, lg);
        }
        dep_wait_once(waited, lg);
        // Drain: every issued load has landed (even CTA's full barriers) and
        // the MMA has released every stage.
        if (rank == 0) {
            const uint32_t n = issued < C::STAGES ? issued : C::STAGES;
            for (uint32_t i = 1; i <= n; ++i) {
                const uint32_t b = issued - i;
                lg.put(PL_WAIT, full_fam, b % C::STAGES, (b / C::STAGES) & 1u);
                wait_drain(full_bar(b % C::STAGES), (b / C::STAGES) & 1u, sm.abort_flag, p);
            }
        }
        for (int i = 0; i < C::STAGES; ++i) {
            lg.put(PL_WAIT, PF_EMPTY, stage, phase ^ 1u);
            if (!wait_drain(sm.empty(stage), phase ^ 1u, sm.abort_flag, p)) break;
            if (fork) {
                lg.put(PL_WAIT, PF_AUX, stage, phase ^ 1u);
                if (!wait_drain(sm.aux_empty(stage), phase ^ 1u, sm.abort_flag, p)) break;
            }
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        lg.close();
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            if constexpr (MG)
                produce(true, false, false, C::TX_A_BYTES);
            else
                produce(true, true, false, C::TX_BYTES);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            Log lg;
            lg.open(p, 1);
            int32_t unit = first_unit;
            uint32_t clc_idx = 0, stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool alive = true, waited = false;
            while (unit >= 0 && alive) {
                const Unit w = decode_unit(unit, p);
                if (w.skip) {  // no accumulator is used for a skipped tile
                    dep_wait_once(waited, lg);
                    unit = next_unit(sm, p, unit, clc_idx, lg);
                    continue;
                }
                lg.put(PL_WAIT, PF_TEMPTY, acc, acc_phase ^ 1u);
                if (!wait_phase(sm.tempty(acc), acc_phase ^ 1u, sm.abort_flag, p, WAIT_MMA_TMEM_EMPTY)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    lg.put(PL_WAIT, PF_FULL, stage, phase);
                    if (!wait_phase(sm.full(stage), phase, sm.abort_flag, p, WAIT_MMA_FULL)) {
                        alive = false;
                        break;
                    }
                    if constexpr (MG) {
                        lg.put(PL_WAIT, PF_AUX, stage, phase);
                        if (!wait_phase(sm.full_b(stage), phase, sm.abort_flag, p, WAIT_MMA_FULL)) {
                            alive = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const uint64_t da = sw128_kmajor_desc(sm.a + stage * C::A_BYTES);
                    const uint64_t db = sw128_kmajor_desc(sm.b + stage * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk) {
                        // +32 bytes per K = 16 step inside the 128-byte swizzle row (encoded >> 4);
                        // the first MMA of a unit overwrites the accumulator
                        mma_bf16<CG>(d_tmem, da + 2u * kk, db + 2u * kk, C::IDESC, (kb != w.kb0) || (kk != 0));
                    }
                    lg.put(PL_MMA, PF_FULL, stage, 0);
                    lg.put(PL_COMMIT, PF_EMPTY, stage, 0);
                    if constexpr (CG == 1)
                        mma_commit(sm.empty(stage));
                    else
                        mma_commit_pair(sm.empty(stage), 0x3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!alive) break;
                lg.put(PL_COMMIT, PF_TFULL, acc, 0);
                if constexpr (CG == 1)
                    mma_commit(sm.tfull(acc));
                else
                    mma_commit_pair(sm.tfull(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                dep_wait_once(waited, lg);
                unit = next_unit(sm, p, unit, clc_idx, lg);
            }
            dep_wait_once(waited, lg);
            // Every MMA issued by this thread has completed before TMEM is freed.
            lg.put(PL_COMMIT, PF_MMA_DONE, 0, 0);
            if constexpr (CG == 1)
                mma_commit(sm.mma_done());
            else
                mma_commit_pair(sm.mma_done(), 0x1);
            lg.put(PL_WAIT, PF_MMA_DONE, 0, 0);
            wait_drain(sm.mma_done(), 0, sm.abort_flag, p);
            lg.close();
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------- CLC scheduler
        if (lane == 0 && p.sched == SCHED_CLC && first_unit >= 0) {
            Log lg;
            lg.open(p, 2);
            uint32_t idx = 0;
            bool outstanding = false, waited = false;
            uint32_t out_r = 0, out_ph = 0;
            const uint32_t depth = static_cast<uint32_t>(p.clc_depth);
            for (;;) {
                const uint32_t r = idx % depth;
                const uint32_t ph = (idx / depth) & 1u;
                if (rank == 0) {
                    lg.put(PL_WAIT, PF_CLC_EMPTY, r, ph ^ 1u);
                    if (!wait_long(sm.clc_empty(r), ph ^ 1u, sm.abort_flag, p, WAIT_SCHED_CLC_EMPTY)) break;
                    // Lazy requests (long K loops): request idx names the unit after this
                    // worker's unit idx, so it waits until the producer has all but the last
                    // kLazyLeadKBlocks of unit idx loaded (completion idx + 1 of prod_began).
                    // A worker then claims its next unit shortly before it needs it, not
                    // when its current unit begins, so the units left late in the launch go
                    // to the workers that finish first.
                    if (p.clc_lazy) {
                        lg.put(PL_WAIT, PF_BEGAN, 0, idx & 1u);
                        if (!wait_long(sm.prod_began(), idx & 1u, sm.abort_flag, p, WAIT_SCHED_PRODUCER)) break;
                    }
                    fence_proxy_async_smem();
                    lg.put(PL_ARRIVE, PF_CLC_FULL, r, 0);
                    mbar_arrive_expect_tx(sm.clc_full(r), C::CLC_RESPONSE_BYTES);
                    lg.put(PL_CREQ, PF_CLC_FULL, r, 0);
                    if constexpr (CG == 1)
                        clc_try_cancel(sm.resp + 16u * r, sm.clc_full(r));
                    else
                        clc_try_cancel_all(sm.resp + 16u * r, sm.clc_full(r));
                    outstanding = true;
                    out_r = r;
                    out_ph = ph;
                } else {
                    // the even CTA's request multicasts its response here: arm our barrier for it
                    lg.put(PL_ARRIVE, PF_CLC_FULL, r, 0);
                    mbar_arrive_expect_tx(sm.clc_full(r), C::CLC_RESPONSE_BYTES);
                }
                const int32_t t = clc_consume(sm, p, idx, lg);
                outstanding = false;
                if (t < 0) {
                    // a failed wait leaves the request possibly in flight
                    if (*sm.abort_flag && rank == 0) outstanding = true;
                    break;
                }
                dep_wait_once(waited, lg);
            }
            dep_wait_once(waited, lg);
            if (outstanding) wait_drain(sm.clc_full(out_r), out_ph, sm.abort_flag, p);
            lg.close();
        }
        __syncwarp();
    } else if (warp == 3 && MG) {
        // ------------------------------------------------- Merge: TMA producer of B
        if (lane == 0) produce(false, true, true, C::TX_B_BYTES);
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------- Fork consumer: row sums of A
        // Reads every ring stage after the MMA issuer's full barrier; on the
        // tiles of the first tile column (n block 0) it adds each row of the A
        // tile (64 bf16 per row; lane L owns rows L, L+32, L+64, L+96) to a
        // running fp32 sum over the unit's k-blocks and stores it at the end.
        if (fork) {
            Log lg;
            if (lane == 0) lg.open(p, 3);
            int32_t unit = first_unit;
            uint32_t clc_idx = 0, stage = 0, phase = 0;
            bool alive = true, waited = false;
            while (unit >= 0 && alive) {
                const Unit w = decode_unit(unit, p);
                int32_t mb, nb;
                raster(w.tile, p, mb, nb);
                const bool active = nb == 0 && !w.skip;
                // eight accumulators per row (one per chunk slot) keep the adds
                // independent; they are combined in slot order at the end
                float sum[4][8];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c) sum[r][c] = 0.f;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    int ok = 1;
                    lg.put(PL_WAIT, PF_FULL, stage, phase);
                    if (lane == 0) ok = wait_phase(sm.full(stage), phase, sm.abort_flag, p, WAIT_MMA_FULL);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        alive = false;
                        break;
                    }
                    if (active) {
                        const uint32_t a_tile = sm.a + stage * C::A_BYTES;
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t row = a_tile + static_cast<uint32_t>(lane + 32 * r) * 128u;
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                // The sum does not care about the order of a row's chunks;
                                // reading slot c ^ (lane & 7) puts every 8 lanes on 8
                                // different 16-byte bank groups (no bank conflicts).
                                uint32_t x0, x1, x2, x3;
                                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                             : "r"(row + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4)));
                                const uint32_t xs[4] = {x0, x1, x2, x3};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    sum[r][c] += __uint_as_float(xs[j] << 16);
                                    sum[r][c] += __uint_as_float(xs[j] & 0xffff0000u);
                                }
                            }
                        }
                    }
                    lg.put(PL_SREAD, PF_FULL, stage, 0);
                    __syncwarp();
                    lg.put(PL_ARRIVE, PF_AUX, stage, 0);
                    if (lane == 0) mbar_arrive(sm.aux_empty(stage));
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!alive) break;
                dep_wait_once(waited, lg);  // before the first row-sum store
                if (active) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float t = sum[r][0];
#pragma unroll
                        for (int c = 1; c < 8; ++c) t += sum[r][c];
                        const int32_t row = mb * C::TILE_M + lane + 32 * r;
                        if (row < p.M) p.row_sums[static_cast<int64_t>(w.group) * p.M + row] = t;
                    }
                }
                int32_t nu = 0;
                if (lane == 0) nu = next_unit(sm, p, unit, clc_idx, lg);
                unit = __shfl_sync(0xffffffffu, nu, 0);
            }
            dep_wait_once(waited, lg);
            lg.close();
        }
        __syncwarp();
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        // Warps 4 .. 4 + EW - 1.  A warp may access TMEM lanes 32 * (warp % 4) onwards:
        // warp 4 + j takes lane quarter q = j % 4 and, with 8 or 16 warps, the
        // subtiles s = h, h + EW / 4, ... (h = j / 4) of that quarter's rows.
        Log lg;
        if (lane == 0) lg.open(p, warp);
        if (p.inputs_ready) {  // D and this task's other outputs wait for the previous kernel
            lg.put(PL_PDL, PF_NONE, 0, 0);
            grid_dep_wait();
            grid_dep_launch();
        }
        constexpr int HALVES = C::EPI_WARPS / 4;
        const int q = (warp - kRoleWarps) & 3;
        const int h = (warp - kRoleWarps) >> 2;
        const uint32_t stg = sm.epi + static_cast<uint32_t>(warp - kRoleWarps) * C::EPI_BUFS * C::EPI_BUF;
        int32_t unit = first_unit;
        uint32_t clc_idx = 0, acc = 0, acc_phase = 0, buf = 0;
        // D is written once and never read back by this kernel: its TMA stores
        // mark their L2 lines evict-first (measured: the output-bound
        // 8192 x 8192 x 64 launch 1.6-6 % shorter, by tile and scheduler; no
        // change at 8192^3).
        const uint64_t store_policy = policy_evict_first();

        // Convert one subtile of fp32 accumulator words and write it to D.
        // Subtiles wholly outside D are skipped (no staging write, no store
        // group).  A TMA store is used only for boxes whose columns lie inside
        // D: the store clips rows exactly but a ragged right edge only to
        // 16-byte granules, so a subtile that crosses N takes plain stores.
        auto emit = [&](const uint32_t (&v)[RAW], int32_t row0, int32_t col, int32_t group) {
            if (row0 >= p.M || col >= p.N) return;
            uint32_t w[32];
            if constexpr (OUT == OUT_F32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = v[j];
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
            }
            if (p.tma_store && col + C::SUB_COLS <= p.N) {
                if (lane == 0) bulk_wait_read<C::EPI_BUFS - 1>();  // the store that used this buffer has read it
                __syncwarp();
                const uint32_t row_addr = stg + buf * C::EPI_BUF + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), w[4 * j], w[4 * j + 1],
                                 w[4 * j + 2], w[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&tmD, stg + buf * C::EPI_BUF, col, row0, group, store_policy);
                    bulk_commit();
                }
                buf = buf + 1u == C::EPI_BUFS ? 0u : buf + 1u;
            } else {
                const int32_t row = row0 + lane;
                if (row < p.M) {
                    if constexpr (OUT == OUT_F32) {
                        float *dst = static_cast<float *>(p.D) + group * p.group_stride +
                                     static_cast<int64_t>(row) * p.ldd + col;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col + j < p.N) dst[j] = __uint_as_float(w[j]);
                    } else {
                        uint16_t *dst = static_cast<uint16_t *>(p.D) + group * p.group_stride +
                                        static_cast<int64_t>(row) * p.ldd + col;
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (col + j < p.N) dst[j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
                    }
                }
            }
        };
        // fp32 partial of one warp slab (32 rows x BN) of a split unit, laid out so
        // that every warp-wide 16-byte access covers 512 contiguous bytes.
        auto slab_of = [&](const Unit &w, int32_t part) -> float4 * {
            const int64_t slab = (static_cast<int64_t>(w.tail) * p.parts + part) * (CG * 4) + rank * 4 + q;
            return reinterpret_cast<float4 *>(p.partials + slab * (32 * BN));
        };

        while (unit >= 0) {
            const Unit w = decode_unit(unit, p);
            int32_t mb, nb;
            raster(w.tile, p, mb, nb);
            // The next unit is taken as soon as this warp holds the accumulator, before
            // its TMEM reads and stores (and a split unit's partial write and
            // reduction): the epilogue is the last consumer of each CLC response, so
            // taking it early frees the slot for the scheduler's next request sooner.
            // Measured at 4096^3, 2-CTA CLC with split tiles: 80.7 -> 76.2 us.  Lane 0
            // parks the unit in shared memory until the end of the tile, so it holds
            // no register through the stores and the reduction.
            bool taken = false;
            const int32_t row0 = mb * C::TILE_M + static_cast<int32_t>(rank) * C::BM + 32 * q;
            const int32_t col0 = nb * BN;
            const bool split = C::SPLIT && w.tail >= 0;  // the host plans no split for 16 warps
            if (!w.skip) {
            int ok = 1;
            lg.put(PL_WAIT, PF_TFULL, acc, acc_phase);
            if (lane == 0) ok = wait_long(sm.tfull(acc), acc_phase, sm.abort_flag, p, WAIT_EPI_TMEM_FULL);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) sm.next_slot[warp - kRoleWarps] = next_unit(sm, p, unit, clc_idx, lg);
            taken = true;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN;
            float4 *const mine = split ? slab_of(w, w.part) : nullptr;
#pragma unroll 1
            for (int s = h; s < C::NUM_SUB; s += HALVES) {
                uint32_t v[RAW];
                if constexpr (RAW == 32) {
                    tmem_ld_32x32b_x32(taddr + s * 32, v);
                } else {
                    uint32_t(&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t(&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    tmem_ld_32x32b_x32(taddr + s * RAW, lo);
                    tmem_ld_32x32b_x32(taddr + s * RAW + 32, hi);
                }
                tmem_ld_wait();
                if (w.kb1 == w.kb0) {
                    // a group with K = 0: the accumulator was never written, D is zero
#pragma unroll
                    for (int j = 0; j < RAW; ++j) v[j] = 0u;
                }
                if (s + HALVES >= C::NUM_SUB) {
                    // this warp's part of the accumulator is read: hand it back to the MMA issuer
                    tc_fence_before();
                    __syncwarp();
                    lg.put(PL_TLOAD, PF_TFULL, acc, 0);
                    lg.put(PL_ARRIVE, PF_TEMPTY, acc, 0);
                    if (lane == 0) {
                        if constexpr (CG == 1)
                            mbar_arrive(sm.tempty(acc));
                        else
                            mbar_arrive_cluster(mapa(sm.tempty(acc), 0));
                    }
                }
                if (split) {
#pragma unroll
                    for (int c = 0; c < RAW / 4; ++c)
                        __stcg(mine + (s * (RAW / 4) + c) * 32 + lane,
                               make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                           __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
                } else {
                    emit(v, row0, col0 + s * C::SUB_COLS, w.group);
                }
            }
            if (split) {
                // The last of the `parts` warps to finish this slab (its subtiles of
                // it, with eight warps) sums the partials in part order and stores
                // D; it also re-arms the counter.
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    int32_t *cnt =
                        p.counters + ((w.tail * CG + static_cast<int32_t>(rank)) * 4 + q) * HALVES + h;
                    last = atomicAdd(cnt, 1) == p.parts - 1;
                    if (last) atomicExch(cnt, 0);
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
#pragma unroll 1
                    for (int s = h; s < C::NUM_SUB; s += HALVES) {
                        uint32_t v[RAW];
                        // F4 float4 (4 * F4 columns) at a time: every part's F4 float4
                        // per lane are in flight together, then summed in part order
                        // 0, 1, ...  Eight epilogue warps leave half the registers.
                        constexpr int F4 = C::EPI_WARPS == 4 ? 8 : 4;
#pragma unroll
                        for (int ch = 0; ch < RAW / (4 * F4); ++ch) {
                            float4 x[kMaxParts][F4];
#pragma unroll
                            for (int pp = 0; pp < kMaxParts; ++pp) {
                                if (pp < p.parts) {
                                    const float4 *src = slab_of(w, pp) + (s * (RAW / 4) + ch * F4) * 32 + lane;
#pragma unroll
                                    for (int c = 0; c < F4; ++c) x[pp][c] = __ldcg(src + c * 32);
                                }
                            }
#pragma unroll
                            for (int c = 0; c < F4; ++c) {
                                float4 a = x[0][c];
#pragma unroll
                                for (int pp = 1; pp < kMaxParts; ++pp) {
                                    if (pp < p.parts) {
                                        a.x += x[pp][c].x;
                                        a.y += x[pp][c].y;
                                        a.z += x[pp][c].z;
                                        a.w += x[pp][c].w;
                                    }
                                }
                                v[ch * 4 * F4 + 4 * c] = __float_as_uint(a.x);
                                v[ch * 4 * F4 + 4 * c + 1] = __float_as_uint(a.y);
                                v[ch * 4 * F4 + 4 * c + 2] = __float_as_uint(a.z);
                                v[ch * 4 * F4 + 4 * c + 3] = __float_as_uint(a.w);
                            }
                        }
                        emit(v, row0, col0 + s * C::SUB_COLS, w.group);
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            }  // !w.skip
            if (p.trace && rank == 0 && q == 0 && h == 0 && lane == 0) {
                atomicAdd(reinterpret_cast<unsigned long long *>(&p.trace[4 * unit]), 1ull);
                p.trace[4 * unit + 1] = worker;
                p.trace[4 * unit + 3] = static_cast<long long>(globaltimer());
            }
            int32_t nu = 0;
            if (lane == 0) nu = taken ? sm.next_slot[warp - kRoleWarps] : next_unit(sm, p, unit, clc_idx, lg);  // a skipped tile
            unit = __shfl_sync(0xffffffffu, nu, 0);
        }
        if (lane == 0) bulk_wait<0>();
        lg.close();
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
}

}  // namespace ts
