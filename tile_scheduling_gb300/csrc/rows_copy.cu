// Jagged int16 copy driven by a work queue.
//
// The two copy examples of CUTLASS TS "Schedules": Dynamic Domain (work tile t
// copies a row whose length comes from an offsets array, offsets[t + 1] -
// offsets[t]) and Skippable Tiles (the oversubscribed copy queue: a per-tile
// predicate decides whether the row copy runs, while every tile still takes
// part in the queue's wait / advance / release).  The work-tile loop runs on
// either scheduler of "Cluster Launch Control": a static grid-stride
// persistent loop (tile = blockIdx.x + i * gridDim.x), or one CTA per tile
// whose running CTAs cancel pending ones; or, non-persistent, one CTA per
// tile that copies its own tile and exits.  The CLC request for the next tile
// is issued before the current row is copied, so its latency hides under the
// copy (the overlap loop of that page).
//
// A row is copied by the whole CTA: a ragged head until src + begin reaches
// the vector alignment, 32-byte (or 16-byte) vectors with two in flight per
// thread, and a ragged tail; when src and dst differ modulo 16 bytes, aligned
// dst vectors joined from two source vectors.  Row bounds are read on the device and checked
// against [0, n] before any access; a row that fails the check is reported in
// the status word and not copied.
//
// Chunked mode (not on the pages): rows are cut into pieces of at most `chunk`
// elements and every piece is a work tile, so that a long row is not left to
// one CTA at the end of the queue.  Two planning kernels scan the piece
// counts (per CTA of 1024 rows, then across those CTAs) and write, per row,
// its first tile (base) and, per tile, its row (map); the copy kernel then
// finds tile t's piece with two loads.  The planning kernels and the copy
// kernel are launched as programmatic dependents, so each is scheduled while
// the one before it finishes.  The
// launch's tile count is an upper bound on the pieces (rows + ceil(n / chunk)
// for rows that do not overlap); tiles past the last piece are skipped like
// the oversubscribed tiles above.
//
// Packed mode (chunk and pack): the kept rows are laid end to end in a
// virtual index space and tile t copies its elements [t * chunk, (t + 1) *
// chunk): a long row spans several tiles and short rows share one, so every
// tile but the last moves `chunk` elements.  The planning kernels write each
// row's virtual start (base) and, per tile, the row holding its first element
// (map).  A tile's CTA takes its rows' segments in batches of one row per
// thread, scans their vector counts in shared memory and copies the vectors
// of all segments as one flat range, so a tile of short rows keeps as many
// loads in flight as a tile of one long row.  Equal tiles also balance the
// static queue's grid-stride assignment.
#include <algorithm>
#include <cstring>

#include "common.h"
#include "ptx.cuh"
#include "shift.cuh"

namespace ts {
namespace {

constexpr int kRowsMaxThreads = 1024;
constexpr int64_t kRowsMaxTiles = 0x7fffffffLL;  // grid x limit
constexpr uint64_t kRowsDefaultTimeoutNs = 1000ull * 1000 * 1000;
constexpr uint64_t kRowsDrainNs = 200ull * 1000 * 1000;
constexpr int64_t kRowsMaxPackChunk = int64_t(1) << 30;  // a packed tile's vector counts stay in int32

// dst[i] = src[i] for b <= i < e when src and dst differ in their offset
// modulo 16 bytes by DELTA (once dst is aligned), by every thread of the CTA:
// each aligned 16-byte vector k of the row's dst is joined from the aligned
// source vectors k and k + 1.  A source vector may lie outside the row but
// never outside src[0, n); the elements not covered by such vectors (at most
// 15 at the head, a few at the tail) are copied one by one.
template <int DELTA>
__device__ __forceinline__ void copy_row_shift(const int16_t *__restrict__ src, int16_t *__restrict__ dst, int64_t n,
                                               int64_t b, int64_t e) {
    const int64_t tid = threadIdx.x, T = blockDim.x;
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst + b), sa = reinterpret_cast<uintptr_t>(src + b);
    int64_t hd = static_cast<int64_t>(((16 - da % 16) % 16) / 2);
    if (hd > e - b) hd = e - b;
    const uintptr_t d0 = da + 2 * hd, sb = sa + 2 * hd - DELTA;
    const uintptr_t s_lo = reinterpret_cast<uintptr_t>(src), s_hi = s_lo + 2 * static_cast<uintptr_t>(n);
    const int64_t k0 = sb >= s_lo ? 0 : 1;
    int64_t k1 = static_cast<int64_t>((s_hi - sb) / 16) - 1;
    const int64_t kd = static_cast<int64_t>((da + 2 * static_cast<uintptr_t>(e - b) - d0) / 16);
    if (kd < k1) k1 = kd;
    if (hd == e - b || k1 - k0 < 1) {  // no whole vector: element by element
        for (int64_t i = b + tid; i < e; i += T) dst[i] = src[i];
        return;
    }
    const int4 *sv = reinterpret_cast<const int4 *>(sb);
    int4 *dv = reinterpret_cast<int4 *>(d0);
    for (int64_t k = k0 + tid; k < k1; k += T) __stcs(dv + k, join16<DELTA>(__ldcs(sv + k), __ldcs(sv + k + 1)));
    for (int64_t i = b + tid; i < b + hd + 8 * k0; i += T) dst[i] = src[i];
    for (int64_t i = b + hd + 8 * k1 + tid; i < e; i += T) dst[i] = src[i];
}

// Division by the chunk size, a launch constant, with a multiply-high (the
// round-up method of Granlund and Montgomery, "Division by invariant integers
// using multiplication", for 64-bit dividends): a 64-bit divide takes about a
// hundred instructions, and the planning kernels need up to two per row.
struct ChunkDiv {
    uint64_t m;  // floor(2^(64 + L) / d) - 2^64 + 1
    int32_t L;   // ceil(log2 d)
    int32_t one; // d == 1
};

ChunkDiv chunk_div(int64_t d) {
    ChunkDiv c{0, 0, d <= 1 ? 1 : 0};
    if (d > 1) {
        c.L = 64 - __builtin_clzll(static_cast<unsigned long long>(d - 1));
        const unsigned __int128 q = (static_cast<unsigned __int128>(1) << (64 + c.L)) / static_cast<uint64_t>(d);
        c.m = static_cast<uint64_t>(q - (static_cast<unsigned __int128>(1) << 64) + 1);
    }
    return c;
}

// floor(n / d) for n >= 0
__device__ __forceinline__ int64_t div_chunk(int64_t n, const ChunkDiv &c) {
    if (c.one) return n;
    const uint64_t u = static_cast<uint64_t>(n);
    const uint64_t t = __umul64hi(c.m, u);
    return static_cast<int64_t>((t + ((u - t) >> 1)) >> (c.L - 1));
}

struct RowsParams {
    const int16_t *src;
    int16_t *dst;
    int64_t n;
    const int64_t *offsets;      // rows + 1 entries
    int64_t rows;                // upper bound on the row count
    const int64_t *rows_device;  // the row count read on the device, or nullptr
    const uint8_t *skip;         // per-row skip mask, or nullptr
    int64_t tiles;               // work tiles (>= rows)
    int32_t sched;
    int32_t pad0;
    int64_t chunk;               // elements per piece, or 0: one tile per row
    int64_t *base;               // chunked: rows + 1 entries, first tile of each row (base[rows] = pieces);
                                 // packed: virtual start of each row (base[rows] = elements in all)
    int32_t *map;                // chunked: tiles entries, the row of each tile (packed: of its first element)
    int64_t *block_sums;         // chunked: per planning CTA, the total of its rows
    int32_t pack;                // packed mode (with chunk > 0)
    int32_t pad1;
    ChunkDiv cdiv;               // division by chunk
    uint64_t timeout_ns;
    uint64_t drain_ns;
    unsigned long long *status;
    long long *trace;  // 2 per tile: visits, block that ran it
};

struct alignas(32) RowVec32 {
    uint32_t w[8];
};

__device__ __forceinline__ void row_ld32(const RowVec32 *p, RowVec32 &v) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                   "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

__device__ __forceinline__ void row_st32(RowVec32 *p, const RowVec32 &v) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}

// dst[i] = src[i] for b <= i < e, by every thread of the CTA.  VEC is the
// vector size in bytes (32 or 16; src and dst share their offset modulo VEC),
// or 2 for element-wise copies.
template <int VEC>
__device__ __forceinline__ void copy_row(const int16_t *__restrict__ src, int16_t *__restrict__ dst, int64_t b,
                                         int64_t e) {
    const int64_t tid = threadIdx.x, T = blockDim.x;
    if constexpr (VEC == 2) {
        for (int64_t i = b + tid; i < e; i += T) dst[i] = src[i];
    } else {
        constexpr int64_t EPV = VEC / 2;  // elements per vector
        const uintptr_t a = reinterpret_cast<uintptr_t>(src + b);
        int64_t head = static_cast<int64_t>(((VEC - a % VEC) % VEC) / 2);
        if (head > e - b) head = e - b;
        const int64_t v0 = b + head;
        const int64_t nv = (e - v0) / EPV;
        const int64_t t0 = v0 + nv * EPV;
        if (tid < head) dst[b + tid] = src[b + tid];
        if (tid < e - t0) dst[t0 + tid] = src[t0 + tid];
        int64_t i = tid;
        if constexpr (VEC == 32) {
            const RowVec32 *s = reinterpret_cast<const RowVec32 *>(src + v0);
            RowVec32 *d = reinterpret_cast<RowVec32 *>(dst + v0);
            for (; i + T < nv; i += 2 * T) {
                RowVec32 x, y;
                row_ld32(s + i, x);
                row_ld32(s + i + T, y);
                row_st32(d + i, x);
                row_st32(d + i + T, y);
            }
            for (; i < nv; i += T) {
                RowVec32 x;
                row_ld32(s + i, x);
                row_st32(d + i, x);
            }
        } else {
            const int4 *s = reinterpret_cast<const int4 *>(src + v0);
            int4 *d = reinterpret_cast<int4 *>(dst + v0);
            for (; i + T < nv; i += 2 * T) {
                const int4 x = __ldcs(s + i), y = __ldcs(s + i + T);
                __stcs(d + i, x);
                __stcs(d + i + T, y);
            }
            for (; i < nv; i += T) __stcs(d + i, __ldcs(s + i));
        }
    }
}

__device__ __forceinline__ void rows_report(const RowsParams &p, unsigned long long code, unsigned long long info) {
    if (atomicCAS(&p.status[0], 0ull, code) == 0ull) atomicExch(&p.status[1], info);
    atomicAdd(&p.status[2], 1ull);
}


// Row copy by vector class: VEC 32, 16 (src and dst share their offset modulo
// VEC bytes) or 2 (element-wise), or -DELTA (they differ modulo 16 bytes by
// DELTA: vectors joined from two source vectors).
template <int VEC>
__device__ __forceinline__ void row_copy(const RowsParams &p, int64_t b, int64_t e) {
    if constexpr (VEC < 0)
        copy_row_shift<-VEC>(p.src, p.dst, p.n, b, e);
    else
        copy_row<VEC>(p.src, p.dst, b, e);
}

// Bounded phase wait on a CTA-local mbarrier.
__device__ __noinline__ bool rows_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t k = 1;; ++k) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((k & 15u) == 0 && globaltimer() - t0 > limit_ns) return false;
    }
}

constexpr int kPlanThreads = 1024;  // one row per thread: a planning CTA covers 1024 rows

// The row count: `rows`, or the device-side count clamped to [0, rows].
__device__ __forceinline__ int64_t row_count(const RowsParams &p) {
    if (!p.rows_device) return p.rows;
    const int64_t r = *p.rows_device;
    return r < 0 ? 0 : (r < p.rows ? r : p.rows);
}

// Chunked: the pieces of row r; packed: its elements.  Rows past the count,
// skipped rows and rows with bad bounds get none (bad bounds are reported
// when `report`).
__device__ __forceinline__ int64_t plan_count(const RowsParams &p, int64_t rows, int64_t r, bool report) {
    if (r >= rows || (p.skip && p.skip[r])) return 0;
    const int64_t b = p.offsets[r], e = p.offsets[r + 1];
    if (b >= 0 && b <= e && e <= p.n) return p.pack ? e - b : div_chunk(e - b + p.chunk - 1, p.cdiv);
    if (report) rows_report(p, 2ull, static_cast<unsigned long long>(r));
    return 0;
}

// Block-wide inclusive scan of one value per thread (kPlanThreads threads).
__device__ __forceinline__ int64_t plan_scan(int64_t x, int64_t *warp_sum) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_sum[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    if (wid > 0) x += warp_sum[wid - 1];
    __syncthreads();  // warp_sum is free again
    return x;
}

// Chunked and packed modes plan with two kernels over CTAs of 1024 rows, each
// launched as a programmatic dependent of the kernel before it in the stream
// (it may be scheduled during that kernel's tail and waits for its results
// before reading memory).  First: the piece (or element) total of each CTA's
// rows.
__global__ void __launch_bounds__(kPlanThreads) rows_plan_sums_kernel(const __grid_constant__ RowsParams p) {
    __shared__ int64_t warp_sum[32];
    grid_dep_wait();  // the offsets, count and mask may come from the previous kernel
    grid_dep_launch();
    const int64_t rows = row_count(p);
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kPlanThreads + threadIdx.x;
    const int64_t total = plan_scan(plan_count(p, rows, r, false), warp_sum);
    if (threadIdx.x == kPlanThreads - 1) p.block_sums[blockIdx.x] = total;
}

// Second: each row's first tile (chunked) or virtual start (packed) in base,
// base[rows] = the pieces (elements) in all, and the tile -> row map.  A row
// with bad bounds or marked in skip_rows gets nothing (bad bounds are
// reported); tiles past the launch's are not mapped, and reported.
__global__ void __launch_bounds__(kPlanThreads) rows_plan_write_kernel(const __grid_constant__ RowsParams p) {
    __shared__ int64_t warp_sum[32];
    __shared__ int64_t start_s;
    grid_dep_wait();
    grid_dep_launch();
    const int64_t rows = row_count(p);
    // this CTA's start: the totals of the CTAs before it
    int64_t part = 0;
    for (int64_t g = threadIdx.x; g < blockIdx.x; g += kPlanThreads) part += p.block_sums[g];
    part = plan_scan(part, warp_sum);
    if (threadIdx.x == kPlanThreads - 1) start_s = part;
    __syncthreads();
    const int64_t start = start_s;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kPlanThreads + threadIdx.x;
    const int64_t cnt = plan_count(p, rows, r, true);
    const int64_t incl = plan_scan(cnt, warp_sum);
    const int64_t first = start + incl - cnt;
    if (r < rows) {
        p.base[r] = first;
        // chunked: the row's pieces are tiles first .. first + cnt - 1; packed:
        // the tiles whose first element lies in the row's virtual range
        const int64_t t0 = p.pack ? div_chunk(first + p.chunk - 1, p.cdiv) : first;
        const int64_t t1 = p.pack ? div_chunk(first + cnt + p.chunk - 1, p.cdiv) : first + cnt;
        for (int64_t t = t0; t < t1; ++t) {
            if (t >= p.tiles) {
                rows_report(p, 3ull, static_cast<unsigned long long>(r));
                break;
            }
            p.map[t] = static_cast<int32_t>(r);
        }
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == kPlanThreads - 1) p.base[rows] = start + incl;
}

// Shared tables of one batch of a packed tile's segments (one per thread).
struct PackTables {
    int64_t first[kRowsMaxThreads];      // element index of the segment's first vector
    int32_t vbase[kRowsMaxThreads + 1];  // exclusive running sum of the segments' vector counts
    int32_t warp_sum[kRowsMaxThreads / 32];
};

// Packed mode: copy the elements [v0, v1) of the virtual row space, starting
// at row r (which holds v0).  Called by every thread of the CTA.
template <int VEC>
__device__ void copy_packed(const RowsParams &p, int64_t v0, int64_t v1, int64_t r, int64_t r_end, PackTables &tb) {
    constexpr int64_t EPV = VEC / 2;  // elements per vector (1: element-wise)
    const int tid = threadIdx.x, T = blockDim.x, lane = tid & 31, wid = tid >> 5;
    for (;;) {
        // this thread's segment: the part of row r + tid inside [v0, v1)
        const int64_t rr = r + tid;
        int64_t b = 0, e = 0;
        if (rr < r_end) {
            const int64_t P0 = p.base[rr], P1 = p.base[rr + 1];
            const int64_t lo = v0 > P0 ? v0 : P0, hi = v1 < P1 ? v1 : P1;
            if (lo < hi) {
                const int64_t o = p.offsets[rr];
                b = o + (lo - P0);
                e = o + (hi - P0);
                if (!(b >= 0 && e <= p.n)) b = e = 0;  // the plan gave rows with bad bounds no elements
            }
        }
        int64_t vb = b, nv = e - b;
        if constexpr (VEC > 2) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(p.src + b);
            int64_t head = static_cast<int64_t>(((VEC - a % VEC) % VEC) / 2);
            if (head > e - b) head = e - b;
            vb = b + head;
            nv = (e - vb) / EPV;
            for (int64_t i = b; i < vb; ++i) p.dst[i] = p.src[i];                   // head
            for (int64_t i = vb + nv * EPV; i < e; ++i) p.dst[i] = p.src[i];        // tail
        }
        // block-wide exclusive scan of the vector counts
        int32_t x = static_cast<int32_t>(nv);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) tb.warp_sum[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t w = lane < T / 32 ? tb.warp_sum[lane] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += y;
            }
            if (lane < T / 32) tb.warp_sum[lane] = w;
        }
        __syncthreads();
        const int32_t excl = (wid > 0 ? tb.warp_sum[wid - 1] : 0) + x - static_cast<int32_t>(nv);
        tb.first[tid] = vb;
        tb.vbase[tid] = excl;
        if (tid == T - 1) tb.vbase[T] = excl + static_cast<int32_t>(nv);
        __syncthreads();
        // the batch's vectors as one flat range; vector j lies in segment i with
        // vbase[i] <= j < vbase[i + 1], found by bisection, then by walking on
        const int32_t NV = tb.vbase[T];
        if (tid < NV) {
            int lo = 0, hi = T;  // vbase[lo] <= j < vbase[hi]
            const int32_t j0 = tid;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (tb.vbase[mid] <= j0) lo = mid; else hi = mid;
            }
            int i = lo;
            for (int32_t j = j0; j < NV; j += T) {
                while (tb.vbase[i + 1] <= j) ++i;
                const int64_t at = tb.first[i] + static_cast<int64_t>(j - tb.vbase[i]) * EPV;
                if constexpr (VEC == 32) {
                    RowVec32 v;
                    row_ld32(reinterpret_cast<const RowVec32 *>(p.src + at), v);
                    row_st32(reinterpret_cast<RowVec32 *>(p.dst + at), v);
                } else if constexpr (VEC == 16) {
                    __stcs(reinterpret_cast<int4 *>(p.dst + at), __ldcs(reinterpret_cast<const int4 *>(p.src + at)));
                } else {
                    p.dst[at] = p.src[at];
                }
            }
        }
        // more rows in the tile past this batch?
        const int64_t next = r + T;
        if (next >= r_end || p.base[next] >= v1) break;
        r = next;
        __syncthreads();  // every thread is done with the tables
    }
}

// PACK: the packed mode's kernel (its own instantiation, so the other modes
// keep their 32 registers per thread and four 512-thread CTAs per SM).
template <int VEC, bool PACK>
__global__ void __launch_bounds__(kRowsMaxThreads, 2) rows_copy_kernel(const __grid_constant__ RowsParams p) {
    __shared__ __align__(16) uint8_t resp[16];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int64_t next_tile;
    const uint32_t resp_a = smem_u32(resp), bar_a = smem_u32(&bar);
    const bool clc = p.sched == SCHED_CLC;
    if (clc && threadIdx.x == 0) {
        mbar_init(bar_a, 1);
        fence_mbar_init();
    }
    // Launched as a programmatic dependent of the kernel before it (the plan, or
    // whatever wrote the offsets): nothing global is read before that kernel's
    // writes are visible.
    grid_dep_wait();
    grid_dep_launch();
    // The row count is read once and holds for the whole launch; tiles past it
    // are the oversubscribed part of the queue and are skipped.
    const int64_t rows = row_count(p);
    // chunked: the planning kernels' piece count (packed: their element total and
    // the tiles that covers), clamped to the tiles it could map
    int64_t pieces = 0, total = 0;
    if (p.chunk > 0) {
        total = p.base[rows];
        pieces = p.pack ? div_chunk(total + p.chunk - 1, p.cdiv) : total;
        if (pieces > p.tiles) pieces = p.tiles;
    }
    extern __shared__ __align__(16) uint8_t dyn_smem[];  // packed mode: PackTables
    __syncthreads();

    int64_t tile = blockIdx.x;
    uint32_t phase = 0;
    while (tile >= 0 && tile < p.tiles) {
        if (clc && threadIdx.x == 0) {
            fence_proxy_async_smem();  // our generic reads of the slot come before the next async write
            mbar_arrive_expect_tx(bar_a, 16);
            clc_try_cancel(resp_a, bar_a);
        }
        // skippable region: the row copy only; the queue bookkeeping below runs for every tile
        if constexpr (PACK) {
            if (tile < pieces) {
                // rows r .. r_end - 1 can hold the tile's elements: r_end is one past
                // the row of the next tile's first element
                const int64_t r = p.map[tile];
                const int64_t r_end = tile + 1 < pieces ? p.map[tile + 1] + 1 : rows;
                const int64_t v0 = tile * p.chunk, v1 = v0 + p.chunk < total ? v0 + p.chunk : total;
                // (packed tiles take element-wise copies when src and dst differ modulo 16)
                copy_packed<(VEC < 0 ? 2 : VEC)>(p, v0, v1, r, r_end, *reinterpret_cast<PackTables *>(dyn_smem));
            }
        } else if (p.chunk > 0) {
            if (tile < pieces) {
                const int64_t r = p.map[tile];
                const int64_t b0 = p.offsets[r], e0 = p.offsets[r + 1];
                const int64_t b = b0 + (tile - p.base[r]) * p.chunk;
                const int64_t e = b + p.chunk < e0 ? b + p.chunk : e0;
                if (b >= 0 && b <= e && e <= p.n) row_copy<VEC>(p, b, e);  // checked by the plan too
            }
        } else if (tile < rows && !(p.skip && p.skip[tile])) {
            const int64_t b = p.offsets[tile], e = p.offsets[tile + 1];
            if (b >= 0 && b <= e && e <= p.n)
                row_copy<VEC>(p, b, e);
            else if (threadIdx.x == 0)
                rows_report(p, 2ull, static_cast<unsigned long long>(tile));
        }
        if (p.trace && threadIdx.x == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&p.trace[2 * tile]), 1ull);
            p.trace[2 * tile + 1] = blockIdx.x;
        }
        if (p.sched == SCHED_NONPERSISTENT) break;  // one tile per CTA, no queue
        if (!clc) {
            tile += gridDim.x;
            continue;
        }
        if (threadIdx.x == 0) {
            int64_t nt = -1;
            if (rows_wait(bar_a, phase, p.timeout_ns)) {
                uint32_t x = 0;
                if (clc_query(resp_a, x)) nt = x;
                fence_proxy_async_smem();
            } else {
                rows_report(p, 1ull, (static_cast<unsigned long long>(WAIT_ROWS_CLC) << 32) | blockIdx.x);
                // the request may still be in flight: let its response land before the CTA exits
                rows_wait(bar_a, phase, p.drain_ns);
            }
            next_tile = nt;
        }
        phase ^= 1u;
        __syncthreads();
        tile = next_tile;
        __syncthreads();  // every thread has read next_tile before thread 0 writes it again
    }
}

struct RowsPlan {
    int vec;
    int threads;
    int64_t tiles, grid, resident;
    // chunked mode: workspace = base[rows + 1], map[tiles], block_sums[plan_ctas], each 256-byte aligned
    int64_t chunk, base_bytes, map_bytes, plan_ctas, workspace_bytes;
    int32_t pack;
    int32_t smem;  // dynamic shared memory per CTA (packed mode's tables)
};

ts_status plan_rows(const int16_t *src, const int16_t *dst, int64_t n, const int64_t *offsets, int64_t rows,
                    int32_t sched, const ts_rows_opts *o, RowsPlan *pl) {
    ts_rows_opts z;
    std::memset(&z, 0, sizeof z);
    if (!o) o = &z;
    if (n < 0 || rows < 0) return fail(TS_ERR_INVALID_ARG, "negative size (n=%lld rows=%lld)",
                                       static_cast<long long>(n), static_cast<long long>(rows));
    if (sched != TS_SCHED_STATIC && sched != TS_SCHED_CLC && sched != TS_SCHED_NONPERSISTENT)
        return fail(TS_ERR_INVALID_ARG, "sched %d", sched);
    if (o->tiles < 0 || o->max_workers < 0 || o->timeout_s < 0 || o->chunk < 0 || o->workspace_bytes < 0)
        return fail(TS_ERR_INVALID_ARG, "negative option");
    if (o->pack != 0 && o->pack != 1) return fail(TS_ERR_INVALID_ARG, "pack = %d (0 or 1)", o->pack);
    if (o->pack && (o->chunk <= 0 || o->chunk > kRowsMaxPackChunk))
        return fail(TS_ERR_INVALID_ARG, "pack needs a chunk in [1, 2^30] (chunk = %lld)",
                    static_cast<long long>(o->chunk));
    // chunked: enough tiles for the pieces of rows that do not overlap; packed:
    // for their elements laid end to end
    const int64_t min_tiles = o->chunk > 0 ? (o->pack ? 0 : rows) + (n + o->chunk - 1) / o->chunk : rows;
    pl->tiles = o->tiles ? o->tiles : min_tiles;
    if (pl->tiles < min_tiles)
        return fail(TS_ERR_INVALID_ARG, "tiles = %lld is below %lld (%s)", static_cast<long long>(pl->tiles),
                    static_cast<long long>(min_tiles),
                    o->chunk > 0 ? (o->pack ? "ceil(n / chunk)" : "rows + ceil(n / chunk)") : "rows");
    if (pl->tiles > kRowsMaxTiles) return fail(TS_ERR_UNSUPPORTED, "more than 2^31 - 1 work tiles");
    pl->chunk = o->chunk;
    pl->pack = o->pack;
    pl->smem = 0;
    pl->base_bytes = 0;
    pl->workspace_bytes = 0;
    if (o->chunk > 0) {
        pl->base_bytes = ((rows + 1) * 8 + 255) / 256 * 256;
        pl->map_bytes = (pl->tiles * 4 + 255) / 256 * 256;
        pl->plan_ctas = rows > 0 ? (rows + kPlanThreads - 1) / kPlanThreads : 1;
        pl->workspace_bytes = pl->base_bytes + pl->map_bytes + pl->plan_ctas * 8;
    }
    if (rows > 0 && !offsets) return fail(TS_ERR_INVALID_ARG, "offsets is NULL");
    if (n > 0 && (!src || !dst)) return fail(TS_ERR_INVALID_ARG, "src or dst is NULL");
    const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
    if (s % 2 || d % 2) return fail(TS_ERR_INVALID_ARG, "src and dst must be 2-byte aligned");
    const uintptr_t bytes = static_cast<uintptr_t>(n) * 2;
    if (s != d && s < d + bytes && d < s + bytes) return fail(TS_ERR_INVALID_ARG, "src and dst overlap");
    pl->threads = o->threads ? o->threads : 512;
    if (pl->threads != 128 && pl->threads != 256 && pl->threads != 512 && pl->threads != 1024)
        return fail(TS_ERR_INVALID_ARG, "threads = %d (128, 256, 512 or 1024)", pl->threads);
    // 32- or 16-byte vectors, or -DELTA: vectors joined across a DELTA-byte shift (src and dst differ modulo 16)
    pl->vec = (s % 32) == (d % 32) ? 32 : (s % 16) == (d % 16) ? 16 : -static_cast<int>((s - d) & 15u);
    pl->grid = 0;
    pl->resident = 0;
    if (pl->tiles == 0) return TS_OK;  // an empty queue: nothing to launch
    const int sms = device_sms(current_device());
    if (sms <= 0) return fail(TS_ERR_CUDA, "cannot query the SM count");
    int per_sm = 0;
    pl->smem = pl->pack ? static_cast<int32_t>(sizeof(PackTables)) : 0;
    cudaError_t e = pl->pack ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rows_copy_kernel<32, true>,
                                                                             pl->threads, pl->smem)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rows_copy_kernel<32, false>,
                                                                             pl->threads, 0);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (per_sm <= 0) return fail(TS_ERR_UNSUPPORTED, "row copy kernel cannot be resident");
    pl->resident = static_cast<int64_t>(per_sm) * sms;
    if (sched != TS_SCHED_STATIC) {  // CLC and non-persistent: one CTA per tile
        pl->grid = pl->tiles;
    } else {
        int64_t w = pl->resident;
        if (o->max_workers > 0) w = std::min<int64_t>(w, o->max_workers);
        pl->grid = std::min<int64_t>(pl->tiles, w);
    }
    return TS_OK;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// during the previous kernel's tail; it waits (griddepcontrol) before reading.
template <class K>
cudaError_t launch_dependent(K kernel, int64_t grid, int threads, int smem, cudaStream_t st, const RowsParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int VEC>
cudaError_t launch_rows(const RowsParams &p, int64_t grid, int threads, int smem, cudaStream_t st) {
    if (p.pack) return launch_dependent(rows_copy_kernel<VEC, true>, grid, threads, smem, st, p);
    return launch_dependent(rows_copy_kernel<VEC, false>, grid, threads, 0, st, p);
}

}  // namespace
}  // namespace ts

extern "C" {

ts_status ts_copy_i16_rows(const int16_t *src, int16_t *dst, int64_t n, const int64_t *offsets, int64_t rows,
                           int32_t sched, const ts_rows_opts *opts, void *stream) {
    using namespace ts;
    RowsPlan pl;
    ts_status s = plan_rows(src, dst, n, offsets, rows, sched, opts, &pl);
    if (s != TS_OK) return s;
    if (pl.grid == 0) return TS_OK;
    unsigned long long *status = device_status_word(&s);
    if (!status) return s;
    RowsParams p;
    std::memset(&p, 0, sizeof p);
    p.src = src;
    p.dst = dst;
    p.n = n;
    p.offsets = offsets;
    p.rows = rows;
    p.rows_device = opts ? opts->rows_device : nullptr;
    p.skip = opts ? opts->skip_rows : nullptr;
    p.tiles = pl.tiles;
    p.sched = sched;
    p.chunk = pl.chunk;
    p.pack = pl.pack;
    p.cdiv = chunk_div(pl.chunk);
    if (pl.chunk > 0) {
        if (!opts->workspace || opts->workspace_bytes < pl.workspace_bytes ||
            reinterpret_cast<uintptr_t>(opts->workspace) % 256 != 0)
            return fail(TS_ERR_INVALID_ARG, "chunked copy needs a 256-byte aligned workspace of %lld bytes",
                        static_cast<long long>(pl.workspace_bytes));
        p.base = static_cast<int64_t *>(opts->workspace);
        p.map = reinterpret_cast<int32_t *>(static_cast<char *>(opts->workspace) + pl.base_bytes);
        p.block_sums =
            reinterpret_cast<int64_t *>(static_cast<char *>(opts->workspace) + pl.base_bytes + pl.map_bytes);
    }
    p.timeout_ns = (opts && opts->timeout_s > 0) ? static_cast<uint64_t>(opts->timeout_s * 1e9) : kRowsDefaultTimeoutNs;
    if (p.timeout_ns == 0) p.timeout_ns = 1;
    p.drain_ns = kRowsDrainNs;
    p.status = status;
    p.trace = opts ? reinterpret_cast<long long *>(opts->trace) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pl.chunk > 0) {
        cudaError_t pe = launch_dependent(rows_plan_sums_kernel, pl.plan_ctas, kPlanThreads, 0, st, p);
        if (pe == cudaSuccess) pe = launch_dependent(rows_plan_write_kernel, pl.plan_ctas, kPlanThreads, 0, st, p);
        if (pe != cudaSuccess) return cuda_fail(pe, "row copy planning launch");
    }
    cudaError_t e = cudaSuccess;
    switch (pl.vec) {
        case 32: e = launch_rows<32>(p, pl.grid, pl.threads, pl.smem, st); break;
        case 16: e = launch_rows<16>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -2: e = launch_rows<-2>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -4: e = launch_rows<-4>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -6: e = launch_rows<-6>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -8: e = launch_rows<-8>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -10: e = launch_rows<-10>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -12: e = launch_rows<-12>(p, pl.grid, pl.threads, pl.smem, st); break;
        case -14: e = launch_rows<-14>(p, pl.grid, pl.threads, pl.smem, st); break;
        default: e = launch_rows<2>(p, pl.grid, pl.threads, pl.smem, st);
    }
    return e == cudaSuccess ? TS_OK : cuda_fail(e, "row copy launch");
}

ts_status ts_copy_rows_launch_info(int64_t n, int64_t rows, int32_t sched, const ts_rows_opts *opts,
                                   ts_launch_info *info) {
    using namespace ts;
    if (!info) return fail(TS_ERR_INVALID_ARG, "info is NULL");
    RowsPlan pl;
    // placeholder aligned, disjoint addresses: the plan only needs their alignment
    const int16_t *a = reinterpret_cast<const int16_t *>(uintptr_t(1) << 40);
    int16_t *b = reinterpret_cast<int16_t *>((uintptr_t(1) << 40) + (uintptr_t(1) << 39));
    static const int64_t dummy_offsets[1] = {0};
    ts_status s = plan_rows(a, b, std::min<int64_t>(n, int64_t(1) << 37), dummy_offsets, rows, sched, opts, &pl);
    if (s != TS_OK) return s;
    std::memset(info, 0, sizeof *info);
    info->cluster = 1;
    info->num_tiles = pl.tiles;
    info->num_units = pl.tiles;
    info->grid_ctas = pl.grid;
    info->workers = pl.grid;
    info->resident = static_cast<int32_t>(pl.resident);
    info->workspace_bytes = pl.workspace_bytes;
    return TS_OK;
}

}  // extern "C"
