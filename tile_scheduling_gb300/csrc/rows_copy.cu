// Jagged int16 copy driven by a work queue.
//
// The two copy examples of CUTLASS TS "Schedules": Dynamic Domain (work tile t
// copies a row whose length comes from an offsets array, offsets[t + 1] -
// offsets[t]) and Skippable Tiles (the oversubscribed copy queue: a per-tile
// predicate decides whether the row copy runs, while every tile still takes
// part in the queue's wait / advance / release).  The work-tile loop runs on
// either scheduler of "Cluster Launch Control": a static grid-stride
// persistent loop (tile = blockIdx.x + i * gridDim.x), or one CTA per tile
// whose running CTAs cancel pending ones.  The CLC request for the next tile
// is issued before the current row is copied, so its latency hides under the
// copy (the overlap loop of that page).
//
// A row is copied by the whole CTA: a ragged head until src + begin reaches
// the vector alignment, 32-byte (or 16-byte) vectors with two in flight per
// thread, and a ragged tail.  Row bounds are read on the device and checked
// against [0, n] before any access; a row that fails the check is reported in
// the status word and not copied.
//
// Chunked mode (not on the pages): rows are cut into pieces of at most `chunk`
// elements and every piece is a work tile, so that a long row is not left to
// one CTA at the end of the queue.  A planning kernel (one CTA) scans the
// piece counts and writes, per row, its first tile (base) and, per tile, its
// row (map); the copy kernel then finds tile t's piece with two loads.  The
// launch's tile count is an upper bound on the pieces (rows + ceil(n / chunk)
// for rows that do not overlap); tiles past the last piece are skipped like
// the oversubscribed tiles above.
#include <algorithm>
#include <cstring>

#include "common.h"
#include "ptx.cuh"

namespace ts {
namespace {

constexpr int kRowsMaxThreads = 1024;
constexpr int64_t kRowsMaxTiles = 0x7fffffffLL;  // grid x limit
constexpr uint64_t kRowsDefaultTimeoutNs = 1000ull * 1000 * 1000;
constexpr uint64_t kRowsDrainNs = 200ull * 1000 * 1000;

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
    int64_t *base;               // chunked: rows + 1 entries, first tile of each row (base[rows] = pieces)
    int32_t *map;                // chunked: tiles entries, the row of each tile
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

// Bounded phase wait on a CTA-local mbarrier.
__device__ __noinline__ bool rows_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t k = 1;; ++k) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((k & 15u) == 0 && globaltimer() - t0 > limit_ns) return false;
    }
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanRows = 8;  // consecutive rows per planning thread: 8192 rows per pass

// Chunked mode, first kernel: piece counts of the rows, their running sum
// (base) and the tile -> row map.  One CTA walks the rows 8192 at a time: each
// thread takes 8 consecutive rows (all their offsets loaded at once), and a
// block-wide exclusive scan of the threads' piece totals places them.  A row
// with bad bounds or marked in skip_rows gets no pieces (bad bounds are
// reported, as in the per-row mode).  Pieces that would not fit in the
// launch's tiles are not mapped, and reported.
__global__ void __launch_bounds__(kPlanThreads) rows_plan_kernel(const __grid_constant__ RowsParams p) {
    __shared__ int64_t warp_sum[kPlanThreads / 32];
    __shared__ int64_t carry_s;
    int64_t rows = p.rows;
    if (p.rows_device) {
        const int64_t r = *p.rows_device;
        rows = r < 0 ? 0 : (r < p.rows ? r : p.rows);
    }
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int64_t r0 = 0; r0 < rows; r0 += kPlanThreads * kPlanRows) {
        const int64_t rt = r0 + static_cast<int64_t>(tid) * kPlanRows;  // this thread's first row
        int64_t off[kPlanRows + 1];
#pragma unroll
        for (int j = 0; j <= kPlanRows; ++j) off[j] = rt + j <= rows ? p.offsets[rt + j] : 0;
        int64_t cnt[kPlanRows];
        int64_t total = 0;
#pragma unroll
        for (int j = 0; j < kPlanRows; ++j) {
            const int64_t r = rt + j;
            cnt[j] = 0;
            if (r < rows && !(p.skip && p.skip[r])) {
                const int64_t b = off[j], e = off[j + 1];
                if (b >= 0 && b <= e && e <= p.n)
                    cnt[j] = (e - b + p.chunk - 1) / p.chunk;
                else
                    rows_report(p, 2ull, static_cast<unsigned long long>(r));
            }
            total += cnt[j];
        }
        // block-wide inclusive scan of the thread totals
        int64_t x = total;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) warp_sum[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int64_t w = lane < kPlanThreads / 32 ? warp_sum[lane] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += y;
            }
            if (lane < kPlanThreads / 32) warp_sum[lane] = w;  // inclusive warp totals
        }
        __syncthreads();
        const int64_t carry = carry_s;
        int64_t first = carry + (wid > 0 ? warp_sum[wid - 1] : 0) + x - total;
#pragma unroll
        for (int j = 0; j < kPlanRows; ++j) {
            const int64_t r = rt + j;
            if (r >= rows) break;
            p.base[r] = first;
            for (int64_t k = 0; k < cnt[j]; ++k) {
                const int64_t t = first + k;
                if (t >= p.tiles) {
                    rows_report(p, 3ull, static_cast<unsigned long long>(r));
                    break;
                }
                p.map[t] = static_cast<int32_t>(r);
            }
            first += cnt[j];
        }
        __syncthreads();  // every thread has read carry_s and warp_sum
        if (tid == kPlanThreads - 1) carry_s = carry + warp_sum[kPlanThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) p.base[rows] = carry_s;
}

template <int VEC>
__global__ void __launch_bounds__(kRowsMaxThreads) rows_copy_kernel(const __grid_constant__ RowsParams p) {
    __shared__ __align__(16) uint8_t resp[16];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int64_t next_tile;
    const uint32_t resp_a = smem_u32(resp), bar_a = smem_u32(&bar);
    const bool clc = p.sched == SCHED_CLC;
    if (clc && threadIdx.x == 0) {
        mbar_init(bar_a, 1);
        fence_mbar_init();
    }
    // The row count is read once and holds for the whole launch; tiles past it
    // are the oversubscribed part of the queue and are skipped.
    int64_t rows = p.rows;
    if (p.rows_device) {
        const int64_t r = *p.rows_device;
        rows = r < 0 ? 0 : (r < p.rows ? r : p.rows);
    }
    // chunked: the planning kernel's piece count, clamped to the tiles it could map
    int64_t pieces = 0;
    if (p.chunk > 0) {
        pieces = p.base[rows];
        if (pieces > p.tiles) pieces = p.tiles;
    }
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
        if (p.chunk > 0) {
            if (tile < pieces) {
                const int64_t r = p.map[tile];
                const int64_t b0 = p.offsets[r], e0 = p.offsets[r + 1];
                const int64_t b = b0 + (tile - p.base[r]) * p.chunk;
                const int64_t e = b + p.chunk < e0 ? b + p.chunk : e0;
                if (b >= 0 && b <= e && e <= p.n) copy_row<VEC>(p.src, p.dst, b, e);  // checked by the plan too
            }
        } else if (tile < rows && !(p.skip && p.skip[tile])) {
            const int64_t b = p.offsets[tile], e = p.offsets[tile + 1];
            if (b >= 0 && b <= e && e <= p.n)
                copy_row<VEC>(p.src, p.dst, b, e);
            else if (threadIdx.x == 0)
                rows_report(p, 2ull, static_cast<unsigned long long>(tile));
        }
        if (p.trace && threadIdx.x == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&p.trace[2 * tile]), 1ull);
            p.trace[2 * tile + 1] = blockIdx.x;
        }
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
    int64_t chunk, base_bytes, workspace_bytes;  // chunked mode: workspace = base[rows + 1], then map[tiles]
};

ts_status plan_rows(const int16_t *src, const int16_t *dst, int64_t n, const int64_t *offsets, int64_t rows,
                    int32_t sched, const ts_rows_opts *o, RowsPlan *pl) {
    ts_rows_opts z;
    std::memset(&z, 0, sizeof z);
    if (!o) o = &z;
    if (n < 0 || rows < 0) return fail(TS_ERR_INVALID_ARG, "negative size (n=%lld rows=%lld)",
                                       static_cast<long long>(n), static_cast<long long>(rows));
    if (sched != TS_SCHED_STATIC && sched != TS_SCHED_CLC) return fail(TS_ERR_INVALID_ARG, "sched %d", sched);
    if (o->tiles < 0 || o->max_workers < 0 || o->timeout_s < 0 || o->chunk < 0 || o->workspace_bytes < 0)
        return fail(TS_ERR_INVALID_ARG, "negative option");
    // chunked: enough tiles for the pieces of rows that do not overlap
    const int64_t min_tiles = o->chunk > 0 ? rows + (n + o->chunk - 1) / o->chunk : rows;
    pl->tiles = o->tiles ? o->tiles : min_tiles;
    if (pl->tiles < min_tiles)
        return fail(TS_ERR_INVALID_ARG, "tiles = %lld is below %lld (%s)", static_cast<long long>(pl->tiles),
                    static_cast<long long>(min_tiles), o->chunk > 0 ? "rows + ceil(n / chunk)" : "rows");
    if (pl->tiles > kRowsMaxTiles) return fail(TS_ERR_UNSUPPORTED, "more than 2^31 - 1 work tiles");
    pl->chunk = o->chunk;
    pl->base_bytes = 0;
    pl->workspace_bytes = 0;
    if (o->chunk > 0) {
        pl->base_bytes = ((rows + 1) * 8 + 255) / 256 * 256;
        pl->workspace_bytes = pl->base_bytes + pl->tiles * 4;
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
    pl->vec = (s % 32) == (d % 32) ? 32 : (s % 16) == (d % 16) ? 16 : 2;
    pl->grid = 0;
    pl->resident = 0;
    if (pl->tiles == 0) return TS_OK;  // an empty queue: nothing to launch
    const int sms = device_sms(current_device());
    if (sms <= 0) return fail(TS_ERR_CUDA, "cannot query the SM count");
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rows_copy_kernel<32>, pl->threads, 0);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (per_sm <= 0) return fail(TS_ERR_UNSUPPORTED, "row copy kernel cannot be resident");
    pl->resident = static_cast<int64_t>(per_sm) * sms;
    if (sched == TS_SCHED_CLC) {
        pl->grid = pl->tiles;
    } else {
        int64_t w = pl->resident;
        if (o->max_workers > 0) w = std::min<int64_t>(w, o->max_workers);
        pl->grid = std::min<int64_t>(pl->tiles, w);
    }
    return TS_OK;
}

template <int VEC>
cudaError_t launch_rows(const RowsParams &p, int64_t grid, int threads, cudaStream_t st) {
    rows_copy_kernel<VEC><<<static_cast<unsigned>(grid), threads, 0, st>>>(p);
    return cudaGetLastError();
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
    if (pl.chunk > 0) {
        if (!opts->workspace || opts->workspace_bytes < pl.workspace_bytes ||
            reinterpret_cast<uintptr_t>(opts->workspace) % 256 != 0)
            return fail(TS_ERR_INVALID_ARG, "chunked copy needs a 256-byte aligned workspace of %lld bytes",
                        static_cast<long long>(pl.workspace_bytes));
        p.base = static_cast<int64_t *>(opts->workspace);
        p.map = reinterpret_cast<int32_t *>(static_cast<char *>(opts->workspace) + pl.base_bytes);
    }
    p.timeout_ns = (opts && opts->timeout_s > 0) ? static_cast<uint64_t>(opts->timeout_s * 1e9) : kRowsDefaultTimeoutNs;
    if (p.timeout_ns == 0) p.timeout_ns = 1;
    p.drain_ns = kRowsDrainNs;
    p.status = status;
    p.trace = opts ? reinterpret_cast<long long *>(opts->trace) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pl.chunk > 0) {
        rows_plan_kernel<<<1, kPlanThreads, 0, st>>>(p);
        const cudaError_t pe = cudaGetLastError();
        if (pe != cudaSuccess) return cuda_fail(pe, "row copy planning launch");
    }
    cudaError_t e = pl.vec == 32   ? launch_rows<32>(p, pl.grid, pl.threads, st)
                    : pl.vec == 16 ? launch_rows<16>(p, pl.grid, pl.threads, st)
                                   : launch_rows<2>(p, pl.grid, pl.threads, st);
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
