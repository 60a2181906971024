// Kernel parameter block and device status layout shared by host and device code.
#pragma once
#include <cstdint>

namespace ts {

enum : int32_t { SCHED_STATIC = 0, SCHED_CLC = 1, SCHED_NONPERSISTENT = 2 };
enum : int32_t { OUT_BF16 = 0, OUT_F32 = 1 };

// Where a bounded wait gave up (reported in the status word).
enum : int32_t {
    WAIT_PRODUCER_EMPTY = 1,
    WAIT_MMA_FULL = 2,
    WAIT_MMA_TMEM_EMPTY = 3,
    WAIT_EPI_TMEM_FULL = 4,
    WAIT_SCHED_CLC_EMPTY = 5,
    WAIT_CLC_FULL = 6,
    WAIT_DRAIN = 7,
    WAIT_ROWS_CLC = 8,
    WAIT_SCHED_PRODUCER = 9,
};

// Device status word (library-owned, one per device):
//   [0] first error code (0 = none, 1 = wait timeout, 2 = row bounds of the
//       jagged copy outside [0, n])
//   [1] code 1: (where << 32) | blockIdx.x;  code 2: the row index
//   [2] number of errors since the last check
constexpr int kStatusWords = 4;

// Most K parts a split tail tile is cut into: the reduction loads every part
// of a 32-column chunk at once, so this bounds its registers.
constexpr int kMaxParts = 4;

// Most groups of a grouped GEMM: the group table travels in the kernel's
// parameter block.
constexpr int kMaxGroups = 256;

// Work units: when the tiles would leave the last wave of workers partly
// empty, split_tiles tiles (tiles 0 .. split_tiles - 1 of the raster) are each
// split along K into `parts` units, and those units come first: unit
// t * parts + p (t < split_tiles) covers k-blocks [p * nk / parts,
// (p + 1) * nk / parts) of tile t.  Units split_tiles * parts onwards are the
// whole tiles split_tiles, split_tiles + 1, ... (full_tiles of them).  Split
// units write fp32 partials to `workspace`; the warp that finishes a 32-row
// slab last (per-slab counter) sums the parts in order 0..parts-1 and stores
// D.  Scheduled first, a split tile's partial write and reduction run in the
// epilogue while the mainloop already computes the worker's next tile, instead
// of after the last wave.
// Division of a non-negative int32 by a divisor fixed at launch, as a
// multiply-high and shift (Granlund and Montgomery, "Division by Invariant
// Integers using Multiplication", 1994): for d >= 1, l = ceil(log2 d),
// s = 31 + l and m = ceil(2^s / d), floor(n / d) = (n * m) >> s for every
// 0 <= n < 2^31.  m < 2^32 always; the product is taken in 64 bits.
struct FastDiv {
    uint64_t m;
    int32_t s;
    int32_t pad;
};

struct GemmParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_tiles, num_k_blocks;
    int32_t num_units, full_tiles, split_tiles, parts;
    int32_t raster_group;  // >= 1
    // 1: the units of odd waves (unit / div_wave odd) load their k-blocks from the
    // last to the first.  A wave then starts on the K end of the operand panels that
    // the wave before it read last, which are still in L2; with every unit walking
    // upwards the next wave finds the start of its A panel evicted by the ~70 MB the
    // previous wave streamed.  Measured at 8192^3 on the 2-CTA tile (ncu, one
    // capture each): DRAM reads 861 -> 797 MB per launch; time per launch, paired
    // A/B over 30 rounds: 2-CTA -0.2 %, 1-CTA 128x256 -1.1 to -1.6 %, 4096^3 and
    // 8192^2 x 4096 within +-0.15 %.  Each unit's sum still runs over every k-block
    // once and the MMA issuer overwrites the accumulator on the unit's first load,
    // whichever it is.
    int32_t k_alt;
    // the raster's divisors: tiles per group of tile rows (raster_group * tiles_n),
    // raster_group, and the height of the last (possibly shorter) group
    FastDiv div_group_tiles, div_group_rows, div_last_rows;
    FastDiv div_wave;      // the workers that fit on the GPU at once (a wave of units)
    int32_t sched;         // SCHED_STATIC / SCHED_CLC / SCHED_NONPERSISTENT
    int32_t tma_store;     // 1: TMA-store epilogue, 0: st.global epilogue
    int32_t clc_depth;     // response slots in flight (1 or 2)
    int32_t clc_lazy;      // 1: the request for the unit after unit j waits until the producer began unit j
    int32_t inputs_ready;  // 1: A, B and skip were final before the previous kernel began (loads skip its barrier)
    int32_t pad2;
    void *D;               // used by the st.global epilogue
    int64_t ldd;           // elements
    uint64_t timeout_ns;   // per-wait limit
    uint64_t drain_ns;     // limit for waiting on copies still in flight at exit
    unsigned long long *status;
    long long *trace;      // 4 int64 per work unit, or nullptr
    int32_t *counters;     // split_tiles * CG * 8 slab counters (zero between launches)
    float *partials;       // split_tiles * parts * CG * 4 slabs of 32 x BN fp32
    // Grouped GEMM (groups > 0): unit u is tile u % tiles_per_group of group
    // group_order[u / tiles_per_group], whose k-blocks are [group_kb[g],
    // group_kb[g + 1]).  D of group g starts group_stride elements after D of
    // group g - 1.
    const uint8_t *skip;   // per tile, row-major by tile row and column per group: nonzero = skip, or nullptr
    float *row_sums;       // Fork consumer output [groups][M]: sum over the K range of each row of A, or nullptr
    // Protocol log (the logged instantiation only): per CTA and role, a count
    // followed by plog_cap event words (PlogOp in gemm_kernel.cuh), or nullptr.
    int32_t *plog;
    int32_t plog_cap;
    int32_t pad3;
    int32_t groups;
    int32_t tiles_per_group;
    int64_t group_stride;
    int32_t group_kb[kMaxGroups + 1];
    // The groups in the order their tiles are scheduled: longest K range first
    // (ties by group index).  Handing out the longest units first is Graham's
    // LPT rule ("Bounds on Multiprocessing Timing Anomalies", 1969): the units
    // left for the end of the launch are the short ones, so the workers finish
    // closer together, under a static round-robin deal and under CLC alike.
    uint8_t group_order[kMaxGroups];
};

#if defined(__CUDACC__)
#define TS_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define TS_HOST_DEVICE inline
#endif

TS_HOST_DEVICE int32_t fast_div(int32_t n, const FastDiv &d) {
    return static_cast<int32_t>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * d.m) >> d.s);
}

// Tile id -> (m block, n block).  Consecutive ids walk `raster_group` tile rows
// down a column band, so workers running at the same time share B tiles in L2.
// Odd groups walk the columns from the right (a serpentine), so a group starts
// on the B panels that the group before it used last.  Measured at 8192^3 on
// the 2-CTA tile (ncu): DRAM reads 880 MB per launch against 953 MB with every
// group walked from the left, in the same time.  The divisions go through
// FastDiv: the epilogue warps decode every tile on their own critical path,
// where the GPU's multi-instruction integer divide cost ~270 cycles per tile.
// The host evaluates the same function to report the mapping
// (ts_gemm_tile_coords).
TS_HOST_DEVICE void raster(int32_t tile, const GemmParams &p, int32_t &mb, int32_t &nb) {
    const int32_t G = p.raster_group;
    const int32_t g = fast_div(tile, p.div_group_tiles);
    const int32_t first_m = g * G;
    const bool last = first_m + G > p.tiles_m;  // the last group may hold fewer tile rows
    const int32_t gsize = last ? p.tiles_m - first_m : G;
    const int32_t local = tile - g * (G * p.tiles_n);
    nb = fast_div(local, last ? p.div_last_rows : p.div_group_rows);
    mb = first_m + (local - nb * gsize);
    if (g & 1) nb = p.tiles_n - 1 - nb;
}

}  // namespace ts
