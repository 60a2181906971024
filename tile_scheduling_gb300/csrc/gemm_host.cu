// Host side of ts_gemm_bf16: argument checks, tile/grid planning, TMA tensor
// maps, and the launch.  The scheduler choice only changes the grid: a static
// persistent grid of resident workers, or (Cluster Launch Control) one block or
// cluster per tile, whose coordinate i is tile i.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.h"

namespace ts {

extern const GemmVariant variant_128_1_bf16_e4, variant_128_1_f32_e4, variant_256_1_bf16_e4, variant_256_1_f32_e4,
    variant_256_2_bf16_e4, variant_256_2_f32_e4, variant_128_1_bf16_e8, variant_128_1_f32_e8, variant_256_1_bf16_e8,
    variant_256_1_f32_e8, variant_256_2_bf16_e8, variant_256_2_f32_e8, variant_128_1_bf16_e4m, variant_128_1_f32_e4m,
    variant_256_1_bf16_e4m, variant_256_1_f32_e4m, variant_256_2_bf16_e4m, variant_256_2_f32_e4m,
    variant_256_1_bf16_e16, variant_256_1_f32_e16, variant_256_2_bf16_e16, variant_256_2_f32_e16,
    variant_128_1_f32_e4_log, variant_128_1_f32_e4m_log, variant_128_1_f32_e8_log, variant_256_1_f32_e16_log,
    variant_256_2_f32_e4_log;

const GemmVariant *find_variant(int bn, int cg, int out, int epi_warps, int merge, int log) {
    static const GemmVariant *const all[] = {
        &variant_128_1_bf16_e4,     &variant_128_1_f32_e4,      &variant_256_1_bf16_e4,  &variant_256_1_f32_e4,
        &variant_256_2_bf16_e4,     &variant_256_2_f32_e4,      &variant_128_1_bf16_e8,  &variant_128_1_f32_e8,
        &variant_256_1_bf16_e8,     &variant_256_1_f32_e8,      &variant_256_2_bf16_e8,  &variant_256_2_f32_e8,
        &variant_128_1_bf16_e4m,    &variant_128_1_f32_e4m,     &variant_256_1_bf16_e4m, &variant_256_1_f32_e4m,
        &variant_256_2_bf16_e4m,    &variant_256_2_f32_e4m,     &variant_256_1_bf16_e16, &variant_256_1_f32_e16,
        &variant_256_2_bf16_e16,    &variant_256_2_f32_e16,     &variant_128_1_f32_e4_log,
        &variant_128_1_f32_e4m_log, &variant_128_1_f32_e8_log,  &variant_256_1_f32_e16_log,
        &variant_256_2_f32_e4_log};
    for (const GemmVariant *v : all)
        if (v->bn == bn && v->cg == cg && v->out == out && v->epi_warps == epi_warps && v->merge == merge &&
            v->log == log)
            return v;
    return nullptr;
}

namespace {

constexpr int64_t kMaxDim = 0x7fffffffLL;
constexpr double kDefaultTimeoutS = 2.0;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr int kDefaultRaster = 8;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(ts_status *err) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t got = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        got = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (got == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) *err = got != cudaSuccess ? cuda_fail(got, "cuTensorMapEncodeTiled lookup")
                                       : fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    return fn;
}

// 2-D row-major tensor [rows][cols] with row pitch `ld` elements, copied in
// boxes of box_rows x box_cols with the 128-byte swizzle.  Out-of-range
// elements of a load read as zero; a store is clipped to the tensor.
ts_status make_map(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int esize, int64_t rows, int64_t cols,
                   int64_t ld, int box_rows, int box_cols) {
    ts_status err = TS_OK;
    auto fn = encode_fn(&err);
    if (!fn) return err;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TS_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld tensor, pitch %lld B",
                    static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols),
                    static_cast<long long>(ld * esize));
    return TS_OK;
}

// D as a 3-D tensor [depth][rows][cols] (depth = groups, 1 for a plain GEMM)
// stored in boxes of box_rows x box_cols x 1 with the 128-byte swizzle; the
// store clips at `rows` inside each group.
ts_status make_map_d(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int esize, int64_t depth, int64_t rows,
                     int64_t cols, int64_t ld, int box_rows, int box_cols) {
    ts_status err = TS_OK;
    auto fn = encode_fn(&err);
    if (!fn) return err;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esize), static_cast<cuuint64_t>(rows * ld * esize)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TS_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d) for D of %lld x %lld x %lld, pitch %lld B",
                    static_cast<int>(r), static_cast<long long>(depth), static_cast<long long>(rows),
                    static_cast<long long>(cols), static_cast<long long>(ld * esize));
    return TS_OK;
}

// Multiplier and shift of FastDiv for divisor d (1 <= d < 2^31; an empty grid's
// divisor 0 is taken as 1, it divides nothing).
FastDiv fast_div_for(int64_t d) {
    if (d < 1) d = 1;
    int l = 0;
    while ((int64_t{1} << l) < d) ++l;
    FastDiv f;
    f.s = 31 + l;
    f.m = ((uint64_t{1} << f.s) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d);
    f.pad = 0;
    return f;
}

template <class T>
__global__ void zero_fill_kernel(T *D, int64_t M, int64_t N, int64_t ldd) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        D[r * ldd + c] = T(0);
    }
}

bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

struct Plan {
    const GemmVariant *v;
    int tile_m, tile_n, cg;
    int64_t tiles_m, tiles_n, num_tiles, workers, grid;
    int64_t lda, ldb, ldd;
    int tma_store;
    int64_t resident;                 // workers that fit at once
    int64_t split_tiles, parts;       // split tiles and their K parts (0, 1 when not split)
    int64_t num_units;
    int64_t split_ws_bytes;           // workspace the split would need (0: no split helps)
    int64_t counter_bytes;            // counter region at the start of the workspace
    bool split;                       // applied (workspace given and large enough)
};

// A split part writes and re-reads an fp32 partial of its tile, a fixed cost
// that only pays off against long parts: with 4 k-blocks per part the split
// made 8192^2 x 512 10 % slower, and it broke even around 32 (K = 2048 per part).
constexpr int64_t kMinKBlocksPerPart = 32;
// The workspace starts with a fixed counter region; partials always follow it,
// so a workspace reused across problem shapes never has partial data where a
// later shape keeps its counters (which every launch leaves at zero).
constexpr int64_t kCounterRegionBytes = 8192;
// K at or below which the automatic choice is eight epilogue warps.  Measured
// on 8192^2 x K: eight win 10-20 % at K <= 192 and up to 10 % at 256; from 384
// on four win by 1-5 % (the extra warps' shared-memory and store traffic slows
// a mainloop that already hides a four-warp epilogue).
constexpr int64_t kShortK = 256;
// K at or below which the automatic choice is sixteen (256-column tiles).
// Measured on 8192^2 x K, bf16 out, against eight: 5-9 % faster at K = 64,
// -1 to +5 % at 128, 2-15 % slower from 256 on.
constexpr int64_t kTinyK = 128;
// K loops of at least this many k-blocks take lazy CLC requests: the producer
// needs the next unit only after loading the current one (>= 32 k-blocks, some
// 8 us), far longer than a request takes.  Shorter loops keep two requests in
// flight: with one k-block per tile the producer runs several tiles ahead.
constexpr int64_t kLazyClcKBlocks = 32;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The raster's group size and division constants for a planned launch.
void set_raster(GemmParams &p, const Plan &pl, const ts_gemm_opts *o) {
    p.tiles_m = static_cast<int32_t>(pl.tiles_m);
    p.tiles_n = static_cast<int32_t>(pl.tiles_n);
    p.raster_group = o->raster_group > 0 ? o->raster_group : kDefaultRaster;
    const int64_t G = p.raster_group;
    const int64_t groups_m = cdiv(pl.tiles_m, G);
    p.div_group_tiles = fast_div_for(G * pl.tiles_n);
    p.div_group_rows = fast_div_for(G);
    p.div_last_rows = fast_div_for(pl.tiles_m - (groups_m - 1) * G);
}

// The longest K range of one group of a grouped GEMM (the K loop the epilogue hides under).
int64_t longest_group(int64_t groups, const int64_t *k_offsets) {
    int64_t m = 0;
    for (int64_t g = 0; g < groups; ++g) m = std::max(m, k_offsets[g + 1] - k_offsets[g]);
    return m;
}

// unit_k: the longest K loop of one work unit (K for a plain GEMM, the longest group's range for
// a grouped one); it picks the epilogue warps.
ts_status plan_gemm(const void *D, int64_t M, int64_t N, int64_t K, int32_t out, int32_t sched,
                    const ts_gemm_opts *o, Plan *pl, int64_t groups = 0, int64_t unit_k = -1) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return fail(TS_ERR_INVALID_ARG, "sizes must be in [0, 2^31-1] (M=%lld N=%lld K=%lld)",
                    static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
    if (out != TS_OUT_BF16 && out != TS_OUT_F32) return fail(TS_ERR_INVALID_ARG, "out_dtype %d", out);
    if (sched != TS_SCHED_STATIC && sched != TS_SCHED_CLC && sched != TS_SCHED_NONPERSISTENT)
        return fail(TS_ERR_INVALID_ARG, "sched %d", sched);
    ts_gemm_opts z;
    std::memset(&z, 0, sizeof z);
    if (!o) o = &z;
    if (o->tile < TS_TILE_AUTO || o->tile > TS_TILE_256x256_2CTA) return fail(TS_ERR_INVALID_ARG, "tile %d", o->tile);
    if (o->max_workers < 0 || o->raster_group < 0 || o->timeout_s < 0)
        return fail(TS_ERR_INVALID_ARG, "negative option");
    if (o->epi_warps != 0 && o->epi_warps != 4 && o->epi_warps != 8 && o->epi_warps != 16)
        return fail(TS_ERR_INVALID_ARG, "epi_warps = %d (0, 4, 8 or 16)", o->epi_warps);
    if (o->merge != 0 && o->merge != 1) return fail(TS_ERR_INVALID_ARG, "merge = %d (0 or 1)", o->merge);
    if (o->inputs_ready != 0 && o->inputs_ready != 1)
        return fail(TS_ERR_INVALID_ARG, "inputs_ready = %d (0 or 1)", o->inputs_ready);
    if (o->merge && o->row_sums)
        return fail(TS_ERR_UNSUPPORTED, "the Merge layout's B producer and the Fork consumer both need warp 3");
    if (o->merge && o->epi_warps > 4)
        return fail(TS_ERR_UNSUPPORTED, "the Merge layout is built with four epilogue warps");
    pl->lda = o->lda ? o->lda : K;
    pl->ldb = o->ldb ? o->ldb : K;
    pl->ldd = o->ldd ? o->ldd : N;
    if (pl->lda < K || pl->ldb < K || pl->ldd < N || pl->lda > (int64_t(1) << 38) || pl->ldb > (int64_t(1) << 38) ||
        pl->ldd > (int64_t(1) << 37))
        return fail(TS_ERR_INVALID_ARG, "leading dimensions must cover a row (lda=%lld ldb=%lld ldd=%lld)",
                    static_cast<long long>(pl->lda), static_cast<long long>(pl->ldb),
                    static_cast<long long>(pl->ldd));

    const int dev = current_device();
    const int sms = device_sms(dev);
    if (sms <= 0) return fail(TS_ERR_CUDA, "cannot query the SM count");
    int tile = o->tile;
    if (o->row_sums && tile == TS_TILE_256x256_2CTA)
        return fail(TS_ERR_UNSUPPORTED, "row sums (the Fork consumer) need a one-CTA tile");
    if (tile == TS_TILE_AUTO) {
        // Largest tile that still gives every SM work: the 2-CTA tile halves
        // each SM's share of B traffic, the 128x128 tile suits small outputs.
        // A grouped launch schedules every group's tiles, so all of them count.
        const int64_t g = groups > 0 ? groups : 1;
        const int64_t t256 = cdiv(M, 256) * cdiv(N, 256) * g;
        const int64_t t128x256 = cdiv(M, 128) * cdiv(N, 256) * g;
        if (t256 * 2 >= sms && !o->row_sums)
            tile = TS_TILE_256x256_2CTA;
        else if (t128x256 >= sms)
            tile = TS_TILE_128x256;
        else
            tile = TS_TILE_128x128;
    }
    int bn = 256, cg = 1;
    if (tile == TS_TILE_128x128) bn = 128;
    if (tile == TS_TILE_256x256_2CTA) cg = 2;
    // Epilogue warps: with a short K loop the epilogue bounds every tile and
    // more warps hide more of its latencies; with a long one the epilogue
    // hides under the mainloop and four leave the SM's issue slots to it.
    // Grouped launches take the same rule on their longest group (measured on 16 groups of
    // 2048 x 2048, 2-CTA tile, static / CLC: K = 64 per group 33.2 / 34.5 us with four warps,
    // 23.0 / 23.9 with sixteen; K = 128 34.2 / 35.2 against 26.9 / 27.7; K = 256 with eight
    // 36.3 / 36.9 against 36.7 / 38.2 with four).
    int epi_warps = o->epi_warps;
    if (epi_warps == 0) {
        epi_warps = 4;
        const int64_t kk = unit_k >= 0 ? unit_k : K;
        if (!o->merge && kk <= kShortK) epi_warps = kk <= kTinyK && bn == 256 ? 16 : 8;
    }
    if (epi_warps == 16 && bn != 256)
        return fail(TS_ERR_UNSUPPORTED, "sixteen epilogue warps are built for 256-column tiles only");
    if (o->protocol_log && o->protocol_log_cap < 1)
        return fail(TS_ERR_INVALID_ARG, "protocol_log_cap = %d (>= 1 with a protocol log)", o->protocol_log_cap);
    const int log = o->protocol_log ? 1 : 0;
    pl->v = find_variant(bn, cg, out, epi_warps, o->merge, log);
    if (!pl->v && log) return fail(TS_ERR_UNSUPPORTED, "no protocol-logging build of tile %d with these options", tile);
    if (!pl->v) return fail(TS_ERR_UNSUPPORTED, "no compiled variant for tile %d", tile);
    pl->cg = cg;
    pl->tile_m = 128 * cg;
    pl->tile_n = bn;
    pl->tiles_m = cdiv(M, pl->tile_m);
    pl->tiles_n = cdiv(N, pl->tile_n);
    pl->num_tiles = pl->tiles_m * pl->tiles_n * (groups > 0 ? groups : 1);
    if (pl->num_tiles * cg > kMaxDim) return fail(TS_ERR_UNSUPPORTED, "too many output tiles");
    int resident = 0;
    cudaError_t e = pl->v->max_workers(&resident);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (resident <= 0) return fail(TS_ERR_UNSUPPORTED, "kernel cannot be resident on this device");
    pl->resident = resident;
    // Split wave: when the tiles do not fill the last wave of W workers, r =
    // tiles mod W tiles are split along K into s = W / r parts, and those parts
    // are scheduled first, so that their partial writes and reduction overlap
    // the next tiles' mainloops rather than trail the launch.
    int64_t W = resident;
    if (sched == TS_SCHED_STATIC && o->max_workers > 0) W = std::min<int64_t>(W, o->max_workers);
    const int64_t nk = cdiv(K, 64);
    pl->split_tiles = 0;
    pl->parts = 1;
    pl->split_ws_bytes = 0;
    pl->counter_bytes = 0;
    pl->split = false;
    // (not with a skip mask: the plan cannot see which tiles of the last wave will run)
    // (nor with sixteen epilogue warps: their variants have no reduction path)
    if (o->split_tail >= 0 && groups == 0 && !o->skip_tiles && !o->row_sums && K > 0 && pl->num_tiles > W &&
        pl->v->epi_warps != 16) {
        const int64_t r = pl->num_tiles % W;
        const int64_t s =
            r > 0 ? std::min<int64_t>(std::min<int64_t>(W / r, nk / kMinKBlocksPerPart), kMaxParts) : 0;
        const int64_t counters = r * cg * 8 * static_cast<int64_t>(sizeof(int32_t));
        if (r > 0 && s >= 2 && counters <= kCounterRegionBytes) {
            pl->counter_bytes = kCounterRegionBytes;
            pl->split_ws_bytes = pl->counter_bytes + r * s * cg * 4 * 32 * static_cast<int64_t>(bn) * 4;
            if (o->workspace && o->workspace_bytes >= pl->split_ws_bytes &&
                reinterpret_cast<uintptr_t>(o->workspace) % 256 == 0) {
                pl->split = true;
                pl->split_tiles = r;
                pl->parts = s;
            }
        }
    }
    pl->num_units = pl->num_tiles - pl->split_tiles + pl->split_tiles * pl->parts;
    if (pl->num_units * cg > kMaxDim) return fail(TS_ERR_UNSUPPORTED, "too many work units");
    if (sched != TS_SCHED_STATIC) {  // CLC and non-persistent: one CTA (cluster) per unit
        pl->workers = pl->num_units;
    } else {
        int64_t w = std::min<int64_t>(pl->num_units, W);
        pl->workers = std::max<int64_t>(w, pl->num_units > 0 ? 1 : 0);
    }
    pl->grid = pl->workers * cg;
    const int esize = out == TS_OUT_F32 ? 4 : 2;
    pl->tma_store = (reinterpret_cast<uintptr_t>(D) % 16 == 0) && ((pl->ldd * esize) % 16 == 0);
    return TS_OK;
}

}  // namespace
}  // namespace ts

namespace ts {
ts_status fill_info(int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts,
                    ts_launch_info *info, int64_t groups, int64_t unit_k = -1) {
    if (!info) return ts::fail(TS_ERR_INVALID_ARG, "info is NULL");
    std::memset(info, 0, sizeof *info);
    ts::Plan pl;
    // alignment of D is unknown here: report the TMA-store epilogue when the pitch allows it
    ts_status s = ts::plan_gemm(reinterpret_cast<const void *>(uintptr_t(256)), M, N, K, out_dtype, sched, opts, &pl,
                                groups, unit_k);
    if (s != TS_OK) return s;
    info->tile_m = pl.tile_m;
    info->tile_n = pl.tile_n;
    info->cluster = pl.cg;
    info->stages = pl.v->stages;
    info->tiles_m = pl.tiles_m;
    info->tiles_n = pl.tiles_n;
    info->num_tiles = pl.num_tiles;
    info->grid_ctas = pl.grid;
    info->workers = pl.workers;
    info->smem_bytes = pl.v->smem_bytes;
    info->tma_store = pl.tma_store;
    info->num_units = pl.num_units;
    info->split_tiles = pl.split_tiles;
    info->split_parts = static_cast<int32_t>(pl.parts);
    info->resident = static_cast<int32_t>(pl.resident);
    info->workspace_bytes = pl.split_ws_bytes;
    info->epi_warps = pl.v->epi_warps;
    info->merge = pl.v->merge;
    info->clc_lazy = (sched == TS_SCHED_CLC && groups == 0 && cdiv(K, 64) >= kLazyClcKBlocks) ? 1 : 0;
    return TS_OK;
}
}  // namespace ts

extern "C" {

ts_status ts_gemm_launch_info(int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                              const ts_gemm_opts *opts, ts_launch_info *info) {
    return ts::fill_info(M, N, K, out_dtype, sched, opts, info, 0);
}

ts_status ts_gemm_tile_coords(int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                              const ts_gemm_opts *opts, int64_t first_tile, int64_t count, int32_t *m_block,
                              int32_t *n_block) {
    ts::Plan pl;
    std::memset(&pl, 0, sizeof pl);
    const int32_t tile = opts ? opts->tile : TS_TILE_AUTO;
    if (tile == TS_TILE_AUTO) {
        // the automatic tile choice depends on the device's SM count
        ts_status s = ts::plan_gemm(reinterpret_cast<const void *>(uintptr_t(256)), M, N, K, out_dtype, sched, opts,
                                    &pl, 0);
        if (s != TS_OK) return s;
    } else {
        // an explicit tile fixes the grid of tiles: no device is needed
        if (M < 0 || N < 0 || K < 0 || M > ts::kMaxDim || N > ts::kMaxDim || K > ts::kMaxDim)
            return ts::fail(TS_ERR_INVALID_ARG, "sizes must be in [0, 2^31-1]");
        if (out_dtype != TS_OUT_BF16 && out_dtype != TS_OUT_F32)
            return ts::fail(TS_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
        if (sched != TS_SCHED_STATIC && sched != TS_SCHED_CLC && sched != TS_SCHED_NONPERSISTENT)
            return ts::fail(TS_ERR_INVALID_ARG, "sched %d", sched);
        if (tile < TS_TILE_AUTO || tile > TS_TILE_256x256_2CTA) return ts::fail(TS_ERR_INVALID_ARG, "tile %d", tile);
        if (opts->raster_group < 0) return ts::fail(TS_ERR_INVALID_ARG, "negative option");
        const int64_t tile_m = tile == TS_TILE_256x256_2CTA ? 256 : 128;
        const int64_t tile_n = tile == TS_TILE_128x128 ? 128 : 256;
        pl.tiles_m = ts::cdiv(M, tile_m);
        pl.tiles_n = ts::cdiv(N, tile_n);
        if (pl.tiles_m * pl.tiles_n * (tile_m / 128) > ts::kMaxDim)
            return ts::fail(TS_ERR_UNSUPPORTED, "too many output tiles");
    }
    const int64_t tiles = pl.tiles_m * pl.tiles_n;
    if (first_tile < 0 || count < 0 || first_tile > tiles || count > tiles - first_tile)
        return ts::fail(TS_ERR_INVALID_ARG, "tiles [%lld, %lld + %lld) outside [0, %lld)",
                        static_cast<long long>(first_tile), static_cast<long long>(first_tile),
                        static_cast<long long>(count), static_cast<long long>(tiles));
    if (count > 0 && (!m_block || !n_block)) return ts::fail(TS_ERR_INVALID_ARG, "m_block or n_block is NULL");
    ts_gemm_opts z;
    std::memset(&z, 0, sizeof z);
    ts::GemmParams p;
    std::memset(&p, 0, sizeof p);
    if (count == 0) return TS_OK;
    ts::set_raster(p, pl, opts ? opts : &z);
    for (int64_t t = 0; t < count; ++t) {
        int32_t mb, nb;
        ts::raster(static_cast<int32_t>(first_tile + t), p, mb, nb);
        m_block[t] = mb;
        n_block[t] = nb;
    }
    return TS_OK;
}

ts_status ts_gemm_protocol_info(int32_t tile, int32_t out_dtype, int32_t epi_warps, int32_t merge,
                                ts_gemm_protocol *proto) {
    if (!proto) return ts::fail(TS_ERR_INVALID_ARG, "proto is NULL");
    if (out_dtype != TS_OUT_BF16 && out_dtype != TS_OUT_F32) return ts::fail(TS_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (epi_warps == 0) epi_warps = 4;
    if (epi_warps != 4 && epi_warps != 8 && epi_warps != 16)
        return ts::fail(TS_ERR_INVALID_ARG, "epi_warps = %d (0, 4, 8 or 16)", epi_warps);
    if (merge != 0 && merge != 1) return ts::fail(TS_ERR_INVALID_ARG, "merge = %d (0 or 1)", merge);
    int bn, cg;
    switch (tile) {
        case TS_TILE_128x128: bn = 128, cg = 1; break;
        case TS_TILE_128x256: bn = 256, cg = 1; break;
        case TS_TILE_256x256_2CTA: bn = 256, cg = 2; break;
        default: return ts::fail(TS_ERR_INVALID_ARG, "tile %d (an explicit tile is required)", tile);
    }
    const ts::GemmVariant *v = ts::find_variant(bn, cg, out_dtype, epi_warps, merge);
    if (!v) return ts::fail(TS_ERR_UNSUPPORTED, "no compiled variant for tile %d", tile);
    *proto = v->protocol;
    return TS_OK;
}

}  // extern "C"

namespace ts {
namespace {

// Validate a grouped GEMM's K offsets (host array of groups + 1 entries).
ts_status check_groups(int64_t groups, const int64_t *k_offsets) {
    if (groups < 1) return fail(TS_ERR_INVALID_ARG, "groups = %lld must be >= 1", static_cast<long long>(groups));
    if (groups > kMaxGroups)
        return fail(TS_ERR_UNSUPPORTED, "%lld groups exceed the %d-group limit", static_cast<long long>(groups),
                    kMaxGroups);
    if (!k_offsets) return fail(TS_ERR_INVALID_ARG, "k_offsets is NULL");
    for (int64_t g = 0; g <= groups; ++g) {
        if (k_offsets[g] < 0 || k_offsets[g] % 64 || k_offsets[g] > kMaxDim)
            return fail(TS_ERR_INVALID_ARG, "k_offsets[%lld] = %lld must be a multiple of 64 in [0, 2^31)",
                        static_cast<long long>(g), static_cast<long long>(k_offsets[g]));
        if (g > 0 && k_offsets[g] < k_offsets[g - 1])
            return fail(TS_ERR_INVALID_ARG, "k_offsets must not decrease (index %lld)", static_cast<long long>(g));
    }
    return TS_OK;
}

// The order in which a grouped GEMM's groups are scheduled (GemmParams::group_order):
// by K range, longest first; equal ranges keep their index order.
void group_order(int64_t groups, const int64_t *k_offsets, uint8_t *order) {
    int32_t idx[kMaxGroups];
    for (int32_t g = 0; g < groups; ++g) idx[g] = g;
    std::stable_sort(idx, idx + groups, [&](int32_t x, int32_t y) {
        return k_offsets[x + 1] - k_offsets[x] > k_offsets[y + 1] - k_offsets[y];
    });
    for (int64_t i = 0; i < groups; ++i) order[i] = static_cast<uint8_t>(idx[i]);
}

// Shared launch path.  groups == 0: plain GEMM over K.  groups > 0: group g
// multiplies columns [k_offsets[g], k_offsets[g + 1]) of A and B into D + g * M * ldd.
ts_status gemm_launch(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, int32_t out_dtype,
                      int32_t sched, const ts_gemm_opts *opts, void *stream, int64_t groups,
                      const int64_t *k_offsets) {
    Plan pl;
    ts_status s = plan_gemm(D, M, N, K, out_dtype, sched, opts, &pl, groups,
                            groups > 0 ? longest_group(groups, k_offsets) : -1);
    if (s != TS_OK) return s;
    if (M == 0 || N == 0) return TS_OK;
    const int64_t depth = groups > 0 ? groups : 1;
    if (!D) return fail(TS_ERR_INVALID_ARG, "D is NULL");
    const int esize = out_dtype == TS_OUT_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(D) % esize) return fail(TS_ERR_INVALID_ARG, "D is not aligned to its element size");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t dbytes = ((depth * M - 1) * pl.ldd + N) * esize;

    if (K == 0) {
        // every group (or the single product) is an empty sum: D = 0
        const int64_t total = depth * M * N;
        const int blocks = static_cast<int>(std::min<int64_t>(cdiv(total, 256), 4096));
        if (out_dtype == TS_OUT_F32)
            zero_fill_kernel<float><<<blocks, 256, 0, st>>>(static_cast<float *>(D), depth * M, N, pl.ldd);
        else
            zero_fill_kernel<uint16_t><<<blocks, 256, 0, st>>>(static_cast<uint16_t *>(D), depth * M, N, pl.ldd);
        cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? TS_OK : cuda_fail(e, "zero-fill launch");
    }
    if (!A || !B) return fail(TS_ERR_INVALID_ARG, "A or B is NULL");
    if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
        return fail(TS_ERR_UNSUPPORTED, "A and B must start on a 16-byte boundary");
    if ((pl.lda * 2) % 16 || (pl.ldb * 2) % 16)
        return fail(TS_ERR_UNSUPPORTED, "rows of A and B must start on 16-byte boundaries (lda, ldb multiples of 8)");
    const int64_t abytes = ((M - 1) * pl.lda + K) * 2, bbytes = ((N - 1) * pl.ldb + K) * 2;
    if (ranges_overlap(D, dbytes, A, abytes) || ranges_overlap(D, dbytes, B, bbytes))
        return fail(TS_ERR_INVALID_ARG, "D overlaps A or B");

    ts_gemm_opts z;
    std::memset(&z, 0, sizeof z);
    const ts_gemm_opts *o = opts ? opts : &z;

    GemmLaunch L;
    std::memset(&L, 0, sizeof L);
    const int b_rows = pl.tile_n / pl.cg;
    if ((s = make_map(&L.a, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, pl.lda, 128, 64)) != TS_OK) return s;
    if ((s = make_map(&L.b, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, pl.ldb, b_rows, 64)) != TS_OK) return s;
    if (pl.tma_store) {
        const CUtensorMapDataType dt =
            out_dtype == TS_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if ((s = make_map_d(&L.d, D, dt, esize, depth, M, N, pl.ldd, 32, 128 / esize)) != TS_OK) return s;
    }
    unsigned long long *status = device_status_word(&s);
    if (!status) return s;

    GemmParams &p = L.p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.tiles_m = static_cast<int32_t>(pl.tiles_m);
    p.tiles_n = static_cast<int32_t>(pl.tiles_n);
    p.num_tiles = static_cast<int32_t>(pl.num_tiles);
    p.num_k_blocks = static_cast<int32_t>(cdiv(K, 64));
    p.num_units = static_cast<int32_t>(pl.num_units);
    p.full_tiles = static_cast<int32_t>(pl.num_tiles - pl.split_tiles);
    p.split_tiles = static_cast<int32_t>(pl.split_tiles);
    p.parts = static_cast<int32_t>(pl.parts);
    if (pl.split) {
        p.counters = static_cast<int32_t *>(o->workspace);
        p.partials = reinterpret_cast<float *>(static_cast<char *>(o->workspace) + pl.counter_bytes);
    }
    set_raster(p, pl, o);
    p.sched = sched;
    p.tma_store = pl.tma_store;
    p.clc_depth = 2;
    p.clc_lazy = (groups == 0 && p.num_k_blocks >= kLazyClcKBlocks) ? 1 : 0;  // (ts_launch_info.clc_lazy)
    // Units of odd waves walk their K range downwards (see GemmParams::k_alt).  The
    // wave length is the number of workers that fit at once, whatever the scheduler
    // or the static cap, so a unit's summation order is a function of the plan alone.
    p.k_alt = 1;
    p.div_wave = fast_div_for(pl.resident);
    p.inputs_ready = o->inputs_ready;
    p.D = D;
    p.ldd = pl.ldd;
    const double tmo = o->timeout_s > 0 ? o->timeout_s : kDefaultTimeoutS;
    p.timeout_ns = static_cast<uint64_t>(std::min(tmo, 60.0) * 1e9);
    if (p.timeout_ns == 0) p.timeout_ns = 1;
    p.drain_ns = kDrainNs;
    p.status = status;
    p.trace = reinterpret_cast<long long *>(o->trace);
    p.skip = o->skip_tiles;
    p.row_sums = o->row_sums;
    p.plog = o->protocol_log;
    p.plog_cap = o->protocol_log_cap;
    p.groups = static_cast<int32_t>(groups);
    p.tiles_per_group = static_cast<int32_t>(pl.tiles_m * pl.tiles_n);
    p.group_stride = M * pl.ldd;
    for (int64_t g = 0; groups > 0 && g <= groups; ++g) p.group_kb[g] = static_cast<int32_t>(k_offsets[g] / 64);
    if (groups > 0) group_order(groups, k_offsets, p.group_order);
    L.grid = static_cast<int>(pl.grid);
    L.stream = st;
    cudaError_t e = pl.v->launch(L);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
    return TS_OK;
}

}  // namespace
}  // namespace ts

extern "C" {

ts_status ts_gemm_bf16_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, int32_t out_dtype,
                          int32_t sched, const ts_gemm_opts *opts, void *stream) {
    return ts::gemm_launch(A, B, D, M, N, K, out_dtype, sched, opts, stream, 0, nullptr);
}

ts_status ts_gemm_bf16_grouped(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t groups,
                               const int64_t *k_offsets, int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts,
                               void *stream) {
    ts_status s = ts::check_groups(groups, k_offsets);
    if (s != TS_OK) return s;
    return ts::gemm_launch(A, B, D, M, N, k_offsets[groups], out_dtype, sched, opts, stream, groups, k_offsets);
}

ts_status ts_gemm_grouped_order(int64_t groups, const int64_t *k_offsets, int32_t *order) {
    ts_status s = ts::check_groups(groups, k_offsets);
    if (s != TS_OK) return s;
    if (!order) return ts::fail(TS_ERR_INVALID_ARG, "order is NULL");
    uint8_t o[ts::kMaxGroups];
    ts::group_order(groups, k_offsets, o);
    for (int64_t i = 0; i < groups; ++i) order[i] = o[i];
    return TS_OK;
}

ts_status ts_gemm_grouped_launch_info(int64_t M, int64_t N, int64_t groups, const int64_t *k_offsets,
                                      int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts,
                                      ts_launch_info *info) {
    ts_status s = ts::check_groups(groups, k_offsets);
    if (s != TS_OK) return s;
    return ts::fill_info(M, N, k_offsets[groups], out_dtype, sched, opts, info, groups,
                         ts::longest_group(groups, k_offsets));
}


ts_status ts_gemm_bf16(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, int32_t out_dtype,
                       int32_t sched, void *stream) {
    return ts_gemm_bf16_ex(A, B, D, M, N, K, out_dtype, sched, nullptr, stream);
}

ts_status ts_gemm_bf16_host(const void *A_host, const void *B_host, void *D_host, void *A_dev, void *B_dev,
                            void *D_dev, int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                            const ts_gemm_opts *opts, void *stream) {
    using namespace ts;
    if (M < 0 || N < 0 || K < 0) return ts_gemm_bf16_ex(A_dev, B_dev, D_dev, M, N, K, out_dtype, sched, opts, stream);
    const int64_t lda = opts && opts->lda ? opts->lda : K, ldb = opts && opts->ldb ? opts->ldb : K;
    const int64_t ldd = opts && opts->ldd ? opts->ldd : N;
    const int64_t esize = out_dtype == TS_OUT_F32 ? 4 : 2;
    // the bytes the device buffers span: every row at its pitch, the last one to its end
    const int64_t a_bytes = M > 0 && K > 0 ? ((M - 1) * lda + K) * 2 : 0;
    const int64_t b_bytes = N > 0 && K > 0 ? ((N - 1) * ldb + K) * 2 : 0;
    const int64_t d_bytes = M > 0 && N > 0 ? ((M - 1) * ldd + N) * esize : 0;
    if ((a_bytes && (!A_host || !A_dev)) || (b_bytes && (!B_host || !B_dev)) || (d_bytes && (!D_host || !D_dev)))
        return fail(TS_ERR_INVALID_ARG, "a host or device buffer is NULL");
    // sizes and options are checked before anything is copied
    ts_launch_info info;
    ts_status s = ts_gemm_launch_info(M, N, K, out_dtype, sched, opts, &info);
    if (s != TS_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (a_bytes) e = cudaMemcpyAsync(A_dev, A_host, static_cast<size_t>(a_bytes), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && b_bytes)
        e = cudaMemcpyAsync(B_dev, B_host, static_cast<size_t>(b_bytes), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "copy of A or B to the device");
    s = ts_gemm_bf16_ex(A_dev, B_dev, D_dev, M, N, K, out_dtype, sched, opts, stream);
    if (s != TS_OK) return s;
    if (d_bytes) e = cudaMemcpyAsync(D_host, D_dev, static_cast<size_t>(d_bytes), cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? TS_OK : cuda_fail(e, "copy of D to the host");
}

}  // extern "C"
