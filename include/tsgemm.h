/*
 * tsgemm -- persistent, warp-specialised bf16 GEMM with static and Cluster
 * Launch Control tile scheduling, plus a vectorised grid-stride int16 copy,
 * for one NVIDIA GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes only.  Every device pointer is owned by
 * the caller; the library never allocates device memory on these paths.  The
 * only library-owned device state is a small per-device status word that
 * records a timed-out barrier wait (see ts_sync_and_check) and the statically
 * sized scratch array of ts_gemm_bf16_checked_noalloc, both module globals.
 *
 * Streams are passed as `void *` holding a cudaStream_t (NULL = the legacy
 * default stream).  Every compute call is asynchronous on that stream and
 * returns once the launch is queued; none of them synchronises.
 *
 * Errors: each call returns a ts_status.  On failure, ts_last_error_detail()
 * gives a human-readable message for the calling thread.  Argument errors are
 * detected before any launch, so a failing call never leaves work queued.
 */
#ifndef TSGEMM_H
#define TSGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TS_OK = 0,
    TS_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, overlapping copy */
    TS_ERR_UNSUPPORTED = 2, /* legal request the library cannot run (TMA alignment, size limits) */
    TS_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed; detail has the CUDA message */
    TS_ERR_TIMEOUT = 4      /* a kernel gave up on a barrier wait (reported by ts_sync_and_check) */
} ts_status;

/* Scheduling shapes (CUTLASS TS "Schedules", Scheduling Shapes): static persistent (a grid of
 * resident workers, tile i of worker w = w + i * workers), dynamic persistent (Cluster Launch
 * Control: one CTA or cluster per tile, running workers take over pending ones), and
 * non-persistent (one CTA or cluster per tile, each computing its own tile and exiting).  The GEMM
 * and the jagged row copy take all three. */
typedef enum { TS_SCHED_STATIC = 0, TS_SCHED_CLC = 1, TS_SCHED_NONPERSISTENT = 2 } ts_sched;
typedef enum { TS_OUT_BF16 = 0, TS_OUT_F32 = 1 } ts_out_dtype;

typedef enum {
    TS_TILE_AUTO = 0,
    TS_TILE_128x128 = 1,      /* one CTA per 128x128 output tile */
    TS_TILE_128x256 = 2,      /* one CTA per 128x256 output tile */
    TS_TILE_256x256_2CTA = 3  /* a 2-CTA cluster per 256x256 output tile (cta_group::2 MMA) */
} ts_tile;

/* Optional knobs for ts_gemm_bf16_ex; zero means "default" for every field. */
typedef struct {
    int32_t tile;         /* ts_tile */
    int32_t max_workers;  /* static scheduler: cap on persistent workers (CTAs or 2-CTA clusters) */
    int64_t lda;          /* row stride of A in elements (>= K); 0 = K */
    int64_t ldb;          /* row stride of B in elements (>= K); 0 = K */
    int64_t ldd;          /* row stride of D in elements (>= N); 0 = N */
    double timeout_s;     /* per-wait limit for every mbarrier wait in the kernel; 0 = 2 s */
    int64_t *trace;       /* device buffer of 4 * num_units int64 (ts_launch_info), zeroed by the
                             caller, or NULL.  Per work unit u: [4u] += 1 per visit,
                             [4u+1] = worker index, [4u+2] = %globaltimer when the producer
                             started the unit, [4u+3] = %globaltimer when the epilogue finished it
                             (for a skipped tile no data passes between the two, so [4u+3] may
                             precede [4u+2]). */
    int32_t raster_group; /* tile raster: consecutive tile ids walk this many tile rows; 0 = 8 */
    int32_t split_tail;   /* 0: split the last, partial wave of tiles along K when `workspace` is
                             large enough; -1: never split */
    void *workspace;      /* device scratch for the split tiles (ts_launch_info.workspace_bytes),
                             256-byte aligned.  Its first 8 KiB hold per-slab counters: zero them
                             before the first use; every normal launch leaves them zero again
                             (after TS_ERR_TIMEOUT zero them once more).  The rest holds fp32
                             partials and needs no initialisation.  Launches that may overlap on
                             the GPU need separate workspaces. */
    int64_t workspace_bytes;
    const uint8_t *skip_tiles; /* device array or NULL: one byte per output tile, entry
                             g * tiles_m * tiles_n + m_block * tiles_n + n_block (g = group, 0 for
                             a plain GEMM; blocks of ts_launch_info.tile_m x tile_n).  A nonzero byte
                             skips the tile: it is neither computed nor stored (D keeps its contents
                             there), but the schedulers still hand it out (CUTLASS TS "Schedules",
                             Skippable Tiles).  A launch with a skip mask does not split its tail. */
    float *row_sums;      /* device fp32 [groups][M] or NULL.  When given, a second consumer task
                             reads every shared-memory ring stage beside the MMA (a Fork pipeline
                             group: CUTLASS TS "Pipeline Groups", Fork) and writes
                             row_sums[g][i] = sum over the group's K range of A[i][k], the
                             correction term of zero-point-quantised products.  Rows whose first
                             tile column is skipped are left untouched.  1-CTA tiles only (AUTO
                             picks one; TS_TILE_256x256_2CTA is TS_ERR_UNSUPPORTED); no split tiles. */
    int32_t epi_warps;    /* epilogue warps per CTA: 4 (one per TMEM lane quarter), 8 or 16 (two or
                             four per quarter, taking its subtiles in turn: more latency hidden
                             when the epilogue bounds the tile); 0 = automatic: 16 with K <= 128
                             on a 256-column tile, 8 with K <= 256, else 4 (K of a grouped GEMM:
                             its longest group's range).
                             16 needs a 256-column tile (else TS_ERR_UNSUPPORTED) and never
                             splits the tail.  Anything else is TS_ERR_INVALID_ARG.  Results do
                             not depend on it. */
    int32_t merge;        /* the ring's barrier layout (CUTLASS TS "Pipeline Groups"): 0 = FusedMerge,
                             one producer thread loads A and B onto one full barrier per stage
                             (2 * S mbarriers); 1 = Merge, separate producer warps for A and for B,
                             each with its own full barrier per stage, sharing the empty barrier
                             (3 * S).  Merge uses four epilogue warps (epi_warps = 8 or 16
                             is TS_ERR_UNSUPPORTED) and cannot run with row_sums (both need warp 3:
                             TS_ERR_UNSUPPORTED).  Results do not depend on it. */
    int32_t inputs_ready; /* 1: the caller guarantees that A, B and skip_tiles held their final contents
                             before the kernel preceding this call in the stream began (none of them
                             is written by that kernel, nor by anything that kernel may run
                             alongside).  Every GEMM launch is a programmatic dependent of the
                             previous kernel; its dependent-launch barrier is one resource of the
                             kernel's dependency graph (CUTLASS TS "Introduction", Core Terms: a PDL
                             barrier).  By default (0) every task waits on it before touching global
                             memory.  With 1 the epilogue (which writes D, the split tiles' workspace
                             and the trace) waits on it first, and every other task runs its first
                             work unit ahead of it and waits on it before its second (the Fork task
                             before its first row_sums store, the producer before its first trace
                             write), so the first tiles' loads and MMAs overlap the previous kernel's
                             tail.  Results do not depend on it when the guarantee holds; when it
                             does not, they are undefined.  Anything else is TS_ERR_INVALID_ARG. */
    int32_t *protocol_log; /* device int32 buffer or NULL: a test instrument.  When given, the launch
                             runs the protocol-logging build of its kernel, in which every role's
                             thread records its barrier operations in program order (waits with
                             their parity, arrivals, TMA loads, MMA k-blocks, tcgen05 commits, CLC
                             requests, the dependent-launch wait, and the units the producer
                             begins), so that a host-side model of the role loops can be compared
                             with them.  Layout: per CTA c and role r (0 producer, 1 MMA issuer,
                             2 CLC scheduler, 3 warp 3, 4 + j epilogue warp j; 20 roles), a block of
                             protocol_log_cap + 1 words at (c * 20 + r) * (protocol_log_cap + 1):
                             the count of events, then the first protocol_log_cap events; the
                             caller zeroes the buffer.  Built for fp32 output on five shapes only:
                             tile 128x128 with four epilogue warps (FusedMerge or Merge) or eight,
                             tile 128x256 with sixteen, and the 2-CTA 256x256 tile with four
                             (others: TS_ERR_UNSUPPORTED).  Results are those of the normal
                             build. */
    int32_t protocol_log_cap; /* events per CTA and role (>= 1 when protocol_log is given) */
} ts_gemm_opts;

/* What ts_gemm_bf16_ex would launch for a problem (host-only query). */
typedef struct {
    int32_t tile_m, tile_n;  /* output tile of one worker */
    int32_t cluster;         /* CTAs per worker: 1, or 2 for the 2-CTA tile */
    int32_t stages;          /* shared-memory ring depth */
    int64_t tiles_m, tiles_n, num_tiles;
    int64_t grid_ctas;       /* CTAs launched */
    int64_t workers;         /* static: persistent workers launched; CLC and non-persistent: num_units */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t tma_store;       /* 1 if D is written through TMA stores, 0 for the st.global epilogue */
    int64_t num_units;       /* work units scheduled: whole tiles plus the K parts of split tiles */
    int64_t split_tiles;     /* tiles split along K, scheduled first (0 if none) */
    int32_t split_parts;     /* K parts per split tile (1 if none) */
    int32_t resident;        /* workers (CTAs or 2-CTA clusters) that fit on the GPU at once */
    int64_t workspace_bytes; /* workspace the split tiles need (0 when no split would help) */
    int32_t epi_warps;       /* epilogue warps per CTA (4, 8 or 16; CTAs have 128 + 32 * epi_warps threads) */
    int32_t merge;           /* 1: Merge barrier layout (A and B producers apart), 0: FusedMerge */
    int32_t clc_lazy;        /* 1: CLC requests wait until the producer has nearly loaded its unit
                                (K loops of 32 k-blocks or more under CLC) */
    int32_t reserved;
} ts_launch_info;

/* The barrier protocol of one kernel variant: the numbers the kernel
 * initialises its mbarriers with.  The host-side protocol checker
 * (tile_scheduling_gb300/protocol.py) models the role loops with them. */
typedef struct {
    int32_t cluster;             /* CTAs per worker */
    int32_t stages;              /* shared-memory ring depth S */
    int32_t tx_bytes;            /* transaction bytes per stage on the even CTA's full barrier */
    int32_t full_arrivals;       /* arrivals that complete a full[s] phase (besides the tx bytes) */
    int32_t empty_arrivals;      /* arrivals that complete an empty[s] phase */
    int32_t accumulators;        /* TMEM accumulator buffers */
    int32_t tmem_full_arrivals;  /* arrivals on tmem_full[a] */
    int32_t tmem_empty_arrivals; /* arrivals on the even CTA's tmem_empty[a] */
    int32_t clc_slots;           /* CLC response slots */
    int32_t clc_full_arrivals;   /* arrivals (besides the response bytes) on a CTA's clc_full[r] */
    int32_t clc_empty_arrivals;  /* arrivals on the even CTA's clc_empty[r]: every consuming role */
    int32_t clc_response_bytes;
    int32_t epilogue_warps;      /* epilogue warps per CTA */
    int32_t stage_bytes;         /* A + B bytes one CTA loads per stage */
    int32_t aux_empty_arrivals;  /* arrivals on aux_empty[s] from the Fork row-sum task (row_sums given) */
    int32_t merge;               /* 1: Merge layout, A on full[s] (a_stage_bytes * cluster) and B on
                                    full_b[s] ((stage_bytes - a_stage_bytes) * cluster), one producer each */
    int32_t a_stage_bytes;       /* A bytes one CTA loads per stage */
} ts_gemm_protocol;

/* Fill *proto for the kernel variant of `tile` (TS_TILE_128x128, _128x256 or
 * _256x256_2CTA; TS_TILE_AUTO is TS_ERR_INVALID_ARG), `out_dtype`, `epi_warps`
 * (4, 8 or 16; 0 = 4; 16 for 256-column tiles only) and `merge` (0 or 1; Merge
 * variants have 4 epilogue warps).
 * Host only; needs no GPU. */
ts_status ts_gemm_protocol_info(int32_t tile, int32_t out_dtype, int32_t epi_warps, int32_t merge,
                                ts_gemm_protocol *proto);

/*
 * ts_protocol_check -- explore every interleaving of a small mbarrier program
 * (host only).  Restates the idea of the Task Scheduling static verifier
 * (CUTLASS TS "Introduction": schedules are checked for deadlocks and races
 * before lowering); tile_scheduling_gb300/protocol.py builds the programs from
 * this kernel's role loops and ts_gemm_protocol_info.
 *
 *   nbars, bar_expected  barriers and the arrivals that complete each phase
 *   nbufs                buffers (ring stages, TMEM accumulators, CLC slots)
 *   nroles, role_group   roles; roles of one group (>= 0) run identical programs
 *   role_offsets         nroles + 1 offsets into ops (in records)
 *   ops                  8-int32 records (see protocol_check.cu)
 *   names                role, barrier and buffer names, '\n'-separated, for messages
 *   max_states           stop after this many distinct states
 * Returns 0 (no deadlock, no race), 1 (violation; msg says which), 2 (state
 * limit reached), -1 (bad arguments).  *states_out = distinct states visited.
 */
int32_t ts_protocol_check(int32_t nbars, const int32_t *bar_expected, int32_t nbufs, int32_t nroles,
                          const int32_t *role_group, const int32_t *role_offsets, const int32_t *ops,
                          const char *names, int64_t max_states, int64_t *states_out, char *msg, int32_t msg_len);

/*
 * ts_protocol_check_ex -- ts_protocol_check with global counters (host only).
 * The split tiles of the GEMM hand their fp32 partials over through a per-slab
 * counter in global memory: each part stores its partial, fences, and adds one
 * to the counter; the part that draws the last ticket re-arms the counter and
 * sums every part.  The programs model that with store, fence and ticket
 * records (see protocol_check.cu).
 *
 *   ncounters            counters (all start at 0)
 *   counter_reductions   per counter, how often its last ticket must be drawn
 * Every other argument and the return value are those of ts_protocol_check; a
 * run that ends with a counter not back at 0, or drawn last a different number
 * of times, is a violation (1).
 */
int32_t ts_protocol_check_ex(int32_t nbars, const int32_t *bar_expected, int32_t nbufs, int32_t nroles,
                             const int32_t *role_group, const int32_t *role_offsets, const int32_t *ops,
                             int32_t ncounters, const int32_t *counter_reductions, const char *names,
                             int64_t max_states, int64_t *states_out, char *msg, int32_t msg_len);

/*
 * ts_gemm_bf16 -- D = A * B^T with bf16 inputs and fp32 accumulation.
 *
 * Definition: D[i][j] = sum_{k<K} A[i][k] * B[j][k] (CUTLASS TS "Pipeline
 * Groups", Overview: the GEMM mainloop resource graph gmem_ab -> smem_a,
 * smem_b -> tmem_c -> gmem_d; TS "Resources", per-work-tile scale_d reset).
 * Tiles are assigned by the static grid-stride rule (TS "Schedules",
 * Scheduling Shapes; "Cluster Launch Control", static persistent scheduler),
 * by Cluster Launch Control work stealing ("Cluster Launch Control", one
 * CLC request and the overlap loop), or not at all (TS_SCHED_NONPERSISTENT:
 * the launch grid maps one CTA or cluster to each work unit, which computes
 * that unit and exits; the pages' non-persistent shape).  Under CLC each worker keeps up to two
 * requests in flight; with K loops of at least 32 k-blocks a request waits
 * until the worker's current unit is nearly loaded (16 k-blocks left), so the
 * last units go to the workers that finish first.  The scheduler changes which
 * CTA computes a tile, never the result.
 *
 *   A     device, bf16 [M][K] row-major (K contiguous), 16-byte aligned
 *   B     device, bf16 [N][K] row-major (K contiguous), 16-byte aligned
 *   D     device, [M][N] row-major, bf16 (out = TS_OUT_BF16, rounded to
 *         nearest even from fp32) or fp32 (TS_OUT_F32)
 *   M, N, K  sizes, each in [0, 2^31 - 1]
 *
 * Work is scheduled in units: whole tiles, and -- when the opts give a
 * workspace -- the tiles of the last, partial wave split along K so that they
 * fill the GPU; a split tile's parts are summed in fixed order by the warp
 * that finishes last, so results do not depend on timing.
 *
 * M == 0 or N == 0: no-op.  K == 0: D is filled with zeros.
 * A and B rows must start on 16-byte boundaries (K a multiple of 8, or lda/ldb
 * via ts_gemm_bf16_ex) or the call returns TS_ERR_UNSUPPORTED.  A D whose row
 * pitch is not a multiple of 16 bytes is written by a plain-store epilogue.
 * D must not overlap A or B.
 */
ts_status ts_gemm_bf16(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                       int32_t out_dtype, int32_t sched, void *stream);

/* As ts_gemm_bf16, with the knobs above; opts may be NULL. */
ts_status ts_gemm_bf16_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                          int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts, void *stream);

/*
 * ts_gemm_bf16_host -- ts_gemm_bf16_ex on operands in host memory: copies A and
 * B from host memory into the caller's device buffers, runs the GEMM on them
 * and copies D back to host memory, all queued on `stream` in that order.
 *
 *   A_host, B_host, D_host  host arrays laid out as the device ones (row pitches
 *                           lda, ldb, ldd of opts, or packed rows); page-locked
 *                           memory makes the copies asynchronous, pageable memory
 *                           makes the calling thread wait for them
 *   A_dev, B_dev, D_dev     device buffers the caller owns, as for ts_gemm_bf16_ex
 * NULL buffers and the problem's sizes and options (as ts_gemm_launch_info
 * checks them) are rejected before anything is copied; the device pointers'
 * alignment and overlap are checked by the GEMM call, after A and B have been
 * queued for copying (D is then not copied back).  Results and the other
 * arguments are as for ts_gemm_bf16_ex.  The host buffers must stay valid
 * until the stream reaches the copies.
 */
ts_status ts_gemm_bf16_host(const void *A_host, const void *B_host, void *D_host, void *A_dev, void *B_dev,
                            void *D_dev, int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                            const ts_gemm_opts *opts, void *stream);

/*
 * ts_gemm_bf16_grouped -- a grouped GEMM whose groups differ in K:
 *
 *   D[g][i][j] = sum_{k_offsets[g] <= k < k_offsets[g+1]} A[i][k] * B[j][k],   0 <= g < groups
 *
 * The per-tile domain of the K loop comes from an offsets array (CUTLASS TS
 * "Schedules", Dynamic Domain: get_domain_size(tile) = offsets[t + 1] - offsets[t]),
 * so tiles of different groups cost different amounts -- the situation in which
 * Cluster Launch Control work stealing pays off ("Cluster Launch Control", when
 * to use CLC).  This is the shape of, e.g., a per-expert weight gradient, where
 * each expert sees a different number of tokens.
 *
 *   A          device, bf16 [M][lda], columns 0 .. k_offsets[groups] used
 *   B          device, bf16 [N][ldb]
 *   D          device, [groups][M][ldd] (group g starts g * M * ldd elements in), bf16 or fp32
 *   k_offsets  HOST array of groups + 1 non-decreasing multiples of 64 (a group
 *              may be empty: its D is zero)
 *   groups     1 .. 256
 * opts as for ts_gemm_bf16_ex (tile, max_workers, lda/ldb/ldd, timeout_s, trace
 * with 4 * num_units entries); no tiles are split.  Work units are the tiles
 * of one group after another, the groups in the order ts_gemm_grouped_order
 * gives: longest K range first, so that the short units are the ones left for
 * the end of the launch (the LPT rule; results do not depend on the order).
 */
ts_status ts_gemm_bf16_grouped(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t groups,
                               const int64_t *k_offsets, int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts,
                               void *stream);

/*
 * ts_gemm_grouped_order -- the order in which ts_gemm_bf16_grouped schedules the
 * groups (host only, no launch): work unit u of the launch is tile
 * u % (tiles_m * tiles_n) of group order[u / (tiles_m * tiles_n)].  Groups are
 * taken by K range (k_offsets[g + 1] - k_offsets[g]), longest first; equal
 * ranges keep their index order.  Handing out the longest units first is
 * Graham's LPT rule for list scheduling, which bounds how far apart the workers
 * finish by the length of the shortest units rather than the longest; it helps
 * the static round-robin deal and CLC work stealing alike (CUTLASS TS
 * "Schedules", Dynamic Domain leaves the order of the units open).
 *
 *   groups, k_offsets   as for ts_gemm_bf16_grouped
 *   order               HOST int32 array of `groups` entries, written with a
 *                       permutation of 0 .. groups - 1
 * Errors: those of ts_gemm_bf16_grouped's offset checks; TS_ERR_INVALID_ARG for
 * a NULL order.
 */
ts_status ts_gemm_grouped_order(int64_t groups, const int64_t *k_offsets, int32_t *order);

/* The launch ts_gemm_bf16_grouped would make (host only). */
ts_status ts_gemm_grouped_launch_info(int64_t M, int64_t N, int64_t groups, const int64_t *k_offsets,
                                      int32_t out_dtype, int32_t sched, const ts_gemm_opts *opts,
                                      ts_launch_info *info);

/* Fill *info with the launch ts_gemm_bf16_ex would make (no launch, no sync). */
ts_status ts_gemm_launch_info(int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                              const ts_gemm_opts *opts, ts_launch_info *info);

/*
 * ts_gemm_tile_coords -- the output tile that each tile id of the launch
 * ts_gemm_bf16_ex would make covers (host only, no launch).  The kernel's
 * raster walks `raster_group` tile rows down one column band before moving to
 * the next band, the bands of odd groups from the right (a build choice for L2
 * reuse; the pages leave tile order open).  The host evaluates the very
 * function the kernel runs.
 *
 *   M, N, K, out_dtype, sched, opts   as for ts_gemm_launch_info (opts->tile and
 *                                     opts->raster_group matter)
 *   first_tile, count   tile ids [first_tile, first_tile + count) within
 *                       [0, tiles_m * tiles_n)
 *   m_block, n_block    HOST int32 arrays of `count` entries, written with the
 *                       tile row and tile column of each id
 * Errors: TS_ERR_INVALID_ARG for a range outside the tile grid or NULL outputs
 * (count > 0), plus the argument errors of ts_gemm_launch_info.
 */
ts_status ts_gemm_tile_coords(int64_t M, int64_t N, int64_t K, int32_t out_dtype, int32_t sched,
                              const ts_gemm_opts *opts, int64_t first_tile, int64_t count, int32_t *m_block,
                              int32_t *n_block);

/*
 * ts_gemm_bf16_checked_noalloc -- ts_gemm_bf16 (default tile choice) plus a
 * check that the tile scheduler computed every output tile exactly once, for
 * callers that cannot allocate device memory.  No counterpart in the pages:
 * it is a packaging of the traced GEMM for such callers.
 *
 * The per-tile trace lives in a fixed array inside this library's device image
 * (room for 65536 output tiles, 2 MiB per device, held until the process
 * exits) instead of caller memory.  The call allocates nothing.  Its first call
 * on a device looks the array's address up and should precede any stream
 * capture; the address is kept for the life of the process, so a
 * cudaDeviceReset after that first call is not supported (the array may move
 * when the module is loaded again).  All calls on a device share the one
 * array: calls that overlap on the GPU race and must be serialised by the
 * caller.
 *
 *   A, B, D, M, N, K, out_dtype, sched   as for ts_gemm_bf16
 *   bad_tiles  device int32, written asynchronously on `stream` with the number
 *              of tiles not visited exactly once (0 on success; 0 when no tile
 *              is scheduled: M, N or K is 0)
 * Problems with more than 65536 output tiles return TS_ERR_UNSUPPORTED.
 */
ts_status ts_gemm_bf16_checked_noalloc(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                                       int32_t out_dtype, int32_t sched, int32_t *bad_tiles, void *stream);

/*
 * ts_copy_i16 -- dst[i] = src[i] for 0 <= i < n (TS "Resources", the int16
 * copy example: get_item / set_item guarded by gid < num_entries; TS
 * "Schedules", the grid-stride domain start = bx * tpb + tx, step = gdimx * tpb).
 *
 *   src, dst  device int16 arrays of n elements.  src == dst is a no-op;
 *             any other overlap is TS_ERR_INVALID_ARG.
 *   n         element count >= 0.
 * 32-byte vectors are used when src and dst share their offset modulo 32
 * bytes, 16-byte vectors when they share it modulo 16 (elements before the
 * first aligned one and after the last whole vector one by one); otherwise
 * every aligned 16-byte dst vector is assembled from two aligned 16-byte
 * source vectors inside src.  Every path gives the same result.
 */
ts_status ts_copy_i16(const int16_t *src, int16_t *dst, int64_t n, void *stream);

/* Optional knobs for ts_copy_i16_rows; zero means "default" for every field. */
typedef struct {
    int64_t tiles;              /* work tiles launched; 0 = the mode's minimum (rows; with a chunk,
                                   see chunk and pack), which it may not be below.  Tiles t >= the
                                   row count (or past the last piece) copy nothing but still take
                                   part in the work queue (the oversubscribed copy queue). */
    const int64_t *rows_device; /* device int64 or NULL: the row count, read once per CTA on the
                                   device and clamped to [0, rows].  Lets one launch shape (tiles,
                                   rows as capacities) serve a count that a previous kernel wrote. */
    const uint8_t *skip_rows;   /* device array of `rows` bytes or NULL: nonzero = skip that row */
    int32_t threads;            /* threads per CTA: 128, 256, 512 or 1024; 0 = 512 */
    int32_t max_workers;        /* static scheduler: cap on persistent CTAs; 0 = all resident */
    double timeout_s;           /* limit on one wait for a CLC response; 0 = 1 s */
    int64_t *trace;             /* device int64 [2 * tiles] zeroed by the caller, or NULL: per tile t,
                                   [2t] += 1 per visit, [2t+1] = blockIdx.x of the CTA that ran it */
    int64_t chunk;              /* 0: work tile t is row t (the Dynamic Domain form below).  > 0: each row
                                   is cut into pieces of at most `chunk` elements and every piece is a work
                                   tile, in row order, so a long row no longer runs on one CTA at the end
                                   of the queue.  Two planning kernels (same stream, CTAs of 1024
                                   rows) read the offsets first.  tiles defaults to, and may not be below,
                                   rows + ceil(n / chunk); tiles past the last piece are skipped. */
    void *workspace;            /* chunk > 0: device scratch of ts_launch_info.workspace_bytes bytes,
                                   256-byte aligned, no initialisation; launches that may overlap on the
                                   GPU need separate workspaces */
    int64_t workspace_bytes;
    int32_t pack;               /* 1 (needs 1 <= chunk <= 2^30): the copied rows are laid end to end and
                                   work tile t copies their elements [t * chunk, (t + 1) * chunk), so
                                   short rows share a tile and long ones span several; every tile but
                                   the last moves chunk elements.  tiles defaults to, and may not be
                                   below, ceil(n / chunk).  0: chunk pieces per row as above.  Other
                                   values are TS_ERR_INVALID_ARG.  Results do not depend on it. */
    int32_t reserved;           /* must be 0 */
} ts_rows_opts;

/*
 * ts_copy_i16_rows -- copy the rows of a jagged int16 array through a work
 * queue: for every row r < R that is not skipped,
 *
 *   dst[i] = src[i]   for offsets[r] <= i < offsets[r + 1]
 *
 * where R is `rows`, or *opts->rows_device clamped to [0, rows].  Work tile t
 * is row t: its loop bound comes from the offsets array (CUTLASS TS
 * "Schedules", Dynamic Domain: get_domain_size(tile) = offsets[t + 1] -
 * offsets[t]); tiles past R and rows marked in skip_rows run no copy, while
 * every tile still waits on, advances and releases the queue (TS "Schedules",
 * Skippable Tiles, whose example is this oversubscribed copy).  sched picks
 * the queue: TS_SCHED_STATIC, a grid-stride persistent loop over the resident
 * CTAs, TS_SCHED_CLC, one CTA per tile with Cluster Launch Control work
 * stealing ("Cluster Launch Control": the request for the next tile is issued
 * before the current row is copied), or TS_SCHED_NONPERSISTENT, one CTA per
 * tile and no queue.  Elements of dst outside the copied rows are never
 * written.
 *
 *   src, dst  device int16 arrays of n elements, 2-byte aligned; src == dst is
 *             allowed (each element is rewritten with itself); any other
 *             overlap is TS_ERR_INVALID_ARG.  32-byte vectors are used when src
 *             and dst share their offset modulo 32 bytes, 16-byte ones modulo
 *             16; otherwise aligned 16-byte dst vectors joined from two source
 *             vectors inside src (packed mode: element-wise copies).
 *   offsets   device int64 array of rows + 1 entries (read on the device).  A
 *             row with offsets[r] < 0, offsets[r + 1] < offsets[r] or
 *             offsets[r + 1] > n is not copied; the next ts_sync_and_check
 *             returns TS_ERR_INVALID_ARG naming the first such row.
 *   rows      row count (upper bound when rows_device is given), >= 0.
 * A CLC response that does not arrive within timeout_s is reported as
 * TS_ERR_TIMEOUT by ts_sync_and_check; the CTA then stops taking tiles.  In
 * chunked or packed mode, rows that overlap can need more tiles than `tiles`:
 * the rows whose pieces do not fit are reported as TS_ERR_INVALID_ARG by
 * ts_sync_and_check (the pieces that fit are copied).  The planning kernels
 * and the copy kernel are launched as programmatic dependents of the kernel
 * before them in the stream: each may be scheduled during that kernel's tail
 * and reads no memory before its writes are visible.
 */
ts_status ts_copy_i16_rows(const int16_t *src, int16_t *dst, int64_t n, const int64_t *offsets, int64_t rows,
                           int32_t sched, const ts_rows_opts *opts, void *stream);

/* The launch ts_copy_i16_rows would make (host only): num_tiles = num_units =
 * tiles, grid_ctas = workers = CTAs launched, resident = CTAs that fit at once,
 * workspace_bytes = the workspace chunked and packed modes need (0 otherwise). */
ts_status ts_copy_rows_launch_info(int64_t n, int64_t rows, int32_t sched, const ts_rows_opts *opts,
                                   ts_launch_info *info);

/*
 * ts_spin -- occupy `ctas` SMs for `duration_ns` nanoseconds (measured with
 * %globaltimer), to make part of the GPU unavailable to a following kernel.
 * Each spinning CTA requests the largest opt-in shared memory so that no
 * GEMM CTA can share its SM.  `started` is a host int32 in page-locked,
 * device-mapped memory (e.g. cudaHostAlloc or a pinned torch tensor); every
 * CTA adds 1 to it when it begins.  duration_ns is capped at 10 s; ctas must
 * be in [1, number of SMs].  This is a measurement helper: the load-imbalance
 * scenario ("Cluster Launch Control", limits of the static scheduler: SMs
 * held by another kernel leave a long launch tail).
 */
ts_status ts_spin(int32_t ctas, int64_t duration_ns, int32_t *started, void *stream);

/* Wait on the host until *started >= expected or timeout_s passes
 * (TS_ERR_TIMEOUT).  Reads the counter with volatile loads. */
ts_status ts_spin_wait_started(const int32_t *started, int32_t expected, double timeout_s);

/* Synchronise `stream`, then report and clear the device status word:
 * TS_ERR_TIMEOUT if a kernel on the current device gave up on a barrier
 * wait since the last check (detail names the wait and the block),
 * TS_ERR_CUDA on an asynchronous CUDA error, TS_OK otherwise. */
ts_status ts_sync_and_check(void *stream);

/* Number of SMs of the current device (cached), or -1 on error. */
int32_t ts_num_sms(void);

const char *ts_status_string(ts_status s);
/* Thread-local message for the last failing call on this thread ("" if none). */
const char *ts_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* TSGEMM_H */
