"""GPU parity of the jagged row copy (ts_copy_i16_rows) against the oracle: bit-exact.

Covers both work queues (static grid-stride and Cluster Launch Control), the
dynamic per-row domain (empty, short, long and unaligned rows), the skippable
tiles (oversubscribed launches, a row count read on the device, a skip mask),
every vector path (src and dst sharing their offset modulo 32, modulo 16, or
neither), and rows whose bounds fail the device-side check.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _jagged(seed: int, rows: int, max_len: int, lead: int = 5, trail: int = 7):
    """Offsets of `rows` rows of lengths in [0, max_len] starting at `lead`, and n = end + trail."""
    z = synth.splitmix64(seed, rows)
    lengths = (z % np.uint64(max_len + 1)).astype(np.int64)
    lengths[::7] = 0  # some empty rows
    offsets = np.concatenate([[lead], lead + np.cumsum(lengths)]).astype(np.int64)
    return offsets, int(offsets[-1]) + trail


def _run(lib, src_h, dst0_h, offsets_h, sched, rows=None, src_off=0, dst_off=0, **kw):
    n = src_h.size
    sbuf = torch.zeros(n + 32, dtype=torch.int16, device="cuda")
    dbuf = torch.full((n + 32,), -7, dtype=torch.int16, device="cuda")
    sbuf[src_off:src_off + n] = torch.from_numpy(src_h).cuda()
    dbuf[dst_off:dst_off + n] = torch.from_numpy(dst0_h).cuda()
    off = torch.from_numpy(np.asarray(offsets_h, dtype=np.int64)).cuda()
    lib.ts_copy_i16_rows(sbuf[src_off:src_off + n], dbuf[dst_off:dst_off + n], off, rows=rows, sched=sched, **kw)
    lib.ts_sync_and_check()
    d = dbuf.cpu().numpy()
    assert np.all(d[:dst_off] == -7) and np.all(d[dst_off + n:] == -7), "write outside dst"
    return d[dst_off:dst_off + n]


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("threads", [128, 512, 1024])
def test_rows_random_jagged(lib, sched, threads):
    offsets, n = _jagged(11 + threads, 300, 5000)
    src = synth.int16_uniform(12, n)
    dst0 = synth.int16_uniform(13, n)
    got = _run(lib, src, dst0, offsets, sched, threads=threads)
    want, bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert bad == -1 and np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (16, 0), (8, 0), (3, 3), (1, 6), (0, 1)])
def test_rows_vector_paths(lib, sched, src_off, dst_off):
    # shared offset mod 32 bytes (16 elements): 32-byte vectors; mod 16: 16-byte; otherwise element-wise
    offsets, n = _jagged(21, 120, 3000, lead=3, trail=9)
    src = synth.int16_uniform(22, n)
    dst0 = synth.int16_uniform(23, n)
    got = _run(lib, src, dst0, offsets, sched, src_off=src_off, dst_off=dst_off)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_oversubscribed_tiles_are_skipped_and_counted(lib, sched):
    offsets, n = _jagged(31, 200, 2000)
    rows = offsets.size - 1
    tiles = 2 * rows + 37
    src = synth.int16_uniform(32, n)
    dst0 = synth.int16_uniform(33, n)
    trace = torch.zeros(2 * tiles, dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, tiles=tiles, trace=trace)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)
    tr = trace.view(tiles, 2).cpu().numpy()
    info = lib.ts_copy_rows_launch_info(n, rows, sched, tiles=tiles)
    if sched == "static":
        assert np.array_equal(tr[:, 0], np.ones(tiles))
        assert np.array_equal(tr[:, 1], oracle.static_owner(tiles, info["grid_ctas"]))
    elif sched == "nonpersistent":  # one CTA per tile, each on its own tile
        assert np.array_equal(tr[:, 0], np.ones(tiles)) and np.array_equal(tr[:, 1], np.arange(tiles))
    else:
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("count", [0, 1, 57, 200, 10_000])
def test_rows_count_read_on_the_device(lib, sched, count):
    offsets, n = _jagged(41, 200, 1500)
    src = synth.int16_uniform(42, n)
    dst0 = synth.int16_uniform(43, n)
    rd = torch.tensor([count], dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, rows_device=rd, tiles=256)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets, rows=min(count, 200))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_skip_mask(lib, sched):
    offsets, n = _jagged(51, 250, 1200)
    src = synth.int16_uniform(52, n)
    dst0 = synth.int16_uniform(53, n)
    skip = (synth.splitmix64(54, 250) % np.uint64(3) == 0).astype(np.uint8)
    got = _run(lib, src, dst0, offsets, sched, skip_rows=torch.from_numpy(skip).cuda())
    want, _ = oracle.copy_rows_i16(src, dst0, offsets, skip=skip)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_empty_queue_and_all_skipped(lib, sched):
    src = synth.int16_uniform(61, 100)
    dst0 = synth.int16_uniform(62, 100)
    # no rows, no tiles: nothing launched
    assert np.array_equal(_run(lib, src, dst0, [0], sched), dst0)
    # no rows but 50 tiles: every tile runs its bookkeeping and copies nothing
    trace = torch.zeros(100, dtype=torch.int64, device="cuda")
    assert np.array_equal(_run(lib, src, dst0, [0], sched, rows=0, tiles=50, trace=trace), dst0)
    assert torch.equal(trace.view(50, 2)[:, 0].cpu(), torch.ones(50, dtype=torch.int64))


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("bad", ["decreasing", "past_n", "negative"])
def test_rows_bad_bounds_are_reported_not_copied(lib, sched, bad):
    n = 1000
    offsets = np.array([0, 100, 300, 600, 1000], dtype=np.int64)
    if bad == "decreasing":
        offsets[2] = 50      # row 1 = [100, 50), row 2 = [50, 600)
    elif bad == "past_n":
        offsets[4] = 1200    # row 3 = [600, 1200)
    else:
        offsets[0] = -10     # row 0 = [-10, 100)
    src = synth.int16_uniform(71, n)
    dst0 = synth.int16_uniform(72, n)
    sbuf = torch.from_numpy(src).cuda()
    dbuf = torch.from_numpy(dst0.copy()).cuda()
    off = torch.from_numpy(offsets).cuda()
    lib.ts_copy_i16_rows(sbuf, dbuf, off, sched=sched)
    with pytest.raises(lib.TsError) as ei:
        lib.ts_sync_and_check()
    assert ei.value.status == lib.TS_ERR_INVALID_ARG
    want, first_bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert first_bad >= 0
    assert np.array_equal(dbuf.cpu().numpy(), want)
    # the status word was cleared: a valid call afterwards succeeds
    good = torch.tensor([0, 500, 1000], dtype=torch.int64, device="cuda")
    lib.ts_copy_i16_rows(sbuf, dbuf, good, sched=sched)
    lib.ts_sync_and_check()
    assert torch.equal(dbuf, sbuf)


def test_rows_same_buffer_rewrites_itself(lib):
    offsets, n = _jagged(81, 50, 900)
    t = torch.from_numpy(synth.int16_uniform(82, n)).cuda()
    before = t.clone()
    lib.ts_copy_i16_rows(t, t, torch.from_numpy(offsets).cuda(), sched="clc")
    lib.ts_sync_and_check()
    assert torch.equal(t, before)


@pytest.mark.slow
@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_full_workload_bit_exact(lib, sched):
    src_h, offsets = synth.ROWS.inputs()
    n = src_h.size
    src = torch.from_numpy(src_h).cuda()
    dst = torch.zeros_like(src)
    trace = torch.zeros(2 * synth.ROWS.rows, dtype=torch.int64, device="cuda")
    lib.ts_copy_i16_rows(src, dst, torch.from_numpy(offsets).cuda(), sched=sched, trace=trace)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)  # the rows tile [0, n): the copy covers every element
    want, bad = oracle.copy_rows_i16(src_h, np.zeros(n, np.int16), offsets)
    idx = np.random.default_rng(1).integers(0, n, 1 << 16)
    assert bad == -1 and np.array_equal(dst[torch.as_tensor(idx, device="cuda")].cpu().numpy(), want[idx])
    assert torch.equal(trace.view(-1, 2)[:, 0].cpu(), torch.ones(synth.ROWS.rows, dtype=torch.int64))


# ------------------------------------------------------------ chunked mode
# Rows cut into work tiles of at most `chunk` elements (a planning kernel maps
# tiles to rows); the result is the same row copy.


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("chunk", [1, 7, 16, 100, 4096, 1 << 20])
def test_rows_chunked_random_jagged(lib, sched, chunk):
    offsets, n = _jagged(91 + chunk, 200 if chunk > 1 else 40, 3000 if chunk > 1 else 300)
    src = synth.int16_uniform(92, n)
    dst0 = synth.int16_uniform(93, n)
    got = _run(lib, src, dst0, offsets, sched, chunk=chunk)
    want, bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert bad == -1 and np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (8, 0), (3, 3), (1, 6)])
def test_rows_chunked_vector_paths(lib, sched, src_off, dst_off):
    offsets, n = _jagged(95, 120, 5000, lead=3, trail=9)
    src = synth.int16_uniform(96, n)
    dst0 = synth.int16_uniform(97, n)
    got = _run(lib, src, dst0, offsets, sched, src_off=src_off, dst_off=dst_off, chunk=33)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_chunked_tiles_visited_once_and_extra_tiles_skipped(lib, sched):
    offsets, n = _jagged(101, 150, 2000)
    rows = offsets.size - 1
    chunk = 250
    info = lib.ts_copy_rows_launch_info(n, rows, sched, chunk=chunk)
    tiles = info["num_tiles"]
    assert tiles == rows + -(-n // chunk) and info["workspace_bytes"] > 0
    pieces = int(sum(-(-(int(offsets[r + 1]) - int(offsets[r])) // chunk) for r in range(rows)))
    assert pieces < tiles  # some tiles are past the last piece
    src = synth.int16_uniform(102, n)
    dst0 = synth.int16_uniform(103, n)
    trace = torch.zeros(2 * tiles, dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, chunk=chunk, trace=trace)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)
    tr = trace.view(tiles, 2).cpu().numpy()
    if sched == "static":
        assert np.array_equal(tr[:, 0], np.ones(tiles))
        assert np.array_equal(tr[:, 1], oracle.static_owner(tiles, info["grid_ctas"]))
    elif sched == "nonpersistent":  # one CTA per tile, each on its own tile
        assert np.array_equal(tr[:, 0], np.ones(tiles)) and np.array_equal(tr[:, 1], np.arange(tiles))
    else:
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("count", [0, 1, 77, 200])
def test_rows_chunked_skip_mask_and_device_count(lib, sched, count):
    offsets, n = _jagged(111, 200, 1500)
    src = synth.int16_uniform(112, n)
    dst0 = synth.int16_uniform(113, n)
    skip = (synth.splitmix64(114, 200) % np.uint64(4) == 0).astype(np.uint8)
    rd = torch.tensor([count], dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, chunk=64, rows_device=rd, skip_rows=torch.from_numpy(skip).cuda())
    want, _ = oracle.copy_rows_i16(src, dst0, offsets, rows=count, skip=skip)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_chunked_bad_bounds_reported(lib, sched):
    n = 1000
    offsets = np.array([0, 100, 300, 600, 1200], dtype=np.int64)  # row 3 runs past n
    src = synth.int16_uniform(121, n)
    dst0 = synth.int16_uniform(122, n)
    sbuf = torch.from_numpy(src).cuda()
    dbuf = torch.from_numpy(dst0.copy()).cuda()
    lib.ts_copy_i16_rows(sbuf, dbuf, torch.from_numpy(offsets).cuda(), sched=sched, chunk=64)
    with pytest.raises(lib.TsError) as ei:
        lib.ts_sync_and_check()
    assert ei.value.status == lib.TS_ERR_INVALID_ARG and "bounds" in ei.value.detail
    want, first_bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert first_bad == 3 and np.array_equal(dbuf.cpu().numpy(), want)


def test_rows_chunked_overlapping_rows_need_more_tiles(lib):
    # rows 0 and 3 are both [0, n) (row 2, which runs backwards, is skipped):
    # 20 pieces, above the default budget of rows + ceil(n / chunk) = 14 tiles
    n, chunk = 1000, 100
    src = torch.from_numpy(synth.int16_uniform(131, n)).cuda()
    off = torch.tensor([0, n, n, 0, n], dtype=torch.int64, device="cuda")
    skip = torch.tensor([0, 0, 1, 0], dtype=torch.uint8, device="cuda")
    dst = torch.zeros(n, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16_rows(src, dst, off, sched="clc", chunk=chunk, skip_rows=skip)
    with pytest.raises(lib.TsError) as ei:
        lib.ts_sync_and_check()
    assert ei.value.status == lib.TS_ERR_INVALID_ARG and "pieces" in ei.value.detail
    # with enough tiles every piece is copied (twice, for the overlap)
    dst = torch.zeros(n, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16_rows(src, dst, off, sched="clc", chunk=chunk, skip_rows=skip, tiles=20)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)


def test_rows_chunked_needs_a_workspace(lib):
    src = torch.zeros(100, dtype=torch.int16, device="cuda")
    dst = torch.zeros(100, dtype=torch.int16, device="cuda")
    off = torch.tensor([0, 100], dtype=torch.int64, device="cuda")
    assert lib.ts_copy_i16_rows_ptr(src.data_ptr(), dst.data_ptr(), 100, off.data_ptr(), 1,
                                    chunk=10) == lib.TS_ERR_INVALID_ARG
    assert "workspace" in lib.ts_last_error_detail()


@pytest.mark.slow
@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_full_workload_chunked_bit_exact(lib, sched):
    src_h, offsets = synth.ROWS.inputs()
    src = torch.from_numpy(src_h).cuda()
    dst = torch.zeros_like(src)
    lib.ts_copy_i16_rows(src, dst, torch.from_numpy(offsets).cuda(), sched=sched, chunk=32768)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)  # the rows tile [0, n)


# ------------------------------------------------------------- packed mode
# The copied rows laid end to end, every work tile `chunk` of their elements:
# short rows share a tile (in batches of one row per thread), long rows span
# several; the result is the same row copy.


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("chunk", [1, 7, 16, 100, 4096, 1 << 20])
@pytest.mark.parametrize("threads", [128, 512])
def test_rows_packed_random_jagged(lib, sched, chunk, threads):
    offsets, n = _jagged(141 + chunk, 200 if chunk > 1 else 40, 3000 if chunk > 1 else 300)
    src = synth.int16_uniform(142, n)
    dst0 = synth.int16_uniform(143, n)
    got = _run(lib, src, dst0, offsets, sched, chunk=chunk, pack=1, threads=threads)
    want, bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert bad == -1 and np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("threads", [128, 1024])
def test_rows_packed_many_tiny_rows_per_tile(lib, sched, threads):
    # 6000 rows of 0-5 elements: a 4096-element tile holds well over a batch of rows
    offsets, n = _jagged(151, 6000, 5)
    src = synth.int16_uniform(152, n)
    dst0 = synth.int16_uniform(153, n)
    got = _run(lib, src, dst0, offsets, sched, chunk=4096, pack=1, threads=threads)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (8, 0), (3, 3), (1, 6)])
def test_rows_packed_vector_paths(lib, sched, src_off, dst_off):
    offsets, n = _jagged(155, 300, 700, lead=3, trail=9)
    src = synth.int16_uniform(156, n)
    dst0 = synth.int16_uniform(157, n)
    got = _run(lib, src, dst0, offsets, sched, src_off=src_off, dst_off=dst_off, chunk=1000, pack=1)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_packed_tiles_visited_once_and_extra_tiles_skipped(lib, sched):
    offsets, n = _jagged(161, 150, 2000, lead=700, trail=900)
    rows = offsets.size - 1
    chunk = 250
    info = lib.ts_copy_rows_launch_info(n, rows, sched, chunk=chunk, pack=1)
    tiles = info["num_tiles"]
    assert tiles == -(-n // chunk) and info["workspace_bytes"] > 0
    total = int(offsets[-1] - offsets[0])
    assert -(-total // chunk) < tiles  # some tiles are past the last packed element
    src = synth.int16_uniform(162, n)
    dst0 = synth.int16_uniform(163, n)
    trace = torch.zeros(2 * tiles, dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, chunk=chunk, pack=1, trace=trace)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)
    tr = trace.view(tiles, 2).cpu().numpy()
    if sched == "static":
        assert np.array_equal(tr[:, 0], np.ones(tiles))
        assert np.array_equal(tr[:, 1], oracle.static_owner(tiles, info["grid_ctas"]))
    elif sched == "nonpersistent":  # one CTA per tile, each on its own tile
        assert np.array_equal(tr[:, 0], np.ones(tiles)) and np.array_equal(tr[:, 1], np.arange(tiles))
    else:
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("count", [0, 1, 77, 200])
def test_rows_packed_skip_mask_and_device_count(lib, sched, count):
    offsets, n = _jagged(171, 200, 1500)
    src = synth.int16_uniform(172, n)
    dst0 = synth.int16_uniform(173, n)
    skip = (synth.splitmix64(174, 200) % np.uint64(4) == 0).astype(np.uint8)
    rd = torch.tensor([count], dtype=torch.int64, device="cuda")
    got = _run(lib, src, dst0, offsets, sched, chunk=300, pack=1, rows_device=rd,
               skip_rows=torch.from_numpy(skip).cuda())
    want, _ = oracle.copy_rows_i16(src, dst0, offsets, rows=count, skip=skip)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_packed_bad_bounds_reported(lib, sched):
    n = 1000
    offsets = np.array([0, 100, 300, 600, 1200], dtype=np.int64)  # row 3 runs past n
    src = synth.int16_uniform(181, n)
    dst0 = synth.int16_uniform(182, n)
    sbuf = torch.from_numpy(src).cuda()
    dbuf = torch.from_numpy(dst0.copy()).cuda()
    lib.ts_copy_i16_rows(sbuf, dbuf, torch.from_numpy(offsets).cuda(), sched=sched, chunk=64, pack=1)
    with pytest.raises(lib.TsError) as ei:
        lib.ts_sync_and_check()
    assert ei.value.status == lib.TS_ERR_INVALID_ARG and "bounds" in ei.value.detail
    want, first_bad = oracle.copy_rows_i16(src, dst0, offsets)
    assert first_bad == 3 and np.array_equal(dbuf.cpu().numpy(), want)


def test_rows_packed_overlapping_rows_need_more_tiles(lib):
    # rows 0 and 3 are both [0, n) (row 2, which runs backwards, is skipped):
    # 2n packed elements need 20 tiles, above the default ceil(n / chunk) = 10
    n, chunk = 1000, 100
    src = torch.from_numpy(synth.int16_uniform(191, n)).cuda()
    off = torch.tensor([0, n, n, 0, n], dtype=torch.int64, device="cuda")
    skip = torch.tensor([0, 0, 1, 0], dtype=torch.uint8, device="cuda")
    dst = torch.zeros(n, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16_rows(src, dst, off, sched="clc", chunk=chunk, pack=1, skip_rows=skip)
    with pytest.raises(lib.TsError) as ei:
        lib.ts_sync_and_check()
    assert ei.value.status == lib.TS_ERR_INVALID_ARG and "pieces" in ei.value.detail
    dst = torch.zeros(n, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16_rows(src, dst, off, sched="clc", chunk=chunk, pack=1, skip_rows=skip, tiles=20)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)


@pytest.mark.slow
@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_rows_full_workload_packed_bit_exact(lib, sched):
    src_h, offsets = synth.ROWS.inputs()
    src = torch.from_numpy(src_h).cuda()
    dst = torch.zeros_like(src)
    lib.ts_copy_i16_rows(src, dst, torch.from_numpy(offsets).cuda(), sched=sched, chunk=32768, pack=1)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)  # the rows tile [0, n)


# Every shift between src and dst within a 16-byte vector, whole rows and
# chunked pieces: rows whose src and dst differ modulo 16 bytes join each dst
# vector from two source vectors (which may lie outside the row, never outside
# src).
@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
@pytest.mark.parametrize("chunk", [0, 333])
@pytest.mark.parametrize("dst_off", range(8))
def test_rows_every_relative_alignment(lib, sched, chunk, dst_off):
    offsets, n = _jagged(1601, 90, 1200, lead=1, trail=2)
    src = synth.int16_uniform(1602, n)
    dst0 = synth.int16_uniform(1603, n)
    got = _run(lib, src, dst0, offsets, sched, src_off=3, dst_off=dst_off, chunk=chunk)
    want, _ = oracle.copy_rows_i16(src, dst0, offsets)
    assert np.array_equal(got, want)
