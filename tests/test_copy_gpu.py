"""GPU parity of ts_copy_i16 against the oracle's scalar copy: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 4096 + 3, 1 << 20, (1 << 20) + 5])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (3, 3), (1, 5), (8, 0)])
def test_copy_sizes_and_alignments(lib, n, src_off, dst_off):
    src_h = synth.int16_uniform(500 + n, n)
    sbuf = torch.zeros(n + 16, dtype=torch.int16, device="cuda")
    dbuf = torch.full((n + 16,), -1, dtype=torch.int16, device="cuda")
    sbuf[src_off:src_off + n] = torch.from_numpy(src_h).cuda()
    lib.ts_copy_i16(sbuf[src_off:src_off + n], dbuf[dst_off:dst_off + n])
    lib.ts_sync_and_check()
    d = dbuf.cpu().numpy()
    assert np.array_equal(d[dst_off:dst_off + n], oracle.copy_i16(src_h))
    assert np.all(d[:dst_off] == -1) and np.all(d[dst_off + n:] == -1)


# Sizes of many rounds of the grid-stride loop, with a partial last round and
# a head and tail of single elements (odd offsets and sizes), on the 32-byte,
# 16-byte and element-wise paths.
@pytest.mark.parametrize("n,src_off,dst_off", [((1 << 23) + 3, 3, 3), (5 * (1 << 22) + 11, 0, 8),
                                               (3 * (1 << 21) + 1, 1, 5), (1 << 24, 0, 0)])
def test_copy_many_chunks_per_cta(lib, n, src_off, dst_off):
    src_h = synth.int16_uniform(900 + n, n)
    sbuf = torch.zeros(n + 16, dtype=torch.int16, device="cuda")
    dbuf = torch.full((n + 16,), -1, dtype=torch.int16, device="cuda")
    sbuf[src_off:src_off + n] = torch.from_numpy(src_h).cuda()
    lib.ts_copy_i16(sbuf[src_off:src_off + n], dbuf[dst_off:dst_off + n])
    lib.ts_sync_and_check()
    d = dbuf.cpu().numpy()
    assert np.array_equal(d[dst_off:dst_off + n], oracle.copy_i16(src_h))
    assert np.all(d[:dst_off] == -1) and np.all(d[dst_off + n:] == -1)


# Every pair of element offsets within a 16-byte vector: the 32- and 16-byte
# vector paths, and for offsets that differ modulo 8 elements the shifted path
# (aligned destination vectors joined from two source vectors), all seven shifts.
@pytest.mark.parametrize("n", [37, 4096 + 5, (1 << 20) + 3])
def test_copy_every_relative_alignment(lib, n):
    src_h = synth.int16_uniform(1300 + n, n)
    sbuf = torch.zeros(n + 16, dtype=torch.int16, device="cuda")
    dbuf = torch.full((n + 16,), -1, dtype=torch.int16, device="cuda")
    want = oracle.copy_i16(src_h)
    for src_off in range(8):
        sbuf.zero_()
        sbuf[src_off:src_off + n] = torch.from_numpy(src_h).cuda()
        for dst_off in range(8):
            dbuf.fill_(-1)
            lib.ts_copy_i16(sbuf[src_off:src_off + n], dbuf[dst_off:dst_off + n])
            lib.ts_sync_and_check()
            d = dbuf.cpu().numpy()
            assert np.array_equal(d[dst_off:dst_off + n], want), (src_off, dst_off)
            assert np.all(d[:dst_off] == -1) and np.all(d[dst_off + n:] == -1), (src_off, dst_off)


@pytest.mark.slow
def test_copy_full_size_bit_exact(lib):
    n = synth.COPY_N
    src_h = synth.int16_uniform(synth.COPY_SEED, n)
    src = torch.from_numpy(src_h).cuda()
    dst = torch.empty_like(src)
    lib.ts_copy_i16(src, dst)
    lib.ts_sync_and_check()
    assert torch.equal(dst, src)  # device-side equality, then the oracle on a sample
    idx = np.random.default_rng(0).integers(0, n, 1 << 16)
    assert np.array_equal(dst[torch.as_tensor(idx, device="cuda")].cpu().numpy(), oracle.copy_i16(src_h)[idx])


def test_copy_same_pointer_is_noop(lib):
    t = torch.arange(100, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16(t, t)
    lib.ts_sync_and_check()
    assert torch.equal(t, torch.arange(100, dtype=torch.int16, device="cuda"))
