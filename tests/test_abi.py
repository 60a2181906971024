"""The C-ABI library loads and exports every entry point its header declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsgemm.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_api():
    names = _declared()
    for n in ("ts_gemm_bf16", "ts_gemm_bf16_ex", "ts_copy_i16", "ts_sync_and_check"):
        assert n in names


def test_library_exports_every_declared_symbol(ts):
    lib = ctypes.CDLL(ts.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_names_match_header(ts):
    for n in _declared():
        assert hasattr(ts, n), f"binding lacks {n}"


def test_status_strings(ts):
    assert ts.ts_status_string(ts.TS_OK) == "TS_OK"
    assert ts.ts_status_string(ts.TS_ERR_TIMEOUT) == "TS_ERR_TIMEOUT"
    assert ts.ts_status_string(99) == "TS_ERR_UNKNOWN"


def test_argument_errors_need_no_gpu(ts):
    # rejected before any CUDA call
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, -1, 4, 4, ts.TS_OUT_F32, stream=0) == ts.TS_ERR_INVALID_ARG
    assert "sizes" in ts.ts_last_error_detail()
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 1 << 31, ts.TS_OUT_F32, stream=0) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 4, 7, stream=0) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 4, ts.TS_OUT_F32, sched=5, stream=0) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 4, ts.TS_OUT_F32, sched=3, stream=0) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 4, ts.TS_OUT_F32, stream=0, tile=9) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 8, ts.TS_OUT_F32, stream=0, lda=4) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 8, ts.TS_OUT_F32, stream=0, epi_warps=6) == ts.TS_ERR_INVALID_ARG
    assert "epi_warps" in ts.ts_last_error_detail()
    assert ts._lib.ts_gemm_bf16_host(None, None, None, None, None, None, 4, 4, 8, ts.TS_OUT_F32, 0, None,
                                     None) == ts.TS_ERR_INVALID_ARG  # NULL buffers, before any CUDA call
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 8, ts.TS_OUT_F32, stream=0, merge=2) == ts.TS_ERR_INVALID_ARG
    assert "merge" in ts.ts_last_error_detail()
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 8, ts.TS_OUT_F32, stream=0, inputs_ready=2) == ts.TS_ERR_INVALID_ARG
    assert "inputs_ready" in ts.ts_last_error_detail()
    # the Merge layout's B producer and the Fork row-sum task would both need warp 3
    o = ts._opts(merge=1)
    o.row_sums = 4096
    assert ts._lib.ts_gemm_bf16_ex(None, None, None, 4, 4, 8, ts.TS_OUT_F32, 0, ctypes.byref(o),
                                   None) == ts.TS_ERR_UNSUPPORTED
    assert ts.ts_gemm_bf16_ptr(0, 0, 0, 4, 4, 8, ts.TS_OUT_F32, stream=0, merge=1,
                               epi_warps=8) == ts.TS_ERR_UNSUPPORTED
    assert ts.ts_copy_i16_ptr(0, 0, -3, stream=0) == ts.TS_ERR_INVALID_ARG
    assert ts.ts_copy_i16_ptr(0, 0, 0, stream=0) == ts.TS_OK
    assert ts.ts_copy_i16_ptr(4096, 4100, 8, stream=0) == ts.TS_ERR_INVALID_ARG  # overlap
    assert ts.ts_copy_i16_ptr(4096, 4096, 8, stream=0) == ts.TS_OK  # src == dst is a no-op


def test_header_is_plain_c():
    # compiles as C99 with no CUDA or torch headers on the include path
    import subprocess
    import tempfile

    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        with open(c, "w") as f:
            f.write('#include "tsgemm.h"\nint main(void){ ts_gemm_opts o = {0}; (void)o; return 0; }\n')
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c", c,
                            "-o", os.path.join(d, "t.o")], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_row_copy_argument_errors_need_no_gpu(ts):
    E = ts.TS_ERR_INVALID_ARG
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, -1, 64, 0, stream=0) == E  # n < 0
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, -2, stream=0) == E  # rows < 0
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, 1, sched=5, stream=0) == E
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, 4, tiles=3, stream=0) == E  # tiles below rows
    assert "tiles" in ts.ts_last_error_detail()
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, 1, threads=100, stream=0) == E
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 0, 1, stream=0) == E  # offsets NULL
    assert ts.ts_copy_i16_rows_ptr(0, 8192, 8, 64, 1, stream=0) == E  # src NULL
    assert ts.ts_copy_i16_rows_ptr(4096, 4100, 8, 64, 1, stream=0) == E  # overlap
    assert ts.ts_copy_i16_rows_ptr(4097, 8192, 8, 64, 1, stream=0) == E  # odd address
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, 1, timeout_s=-1.0, stream=0) == E
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 8, 64, 1, chunk=-1, stream=0) == E
    # chunked: tiles may not be below rows + ceil(n / chunk) = 2 + 3
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 9, 64, 2, chunk=4, tiles=4, stream=0) == E
    assert "ceil(n / chunk)" in ts.ts_last_error_detail()
    # packed: a chunk in [1, 2^30] is required, pack is 0 or 1, and tiles may not be
    # below ceil(n / chunk) = 3 (the rows do not count)
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 9, 64, 2, pack=1, stream=0) == E
    assert "pack" in ts.ts_last_error_detail()
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 9, 64, 2, chunk=(1 << 30) + 1, pack=1, stream=0) == E
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 9, 64, 2, chunk=4, pack=2, stream=0) == E
    assert ts.ts_copy_i16_rows_ptr(4096, 8192, 9, 64, 2, chunk=4, pack=1, tiles=2, stream=0) == E
    assert "ceil(n / chunk)" in ts.ts_last_error_detail()
    # an empty queue launches nothing
    assert ts.ts_copy_i16_rows_ptr(0, 0, 0, 0, 0, stream=0) == ts.TS_OK


def test_binding_structs_match_the_header_layout(ts):
    # the ctypes mirrors of the option and info structs have the C layout (size and every offset)
    import subprocess
    import tempfile

    structs = {"ts_gemm_opts": ts.GemmOpts, "ts_launch_info": ts.LaunchInfo, "ts_rows_opts": ts.RowsOpts,
               "ts_gemm_protocol": ts.GemmProtocol}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tsgemm.h"', 'int main(void) {']
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        with open(c, "w") as fh:
            fh.write("\n".join(lines))
        exe = os.path.join(d, "layout")
        r = subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(line.split()[:2]): int(line.split()[2]) for line in out if line}
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, f"{cname}.{f}"
