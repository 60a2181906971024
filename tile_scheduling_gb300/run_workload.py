"""Run one named workload a few times (for profilers such as ncu); prints nothing but a summary line.

Usage: python -m tile_scheduling_gb300.run_workload {gemm256,gemm4096,gemm8192,ragged,smallk,grouped,copy,rows}
           [--launches N] [--sched static|clc|nonpersistent] [--tile auto|128x128|128x256|256x256]
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

import tile_scheduling_gb300 as ts  # noqa: E402

GEMMS = {"gemm256": synth.GEMM_256, "gemm4096": synth.GEMM_4096, "gemm8192": synth.GEMM_8192,
         "ragged": synth.GEMM_RAGGED, "smallk": synth.GEMM_SMALLK}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", choices=sorted(GEMMS) + ["grouped", "copy", "rows"])
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--sched", default=None, choices=["static", "clc", "nonpersistent"])
    ap.add_argument("--tile", default=None)
    ap.add_argument("--chunk", type=int, default=0, help="rows: elements per work tile (0: one tile per row)")
    ap.add_argument("--pack", type=int, default=0, choices=[0, 1], help="rows: lay the rows end to end (with --chunk)")
    ap.add_argument("--merge", type=int, default=0, choices=[0, 1], help="GEMM: the Merge barrier layout")
    a = ap.parse_args(argv)
    if a.workload == "copy":
        src = torch.from_numpy(synth.int16_uniform(synth.COPY_SEED, synth.COPY_N)).cuda()
        dst = torch.empty_like(src)
        for _ in range(a.launches):
            ts.ts_copy_i16(src, dst)
        ts.ts_sync_and_check()
        print(f"copy n={synth.COPY_N} x{a.launches} ok")
        return 0
    if a.workload == "rows":
        src_h, off_h = synth.ROWS.inputs()
        src = torch.from_numpy(src_h).cuda()
        dst = torch.empty_like(src)
        off = torch.from_numpy(off_h).cuda()
        sched = a.sched or "clc"
        ws = None
        if a.chunk:
            need = ts.ts_copy_rows_launch_info(src.numel(), synth.ROWS.rows, sched, chunk=a.chunk,
                                               pack=a.pack)["workspace_bytes"]
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        for _ in range(a.launches):
            ts.ts_copy_i16_rows(src, dst, off, sched=sched, chunk=a.chunk, workspace=ws, pack=a.pack)
        ts.ts_sync_and_check()
        print(f"{synth.ROWS.name}: {sched} chunk {a.chunk} pack {a.pack} x{a.launches} ok")
        return 0
    if a.workload == "grouped":
        w = synth.GROUPED
        off = w.k_offsets()
        A_bits, B_bits = w.inputs()
        A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
        B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
        D = torch.empty((w.groups, w.M, w.N), dtype=torch.bfloat16, device="cuda")
        sched = a.sched or "clc"
        tile = a.tile or "auto"
        for _ in range(a.launches):
            ts.ts_gemm_bf16_grouped(A, B, D, off, sched=sched, tile=tile)
        ts.ts_sync_and_check()
        print(f"{w.name}: {sched} {tile} x{a.launches} ok")
        return 0
    w = GEMMS[a.workload]
    A_bits, B_bits = w.inputs()
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.float32 if w.out == "f32" else torch.bfloat16
    D = torch.empty((w.M, w.N), dtype=out, device="cuda")
    sched = a.sched or w.sched[-1]
    tile = a.tile or w.tile
    for _ in range(a.launches):
        ts.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile, merge=a.merge)
    ts.ts_sync_and_check()
    print(f"{w.name}: {sched} {tile} merge {a.merge} x{a.launches} ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
