"""Helpers shared by the GPU parity tests (tolerances, transfers)."""
import numpy as np
import torch

import oracle

# Error bound for random inputs: the tensor core's fp32 accumulation order is
# not specified, so bit equality is not expected; instead
#   |D - ref| <= 2^-10 * sum_k |a_ik b_jk|                 (fp32 output)
#   |D - ref| <= 2^-10 * sum_k |a_ik b_jk| + 2^-8 |ref|    (bf16 output: one more rounding)
FP32_REL = 2.0 ** -10
BF16_ROUND = 2.0 ** -8


def to_device_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f64(bf16_bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def bound(ref: np.ndarray, absprod: np.ndarray, out_dtype) -> np.ndarray:
    b = FP32_REL * absprod
    if out_dtype == torch.bfloat16:
        b = b + BF16_ROUND * np.abs(ref)
    return b


def assert_within_bound(got: np.ndarray, ref: np.ndarray, absprod: np.ndarray, out_dtype, what=""):
    err = np.abs(got - ref)
    lim = bound(ref, absprod, out_dtype)
    bad = ~(err <= lim)  # NaN counts as a violation
    if bad.any():
        idx = np.argwhere(bad)[:5]
        rows = [(tuple(i), float(got[tuple(i)]), float(ref[tuple(i)]), float(lim[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} entries outside the bound; first (idx, got, ref, bound): {rows}")


def assert_bit_exact(D: torch.Tensor, ref: np.ndarray, what=""):
    """Exact comparison for integer-valued results: fp32 equal, bf16 equal to the RNE of the exact value."""
    if D.dtype == torch.bfloat16:
        want = oracle.bf16_rne(ref)
        got = bf16_bits(D)
    else:
        want = ref.astype(np.float32)
        got = D.detach().cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)[:5]
        raise AssertionError(f"{what}: {int((got != want).sum())} mismatches; first {bad.tolist()}")


# Kernel layouts the parametrised GPU tests run: (epilogue warps, barrier
# layout), 0 = FusedMerge (A and B on one full barrier per stage), 1 = Merge
# (separate producers and full barriers for A and B; four epilogue warps).
LAYOUTS = [(4, 0), (8, 0), (4, 1)]


def tile_layouts(tiles):
    """(tile, epilogue warps, barrier layout) cases: every layout on every tile,
    and sixteen epilogue warps on the 256-column tiles (the only ones built)."""
    return [(t, ew, mg) for t in tiles for ew, mg in LAYOUTS + ([(16, 0)] if t != "128x128" else [])]
