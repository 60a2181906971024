// GEMM variant: BN = 128, 1-CTA worker, bf16 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_128_1_bf16, 128, 1, OUT_BF16)
