// GEMM variant: BN = 256, 1-CTA worker, bf16 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_1_bf16, 256, 1, OUT_BF16)
