// GEMM variant: BN = 256, 2-CTA worker, bf16 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_2_bf16, 256, 2, OUT_BF16)
