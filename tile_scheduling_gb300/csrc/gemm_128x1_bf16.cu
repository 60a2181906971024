// GEMM variant: BN = 128, 1-CTA worker, bf16 output; 4 and 8 epilogue warps; the Merge
// barrier layout with 4.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_128_1_bf16_e4, 128, 1, OUT_BF16, 4, 0)
TS_GEMM_VARIANT(variant_128_1_bf16_e4m, 128, 1, OUT_BF16, 4, 1)
TS_GEMM_VARIANT(variant_128_1_bf16_e8, 128, 1, OUT_BF16, 8, 0)
