// GEMM variant: BN = 256, 2-CTA worker, bf16 output; 4, 8 and 16 epilogue warps; the Merge
// barrier layout with 4.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_2_bf16_e4, 256, 2, OUT_BF16, 4, 0)
TS_GEMM_VARIANT(variant_256_2_bf16_e4m, 256, 2, OUT_BF16, 4, 1)
TS_GEMM_VARIANT(variant_256_2_bf16_e8, 256, 2, OUT_BF16, 8, 0)
TS_GEMM_VARIANT(variant_256_2_bf16_e16, 256, 2, OUT_BF16, 16, 0)
