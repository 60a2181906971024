// GEMM variant: BN = 256, 1-CTA worker, f32 output; 4, 8 and 16 epilogue warps; the Merge
// barrier layout with 4.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_1_f32_e4, 256, 1, OUT_F32, 4, 0)
TS_GEMM_VARIANT(variant_256_1_f32_e4m, 256, 1, OUT_F32, 4, 1)
TS_GEMM_VARIANT(variant_256_1_f32_e8, 256, 1, OUT_F32, 8, 0)
TS_GEMM_VARIANT(variant_256_1_f32_e16, 256, 1, OUT_F32, 16, 0)
