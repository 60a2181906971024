// GEMM variant: BN = 128, 1-CTA worker, f32 output; 4 and 8 epilogue warps; the Merge
// barrier layout with 4.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_128_1_f32_e4, 128, 1, OUT_F32, 4, 0)
TS_GEMM_VARIANT(variant_128_1_f32_e4m, 128, 1, OUT_F32, 4, 1)
TS_GEMM_VARIANT(variant_128_1_f32_e8, 128, 1, OUT_F32, 8, 0)
