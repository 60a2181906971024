// GEMM variant: BN = 256, 1-CTA worker, f32 output; 4 and 8 epilogue warps.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_1_f32_e4, 256, 1, OUT_F32, 4)
TS_GEMM_VARIANT(variant_256_1_f32_e8, 256, 1, OUT_F32, 8)
