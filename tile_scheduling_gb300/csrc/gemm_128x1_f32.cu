// GEMM variant: BN = 128, 1-CTA worker, f32 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_128_1_f32, 128, 1, OUT_F32)
