// GEMM variant: BN = 256, 1-CTA worker, f32 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_1_f32, 256, 1, OUT_F32)
