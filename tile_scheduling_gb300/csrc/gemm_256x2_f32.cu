// GEMM variant: BN = 256, 2-CTA worker, f32 output.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT(variant_256_2_f32, 256, 2, OUT_F32)
