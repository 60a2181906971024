// Protocol-logging instantiation (a test instrument): the 2-CTA 256x256 fp32 tile with four
// epilogue warps per CTA.
#include "gemm_launch.cuh"

TS_GEMM_VARIANT_LOG(variant_256_2_f32_e4_log, 256, 2, OUT_F32, 4, 0, 1)
