// Protocol-logging instantiation (a test instrument): the 1-CTA 128x256 fp32 tile with sixteen
// epilogue warps (the short-K epilogue).
#include "gemm_launch.cuh"

TS_GEMM_VARIANT_LOG(variant_256_1_f32_e16_log, 256, 1, OUT_F32, 16, 0, 1)
