// Protocol-logging instantiations (a test instrument): the 1-CTA 128x128 fp32 tile with four
// epilogue warps in the FusedMerge and the Merge barrier layouts and with eight, and the 1-CTA
// 128x256 fp32 tile with sixteen (the short-K epilogue).
#include "gemm_launch.cuh"

TS_GEMM_VARIANT_LOG(variant_128_1_f32_e4_log, 128, 1, OUT_F32, 4, 0, 1)
TS_GEMM_VARIANT_LOG(variant_128_1_f32_e4m_log, 128, 1, OUT_F32, 4, 1, 1)
TS_GEMM_VARIANT_LOG(variant_128_1_f32_e8_log, 128, 1, OUT_F32, 8, 0, 1)
