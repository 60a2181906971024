// Host-side helpers shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tsgemm.h"
#include "gemm_params.h"

namespace ts {

// Record a thread-local error message and return `s`.
ts_status fail(ts_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// Map a CUDA runtime error to TS_ERR_CUDA with context.
ts_status cuda_fail(cudaError_t e, const char *what);

int current_device();
int device_sms(int dev);
int device_smem_optin(int dev);
// Device address of the library-owned status word on the current device.
unsigned long long *device_status_word(ts_status *err);

// One compiled GEMM variant (tile shape, cluster size, output type).
struct GemmLaunch {
    CUtensorMap a, b, d;
    GemmParams p;
    int grid;
    cudaStream_t stream;
};

struct GemmVariant {
    int bn, cg, out, epi_warps, merge, log, stages, smem_bytes;
    ts_gemm_protocol protocol;  // barrier layout and arrival counts of this variant
    cudaError_t (*launch)(const GemmLaunch &);
    // Workers (CTAs, or 2-CTA clusters) that can be resident at once.
    cudaError_t (*max_workers)(int *);
};

// log = 1: the protocol-logging instantiation (a test instrument; few shapes have one).
const GemmVariant *find_variant(int bn, int cg, int out, int epi_warps, int merge, int log = 0);

}  // namespace ts
