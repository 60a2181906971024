// Host launcher for one instantiation of the GEMM kernel.  Each instance
// translation unit includes this file and expands TS_GEMM_VARIANT once, so the
// variants compile in parallel.
#pragma once
#include <atomic>

#include "common.h"
#include "gemm_kernel.cuh"

namespace ts {
// Internal linkage: each variant translation unit has its own instance, and
// the per-device "prepared" flag below is not merged with a same-named one in
// another copy of this library loaded into the process (function-local
// statics of templates otherwise become process-unique symbols).
namespace {

template <int BN, int CG, int OUT, int EW, int MG, int LOG>
struct GemmInstance {
    using C = GemmCfg<BN, CG, OUT, EW, MG, LOG>;

    // cudaFuncSetAttribute once per device (bit per device ordinal).
    static cudaError_t prepare() {
        static std::atomic<uint64_t> done{0};
        const int dev = current_device();
        const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
        if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        cudaError_t e = cudaFuncSetAttribute(gemm_ws_kernel<BN, CG, OUT, EW, MG, LOG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }

    static constexpr ts_gemm_protocol protocol() {
        return ts_gemm_protocol{CG,
                                C::STAGES,
                                C::TX_BYTES,
                                C::FULL_ARRIVALS,
                                C::EMPTY_ARRIVALS,
                                C::ACCUMULATORS,
                                C::TFULL_ARRIVALS,
                                C::TEMPTY_ARRIVALS,
                                kMaxClcDepth,
                                C::CLC_FULL_ARRIVALS,
                                C::CLC_CONSUMERS,
                                C::CLC_RESPONSE_BYTES,
                                C::EPI_WARPS,
                                C::A_BYTES + C::B_BYTES,
                                C::AUX_EMPTY_ARRIVALS,
                                C::MERGE,
                                C::A_BYTES};
    }

    static cudaError_t launch(const GemmLaunch &L) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(L.grid), 1, 1);
        cfg.blockDim = dim3(C::THREADS, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = L.stream;
        // Programmatic stream serialization: the kernel's prologue may overlap the
        // previous kernel in the stream; the kernel waits for it (griddepcontrol)
        // before its first global memory access.
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (CG == 2) {
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = 2;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        return cudaLaunchKernelEx(&cfg, gemm_ws_kernel<BN, CG, OUT, EW, MG, LOG>, L.a, L.b, L.d, L.p);
    }

    static cudaError_t max_workers(int *out) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        if (CG == 1) {
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_ws_kernel<BN, CG, OUT, EW, MG, LOG>, C::THREADS,
                                                              C::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            *out = per_sm * device_sms(current_device());
            return cudaSuccess;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        cfg.blockDim = dim3(C::THREADS, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(gemm_ws_kernel<BN, CG, OUT, EW, MG, LOG>),
                                           &cfg);
        if (e != cudaSuccess) return e;
        *out = clusters;
        return cudaSuccess;
    }
};

}  // namespace
}  // namespace ts

#define TS_GEMM_VARIANT_LOG(NAME, BN, CG, OUT, EW, MG, LOG)                                                \
    namespace ts {                                                                                         \
    extern const GemmVariant NAME;                                                                         \
    const GemmVariant NAME = {BN,                                                                          \
                              CG,                                                                          \
                              OUT,                                                                         \
                              EW,                                                                          \
                              MG,                                                                          \
                              LOG,                                                                         \
                              GemmCfg<BN, CG, OUT, EW, MG, LOG>::STAGES,                                   \
                              GemmCfg<BN, CG, OUT, EW, MG, LOG>::SMEM_BYTES,                               \
                              GemmInstance<BN, CG, OUT, EW, MG, LOG>::protocol(),                          \
                              &GemmInstance<BN, CG, OUT, EW, MG, LOG>::launch,                             \
                              &GemmInstance<BN, CG, OUT, EW, MG, LOG>::max_workers};                       \
    }
// A product variant; TS_GEMM_VARIANT_LOG with LOG = 1 instantiates the protocol-logging kernel.
#define TS_GEMM_VARIANT(NAME, BN, CG, OUT, EW, MG) TS_GEMM_VARIANT_LOG(NAME, BN, CG, OUT, EW, MG, 0)
