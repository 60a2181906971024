// Measurement helper: hold `ctas` SMs for a bounded time.
//
// This recreates the situation in which a static persistent schedule leaves a
// long launch tail ("Cluster Launch Control", limits of the static persistent
// scheduler: some SMs are held by another kernel, so a pre-assigned worker
// starts late and runs its tiles alone).  Each CTA takes the largest opt-in
// shared memory, so no GEMM CTA can share its SM, announces itself through a
// host-mapped counter, and sleeps in short steps until %globaltimer says its
// time is up.  It never waits on anything else.
#include <chrono>
#include <thread>

#include "common.h"

namespace ts {
namespace {

constexpr int64_t kMaxSpinNs = 10ll * 1000 * 1000 * 1000;

__global__ void spin_kernel(uint64_t duration_ns, int32_t *started) {
    extern __shared__ uint8_t hold[];
    if (threadIdx.x == 0) {
        uint64_t t0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        atomicAdd_system(started, 1);
        __threadfence_system();
        for (;;) {
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (t - t0 >= duration_ns) break;
            __nanosleep(1000);
        }
        hold[0] = 1;
    }
}

}  // namespace
}  // namespace ts

extern "C" {

ts_status ts_spin(int32_t ctas, int64_t duration_ns, int32_t *started, void *stream) {
    using namespace ts;
    const int dev = current_device();
    const int sms = device_sms(dev);
    if (ctas < 1 || ctas > sms) return fail(TS_ERR_INVALID_ARG, "ctas = %d must be in [1, %d]", ctas, sms);
    if (duration_ns < 0 || duration_ns > kMaxSpinNs)
        return fail(TS_ERR_INVALID_ARG, "duration_ns must be in [0, 1e10]");
    if (!started) return fail(TS_ERR_INVALID_ARG, "started is NULL");
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, started);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(started)");
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer)
        return fail(TS_ERR_INVALID_ARG, "started must be page-locked, device-mapped host memory");
    const int smem = device_smem_optin(dev);
    if (smem <= 0) return fail(TS_ERR_CUDA, "cannot query shared memory per block");
    e = cudaFuncSetAttribute(spin_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(spin)");
    spin_kernel<<<ctas, 32, smem, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(duration_ns),
                                                                      static_cast<int32_t *>(attr.devicePointer));
    e = cudaGetLastError();
    return e == cudaSuccess ? TS_OK : cuda_fail(e, "spin launch");
}

ts_status ts_spin_wait_started(const int32_t *started, int32_t expected, double timeout_s) {
    using namespace ts;
    if (!started) return fail(TS_ERR_INVALID_ARG, "started is NULL");
    const volatile int32_t *p = started;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        if (*p >= expected) return TS_OK;
        const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (el > timeout_s)
            return fail(TS_ERR_TIMEOUT, "only %d of %d spinning CTAs started within %.3f s", *p, expected, timeout_s);
        std::this_thread::yield();
    }
}

}  // extern "C"
