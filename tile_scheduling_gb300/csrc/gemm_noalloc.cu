// Self-checking GEMM for callers that cannot allocate device memory.
//
// ts_gemm_bf16_ex can record a per-tile trace (visit count, worker, start and
// end time) into a scratch buffer the caller allocates.  Some callers cannot
// call cudaMalloc at all -- for example a plugin running inside a host process
// whose own allocator owns all device memory, or a latency-critical path that
// must never enter the CUDA allocator.  This entry point gives them the same
// GEMM plus a check that the tile scheduler computed every output tile exactly
// once, with the trace kept in a fixed-size array that lives in this library's
// device image instead of caller memory.
//
// The scratch array is a file-scope __device__ variable: every device that
// loads the library holds it (2 MiB) until the process exits.  Its device
// address is looked up once per device, on the first call made with that
// device current; that first call should therefore come before any stream
// capture.  The address is kept for the life of the process: a cudaDeviceReset
// after the first call (which may load the module, and the array, elsewhere)
// is not supported.  Every call shares the one array per device: calls that overlap on
// the GPU (two streams, or two host threads) race on it, so serialise them.
// Each call clears the part it uses before the GEMM runs.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.h"

namespace ts {
namespace {

constexpr int64_t kNoAllocMaxTiles = int64_t(1) << 16;  // 4 int64 per tile: 2 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) long long g_noalloc_trace[4 * kNoAllocMaxTiles];

std::mutex g_setup_mu;
long long *g_trace_addr[kMaxDevices];

// Device address of the scratch array for the current device (looked up once).
ts_status scratch_address(long long **out) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return fail(TS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> g(g_setup_mu);
    if (!g_trace_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_trace);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
        g_trace_addr[dev] = static_cast<long long *>(p);
    }
    *out = g_trace_addr[dev];
    return TS_OK;
}

__global__ void clear_trace_kernel(long long *trace, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        trace[i] = 0;
}

// *bad = number of tiles whose visit count is not exactly one.
__global__ void count_bad_tiles_kernel(const long long *trace, int64_t tiles, int32_t *bad) {
    __shared__ int32_t partial[256];
    int32_t c = 0;
    for (int64_t t = threadIdx.x; t < tiles; t += blockDim.x) c += trace[4 * t] != 1;
    partial[threadIdx.x] = c;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) partial[threadIdx.x] += partial[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) *bad = partial[0];
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_gemm_bf16_checked_noalloc(const void *A, const void *B, void *D, int64_t M, int64_t N,
                                                  int64_t K, int32_t out_dtype, int32_t sched, int32_t *bad_tiles,
                                                  void *stream) {
    using namespace ts;
    if (!bad_tiles) return fail(TS_ERR_INVALID_ARG, "bad_tiles is NULL");
    ts_launch_info info;
    ts_status s = ts_gemm_launch_info(M, N, K, out_dtype, sched, nullptr, &info);
    if (s != TS_OK) return s;
    if (info.num_units > kNoAllocMaxTiles)
        return fail(TS_ERR_UNSUPPORTED,
                    "%lld output tiles exceed the %lld-tile scratch of the no-allocation entry point; "
                    "use ts_gemm_bf16_ex with a caller-allocated trace",
                    static_cast<long long>(info.num_units), static_cast<long long>(kNoAllocMaxTiles));
    long long *trace = nullptr;
    if ((s = scratch_address(&trace)) != TS_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // No tile is scheduled when the output is empty or K == 0 (zero fill).
    const int64_t tiles = (M == 0 || N == 0 || K == 0) ? 0 : info.num_units;
    if (tiles > 0) {
        const int blocks = static_cast<int>(std::min<int64_t>((4 * tiles + 255) / 256, 1024));
        clear_trace_kernel<<<blocks, 256, 0, st>>>(trace, 4 * tiles);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "scratch clear launch");
    }
    ts_gemm_opts o;
    std::memset(&o, 0, sizeof o);
    o.trace = reinterpret_cast<int64_t *>(trace);
    if ((s = ts_gemm_bf16_ex(A, B, D, M, N, K, out_dtype, sched, &o, stream)) != TS_OK) return s;
    count_bad_tiles_kernel<<<1, 256, 0, st>>>(trace, tiles, bad_tiles);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TS_OK : cuda_fail(e, "tile check launch");
}
