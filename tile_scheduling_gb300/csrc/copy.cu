// Grid-stride int16 copy: dst[gid] = src[gid] for gid < n.
//
// The domain is the grid-stride loop of TS "Schedules" (start = bx * tpb + tx,
// step = gdimx * tpb) over the elements of the int16 copy example of TS
// "Resources" (get_item / set_item, both guarded by gid < num_entries).  On
// this GPU the loop runs over 16-byte vectors (8 elements), keeps four
// independent vectors in flight per thread, and the grid is sized to the
// resident capacity (SM count x blocks per SM) so every CTA is persistent.
// The ragged head (until src is 16-byte aligned) and tail are copied element
// by element with the same guard.
#include <algorithm>

#include "common.h"

namespace ts {
namespace {

constexpr int kCopyThreads = 256;

__device__ __forceinline__ int4 ld_stream(const int4 *p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(int4 *p, int4 v) {
    asm volatile("st.global.cs.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__global__ void __launch_bounds__(kCopyThreads) copy_i16_vec_kernel(const int16_t *__restrict__ src,
                                                                    int16_t *__restrict__ dst, int64_t head,
                                                                    int64_t nvec, int64_t n) {
    const int64_t gid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int4 *s4 = reinterpret_cast<const int4 *>(src + head);
    int4 *d4 = reinterpret_cast<int4 *>(dst + head);
    int64_t i = gid;
    for (; i + 3 * step < nvec; i += 4 * step) {
        const int4 v0 = ld_stream(s4 + i);
        const int4 v1 = ld_stream(s4 + i + step);
        const int4 v2 = ld_stream(s4 + i + 2 * step);
        const int4 v3 = ld_stream(s4 + i + 3 * step);
        st_stream(d4 + i, v0);
        st_stream(d4 + i + step, v1);
        st_stream(d4 + i + 2 * step, v2);
        st_stream(d4 + i + 3 * step, v3);
    }
    for (; i < nvec; i += step) st_stream(d4 + i, ld_stream(s4 + i));
    // ragged head [0, head) and tail [head + 8 * nvec, n)
    const int64_t tail0 = head + 8 * nvec;
    if (gid < head) dst[gid] = src[gid];
    if (gid < n - tail0) dst[tail0 + gid] = src[tail0 + gid];
}

__global__ void __launch_bounds__(kCopyThreads) copy_i16_scalar_kernel(const int16_t *__restrict__ src,
                                                                       int16_t *__restrict__ dst, int64_t n) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t gid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; gid < n; gid += step)
        dst[gid] = src[gid];
}

int resident_blocks(const void *kernel) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCopyThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return per_sm * std::max(1, device_sms(current_device()));
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_copy_i16(const int16_t *src, int16_t *dst, int64_t n, void *stream) {
    using namespace ts;
    if (n < 0) return fail(TS_ERR_INVALID_ARG, "n = %lld < 0", static_cast<long long>(n));
    if (n == 0) return TS_OK;
    if (!src || !dst) return fail(TS_ERR_INVALID_ARG, "src or dst is NULL");
    if (src == dst) return TS_OK;
    const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t bytes = static_cast<uintptr_t>(n) * 2;
    if (s < d + bytes && d < s + bytes) return fail(TS_ERR_INVALID_ARG, "src and dst overlap");
    if (s % 2 || d % 2) return fail(TS_ERR_INVALID_ARG, "src and dst must be 2-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s % 16) == (d % 16)) {
        const int64_t head = std::min<int64_t>(n, static_cast<int64_t>(((16 - s % 16) % 16) / 2));
        const int64_t nvec = (n - head) / 8;
        static int grid_cache[64];
        const int dev = current_device();
        int grid = dev < 64 ? grid_cache[dev] : 0;
        if (grid == 0) {
            grid = resident_blocks(reinterpret_cast<const void *>(copy_i16_vec_kernel));
            if (dev < 64) grid_cache[dev] = grid;
        }
        // enough threads for the head and tail (< 16 elements in all)
        grid = std::max(grid, 1);
        copy_i16_vec_kernel<<<grid, kCopyThreads, 0, st>>>(src, dst, head, nvec, n);
    } else {
        const int grid = resident_blocks(reinterpret_cast<const void *>(copy_i16_scalar_kernel));
        copy_i16_scalar_kernel<<<grid, kCopyThreads, 0, st>>>(src, dst, n);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TS_OK : cuda_fail(e, "copy launch");
}
