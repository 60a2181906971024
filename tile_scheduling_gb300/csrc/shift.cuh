// Joining two aligned 16-byte vectors into the 16 bytes that start DELTA
// bytes into the first: the copy kernels' path for a source and destination
// that differ in their offset modulo 16 bytes (every destination vector is
// aligned, the two source vectors around its bytes are).
#pragma once
#include <cstdint>

namespace ts {

template <int DELTA>
__device__ __forceinline__ int4 join16(const int4 &a, const int4 &b) {
    static_assert(DELTA > 0 && DELTA < 16 && DELTA % 2 == 0, "an even byte shift inside a vector");
    const uint32_t w[8] = {static_cast<uint32_t>(a.x), static_cast<uint32_t>(a.y), static_cast<uint32_t>(a.z),
                           static_cast<uint32_t>(a.w), static_cast<uint32_t>(b.x), static_cast<uint32_t>(b.y),
                           static_cast<uint32_t>(b.z), static_cast<uint32_t>(b.w)};
    constexpr int q = DELTA / 4, r = DELTA % 4;  // whole words, then 0 or 2 bytes
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = r == 0 ? w[q + i] : __funnelshift_r(w[q + i], w[q + i + 1], 8 * r);
    return make_int4(static_cast<int>(o[0]), static_cast<int>(o[1]), static_cast<int>(o[2]), static_cast<int>(o[3]));
}

}  // namespace ts
