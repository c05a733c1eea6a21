// tile_load.cuh -- global -> shared tile loads for the CUDA-core chunk kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dn {

// 16 bytes of T from global memory (16-byte aligned) as floats.
__device__ __forceinline__ void load16(const float* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

// Rows [r0, r0 + R) of a row-major tensor with row length D, columns
// c0 .. c0 + W - 1, into shared memory with row pitch LD; rows at or past
// n (relative to r0) read as zeros.  16-byte loads, several in flight per
// thread (row starts and c0 are multiples of 16 bytes).
template <int NT, int R, int W, int LD, int D, typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* __restrict__ src, size_t r0,
                                          int n, int c0) {
    constexpr int V = 16 / sizeof(T), PER = W / V;
    static_assert(W % V == 0, "whole 16-byte groups");
#pragma unroll 4
    for (int e = threadIdx.x; e < R * PER; e += NT) {
        const int t = e / PER, i = (e % PER) * V;
        float x[V];
        if (t < n) {
            load16(src + (r0 + t) * D + c0 + i, x);
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j) x[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < V; ++j) dst[t * LD + i + j] = x[j];
    }
}

}  // namespace dn
