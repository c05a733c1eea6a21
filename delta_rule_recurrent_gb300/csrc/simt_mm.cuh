// simt_mm.cuh -- register-tiled fp32 products for the CUDA-core chunk kernels.
//
// A CTA of 256 threads is viewed as a 16 x 16 grid (tx = tid % 16,
// ty = tid / 16); thread (ty, tx) owns the elements (ty + 16 i, tx + 16 j) of
// an M x N result.  Operands are read through accessors, so the same loop
// serves plain, transposed and masked operands in shared memory.
#pragma once

namespace dn {
namespace simt {

constexpr int kThreads = 256;

// acc[i][j] += sum_kk a(ty + 16 i, kk) * b(kk, tx + 16 j).
template <int M, int N, int K, typename FA, typename FB>
__device__ __forceinline__ void mm_acc(float (&acc)[M / 16][N / 16], FA a, FB b) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
    for (int kk = 0; kk < K; ++kk) {
        float av[M / 16], bv[N / 16];
#pragma unroll
        for (int i = 0; i < M / 16; ++i) av[i] = a(ty + 16 * i, kk);
#pragma unroll
        for (int j = 0; j < N / 16; ++j) bv[j] = b(kk, tx + 16 * j);
#pragma unroll
        for (int i = 0; i < M / 16; ++i)
#pragma unroll
            for (int j = 0; j < N / 16; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

template <int M, int N>
__device__ __forceinline__ void zero(float (&acc)[M / 16][N / 16]) {
#pragma unroll
    for (int i = 0; i < M / 16; ++i)
#pragma unroll
        for (int j = 0; j < N / 16; ++j) acc[i][j] = 0.f;
}

// f(m, n, acc[i][j]) for every element the calling thread owns.
template <int M, int N, typename F>
__device__ __forceinline__ void for_each(const float (&acc)[M / 16][N / 16], F f) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < M / 16; ++i)
#pragma unroll
        for (int j = 0; j < N / 16; ++j) f(ty + 16 * i, tx + 16 * j, acc[i][j]);
}

}  // namespace simt
}  // namespace dn
