// simt_mm.cuh -- register-tiled products for the CUDA-core chunk kernels.
//
// A CTA of kThreads threads forms M x N products (M a multiple of 64, N of
// 16 or 32) from operands in shared memory, read through accessors a(m, k)
// and b(k, n), so the same loop serves plain, transposed and masked operands.
// Two interchangeable policies with the same interface:
//   Fp32Ops      fp32 FMA on CUDA cores, 256 threads: thread (ty, tx) =
//                (tid / 16, tid % 16) owns the elements (ty + 16 i, tx + 16 j);
//   Tf32Ops<NW>  warp-level m16n8k8 tensor-core MMAs with tf32 operands and
//                fp32 accumulation, NW warps: warp w owns row blocks
//                (w % 4) + 4 i of 16 rows and column part w / 4 of NW / 4,
//                in the m16n8 accumulator layout (lane 4g + q holds rows g,
//                g + 8 at columns 2q, 2q + 1).
// Each holds M N / kThreads floats per thread; an accumulator is only ever
// read through the for_each, update2 or row_sums of the policy that filled it.  kPad is the row padding
// (floats) that keeps the policy's shared-memory operand reads free of bank
// conflicts: an odd pitch for the per-thread FMA pattern, a pitch of 4 mod 32
// for the fragment pattern (rows g = 0..7 by columns q = 0..3).
#pragma once

#include <stdint.h>

namespace dn {
namespace simt {

constexpr int kThreads = 256;

struct Fp32Ops {
    static constexpr int kPad = 1;
    static constexpr int kThreads = 256;

    template <int M, int N>
    struct Acc {
        float v[M / 16][N / 16];
    };

    template <int M, int N>
    static __device__ __forceinline__ void zero(Acc<M, N>& acc) {
#pragma unroll
        for (int i = 0; i < M / 16; ++i)
#pragma unroll
            for (int j = 0; j < N / 16; ++j) acc.v[i][j] = 0.f;
    }

    // acc += sum_kk a(m, kk) * b(kk, n)
    template <int M, int N, int K, typename FA, typename FB>
    static __device__ __forceinline__ void mm(Acc<M, N>& acc, FA a, FB b) {
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
                for (int j = 0; j < N / 16; ++j) acc.v[i][j] = fmaf(av[i], bv[j], acc.v[i][j]);
        }
    }

    // f(m, n, value) for every element the calling thread owns
    template <int M, int N, typename F>
    static __device__ __forceinline__ void for_each(const Acc<M, N>& acc, F f) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
        for (int i = 0; i < M / 16; ++i)
#pragma unroll
            for (int j = 0; j < N / 16; ++j) f(ty + 16 * i, tx + 16 * j, acc.v[i][j]);
    }

    // f(m, n, a&, b&) for every element the calling thread owns in two
    // accumulators of one shape (in place)
    template <int M, int N, typename F>
    static __device__ __forceinline__ void update2(Acc<M, N>& a, Acc<M, N>& b, F f) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
        for (int i = 0; i < M / 16; ++i)
#pragma unroll
            for (int j = 0; j < N / 16; ++j) f(ty + 16 * i, tx + 16 * j, a.v[i][j], b.v[i][j]);
    }

    // Row sums of f(m, n, value) in a fixed order: out[p * M + m] is the sum
    // over the columns of part p (kRowParts parts), each written by exactly
    // one thread.  Row ty + 16 i lives on the 16 lanes of one half-warp.
    static constexpr int kRowParts = 1;
    template <int M, int N, typename F>
    static __device__ __forceinline__ void row_sums(const Acc<M, N>& acc, F f, float* out) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
        for (int i = 0; i < M / 16; ++i) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < N / 16; ++j) s += f(ty + 16 * i, tx + 16 * j, acc.v[i][j]);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (tx == 0) out[ty + 16 * i] = s;
        }
    }
};

template <int NW>
struct Tf32Ops {
    static constexpr int kPad = 4;
    static constexpr int kThreads = 32 * NW;
    static constexpr int kParts = NW / 4;  // column parts

    template <int M, int N>
    struct Acc {
        static_assert(N % (8 * kParts) == 0, "whole n8 tiles per warp");
        float v[M / 64][N / (8 * kParts)][4];
    };

    // The fp32 bit pattern as a tf32 operand: the MMA reads its upper 19
    // bits, i.e. the value truncated to tf32 (no separate rounding step).
    static __device__ __forceinline__ uint32_t tf32(float x) { return __float_as_uint(x); }

    template <int M, int N>
    static __device__ __forceinline__ void zero(Acc<M, N>& acc) {
#pragma unroll
        for (int i = 0; i < M / 64; ++i)
#pragma unroll
            for (int j = 0; j < N / (8 * kParts); ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc.v[i][j][r] = 0.f;
    }

    template <int M, int N, int K, typename FA, typename FB>
    static __device__ __forceinline__ void mm(Acc<M, N>& acc, FA a, FB b) {
        static_assert(K % 8 == 0, "K in steps of 8");
        constexpr int NJ = N / (8 * kParts);
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
        const int m0 = 16 * (w & 3), n0 = (w >> 2) * (N / kParts);
#pragma unroll 2
        for (int k = 0; k < K; k += 8) {
            uint32_t af[M / 64][4], bf[NJ][2];
#pragma unroll
            for (int i = 0; i < M / 64; ++i) {
                const int r = m0 + 64 * i + g;
                af[i][0] = tf32(a(r, k + q));
                af[i][1] = tf32(a(r + 8, k + q));
                af[i][2] = tf32(a(r, k + q + 4));
                af[i][3] = tf32(a(r + 8, k + q + 4));
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                bf[j][0] = tf32(b(k + q, n0 + 8 * j + g));
                bf[j][1] = tf32(b(k + q + 4, n0 + 8 * j + g));
            }
#pragma unroll
            for (int i = 0; i < M / 64; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j)
                    asm volatile(
                        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, "
                        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                        : "+f"(acc.v[i][j][0]), "+f"(acc.v[i][j][1]), "+f"(acc.v[i][j][2]),
                          "+f"(acc.v[i][j][3])
                        : "r"(af[i][0]), "r"(af[i][1]), "r"(af[i][2]), "r"(af[i][3]),
                          "r"(bf[j][0]), "r"(bf[j][1]));
        }
    }

    template <int M, int N, typename F>
    static __device__ __forceinline__ void for_each(const Acc<M, N>& acc, F f) {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
        const int m0 = 16 * (w & 3), n0 = (w >> 2) * (N / kParts);
#pragma unroll
        for (int i = 0; i < M / 64; ++i)
#pragma unroll
            for (int j = 0; j < N / (8 * kParts); ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    f(m0 + 64 * i + g + 8 * (r >> 1), n0 + 8 * j + 2 * q + (r & 1), acc.v[i][j][r]);
    }

    template <int M, int N, typename F>
    static __device__ __forceinline__ void update2(Acc<M, N>& a, Acc<M, N>& b, F f) {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
        const int m0 = 16 * (w & 3), n0 = (w >> 2) * (N / kParts);
#pragma unroll
        for (int i = 0; i < M / 64; ++i)
#pragma unroll
            for (int j = 0; j < N / (8 * kParts); ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    f(m0 + 64 * i + g + 8 * (r >> 1), n0 + 8 * j + 2 * q + (r & 1), a.v[i][j][r],
                      b.v[i][j][r]);
    }

    // Row sums as Fp32Ops::row_sums; part p is the column part of warps
    // w / 4 = p, and row g (g + 8) of a warp's block lives on its lanes 4 g .. 4 g + 3.
    static constexpr int kRowParts = kParts;
    template <int M, int N, typename F>
    static __device__ __forceinline__ void row_sums(const Acc<M, N>& acc, F f, float* out) {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
        const int m0 = 16 * (w & 3), n0 = (w >> 2) * (N / kParts), part = w >> 2;
#pragma unroll
        for (int i = 0; i < M / 64; ++i) {
            float s[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < N / (8 * kParts); ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    s[r >> 1] += f(m0 + 64 * i + g + 8 * (r >> 1), n0 + 8 * j + 2 * q + (r & 1),
                                   acc.v[i][j][r]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
                s[h] += __shfl_xor_sync(0xffffffffu, s[h], 2);
                if (q == 0) out[part * M + m0 + 64 * i + g + 8 * h] = s[h];
            }
        }
    }
};

// The CUDA-core forward's helpers (fp32 FMA, plain arrays).
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

}  // namespace simt
}  // namespace dn
