// qk_prep.cu -- optional input preparation (dn_qk_prepare): per row of the
// head dimension, q and k become x / sqrt(sum x^2 + eps), then q is
// multiplied by the query scale.  This is the l2norm helper and the
// 1/sqrt(head_dim) query factor of the Gated DeltaNet PyTorch code on
// "DeltaNet 引入 Delta Rule" (garden.houmin.site/infra/delta-net), and the
// d_k^{-1/2} read of "Kimi Delta Attention" (fr.news.hada.io/topic?id=31925).
//
// An HBM-bound elementwise pass (2 bytes in and 2 out per element for bf16):
// one warp per row, each lane owning D/32 contiguous elements, so a warp's
// access to a row is one contiguous 128- or 256-byte segment.  Each warp
// loads kRows rows before reducing any of them; the sum of squares is a
// butterfly shuffle in fp32.  The
// grid strides over the q rows and then the k rows in one wave of blocks
// (the SM count times the blocks that fit on an SM at once).
#include <string.h>

#include "dn_common.cuh"
#include "dn_internal.h"

namespace dn {
namespace {

constexpr int kThreads = 256;
// Rows per warp in flight.  Measured on the 1.3B-layer shape (bf16, d = 128):
// 2 rows (32 registers, 8 blocks per SM) 57.8 us; 4 rows (48 registers)
// 74.1 us; 8 rows 106.9 us.  Resident warps matter more than rows per warp.
constexpr int kRows = 2;

// A lane's E = D / 32 contiguous elements, moved as one vector access and
// widened to fp32 (bf16 pairs travel as 32-bit words, element 2i in the low
// half, as they lie in memory).
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    __nv_bfloat162 h;
    memcpy(&h, &w, 4);
    return __bfloat1622float2(h);
}
__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    uint32_t w;
    memcpy(&w, &h, 4);
    return w;
}

__device__ __forceinline__ void load_lane(const float* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load_lane(const float* p, float (&x)[2]) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
}
__device__ __forceinline__ void load_lane(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 a = bf2_to_f2(w.x), b = bf2_to_f2(w.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
__device__ __forceinline__ void load_lane(const __nv_bfloat16* p, float (&x)[2]) {
    const float2 a = bf2_to_f2(*reinterpret_cast<const uint32_t*>(p));
    x[0] = a.x; x[1] = a.y;
}

__device__ __forceinline__ void store_lane(float* p, const float (&y)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void store_lane(float* p, const float (&y)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(y[0], y[1]);
}
__device__ __forceinline__ void store_lane(__nv_bfloat16* p, const float (&y)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(f2_to_bf2(y[0], y[1]), f2_to_bf2(y[2], y[3]));
}
__device__ __forceinline__ void store_lane(__nv_bfloat16* p, const float (&y)[2]) {
    *reinterpret_cast<uint32_t*>(p) = f2_to_bf2(y[0], y[1]);
}

// Rows [0, rows) are q rows (scaled), rows [rows, 2 rows) k rows; with
// normalize == 0 only the q rows are visited.  src may equal dst: every lane
// reads its elements before it writes them, and with normalize != 0 the
// shuffles order all of a row's reads before any of its writes.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
qk_prepare_kernel(const T* q, const T* k, T* q_out, T* k_out, long long rows,
                  int normalize, float scale, float eps) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long nrows = normalize ? 2 * rows : rows;
    const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * kThreads) >> 5;
    for (long long r0 = warp * kRows; r0 < nrows; r0 += nwarps * kRows) {
        float x[kRows][E];
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const long long r = r0 + j;  // warp-uniform
            if (r < nrows) {
                const T* src = (r < rows ? q + r * D : k + (r - rows) * D) + lane * E;
                load_lane(src, x[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const long long r = r0 + j;  // warp-uniform
            if (r < nrows) {
                float f = r < rows ? scale : 1.0f;
                if (normalize) {
                    float ss = 0.0f;
#pragma unroll
                    for (int e = 0; e < E; ++e) ss = fmaf(x[j][e], x[j][e], ss);
                    f *= rsqrtf(warp_sum(ss) + eps);
                }
                float y[E];
#pragma unroll
                for (int e = 0; e < E; ++e) y[e] = x[j][e] * f;
                T* dst = (r < rows ? q_out + r * D : k_out + (r - rows) * D) + lane * E;
                store_lane(dst, y);
            }
        }
    }
}

// Gradient of the preparation with respect to its raw rows.  For a row x
// with output y = f x, f = scale / n and n = sqrt(sum x^2 + eps) (chain rule
// through dn/dx_i = x_i / n):
//     dx = f (dy - x (x . dy) / n^2)      (normalize != 0)
//     dx = scale dy                       (normalize == 0; k rows not visited)
// Rows [0, rows) are q rows, [rows, 2 rows) k rows (no scale).  dx may equal
// dy: each lane reads its elements of x and dy before the shuffles that end
// with its own writes.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
qk_prepare_bwd_kernel(const T* q, const T* k, const T* dq_out, const T* dk_out, T* dq, T* dk,
                      long long rows, int normalize, float scale, float eps) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long nrows = normalize ? 2 * rows : rows;
    const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * kThreads) >> 5;
    for (long long r = warp; r < nrows; r += nwarps) {  // warp-uniform
        const bool is_q = r < rows;
        const long long off = (is_q ? r : r - rows) * D + lane * E;
        float g[E];
        load_lane((is_q ? dq_out : dk_out) + off, g);
        const float s = is_q ? scale : 1.0f;
        float y[E];
        if (normalize) {
            float x[E];
            load_lane((is_q ? q : k) + off, x);
            float ss = 0.0f, xg = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ss = fmaf(x[e], x[e], ss);
                xg = fmaf(x[e], g[e], xg);
            }
            const float n2 = warp_sum(ss) + eps;
            const float inv = rsqrtf(n2);
            const float c = warp_sum(xg) / n2;
#pragma unroll
            for (int e = 0; e < E; ++e) y[e] = s * inv * fmaf(-x[e], c, g[e]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) y[e] = s * g[e];
        }
        store_lane((is_q ? dq : dk) + off, y);
    }
}

template <typename T, int D>
cudaError_t launch_bwd_typed(const void* q, const void* k, const void* dq_out, const void* dk_out,
                             void* dq, void* dk, long long rows, int normalize, float scale,
                             float eps, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qk_prepare_bwd_kernel<T, D>,
                                                          kThreads, 0);
    if (e != cudaSuccess) return e;
    const long long nrows = normalize ? 2 * rows : rows;
    const long long per_block = kThreads / 32;
    const long long need = (nrows + per_block - 1) / per_block;
    const long long full = (long long)sms * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(need < full ? need : full);
    qk_prepare_bwd_kernel<T, D><<<grid, kThreads, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(dq_out),
        static_cast<const T*>(dk_out), static_cast<T*>(dq), static_cast<T*>(dk), rows,
        normalize, scale, eps);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_typed(const void* q, const void* k, void* q_out, void* k_out,
                         long long rows, int normalize, float scale, float eps,
                         cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qk_prepare_kernel<T, D>,
                                                          kThreads, 0);
    if (e != cudaSuccess) return e;
    const long long nrows = normalize ? 2 * rows : rows;
    const long long per_block = (kThreads / 32) * kRows;
    const long long need = (nrows + per_block - 1) / per_block;
    // one wave: every SM holding as many blocks as fit at once
    const long long full = (long long)sms * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(need < full ? need : full);
    qk_prepare_kernel<T, D><<<grid, kThreads, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<T*>(q_out),
        static_cast<T*>(k_out), rows, normalize, scale, eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_prepare(const void* q, const void* k, void* q_out, void* k_out,
                              long long rows, int d, int normalize, float scale, float eps,
                              int dt, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    if (dt == 0) {
        if (d == 128)
            return launch_typed<float, 128>(q, k, q_out, k_out, rows, normalize, scale, eps, stream);
        return launch_typed<float, 64>(q, k, q_out, k_out, rows, normalize, scale, eps, stream);
    }
    if (d == 128)
        return launch_typed<__nv_bfloat16, 128>(q, k, q_out, k_out, rows, normalize, scale, eps,
                                                stream);
    return launch_typed<__nv_bfloat16, 64>(q, k, q_out, k_out, rows, normalize, scale, eps,
                                           stream);
}

cudaError_t launch_qk_prepare_bwd(const void* q, const void* k, const void* dq_out,
                                  const void* dk_out, void* dq, void* dk, long long rows, int d,
                                  int normalize, float scale, float eps, int dt,
                                  cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
#define DN_PREP_BWD(T_, D_)                                                                    \
    return launch_bwd_typed<T_, D_>(q, k, dq_out, dk_out, dq, dk, rows, normalize, scale, eps, \
                                    stream)
    if (dt == 0) {
        if (d == 128) DN_PREP_BWD(float, 128);
        DN_PREP_BWD(float, 64);
    }
    if (d == 128) DN_PREP_BWD(__nv_bfloat16, 128);
    DN_PREP_BWD(__nv_bfloat16, 64);
#undef DN_PREP_BWD
}

}  // namespace dn
