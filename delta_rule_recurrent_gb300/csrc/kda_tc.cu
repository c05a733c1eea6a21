// kda_tc.cu -- the CUDA-core kernels around the tensor-core form of Kimi Delta
// Attention (dn_chunk_fwd_kda with a workspace).
//
// KDA decays every key channel d of the state by its own keep rate
// exp(g_t[d]) ("Kimi Delta Attention : atténuation par canal",
// fr.news.hada.io/topic?id=31925).  With G_t[d] the cumulative log decay from
// the chunk start, the chunk algebra carries the ratios exp(G_i[d] - G_j[d])
// inside the sums over d ("Chunkwise KDA : réorganiser la récurrence en
// multiplications matricielles", same page):
//     A[i][j] = beta_i sum_d k_i[d] k_j[d] exp(G_i[d] - G_j[d])   (j < i)
//     P[i][j] = sum_d q_i[d] k_j[d] exp(G_i[d] - G_j[d])          (j <= i)
//     U' = (I + A)^{-1} diag(beta) (V - (K . exp G) S)
//     O = (Q . exp G) S + P U',   S <- diag(exp G_C) S + (K . exp(G_C - G))^T U'
// While every channel's decay over the chunk stays within exp(-80) the ratio
// separates as exp(G_i[d]) exp(-G_j[d]), a product of two numbers bf16 holds
// (bf16 has fp32's exponent range), so A and P are one tensor-core product of
// [K . exp G; Q . exp G] with (K . exp(-G))^T, and the rest is the plain
// two-pass algebra on the decayed operands:
//   kda_decay_kernel   per chunk: G (prefix sums per channel), the optional
//                      q/k L2 normalisation and query scale, and the bf16
//                      operands K~ = K . exp G, Q~ = Q . exp G (the scan's [K; Q]),
//                      K^ = K . exp(G_C - G) (the scan's state update), K- =
//                      K . exp(-G) (the prepare pass's right factor), plus
//                      exp G_C per channel and the chunk's separability flag;
//   (tensor cores)     the prepare pass on [K~; Q~] (K-)^T, the scan;
//   kda_fix_kernel     for a chunk whose decay exceeds exp(-80) on some channel
//                      (where exp(-G) would leave the range) the [PT; Tm] tile
//                      again in fp32 on CUDA cores, every ratio its own clamped
//                      exponential, over the tensor-core pass's tile.
#include <cuda_bf16.h>

#include "dn_common.cuh"
#include "dn_internal.h"
#include "simt_mm.cuh"
#include "tri_inverse.cuh"

namespace dn {
namespace {

constexpr int kC = 64, kD = 128;
constexpr int kSide = 256;  // fp32 per chunk: exp G_C [128], then the separability flag

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// One CTA of 256 threads per (head, chunk).  Warp w first forms the row
// factors of the optional preparation for rows 8w .. 8w + 7 of k and q (16
// bytes per lane, two rows per load).  Then thread (u, p), u = tid / 64 the
// token quarter and p = tid % 64 the channel pair (2p, 2p + 1), sums its 16
// tokens' log keep rates; the quarters' sums give each quarter its starting
// G and the chunk's G_C; and a second walk over the 16 tokens writes the four
// operands (4-byte accesses, a warp covering 128 contiguous bytes of a row).
// A chunk whose decay passes exp(-80) on some channel is appended to `fix`
// (count in fix[0], chunk indices after it).
__global__ void __launch_bounds__(256)
kda_decay_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                 const float* __restrict__ g, __nv_bfloat16* __restrict__ qt,
                 __nv_bfloat16* __restrict__ kt, __nv_bfloat16* __restrict__ kh,
                 __nv_bfloat16* __restrict__ kb, float* __restrict__ side, int* __restrict__ fix,
                 int T, int nchunks, QkNorm nm) {
    __shared__ float fk[kC], fq[kC];
    __shared__ float2 part[4][64];
    __shared__ int nonsep;
    const int item = blockIdx.x, bh = item / nchunks, c = item % nchunks;
    const int t0 = c * kC, n = min(kC, T - t0);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const size_t row0 = (size_t)bh * T + t0;
    if (tid == 0) nonsep = 0;
    {   // row factors: lanes 0-15 row 8w + 2i, lanes 16-31 row 8w + 2i + 1
        const int half = lane >> 4, l = lane & 15;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 8 * w + 2 * i + half;
            float sk = 0.f, sq = 0.f;
            if (nm.l2norm && r < n) {
                const uint4 a = *reinterpret_cast<const uint4*>(k + (row0 + r) * kD + 8 * l);
                const uint4 b = *reinterpret_cast<const uint4*>(q + (row0 + r) * kD + 8 * l);
                const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ua[j]));
                    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ub[j]));
                    sk = fmaf(x.x, x.x, fmaf(x.y, x.y, sk));
                    sq = fmaf(y.x, y.x, fmaf(y.y, y.y, sq));
                }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) {  // within each 16-lane half
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
            }
            if (l == 0) {
                fk[r] = nm.l2norm ? rsqrtf(sk + nm.eps) : 1.f;
                fq[r] = nm.qscale * (nm.l2norm ? rsqrtf(sq + nm.eps) : 1.f);
            }
        }
    }
    const int u = tid >> 6, p = tid & 63, ta = 16 * u;
    float2 sum = make_float2(0.f, 0.f);  // this quarter's log keep rates, channels 2p, 2p + 1
#pragma unroll 4
    for (int t = ta; t < ta + 16; ++t) {
        if (t < n) {
            const float2 x = *reinterpret_cast<const float2*>(g + (row0 + t) * kD + 2 * p);
            sum.x += x.x;
            sum.y += x.y;
        }
    }
    part[u][p] = sum;
    __syncthreads();
    float2 G = make_float2(0.f, 0.f), GC = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float2 s = part[v][p];
        if (v < u) G.x += s.x, G.y += s.y;
        GC.x += s.x;
        GC.y += s.y;
    }
    if (GC.x < -80.f || GC.y < -80.f) nonsep = 1;  // (every writer writes 1)
    const float2 eC = make_float2(__expf(GC.x), __expf(GC.y));
    if (u == 0) *reinterpret_cast<float2*>(side + (size_t)item * kSide + 2 * p) = eC;
#pragma unroll 2
    for (int t = ta; t < ta + 16; ++t) {
        if (t < n) {
            const size_t e = (row0 + t) * kD + 2 * p;
            const float2 x = *reinterpret_cast<const float2*>(g + e);
            G.x += x.x;
            G.y += x.y;
            const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(k + e));
            const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(q + e));
            const float a = fk[t], b = fq[t];
            const float k0 = kv.x * a, k1 = kv.y * a, q0 = qv.x * b, q1 = qv.y * b;
            const float e0 = __expf(G.x), e1 = __expf(G.y);
            const float i0 = __expf(fminf(-G.x, 80.f)), i1 = __expf(fminf(-G.y, 80.f));
            *reinterpret_cast<__nv_bfloat162*>(kt + e) = __floats2bfloat162_rn(k0 * e0, k1 * e1);
            *reinterpret_cast<__nv_bfloat162*>(qt + e) = __floats2bfloat162_rn(q0 * e0, q1 * e1);
            *reinterpret_cast<__nv_bfloat162*>(kh + e) =
                __floats2bfloat162_rn(k0 * __expf(GC.x - G.x), k1 * __expf(GC.y - G.y));
            // exp(-G) capped at exp(80): only a separable chunk's product is used
            *reinterpret_cast<__nv_bfloat162*>(kb + e) = __floats2bfloat162_rn(k0 * i0, k1 * i1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        side[(size_t)item * kSide + kD] = nonsep ? 0.f : 1.f;
        if (nonsep) fix[1 + atomicAdd(fix, 1)] = item;
    }
}

// The [PT; Tm] tile of one chunk in fp32 on CUDA cores, for the chunks the
// separable product does not cover (flag 0); every other CTA returns at once.
// 256 threads (a 16 x 16 grid for the products), all operands in shared memory.
constexpr int kLK = kD + 1, kLA = kC + 1;
struct FixSmem {
    static constexpr int kK = 0, kQ = kK + kC * kLK, kG = kQ + kC * kLK;
    static constexpr int kA = kG + kC * kLK, kX = kA + kC * kLA, kP = kX + kC * kLA;
    static constexpr int kT = kP + kC * kLA, kY = kT + kC * kLA, kB = kY + 3 * 16 * 17;
    static constexpr int kF = kB + kC;  // 2 x 64 row factors
    static constexpr size_t kBytes = sizeof(float) * (kF + 2 * kC);
};

__device__ void fix_one(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                        const __nv_bfloat16* __restrict__ beta, const float* __restrict__ g,
                        __nv_bfloat16* __restrict__ tiles, int item, int T, int nchunks,
                        const QkNorm& nm) {
    using L = FixSmem;
    extern __shared__ float sm[];
    float *Ks = sm + L::kK, *Qs = sm + L::kQ, *Gs = sm + L::kG, *Am = sm + L::kA;
    float *Xm = sm + L::kX, *Pm = sm + L::kP, *Tm = sm + L::kT, *Ys = sm + L::kY;
    float *bs = sm + L::kB, *fr = sm + L::kF;
    const int bh = item / nchunks, c = item % nchunks, t0 = c * kC, n = min(kC, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    const int tid = threadIdx.x;
    for (int e = tid; e < kC * kD; e += 256) {
        const int t = e / kD, d = e % kD;
        const bool in = t < n;
        Ks[t * kLK + d] = in ? bf(k + (row0 + t) * kD + d) : 0.f;
        Qs[t * kLK + d] = in ? bf(q + (row0 + t) * kD + d) : 0.f;
        Gs[t * kLK + d] = in ? g[(row0 + t) * kD + d] : 0.f;
    }
    if (tid < kC) bs[tid] = tid < n ? __bfloat162float(beta[row0 + tid]) : 0.f;
    __syncthreads();
    if (tid < 2 * kC) {  // row factors of the preparation
        const float* row = tid < kC ? Ks + tid * kLK : Qs + (tid - kC) * kLK;
        float f = tid < kC ? 1.f : nm.qscale;
        if (nm.l2norm) {
            float ss = 0.f;
            for (int d = 0; d < kD; ++d) ss = fmaf(row[d], row[d], ss);
            f *= rsqrtf(ss + nm.eps);
        }
        fr[tid] = f;
    } else if (tid < 2 * kC + kD) {  // prefix sums of channel d
        const int d = tid - 2 * kC;
        float acc = 0.f;
        for (int t = 0; t < kC; ++t) {
            acc += Gs[t * kLK + d];
            Gs[t * kLK + d] = acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < kC * kD; e += 256) {
        const int t = e / kD, d = e % kD;
        Ks[t * kLK + d] *= fr[t];
        Qs[t * kLK + d] *= fr[kC + t];
    }
    __syncthreads();
    {   // A and P with one clamped exponential per ratio (pairs past the diagonal masked)
        const int tx = tid & 15, ty = tid >> 4;
        float aa[4][4] = {}, ap[4][4] = {};
        for (int d = 0; d < kD; ++d) {
            float ki[4], qi[4], gi[4], kj[4], gj[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ki[i] = Ks[(ty + 16 * i) * kLK + d];
                qi[i] = Qs[(ty + 16 * i) * kLK + d];
                gi[i] = Gs[(ty + 16 * i) * kLK + d];
                kj[i] = Ks[(tx + 16 * i) * kLK + d];
                gj[i] = Gs[(tx + 16 * i) * kLK + d];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float e = __expf(fminf(gi[i] - gj[j], 0.f)) * kj[j];
                    aa[i][j] = fmaf(ki[i], e, aa[i][j]);
                    ap[i][j] = fmaf(qi[i], e, ap[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = ty + 16 * i, nn = tx + 16 * j;
                Am[m * kLA + nn] = nn < m ? bs[m] * aa[i][j] : 0.f;
                Pm[m * kLA + nn] = nn <= m ? ap[i][j] : 0.f;
            }
    }
    __syncthreads();
    unit_lower_inverse64<256, kLA>(Am, Xm, Ys);  // ends with a barrier
    for (int e = tid; e < kC * kC; e += 256) {   // Tm = X diag(beta)
        const int i = e / kC, j = e % kC;
        Tm[i * kLA + j] = Xm[i * kLA + j] * bs[j];
    }
    __syncthreads();
    {   // PT = P Tm; the tile: rows 0-63 PT, rows 64-127 Tm, bf16
        float acc[4][4];
        simt::zero<64, 64>(acc);
        simt::mm_acc<64, 64, kC>(acc, [&](int m, int kk) { return Pm[m * kLA + kk]; },
                                 [&](int kk, int nn) { return Tm[kk * kLA + nn]; });
        const int tx = tid & 15, ty = tid >> 4;
        __nv_bfloat16* const tile = tiles + (size_t)item * 128 * kC;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = ty + 16 * i, nn = tx + 16 * j;
                tile[m * kC + nn] = __float2bfloat16_rn(acc[i][j]);
                tile[(kC + m) * kC + nn] = __float2bfloat16_rn(Tm[m * kLA + nn]);
            }
    }
    __syncthreads();  // the shared arrays are reused for the next chunk
}

// The chunks listed by kda_decay_kernel (fix[0] of them), one at a time per CTA.
__global__ void __launch_bounds__(256)
kda_fix_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
               const __nv_bfloat16* __restrict__ beta, const float* __restrict__ g,
               const int* __restrict__ fix, __nv_bfloat16* __restrict__ tiles, int T,
               int nchunks, QkNorm nm) {
    const int count = fix[0];
    for (int i = blockIdx.x; i < count; i += gridDim.x)
        fix_one(q, k, beta, g, tiles, fix[1 + i], T, nchunks, nm);
}

}  // namespace

cudaError_t launch_kda_decay(const void* q, const void* k, const float* g, void* qt, void* kt,
                             void* kh, void* kb, float* side, int* fix, int BH, int T,
                             const QkNorm& nm, cudaStream_t stream) {
    const int nchunks = (T + kC - 1) / kC;
    const long long items = (long long)BH * nchunks;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(fix, 0, sizeof(int), stream);  // the list starts empty
    if (e != cudaSuccess) return e;
    kda_decay_kernel<<<(unsigned)items, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g,
        static_cast<__nv_bfloat16*>(qt), static_cast<__nv_bfloat16*>(kt),
        static_cast<__nv_bfloat16*>(kh), static_cast<__nv_bfloat16*>(kb), side, fix, T, nchunks,
        nm);
    return cudaGetLastError();
}

cudaError_t launch_kda_fix(const void* q, const void* k, const void* beta, const float* g,
                           const int* fix, void* tiles, int BH, int T, const QkNorm& nm,
                           cudaStream_t stream) {
    const int nchunks = (T + kC - 1) / kC;
    const long long items = (long long)BH * nchunks;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kda_fix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)FixSmem::kBytes);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(items < sms ? items : sms);  // one wave; most calls list none
    kda_fix_kernel<<<grid, 256, FixSmem::kBytes, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(beta), g, fix, static_cast<__nv_bfloat16*>(tiles), T,
        nchunks, nm);
    return cudaGetLastError();
}

}  // namespace dn
