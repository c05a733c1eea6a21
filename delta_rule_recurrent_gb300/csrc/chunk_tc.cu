// chunk_tc.cu -- chunkwise delta-rule forward on tcgen05 tensor cores
// (bf16 operands, fp32 accumulation in TMEM), dk = dv = 128, chunk C = 64.
//
// Chunk algebra ("Chunkwise KDA : réorganiser la récurrence en
// multiplications matricielles", fr.news.hada.io/topic?id=31925, decay D = I;
// appendix B.2 "UT transform", paperlayer.ai/abs/2406.06484v6).  For a chunk
// with rows K, Q, V (C x 128), write strengths beta and incoming state S
// ([dk][dv], fp32):
//     A    = tril(diag(beta) K K^T, -1),   P = tril(Q K^T)      (incl. diagonal)
//     Tm   = (I + A)^{-1} diag(beta)        W = Tm K,  U = Tm V
//     U'   = U - W S                        (true per-token errors)
//     O    = Q S + P U'                     S <- S + K^T U'
// This kernel regroups the output as O = (Q - PT K) S + PT V with PT = P Tm,
// which equals Q S + P U' exactly and lets one MMA produce O and U' together:
//     D1 = [PT; Tm] V  (+)  [Q - PT K; -W] S    ->  rows 0-63: O, rows 64-127: U'
// so the state-dependent chain per chunk is: S -> bf16 -> one MMA (K = dk) ->
// U' -> bf16 -> S += K^T U' (K = C).
//
// One CTA (8 warps) owns one (batch, head) and walks its chunks in order with
// S resident in TMEM.  Operand tiles live in shared memory in the 128-byte
// swizzled layout TMA writes; q, k, v arrive by TMA (3-D maps, so rows past
// the end of a sequence read as zeros) and o leaves by TMA store (rows past
// the end are not written).  Every mbarrier wait is bounded; on a timeout the
// CTA records an error code, drains what it has in flight and exits.
#include <cudaTypedefs.h>
#include <cuda.h>

#include <mutex>

#include "dn_common.cuh"
#include "dn_internal.h"
#include "tc_ptx.cuh"
#include "tri_inverse.cuh"

namespace dn {

// First device-side error recorded by a tensor-core chunk kernel (0 = none).
__device__ unsigned int g_chunk_tc_error = 0;

namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // dk = dv
constexpr int kThreads = 256;   // 8 warps: warp w reads TMEM lanes 32*(w%4).., columns half w/4
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

// Shared-memory layout (byte offsets from a 1024-aligned base).
constexpr uint32_t kRegKQW = 192 * 128;           // one dk half of [K; Q'; -W]: 192 rows x 128 B
constexpr uint32_t kStageKQW = 2 * kRegKQW;       // both dk halves
constexpr uint32_t OFF_KQW = 0;                   // 2 stages
constexpr uint32_t OFF_V = 2 * kStageKQW;         // V: 2 dv halves x 64 rows x 128 B
constexpr uint32_t OFF_TP = OFF_V + 16384;        // [PT; Tm] 128 rows x 128 B; later the O tile
constexpr uint32_t OFF_SB = OFF_TP + 16384;       // S in bf16 (2 x 128 rows x 128 B); later U'
constexpr uint32_t OFF_AM = OFF_SB + 32768;       // A   fp32 64 x 65
constexpr uint32_t OFF_XM = OFF_AM + 64 * kTriPitch * 4;  // X fp32 64 x 65
constexpr uint32_t OFF_YS = OFF_XM + 64 * kTriPitch * 4;  // solve scratch 816 floats
constexpr uint32_t OFF_BETA = OFF_YS + 816 * 4;   // beta, 64 floats
constexpr uint32_t OFF_BAR = OFF_BETA + 256;      // 4 mbarriers
constexpr uint32_t OFF_TMEMPTR = OFF_BAR + 32;
constexpr uint32_t kSmemBytes = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
static_assert(OFF_V % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_SB % 1024 == 0, "tile alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns (512 allocated): S | D1 (O, U') | DW (PT K, W) | G (K K^T, Q K^T; then PT).
constexpr uint32_t COL_S = 0, COL_D1 = 128, COL_DW = 256, COL_G = 384;

constexpr uint32_t IDESC_G = idesc_bf16_f32(128, 64, 0, 0);     // [K;Q] K^T
constexpr uint32_t IDESC_PT = idesc_bf16_f32(128, 64, 0, 1);    // [P;Tm] Tm
constexpr uint32_t IDESC_KB = idesc_bf16_f32(128, 128, 0, 1);   // A K-major, B MN-major
constexpr uint32_t IDESC_MM = idesc_bf16_f32(128, 128, 1, 1);   // both MN-major

enum : unsigned { kErrTimeoutLoad = 1, kErrTimeoutMma = 2 };

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
}
// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a 128B-swizzled region.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
    return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
// Writes 32 fp32 values as bf16 into 4 consecutive chunks (starting at ch0)
// of row r of a swizzled region.
__device__ __forceinline__ void store_row32_bf16(uint32_t region, int r, int ch0,
                                                 const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(region + sw128(r, ch0 + c), pack_bf16(x[8 * c + 0], x[8 * c + 1]),
                     pack_bf16(x[8 * c + 2], x[8 * c + 3]), pack_bf16(x[8 * c + 4], x[8 * c + 5]),
                     pack_bf16(x[8 * c + 6], x[8 * c + 7]));
}
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&x)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const __nv_bfloat16* __restrict__ beta, const float* __restrict__ S0,
                float* __restrict__ S_T, int T) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw_addr);
    float* const Am = reinterpret_cast<float*>(gbase + OFF_AM);
    float* const Xm = reinterpret_cast<float*>(gbase + OFF_XM);
    float* const Ys = reinterpret_cast<float*>(gbase + OFF_YS);
    float* const betas = reinterpret_cast<float*>(gbase + OFF_BETA);
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(gbase + OFF_TMEMPTR);
    const uint32_t bar_kq0 = base + OFF_BAR, bar_v = base + OFF_BAR + 16,
                   bar_mma = base + OFF_BAR + 24;
    const uint32_t sTP = base + OFF_TP, sSB = base + OFF_SB, sV = base + OFF_V;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, half = warp >> 2;  // TMEM lane quarter, column half
    const int bh = blockIdx.x;
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        mbar_init(bar_kq0, 1);
        mbar_init(bar_kq0 + 8, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

    // Loads issued by thread 0, tracked so an abort can drain them.
    auto issue_kq = [&](int c) {
        const uint32_t st = base + OFF_KQW + (uint32_t)(c & 1) * kStageKQW;
        const uint32_t bar = bar_kq0 + 8u * (uint32_t)(c & 1);
        mbar_arrive_expect_tx(bar, 4 * 8192);
        tma_load_3d(st, &tm_k, bar, 0, c * kC, bh);
        tma_load_3d(st + kRegKQW, &tm_k, bar, 64, c * kC, bh);
        tma_load_3d(st + 8192, &tm_q, bar, 0, c * kC, bh);
        tma_load_3d(st + kRegKQW + 8192, &tm_q, bar, 64, c * kC, bh);
    };
    auto issue_v = [&](int c) {
        mbar_arrive_expect_tx(bar_v, 2 * 8192);
        tma_load_3d(sV, &tm_v, bar_v, 0, c * kC, bh);
        tma_load_3d(sV + 8192, &tm_v, bar_v, 64, c * kC, bh);
    };
    int kq_issued = 0, v_issued = 0;  // loads issued (thread 0's view)
    int kq_waited = 0, v_waited = 0;  // loads waited for
    uint32_t mma_phase = 0;  // MMA-barrier phases waited for (all threads)
    uint32_t mma_commits = 0;  // commits issued (thread 0); each is waited for at once
    bool fail = false;
    unsigned err_code = 0;

    if (tid == 0 && nchunks > 0) {
        issue_kq(0);
        issue_v(0);
        kq_issued = v_issued = 1;
    }
    // S0 (or zeros) into TMEM: thread owns state row 32*q4 + lane, columns 64*half ..
    {
        const int i = 32 * q4 + lane;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t r[32];
            const int j0 = 64 * half + 32 * part;
            if (S0) {
                const float4* src =
                    reinterpret_cast<const float4*>(S0 + ((size_t)bh * kD + i) * kD + j0);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4) {
                    const float4 f = src[v4];
                    r[4 * v4 + 0] = __float_as_uint(f.x);
                    r[4 * v4 + 1] = __float_as_uint(f.y);
                    r[4 * v4 + 2] = __float_as_uint(f.z);
                    r[4 * v4 + 3] = __float_as_uint(f.w);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = 0u;
            }
            tmem_st32(tmem + lane_base + COL_S + (uint32_t)j0, r);
        }
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    auto wait_mma = [&]() {
        if (!mbar_wait(bar_mma, mma_phase & 1u, kTimeoutNs)) {
            fail = true;
            err_code = kErrTimeoutMma;
        }
        ++mma_phase;
        tc_fence_after_sync();
    };

    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        const int t0 = c * kC;
        const int n = min(kC, T - t0);
        const uint32_t sKQW = base + OFF_KQW + (uint32_t)s * kStageKQW;

        if (tid == 0) {
            // The previous chunk's o store must have read the tile before TP is reused.
            bulk_wait_group_read0();
            if (c + 1 < nchunks) {
                issue_kq(c + 1);
                ++kq_issued;
            }
        }
        if (tid < kC) {
            betas[tid] = tid < n ? __bfloat162float(beta[(size_t)bh * T + t0 + tid]) : 0.f;
        }
        if (mbar_wait(bar_kq0 + 8u * (uint32_t)s, (uint32_t)(c >> 1) & 1u, kTimeoutNs)) {
            if (tid == 0) ++kq_waited;
        } else {
            fail = true;
            err_code = kErrTimeoutLoad;
        }

        // ---- S (fp32, TMEM) -> bf16 operand tile: row i = dk index, dv halves as regions.
        {
            const int i = 32 * q4 + lane;
            const uint32_t region = sSB + (uint32_t)half * 16384u;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                tmem_ld32f(tmem + lane_base + COL_S + 64 * half + 32 * part, x);
                store_row32_bf16(region, i, 4 * part, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(fail)) goto bail;

        // ---- G = [K; Q] K^T  (rows 0-63: K K^T, rows 64-127: Q K^T)
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = sKQW + (uint32_t)(kk >> 2) * kRegKQW + (uint32_t)(kk & 3) * 32u;
                mma_bf16_ss(tmem + COL_G, sw128_desc(a, 16, 1024), sw128_desc(a, 16, 1024), IDESC_G,
                            kk > 0);
            }
            mma_commit(bar_mma);
            ++mma_commits;
        }
        wait_mma();
        {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_G + 32 * half, x);
            if (q4 < 2) {  // A = beta_i (k_i . k_j) for j < i
                const int i = 32 * q4 + lane;
                const float bi = betas[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    Am[i * kTriPitch + j] = j < i ? bi * x[jj] : 0.f;
                }
            } else {  // P = q_t . k_j for j <= t, as bf16 into rows 0-63 of TP
                const int t = 32 * (q4 - 2) + lane;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    if (j > t) x[jj] = 0.f;
                }
                store_row32_bf16(sTP, t, 4 * half, x);
            }
        }
        tc_fence_before_sync();
        if (__syncthreads_or(fail)) goto bail;

        // ---- X = (I + A)^{-1}; Tm = X diag(beta) as bf16 into rows 64-127 of TP
        unit_lower_inverse64<kThreads>(Am, Xm, Ys);
        {
            const int i = tid >> 2, c0 = (tid & 3) * 16;
            float x[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = Xm[i * kTriPitch + c0 + e] * betas[c0 + e];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
                st_shared_v4(sTP + sw128(64 + i, c0 / 8 + cc), pack_bf16(x[8 * cc + 0], x[8 * cc + 1]),
                             pack_bf16(x[8 * cc + 2], x[8 * cc + 3]),
                             pack_bf16(x[8 * cc + 4], x[8 * cc + 5]),
                             pack_bf16(x[8 * cc + 6], x[8 * cc + 7]));
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(fail)) goto bail;

        // ---- PT = P Tm (rows 0-63 of the result)
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_G, sw128_desc(sTP + 32u * kk, 16, 1024),
                            sw128_desc(sTP + 8192u + 2048u * kk, 8192, 1024), IDESC_PT, kk > 0);
            mma_commit(bar_mma);
            ++mma_commits;
        }
        wait_mma();
        if (q4 < 2) {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_G + 32 * half, x);
            store_row32_bf16(sTP, 32 * q4 + lane, 4 * half, x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(fail)) goto bail;

        // ---- DW = [PT; Tm] K  and  D1 = [PT; Tm] V
        if (tid == 0) {
            if (mbar_wait(bar_v, (uint32_t)c & 1u, kTimeoutNs)) {
                ++v_waited;
            } else {
                fail = true;
                err_code = kErrTimeoutLoad;
            }
            tc_fence_after_sync();
            if (!fail) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + COL_DW, sw128_desc(sTP + 32u * kk, 16, 1024),
                                sw128_desc(sKQW + 2048u * kk, kRegKQW, 1024), IDESC_KB, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + COL_D1, sw128_desc(sTP + 32u * kk, 16, 1024),
                                sw128_desc(sV + 2048u * kk, 8192, 1024), IDESC_KB, kk > 0);
                mma_commit(bar_mma);
                ++mma_commits;
            }
        }
        if (__syncthreads_or(fail)) goto bail;
        wait_mma();
        if (tid == 0 && c + 1 < nchunks) {
            issue_v(c + 1);
            ++v_issued;
        }
        // ---- rows 0-63: Q' = Q - PT K over the Q rows; rows 64-127: -W into the W rows
        {
            float x[64];
            {
                float a[32], b[32];
                tmem_ld32f(tmem + lane_base + COL_DW + 64 * half, a);
                tmem_ld32f(tmem + lane_base + COL_DW + 64 * half + 32, b);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = a[e];
                    x[32 + e] = b[e];
                }
            }
            const uint32_t region = sKQW + (uint32_t)half * kRegKQW;
            if (q4 < 2) {
                const int row = 64 + 32 * q4 + lane;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t addr = region + sw128(row, ch);
                    const uint4 qv = ld_shared_v4(addr);
                    const float2 q0 = unpack_bf16(qv.x), q1 = unpack_bf16(qv.y),
                                 q2 = unpack_bf16(qv.z), q3 = unpack_bf16(qv.w);
                    const float* d = x + 8 * ch;
                    st_shared_v4(addr, pack_bf16(q0.x - d[0], q0.y - d[1]),
                                 pack_bf16(q1.x - d[2], q1.y - d[3]),
                                 pack_bf16(q2.x - d[4], q2.y - d[5]),
                                 pack_bf16(q3.x - d[6], q3.y - d[7]));
                }
            } else {
                const int row = 128 + 32 * (q4 - 2) + lane;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float* d = x + 8 * ch;
                    st_shared_v4(region + sw128(row, ch), pack_bf16(-d[0], -d[1]),
                                 pack_bf16(-d[2], -d[3]), pack_bf16(-d[4], -d[5]),
                                 pack_bf16(-d[6], -d[7]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(fail)) goto bail;

        // ---- D1 += [Q'; -W] S   ->  rows 0-63: O, rows 64-127: U'
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a =
                    sKQW + (uint32_t)(kk >> 2) * kRegKQW + 8192u + (uint32_t)(kk & 3) * 32u;
                mma_bf16_ss(tmem + COL_D1, sw128_desc(a, 16, 1024),
                            sw128_desc(sSB + 2048u * kk, 16384, 1024), IDESC_KB, 1);
            }
            mma_commit(bar_mma);
            ++mma_commits;
        }
        wait_mma();
        // ---- O -> tile for the TMA store (reusing TP); U' -> operand tile (reusing SB)
        {
            const int t = 32 * (q4 & 1) + lane;
            const uint32_t region = (q4 < 2 ? sTP : sSB) + (uint32_t)half * 8192u;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                tmem_ld32f(tmem + lane_base + COL_D1 + 64 * half + 32 * part, x);
                store_row32_bf16(region, t, 4 * part, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(fail)) goto bail;

        // ---- S += K^T U'; store o
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_S, sw128_desc(sKQW + 2048u * kk, kRegKQW, 1024),
                            sw128_desc(sSB + 2048u * kk, 8192, 1024), IDESC_MM, 1);
            mma_commit(bar_mma);
            ++mma_commits;
            tma_store_3d(&tm_o, sTP, 0, t0, bh);
            tma_store_3d(&tm_o, sTP + 8192u, 64, t0, bh);
            bulk_commit_group();
        }
        wait_mma();
        if (__syncthreads_or(fail)) goto bail;
    }

    if (S_T) {
        const int i = 32 * q4 + lane;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float x[32];
            const int j0 = 64 * half + 32 * part;
            tmem_ld32f(tmem + lane_base + COL_S + (uint32_t)j0, x);
            float4* dst = reinterpret_cast<float4*>(S_T + ((size_t)bh * kD + i) * kD + j0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(x[4 * v4], x[4 * v4 + 1], x[4 * v4 + 2], x[4 * v4 + 3]);
        }
    }
    if (tid == 0) bulk_wait_group0();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
    return;

bail:
    // A wait ran out: record it, let everything this CTA started finish
    // (bounded again), release TMEM and leave.
    if (tid == 0) {
        atomicCAS(&g_chunk_tc_error, 0u, err_code ? err_code : kErrTimeoutMma);
        // Only the most recent commit can still be pending; re-wait for it.
        if (mma_commits > 0) mbar_wait(bar_mma, (mma_commits - 1u) & 1u, kTimeoutNs);
        for (int c = kq_waited; c < kq_issued; ++c)
            mbar_wait(bar_kq0 + 8u * (uint32_t)(c & 1), (uint32_t)(c >> 1) & 1u, kTimeoutNs);
        for (int c = v_waited; c < v_issued; ++c) mbar_wait(bar_v, (uint32_t)c & 1u, kTimeoutNs);
        bulk_wait_group0();
    } else if (err_code) {
        atomicCAS(&g_chunk_tc_error, 0u, err_code);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a [BH][T][128] bf16 tensor with 64 x 64 x 1 boxes, 128B swizzle.
bool make_map(CUtensorMap* map, const void* ptr, int BH, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)T * kD * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supports(int dk, int dv, int dt) { return dk == kD && dv == kD && dt == 1; }

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const void* beta,
                            const float* S0, void* o, float* S_T, int BH, int T, int dk, int dv,
                            int dt, cudaStream_t stream) {
    if (!chunk_tc_supports(dk, dv, dt)) return cudaErrorNotSupported;
    if (BH <= 0 || T <= 0) return cudaSuccess;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, q, BH, T) || !make_map(&mk, k, BH, T) || !make_map(&mv, v, BH, T) ||
        !make_map(&mo, o, BH, T))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(chunk_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    chunk_tc_kernel<<<BH, kThreads, kSmemBytes, stream>>>(
        mq, mk, mv, mo, static_cast<const __nv_bfloat16*>(beta), S0, S_T, T);
    return cudaGetLastError();
}

unsigned int chunk_tc_take_device_error() {
    unsigned int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_chunk_tc_error, sizeof(h)) != cudaSuccess) return ~0u;
    if (h) cudaMemcpyToSymbol(g_chunk_tc_error, &zero, sizeof(zero));
    return h;
}

}  // namespace dn
