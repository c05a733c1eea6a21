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
// The kernel regroups the output as O = (Q - PT K) S + PT V with PT = P Tm,
// which equals Q S + P U' exactly and lets one MMA produce O and U' together:
//     D1 = [PT; Tm] V  (+)  [Q - PT K; -W] S    ->  rows 0-63: O, rows 64-127: U'
// so the state-dependent chain per chunk is only: S -> bf16 -> one MMA over
// dk -> U' -> bf16 -> S += K^T U'.
//
// One CTA owns one (batch, head) and keeps S in TMEM for the whole sequence.
// Its 16 warps have fixed roles so the serial chain of chunk c overlaps the
// state-independent work of chunks c+1 and c+2:
//   warp 0      TMA producer (q, k, v tiles; 3-D maps, rows past the end read 0)
//   warp 1      TMEM owner and the single MMA-issuing thread; it polls the
//               readiness of every pending MMA and issues the state chain first
//   warp 2      TMA store of o tiles (rows past the end are not written)
//   warps 4-7   state group: S -> bf16 operand, O and U' epilogues, final state
//   warps 8-11, 12-15   chunk groups for even and odd chunks: A, P, the
//               triangular solve, Tm, PT, and the Q' / -W operands
// Operand tiles use the 128-byte swizzled shared-memory layout that TMA
// writes.  Every wait is bounded: on a timeout the CTA records an error code
// (read back with dn_device_error), drains what it started and exits.
#include <cudaTypedefs.h>
#include <cuda.h>

#include <mutex>

#include "dn_common.cuh"
#include "dn_internal.h"
#include "tc_ptx.cuh"

namespace dn {

// First device-side error recorded by a tensor-core chunk kernel (0 = none).
__device__ unsigned int g_chunk_tc_error = 0;

namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // dk = dv
constexpr int kThreads = 512;   // 16 warps
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s without progress
constexpr int kP = 65;          // row pitch (floats) of the fp32 solve array

// ---------------------------------------------------------------- smem map
constexpr uint32_t kRegKQW = 192 * 128;              // one dk half of [K; Q'; -W]
constexpr uint32_t kStageKQW = 2 * kRegKQW;
constexpr uint32_t OFF_KQW = 0;                      // 2 stages
constexpr uint32_t OFF_V = OFF_KQW + 2 * kStageKQW;  // V, 2 dv halves x 64 rows
constexpr uint32_t OFF_TP = OFF_V + 16384;           // 2 stages of [PT; Tm]; then the O tile
constexpr uint32_t OFF_SB = OFF_TP + 2 * 16384;      // S as bf16 (2 x 128 rows); then U'
constexpr uint32_t OFF_X = OFF_SB + 32768;           // 2 x fp32 64 x kP: A, overwritten by X
constexpr uint32_t kXBytes = 64 * kP * 4;
constexpr uint32_t OFF_Y = OFF_X + 2 * kXBytes;      // 2 x 3 x 16 x 16 fp32 solve scratch
constexpr uint32_t OFF_BETA = OFF_Y + 2 * 3072;      // 2 x 64 fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 512;         // mbarriers, 8 bytes each
constexpr int kNumBars = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * kNumBars;  // abort flag, TMEM address
constexpr uint32_t kSmemBytes = OFF_MISC + 16 + 1024;  // + 1024-byte alignment slack
static_assert(OFF_V % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_SB % 1024 == 0, "tile alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// mbarrier indices ([2] = one per chunk parity)
enum : int {
    B_KQ_FULL = 0,    // [2] q, k tiles landed
    B_KQ_EMPTY = 2,   // [2] stage's last reader (S += K^T U') completed
    B_TP_READY = 4,   // [2] P and Tm written (chunk group)
    B_TP_FULL = 6,    // [2] PT written over P (chunk group)
    B_QW_READY = 8,   // [2] Q' and -W written (chunk group)
    B_O_FULL = 10,    // [2] O tile written (state group)
    B_O_FREE = 12,    // [2] O tile stored (store warp)
    B_G_FULL = 14,    // [2] G = [K;Q] K^T done
    B_PT_FULL = 16,   // [2] PT = P Tm done
    B_G_EMPTY = 18,   // [2] chunk group finished with its G / PT columns
    B_V_FULL = 20,    // v tile landed
    B_V_EMPTY = 21,   // D1 = [PT;Tm] V done (v tile free)
    B_DW_FULL = 22,   // [2] DW = [PT;Tm] K done (one per chunk group)
    B_DW_EMPTY = 24,  // chunk group finished reading DW
    B_SB_FULL = 25,   // S bf16 operand written
    B_D1_FULL = 26,   // D1 += [Q';-W] S done
    B_U_FULL = 27,    // U' written
    B_D1_EMPTY = 28,  // state group finished reading D1
    B_S_READY = 29,   // S += K^T U' done
    B_DRAIN = 30,     // final drain of the MMA pipe
};
// Parity waits are only unambiguous when a barrier cannot run two phases
// ahead of its waiter, so every barrier has exactly one waiting role, which
// consumes its phases in order.

// TMEM columns (512 allocated): S | D1 (O, U') | DW (PT K, W) | G/PT even | G/PT odd
constexpr uint32_t COL_S = 0, COL_D1 = 128, COL_DW = 256, COL_G = 384;

constexpr uint32_t IDESC_G = idesc_bf16_f32(128, 64, 0, 0);    // [K;Q] K^T
constexpr uint32_t IDESC_PT = idesc_bf16_f32(128, 64, 0, 1);   // [P;Tm] Tm
constexpr uint32_t IDESC_KB = idesc_bf16_f32(128, 128, 0, 1);  // A K-major, B MN-major
constexpr uint32_t IDESC_MM = idesc_bf16_f32(128, 128, 1, 1);  // both MN-major

enum : unsigned { kErrTimeout = 1 };

// ----------------------------------------------------------- small helpers
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
// 32 fp32 values -> bf16 into 4 consecutive chunks (from ch0) of row r.
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
// Named barrier over one 128-thread warpgroup.
__device__ __forceinline__ void wg_sync(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
// Named barrier over one warpgroup that also ORs a flag across it, so every
// thread of the group takes the same branch after a bounded wait.
__device__ __forceinline__ bool wg_sync_or(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

struct Ctl {
    uint32_t bars;             // shared address of mbarrier 0
    volatile int* abort_flag;  // set by whichever role times out first
    __device__ uint32_t bar(int i) const { return bars + 8u * (uint32_t)i; }
    __device__ bool aborted() const { return *abort_flag != 0; }
    __device__ void raise() const {
        *abort_flag = 1;
        atomicCAS(&g_chunk_tc_error, 0u, (unsigned)kErrTimeout);
    }
    // Bounded wait for the phase of barrier b with the given parity.  Gives up
    // when another role has aborted, or after kTimeoutNs (raising the abort).
    __device__ bool wait(int b, uint32_t parity) const {
        const uint32_t a = bar(b);
        if (mbar_try_wait(a, parity & 1u)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
#pragma unroll 1
            for (int i = 0; i < 32; ++i)
                if (mbar_try_wait(a, parity & 1u)) return true;
            if (aborted()) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                raise();
                return false;
            }
        }
    }
};

struct Smem {
    uint32_t base;   // shared address of the 1024-aligned base
    uint8_t* gbase;  // generic pointer to it
    __device__ uint32_t kqw(int s) const { return base + OFF_KQW + (uint32_t)s * kStageKQW; }
    __device__ uint32_t tp(int s) const { return base + OFF_TP + (uint32_t)s * 16384u; }
    __device__ uint32_t v() const { return base + OFF_V; }
    __device__ uint32_t sb() const { return base + OFF_SB; }
    __device__ float* x(int s) const {
        return reinterpret_cast<float*>(gbase + OFF_X + (uint32_t)s * kXBytes);
    }
    __device__ float* y(int s) const {
        return reinterpret_cast<float*>(gbase + OFF_Y + (uint32_t)s * 3072u);
    }
    __device__ float* beta(int s) const {
        return reinterpret_cast<float*>(gbase + OFF_BETA + (uint32_t)s * 256u);
    }
};

// ------------------------------------------------- triangular solve, in place
// X <- (I + A)^{-1} for a strictly lower-triangular 64 x 64 A held in X (row
// pitch kP, zeros on and above the diagonal), by one warpgroup (t = 0..127).
// The pages compute this inverse by forward substitution, in blocks of 16
// tokens ("Hardware-efficient implementation", section 3 of
// paperlayer.ai/abs/2406.06484v6; "Pipeline Triton Chunkwise",
// fr.news.hada.io/topic?id=31925).  Diagonal 16 x 16 blocks: right-looking
// column substitution in registers.  Block rows i = 1..3 then follow from
// X_ij = -X_ii sum_{k=j}^{i-1} A_ik X_kj; block row i of A is only read
// while forming block row i of X, so X overwrites it in place.
__device__ __forceinline__ void solve_unit_lower64(float* X, float* Ys, int t, int barid) {
    if (t < 64) {
        const int base = (t >> 4) * 16, c = t & 15;
        float x[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) x[l] = (l == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r)
#pragma unroll
            for (int l = r + 1; l < 16; ++l)
                x[l] = fmaf(-X[(base + l) * kP + base + r], x[r], x[l]);
        wg_sync(barid);
#pragma unroll
        for (int l = 0; l < 16; ++l) X[(base + l) * kP + base + c] = x[l];
    } else {
        wg_sync(barid);
    }
    wg_sync(barid);
    const int r0 = t >> 4, c = t & 15;
#pragma unroll
    for (int i = 1; i < 4; ++i) {
#pragma unroll
        for (int m = 0; m < 2 * i; ++m) {
            const int j = m >> 1, r = r0 + 8 * (m & 1);
            const float* arow = X + (16 * i + r) * kP;
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int k = 16 * j; k < 16 * i; k += 2) {
                y0 = fmaf(arow[k], X[k * kP + 16 * j + c], y0);
                y1 = fmaf(arow[k + 1], X[(k + 1) * kP + 16 * j + c], y1);
            }
            Ys[(j * 16 + r) * 16 + c] = y0 + y1;
        }
        wg_sync(barid);
#pragma unroll
        for (int m = 0; m < 2 * i; ++m) {
            const int j = m >> 1, r = r0 + 8 * (m & 1);
            const float* xrow = X + (16 * i + r) * kP + 16 * i;
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int mm = 0; mm < 16; mm += 2) {
                x0 = fmaf(xrow[mm], Ys[(j * 16 + mm) * 16 + c], x0);
                x1 = fmaf(xrow[mm + 1], Ys[(j * 16 + mm + 1) * 16 + c], x1);
            }
            X[(16 * i + r) * kP + 16 * j + c] = -(x0 + x1);
        }
        wg_sync(barid);
    }
}

// ----------------------------------------------------------------- roles
__device__ void producer_role(const Ctl& ctl, const Smem& sm, const CUtensorMap* tm_q,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, int bh,
                              int nchunks) {
    int nkq = 0, nv = 0;
    uint64_t t0 = globaltimer_ns();
    while ((nkq < nchunks || nv < nchunks) && !ctl.aborted()) {
        bool progressed = false;
        if (nkq < nchunks &&
            (nkq < 2 || mbar_test_wait(ctl.bar(B_KQ_EMPTY + (nkq & 1)), ((nkq >> 1) - 1) & 1))) {
            const int s = nkq & 1;
            const uint32_t st = sm.kqw(s), bar = ctl.bar(B_KQ_FULL + s);
            mbar_arrive_expect_tx(bar, 4 * 8192);
            tma_load_3d(st, tm_k, bar, 0, nkq * kC, bh);
            tma_load_3d(st + kRegKQW, tm_k, bar, 64, nkq * kC, bh);
            tma_load_3d(st + 8192, tm_q, bar, 0, nkq * kC, bh);
            tma_load_3d(st + kRegKQW + 8192, tm_q, bar, 64, nkq * kC, bh);
            if (nkq + 2 < nchunks) {  // warm L2 for the load after next
                tma_prefetch_l2_3d(tm_k, 0, (nkq + 2) * kC, bh);
                tma_prefetch_l2_3d(tm_k, 64, (nkq + 2) * kC, bh);
                tma_prefetch_l2_3d(tm_q, 0, (nkq + 2) * kC, bh);
                tma_prefetch_l2_3d(tm_q, 64, (nkq + 2) * kC, bh);
            }
            ++nkq;
            progressed = true;
        }
        if (nv < nchunks && (nv < 1 || mbar_test_wait(ctl.bar(B_V_EMPTY), (nv - 1) & 1))) {
            const uint32_t bar = ctl.bar(B_V_FULL);
            mbar_arrive_expect_tx(bar, 2 * 8192);
            tma_load_3d(sm.v(), tm_v, bar, 0, nv * kC, bh);
            tma_load_3d(sm.v() + 8192, tm_v, bar, 64, nv * kC, bh);
            if (nv + 1 < nchunks) {  // v tile is single-buffered: warm L2 for the next one
                tma_prefetch_l2_3d(tm_v, 0, (nv + 1) * kC, bh);
                tma_prefetch_l2_3d(tm_v, 64, (nv + 1) * kC, bh);
            }
            ++nv;
            progressed = true;
        }
        if (progressed) {
            t0 = globaltimer_ns();
        } else if (globaltimer_ns() - t0 > kTimeoutNs) {
            ctl.raise();
        }
    }
    // Leave nothing in flight: wait (bounded) for the last load on each barrier.
    for (int s = 0; s < 2; ++s) {
        const int n_s = (nkq - s + 1) / 2;  // loads issued into stage s
        if (n_s > 0) mbar_wait(ctl.bar(B_KQ_FULL + s), (uint32_t)(n_s - 1) & 1u, kTimeoutNs);
    }
    if (nv > 0) mbar_wait(ctl.bar(B_V_FULL), (uint32_t)(nv - 1) & 1u, kTimeoutNs);
}

// The single MMA-issuing thread.  Each pending MMA group becomes issuable
// when the barriers it depends on have completed; the state chain
// (S += K^T U', then D1 += [Q';-W] S) has priority over chunk-local work.
// Every barrier checked here can complete at most once between two checks
// of the same phase, so parity tests are unambiguous.
__device__ void mma_role(const Ctl& ctl, const Smem& sm, uint32_t tmem, int nchunks) {
    int nG = 0, nPT = 0, nDW = 0, nD1 = 0, nM2 = 0, nM3 = 0;
    uint64_t t0 = globaltimer_ns();
    auto ready = [&](int b, int phase) {
        return mbar_test_wait(ctl.bar(b), (uint32_t)phase & 1u);
    };
    while (nM3 < nchunks && !ctl.aborted()) {
        bool issued = false;
        if (nM3 < nM2 && ready(B_U_FULL, nM3)) {
            // S += K^T U'
            const uint32_t kqw = sm.kqw(nM3 & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_S, sw128_desc(kqw + 2048u * kk, kRegKQW, 1024),
                            sw128_desc(sm.sb() + 2048u * kk, 8192, 1024), IDESC_MM, 1);
            mma_commit(ctl.bar(B_S_READY));
            mma_commit(ctl.bar(B_KQ_EMPTY + (nM3 & 1)));
            ++nM3;
            issued = true;
        } else if (nM2 < nD1 && ready(B_QW_READY + (nM2 & 1), nM2 >> 1) &&
                   ready(B_SB_FULL, nM2)) {
            // D1 += [Q'; -W] S
            const uint32_t kqw = sm.kqw(nM2 & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a =
                    kqw + (uint32_t)(kk >> 2) * kRegKQW + 8192u + (uint32_t)(kk & 3) * 32u;
                mma_bf16_ss(tmem + COL_D1, sw128_desc(a, 16, 1024),
                            sw128_desc(sm.sb() + 2048u * kk, 16384, 1024), IDESC_KB, 1);
            }
            mma_commit(ctl.bar(B_D1_FULL));
            ++nM2;
            issued = true;
        } else if (nD1 < nDW && nD1 == nM2 && ready(B_V_FULL, nD1) &&
                   (nD1 == 0 || ready(B_D1_EMPTY, nD1 - 1))) {
            // D1 = [PT; Tm] V   (the chunk's TP_FULL was seen when its DW was issued)
            const uint32_t tp = sm.tp(nD1 & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_D1, sw128_desc(tp + 32u * kk, 16, 1024),
                            sw128_desc(sm.v() + 2048u * kk, 8192, 1024), IDESC_KB, kk > 0);
            mma_commit(ctl.bar(B_V_EMPTY));
            ++nD1;
            issued = true;
        } else if (nDW < nPT && ready(B_TP_FULL + (nDW & 1), nDW >> 1) &&
                   (nDW == 0 || ready(B_DW_EMPTY, nDW - 1))) {
            // DW = [PT; Tm] K
            const uint32_t tp = sm.tp(nDW & 1), kqw = sm.kqw(nDW & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_DW, sw128_desc(tp + 32u * kk, 16, 1024),
                            sw128_desc(kqw + 2048u * kk, kRegKQW, 1024), IDESC_KB, kk > 0);
            mma_commit(ctl.bar(B_DW_FULL + (nDW & 1)));
            ++nDW;
            issued = true;
        } else if (nPT < nG && ready(B_TP_READY + (nPT & 1), nPT >> 1)) {
            // PT = P Tm into the chunk group's G columns
            const uint32_t tp = sm.tp(nPT & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_G + 64u * (nPT & 1), sw128_desc(tp + 32u * kk, 16, 1024),
                            sw128_desc(tp + 8192u + 2048u * kk, 8192, 1024), IDESC_PT, kk > 0);
            mma_commit(ctl.bar(B_PT_FULL + (nPT & 1)));
            ++nPT;
            issued = true;
        } else if (nG < nchunks && ready(B_KQ_FULL + (nG & 1), nG >> 1) &&
                   (nG < 2 || ready(B_G_EMPTY + (nG & 1), (nG >> 1) - 1))) {
            // G = [K; Q] K^T
            const uint32_t kqw = sm.kqw(nG & 1);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = kqw + (uint32_t)(kk >> 2) * kRegKQW + (uint32_t)(kk & 3) * 32u;
                mma_bf16_ss(tmem + COL_G + 64u * (nG & 1), sw128_desc(a, 16, 1024),
                            sw128_desc(a, 16, 1024), IDESC_G, kk > 0);
            }
            mma_commit(ctl.bar(B_G_FULL + (nG & 1)));
            ++nG;
            issued = true;
        }
        if (issued) {
            t0 = globaltimer_ns();
        } else if (globaltimer_ns() - t0 > kTimeoutNs) {
            ctl.raise();
        }
    }
    // Drain the MMA pipe before anyone releases TMEM or shared memory.
    mma_commit(ctl.bar(B_DRAIN));
    mbar_wait(ctl.bar(B_DRAIN), 0, kTimeoutNs);
}

__device__ void store_role(const Ctl& ctl, const Smem& sm, const CUtensorMap* tm_o, int bh,
                           int nchunks) {
    for (int c = 0; c < nchunks; ++c) {
        if (!ctl.wait(B_O_FULL + (c & 1), (uint32_t)(c >> 1))) break;
        const uint32_t tile = sm.tp(c & 1);
        tma_store_3d(tm_o, tile, 0, c * kC, bh);
        tma_store_3d(tm_o, tile + 8192u, 64, c * kC, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(ctl.bar(B_O_FREE + (c & 1)));
    }
    bulk_wait_group0();
}

// State group (warps 4-7): thread t owns state row t = TMEM lane t.
__device__ void state_role(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t,
                           const float* __restrict__ S0, float* __restrict__ S_T, int bh,
                           int nchunks) {
    constexpr int kBar = 1;
    const uint32_t lane_base = (uint32_t)(32 * (t >> 5)) << 16;
    // S0 (or zeros) into TMEM.
#pragma unroll
    for (int part = 0; part < 4; ++part) {
        uint32_t r[32];
        if (S0) {
            const float4* src =
                reinterpret_cast<const float4*>(S0 + ((size_t)bh * kD + t) * kD + 32 * part);
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
        tmem_st32(tmem + lane_base + COL_S + 32u * part, r);
    }
    tmem_wait_st();

    for (int c = 0; c < nchunks; ++c) {
        if (c > 0) {
            const bool ok = ctl.wait(B_S_READY, (uint32_t)(c - 1));
            if (wg_sync_or(kBar, !ok)) return;
        }
        tc_fence_after_sync();
        // S (fp32) -> bf16 operand tile: dv halves as regions, row t.
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_S + 32u * part, x);
            store_row32_bf16(sm.sb() + (uint32_t)(part >> 1) * 16384u, t, 4 * (part & 1), x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(kBar);
        if (t == 0) mbar_arrive(ctl.bar(B_SB_FULL));

        const bool ok = ctl.wait(B_D1_FULL, (uint32_t)c);
        if (wg_sync_or(kBar, !ok)) return;
        tc_fence_after_sync();
        // rows 0-63: O into the chunk's o tile; rows 64-127: U' over the S operand.
        const int row = t & 63;
        const uint32_t dst = (t < 64) ? sm.tp(c & 1) : sm.sb();
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_D1 + 32u * part, x);
            store_row32_bf16(dst + (uint32_t)(part >> 1) * 8192u, row, 4 * (part & 1), x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(kBar);
        if (t == 0) {
            mbar_arrive(ctl.bar(B_U_FULL));
            mbar_arrive(ctl.bar(B_D1_EMPTY));
            mbar_arrive(ctl.bar(B_O_FULL + (c & 1)));
        }
    }
    if (nchunks > 0) {
        const bool ok = ctl.wait(B_S_READY, (uint32_t)(nchunks - 1));
        if (wg_sync_or(kBar, !ok)) return;
    }
    tc_fence_after_sync();
    if (S_T) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_S + 32u * part, x);
            float4* dst = reinterpret_cast<float4*>(S_T + ((size_t)bh * kD + t) * kD + 32 * part);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(x[4 * v4], x[4 * v4 + 1], x[4 * v4 + 2], x[4 * v4 + 3]);
        }
    }
}

// Chunk group g (0: even chunks, warps 8-11; 1: odd chunks, warps 12-15).
__device__ void chunk_role(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t, int g,
                           const __nv_bfloat16* __restrict__ beta, int bh, int T, int nchunks) {
    const int barid = 2 + g;
    const uint32_t lane_base = (uint32_t)(32 * (t >> 5)) << 16;
    const uint32_t colG = COL_G + 64u * (uint32_t)g;
    float* const X = sm.x(g);
    float* const Ys = sm.y(g);
    float* const betas = sm.beta(g);
    const uint32_t tp = sm.tp(g), kqw = sm.kqw(g);
    const int row = t & 63;

    for (int c = g, it = 0; c < nchunks; c += 2, ++it) {
        const int t0 = c * kC;
        const int n = min(kC, T - t0);
        if (t < kC) betas[t] = t < n ? __bfloat162float(beta[(size_t)bh * T + t0 + t]) : 0.f;
        bool ok = true;
        if (it > 0) ok = ctl.wait(B_O_FREE + g, (uint32_t)(it - 1));  // o tile of c-2 stored
        ok = ok && ctl.wait(B_G_FULL + g, (uint32_t)it);
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        // A = beta_i (k_i . k_j) for j < i (TMEM rows 0-63) as fp32;
        // P = q_t . k_j for j <= t (rows 64-127) as bf16 over rows 0-63 of [PT; Tm].
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float x[32];
            tmem_ld32f(tmem + lane_base + colG + 32u * part, x);
            if (t < 64) {
                const float bi = betas[row];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * part + jj;
                    X[row * kP + j] = j < row ? bi * x[jj] : 0.f;
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (32 * part + jj > row) x[jj] = 0.f;
                store_row32_bf16(tp, row, 4 * part, x);
            }
        }
        tc_fence_before_sync();
        wg_sync(barid);
        solve_unit_lower64(X, Ys, t, barid);
        // Tm = X diag(beta) -> bf16 rows 64-127 of [PT; Tm]
        {
            const int i = t >> 1, c0 = 32 * (t & 1);
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = X[i * kP + c0 + e] * betas[c0 + e];
            store_row32_bf16(tp, 64 + i, c0 / 8, x);
        }
        fence_proxy_async_smem();
        wg_sync(barid);
        if (t == 0) mbar_arrive(ctl.bar(B_TP_READY + g));

        ok = ctl.wait(B_PT_FULL + g, (uint32_t)it);
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        if (t < 64) {  // PT -> bf16 over P
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                tmem_ld32f(tmem + lane_base + colG + 32u * part, x);
                store_row32_bf16(tp, t, 4 * part, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(barid);
        if (t == 0) {
            mbar_arrive(ctl.bar(B_TP_FULL + g));
            mbar_arrive(ctl.bar(B_G_EMPTY + g));
        }

        ok = ctl.wait(B_DW_FULL + g, (uint32_t)it);
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        // rows 0-63: Q' = Q - PT K over the Q rows; rows 64-127: -W into the W rows.
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float x[32];
            tmem_ld32f(tmem + lane_base + COL_DW + 32u * part, x);
            const uint32_t region = kqw + (uint32_t)(part >> 1) * kRegKQW;
            const int ch0 = 4 * (part & 1);
            if (t < 64) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint32_t addr = region + sw128(64 + row, ch0 + cc);
                    const uint4 qv = ld_shared_v4(addr);
                    const float2 a0 = unpack_bf16(qv.x), a1 = unpack_bf16(qv.y),
                                 a2 = unpack_bf16(qv.z), a3 = unpack_bf16(qv.w);
                    const float* d = x + 8 * cc;
                    st_shared_v4(addr, pack_bf16(a0.x - d[0], a0.y - d[1]),
                                 pack_bf16(a1.x - d[2], a1.y - d[3]),
                                 pack_bf16(a2.x - d[4], a2.y - d[5]),
                                 pack_bf16(a3.x - d[6], a3.y - d[7]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = -x[e];
                store_row32_bf16(region, 128 + row, ch0, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(barid);
        if (t == 0) {
            mbar_arrive(ctl.bar(B_DW_EMPTY));
            mbar_arrive(ctl.bar(B_QW_READY + g));
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const __nv_bfloat16* __restrict__ beta, const float* __restrict__ S0,
                float* __restrict__ S_T, int T) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    const Smem sm{base, smem_raw + (base - raw_addr)};
    int* const misc = reinterpret_cast<int*>(sm.gbase + OFF_MISC);
    const Ctl ctl{base + OFF_BAR, reinterpret_cast<volatile int*>(misc)};
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(misc + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        misc[0] = 0;
        for (int b = 0; b < kNumBars; ++b) mbar_init(ctl.bar(b), 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) producer_role(ctl, sm, &tm_q, &tm_k, &tm_v, bh, nchunks);
    } else if (warp == 1) {
        if (lane == 0) mma_role(ctl, sm, tmem, nchunks);
    } else if (warp == 2) {
        if (lane == 0) store_role(ctl, sm, &tm_o, bh, nchunks);
    } else if (warp >= 4 && warp < 8) {
        state_role(ctl, sm, tmem, tid - 128, S0, S_T, bh, nchunks);
    } else if (warp >= 8) {
        const int g = (warp - 8) >> 2;
        chunk_role(ctl, sm, tmem, tid - 256 - 128 * g, g, beta, bh, T, nchunks);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
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
