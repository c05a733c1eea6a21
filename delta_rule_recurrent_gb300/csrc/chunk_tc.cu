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
// which equals Q S + P U' exactly and lets one accumulator produce O and U':
//     D1 = [PT; Tm] V  (+)  [Q - PT K; -W] S    ->  rows 0-63: O, rows 64-127: U'
// Everything left of the (+) depends only on the chunk's own inputs, so the
// state-dependent chain per chunk is: S -> bf16 -> the D1 MMAs -> U' -> bf16
// -> S += K^T U'.
//
// One CTA owns one (batch, head) and keeps S in TMEM for the whole sequence.
// Its warps have fixed roles:
//   warp 0      TMA producer: [K; Q] tiles into a 3-stage ring, v tiles
//               (3-D maps, so rows past the end of a sequence read as zeros)
//   warp 1      TMEM owner
//   warps 4-7   state group: S -> bf16 operand, the D1 MMAs, the o tile
//               (TMA store from the spent half of the S operand), U',
//               S += K^T U', final state
//   warps 8-11, 12-15   chunk groups for even and odd chunks: G = [K; Q] K^T,
//               A and P, the triangular solve, Tm, PT and the [Q'; -W]
//               operand, which each group leaves in a TMEM buffer of its own
// A chunk group meets the state group only at the hand-over of its chunk and
// when it reuses its buffers two chunks later, so the groups run ahead of the
// state chain by up to a chunk each.  Each elected thread issues its role's
// MMAs and waits on its own commits.  Operand tiles in shared memory use the
// 128-byte swizzled layout TMA writes.
// Every wait is bounded: on a timeout the CTA records an error code (read
// back with dn_device_error), drains what it started and exits.
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

constexpr int kC = 64;         // chunk length
constexpr int kD = 128;        // dk = dv
constexpr int kThreads = 512;  // 16 warps
constexpr int kStages = 3;     // [K; Q] ring depth
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s without progress
// The polling roles count SM cycles (clock64 is cheap to read); at the
// GB300's clocks 4e9 cycles is 2 s or more.
constexpr long long kTimeoutCycles = 4000000000ll;
constexpr int kP = 68;   // row pitch (floats) of the fp32 solve array: 16-byte rows,
                         // and 8 consecutive rows of a 128-bit access hit 8 distinct bank groups
constexpr int kYP = 36;  // row pitch of the 32 x 32 solve scratch

// ---------------------------------------------------------------- smem map
constexpr uint32_t kRegKQ = 128 * 128;               // one dk half of [K; Q]: 128 rows x 128 B
constexpr uint32_t kStageKQ = 2 * kRegKQ;            // 32 KB
constexpr uint32_t OFF_KQ = 0;                       // kStages stages
constexpr uint32_t OFF_V = OFF_KQ + kStages * kStageKQ;  // V, 2 dv halves x 64 rows
constexpr uint32_t OFF_TP = OFF_V + 16384;           // 2 x [PT; Tm] (one per chunk group)
constexpr uint32_t OFF_SB = OFF_TP + 2 * 16384;      // S as bf16 (2 x 128 rows); then U', o tile
constexpr uint32_t OFF_X = OFF_SB + 32768;           // 2 x fp32 64 x kP: A, overwritten by X
constexpr uint32_t kXBytes = 64 * kP * 4;
constexpr uint32_t OFF_Y = OFF_X + 2 * kXBytes;      // 2 x fp32 32 x kYP solve scratch
constexpr uint32_t kYBytes = 32 * kYP * 4;
constexpr uint32_t OFF_BETA = OFF_Y + 2 * kYBytes;   // 2 x 64 fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 512;         // mbarriers, 8 bytes each
constexpr int kNumBars = 26;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * kNumBars;  // abort flag, TMEM address
constexpr uint32_t kSmemBytes = OFF_MISC + 16 + 1024;  // + 1024-byte alignment slack
static_assert(OFF_V % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_SB % 1024 == 0, "tile alignment");
static_assert(OFF_X % 16 == 0 && OFF_Y % 16 == 0 && OFF_BETA % 16 == 0, "vector alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// mbarrier indices.  Every barrier has exactly one waiting role, which
// consumes its phases in order, so a parity test can never see a phase two
// ahead of the one it asks for.  Barriers indexed [2] belong to the chunk
// group of that parity; [6] is (stage, group): chunk c uses c % 6.
enum : int {
    B_KQ_FULL = 0,     // [6] q, k tiles landed               (producer -> chunk group)
    B_KQ_EMPTY = 6,    // [3] stage's last reader done         (state MMA -> producer)
    B_V_FULL = 9,      // v tile landed                        (producer -> state group)
    B_V_EMPTY = 10,    // D1 MMAs done, v tile free            (state MMA -> producer)
    B_G_FULL = 11,     // [2] G = [K;Q] K^T done               (own commit)
    B_PT_FULL = 13,    // [2] PT = P Tm done                   (own commit)
    B_DW_FULL = 15,    // [2] DW = [PT;Tm] K done              (own commit)
    B_QW_READY = 17,   // [2] [PT; Tm] and [Q'; -W] ready      (chunk group -> state group)
    B_FREE = 19,       // [2] D1 MMAs read them; both free     (state MMA -> chunk group)
    B_D1_FULL = 21,    // D1 done                              (own commit, state group)
    B_S_READY = 22,    // S += K^T U' done                     (own commit, state group)
    B_DRAIN = 23,      // [3] final drain of each issuer's MMAs (state, group 0, group 1)
};

// TMEM columns (512 allocated):
//   S | D1 (O, U') | per chunk group g: [Q'; -W] bf16 (64), then G / PT (64)
// DW = [PT; Tm] K spans a group's 128 columns (dk 0-63 in the [Q'; -W]
// columns, dk 64-127 in the G columns) before being packed into the first 64.
constexpr uint32_t COL_S = 0, COL_D1 = 128, COL_GRP = 256;

constexpr uint32_t IDESC_G = idesc_bf16_f32(128, 64, 0, 0);    // [K;Q] K^T
constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0, 1);  // A K-major, B MN-major, N = 64
constexpr uint32_t IDESC_KB = idesc_bf16_f32(128, 128, 0, 1);  // A K-major (smem or TMEM), B MN-major
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
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&x)[64]) {
    uint32_t r[64];
    tmem_ld64(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i]);
}
// 64 fp32 values -> bf16 into the 8 chunks of row r of a swizzled region.
__device__ __forceinline__ void store_row64_bf16(uint32_t region, int r, const float (&x)[64]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(region + sw128(r, c), pack_bf16(x[8 * c + 0], x[8 * c + 1]),
                     pack_bf16(x[8 * c + 2], x[8 * c + 3]), pack_bf16(x[8 * c + 4], x[8 * c + 5]),
                     pack_bf16(x[8 * c + 6], x[8 * c + 7]));
}
__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void sts4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void fma4(float4& acc, float a, const float4& b) {
    acc.x = fmaf(a, b.x, acc.x);
    acc.y = fmaf(a, b.y, acc.y);
    acc.z = fmaf(a, b.z, acc.z);
    acc.w = fmaf(a, b.w, acc.w);
}
__device__ __forceinline__ float4 neg4(float4 v) { return make_float4(-v.x, -v.y, -v.z, -v.w); }
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
// 16-bit read-only global load that the compiler keeps in program order.
__device__ __forceinline__ uint16_t ld_nc_u16(const void* p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
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

// Group wait: thread 0 of the warpgroup polls the barrier, the others sleep
// in the named barrier.  True for the whole group, or false for the whole
// group if the wait gave up.
__device__ __forceinline__ bool wg_wait(const Ctl& ctl, int b, uint32_t parity, int t, int barid) {
    bool ok = true;
    if (t == 0) ok = ctl.wait(b, parity);
    return !wg_sync_or(barid, !ok);
}

struct Smem {
    uint32_t base;   // shared address of the 1024-aligned base
    uint8_t* gbase;  // generic pointer to it
    __device__ uint32_t kq(int s) const { return base + OFF_KQ + (uint32_t)s * kStageKQ; }
    __device__ uint32_t tp(int g) const { return base + OFF_TP + (uint32_t)g * 16384u; }
    __device__ uint32_t v() const { return base + OFF_V; }
    __device__ uint32_t sb() const { return base + OFF_SB; }
    __device__ float* x(int g) const {
        return reinterpret_cast<float*>(gbase + OFF_X + (uint32_t)g * kXBytes);
    }
    __device__ float* y(int g) const {
        return reinterpret_cast<float*>(gbase + OFF_Y + (uint32_t)g * kYBytes);
    }
    __device__ float* beta(int g) const {
        return reinterpret_cast<float*>(gbase + OFF_BETA + (uint32_t)g * 256u);
    }
};

// ------------------------------------------------- triangular solve, in place
// X <- (I + A)^{-1} for a strictly lower-triangular 64 x 64 A held in X (row
// pitch kP, zeros on and above the diagonal), by one warpgroup (t = 0..127).
// The pages compute this inverse by forward substitution, in blocks of 16
// tokens ("Hardware-efficient implementation", section 3 of
// paperlayer.ai/abs/2406.06484v6; "Pipeline Triton Chunkwise",
// fr.news.hada.io/topic?id=31925).  Here:
//   - the four 16 x 16 diagonal blocks by right-looking column substitution;
//   - 16 -> 32: inside each 32-row half, X_10 = -X_11 A_10 X_00;
//   - 32 -> 64: X_[10] = -X_[11] A_[10] X_[00] with 32 x 32 blocks, skipping
//     the known zero quarter of X_[00] and of X_[11].
// A block of A is only read while forming the block of X at its position, so
// X overwrites A in place.  Ys (32 x kYP floats) holds the intermediate
// products.  Shared-memory bandwidth bounds this routine, so every thread
// keeps a small register tile and reads with 128-bit loads.
__device__ __forceinline__ void solve_unit_lower64(float* X, float* Ys, int t, int barid) {
    if (t < 64) {
        const int base = (t >> 4) * 16, c = t & 15;
        const float* blk = X + base * (kP + 1);  // &X[base][base]
        float x[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) x[l] = (l == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r)
#pragma unroll
            for (int l = r + 1; l < 16; ++l) x[l] = fmaf(-blk[l * kP + r], x[r], x[l]);
        wg_sync(barid);
#pragma unroll
        for (int l = 0; l < 16; ++l) X[(base + l) * kP + base + c] = x[l];
    } else {
        wg_sync(barid);
    }
    wg_sync(barid);
    {   // 16 -> 32 in both halves: thread (half h, row r, 4 columns c4)
        const int h = t >> 6, r = (t >> 2) & 15, c4 = (t & 3) * 4;
        const int o = 32 * h;
        const float* arow = X + (o + 16 + r) * kP + o;
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
            const float4 a = lds4(arow + k);
            fma4(y, a.x, lds4(X + (o + k + 0) * kP + o + c4));
            fma4(y, a.y, lds4(X + (o + k + 1) * kP + o + c4));
            fma4(y, a.z, lds4(X + (o + k + 2) * kP + o + c4));
            fma4(y, a.w, lds4(X + (o + k + 3) * kP + o + c4));
        }
        sts4(Ys + (16 * h + r) * kYP + c4, y);
        wg_sync(barid);
        const float* xrow = X + (o + 16 + r) * kP + o + 16;
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 a = lds4(xrow + m);
            fma4(z, a.x, lds4(Ys + (16 * h + m + 0) * kYP + c4));
            fma4(z, a.y, lds4(Ys + (16 * h + m + 1) * kYP + c4));
            fma4(z, a.z, lds4(Ys + (16 * h + m + 2) * kYP + c4));
            fma4(z, a.w, lds4(Ys + (16 * h + m + 3) * kYP + c4));
        }
        sts4(X + (o + 16 + r) * kP + o + c4, neg4(z));
        wg_sync(barid);
    }
    {   // 32 -> 64: thread (rows r and r + 16, 4 columns c); c is warp-uniform
        const int r = t & 15, c = (t >> 4) * 4;
        const float* a0 = X + (32 + r) * kP;
        const float* a1 = X + (48 + r) * kP;
        float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
        auto ystep = [&](int k) {
            const float4 p = lds4(a0 + k), q = lds4(a1 + k);
            const float4 x0 = lds4(X + (k + 0) * kP + c), x1 = lds4(X + (k + 1) * kP + c);
            const float4 x2 = lds4(X + (k + 2) * kP + c), x3 = lds4(X + (k + 3) * kP + c);
            fma4(y0, p.x, x0); fma4(y0, p.y, x1); fma4(y0, p.z, x2); fma4(y0, p.w, x3);
            fma4(y1, q.x, x0); fma4(y1, q.y, x1); fma4(y1, q.z, x2); fma4(y1, q.w, x3);
        };
        if (c < 16) {
#pragma unroll
            for (int k = 0; k < 32; k += 4) ystep(k);
        } else {  // rows 0-15 of X_[00] are zero in columns 16-31
#pragma unroll
            for (int k = 16; k < 32; k += 4) ystep(k);
        }
        sts4(Ys + r * kYP + c, y0);
        sts4(Ys + (16 + r) * kYP + c, y1);
        wg_sync(barid);
        const float* x0r = X + (32 + r) * kP + 32;
        const float* x1r = X + (48 + r) * kP + 32;
        float4 z0 = make_float4(0.f, 0.f, 0.f, 0.f), z1 = z0;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {  // row r of X_[11] is zero past column 15
            const float4 p = lds4(x0r + m), q = lds4(x1r + m);
            const float4 y_0 = lds4(Ys + (m + 0) * kYP + c), y_1 = lds4(Ys + (m + 1) * kYP + c);
            const float4 y_2 = lds4(Ys + (m + 2) * kYP + c), y_3 = lds4(Ys + (m + 3) * kYP + c);
            fma4(z0, p.x, y_0); fma4(z0, p.y, y_1); fma4(z0, p.z, y_2); fma4(z0, p.w, y_3);
            fma4(z1, q.x, y_0); fma4(z1, q.y, y_1); fma4(z1, q.z, y_2); fma4(z1, q.w, y_3);
        }
#pragma unroll
        for (int m = 16; m < 32; m += 4) {
            const float4 q = lds4(x1r + m);
            fma4(z1, q.x, lds4(Ys + (m + 0) * kYP + c));
            fma4(z1, q.y, lds4(Ys + (m + 1) * kYP + c));
            fma4(z1, q.z, lds4(Ys + (m + 2) * kYP + c));
            fma4(z1, q.w, lds4(Ys + (m + 3) * kYP + c));
        }
        sts4(X + (32 + r) * kP + c, neg4(z0));
        sts4(X + (48 + r) * kP + c, neg4(z1));
        wg_sync(barid);
    }
}


// ----------------------------------------------------------------- roles
__device__ void producer_role(const Ctl& ctl, const Smem& sm, const CUtensorMap* tm_q,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, int bh,
                              int nchunks) {
    int nkq = 0, nv = 0;
    long long t0 = clock64();
    while ((nkq < nchunks || nv < nchunks) && !ctl.aborted()) {
        bool progressed = false;
        const int s = nkq % kStages;
        if (nkq < nchunks &&
            (nkq < kStages ||
             mbar_test_wait(ctl.bar(B_KQ_EMPTY + s), (uint32_t)(nkq / kStages - 1) & 1u))) {
            const uint32_t st = sm.kq(s), bar = ctl.bar(B_KQ_FULL + nkq % 6);
            mbar_arrive_expect_tx(bar, 4 * 8192);
            tma_load_3d(st, tm_k, bar, 0, nkq * kC, bh);
            tma_load_3d(st + kRegKQ, tm_k, bar, 64, nkq * kC, bh);
            tma_load_3d(st + 8192, tm_q, bar, 0, nkq * kC, bh);
            tma_load_3d(st + kRegKQ + 8192, tm_q, bar, 64, nkq * kC, bh);
            if (nkq + kStages < nchunks) {  // warm L2 for this stage's next tiles
                const int y = (nkq + kStages) * kC;
                tma_prefetch_l2_3d(tm_k, 0, y, bh);
                tma_prefetch_l2_3d(tm_k, 64, y, bh);
                tma_prefetch_l2_3d(tm_q, 0, y, bh);
                tma_prefetch_l2_3d(tm_q, 64, y, bh);
            }
            ++nkq;
            progressed = true;
        }
        if (nv < nchunks && (nv < 1 || mbar_test_wait(ctl.bar(B_V_EMPTY), (uint32_t)(nv - 1) & 1u))) {
            const uint32_t bar = ctl.bar(B_V_FULL);
            mbar_arrive_expect_tx(bar, 2 * 8192);
            tma_load_3d(sm.v(), tm_v, bar, 0, nv * kC, bh);
            tma_load_3d(sm.v() + 8192, tm_v, bar, 64, nv * kC, bh);
            if (nv + 1 < nchunks) {  // the v tile is single-buffered: warm L2 for the next one
                tma_prefetch_l2_3d(tm_v, 0, (nv + 1) * kC, bh);
                tma_prefetch_l2_3d(tm_v, 64, (nv + 1) * kC, bh);
            }
            ++nv;
            progressed = true;
        }
        if (progressed) {
            t0 = clock64();
        } else {
            __nanosleep(64);  // loads run well ahead; stay off the issue slots
            if (clock64() - t0 > kTimeoutCycles) ctl.raise();
        }
    }
    // Leave nothing in flight: wait (bounded) for the last load on each barrier.
    for (int b = 0; b < 6; ++b) {
        const int n_b = (nkq - b + 5) / 6;  // loads that completed on barrier b
        if (n_b > 0) mbar_wait(ctl.bar(B_KQ_FULL + b), (uint32_t)(n_b - 1) & 1u, kTimeoutNs);
    }
    if (nv > 0) mbar_wait(ctl.bar(B_V_FULL), (uint32_t)(nv - 1) & 1u, kTimeoutNs);
}

// Lets everything a thread issued to the tensor core finish (bounded), so
// TMEM and shared memory can be released safely.
__device__ __forceinline__ void drain_mmas(const Ctl& ctl, int b) {
    mma_commit(ctl.bar(b));
    mbar_wait(ctl.bar(b), 0, kTimeoutNs);
}

// State group (warps 4-7): thread t owns state row t = TMEM lane t; thread 0
// issues the state group's MMAs.
__device__ void state_role_body(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t,
                                const float* __restrict__ S0, float* __restrict__ S_T,
                                const CUtensorMap* tm_o, int bh, int nchunks) {
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
        const int g = c & 1;
        // S += K^T U' of the previous chunk done, and its o tile read out by TMA.
        if (c > 0) {
            bool ok0 = true;
            if (t == 0) {
                ok0 = ctl.wait(B_S_READY, (uint32_t)(c - 1));
                bulk_wait_group_read0();
            }
            if (wg_sync_or(kBar, !ok0)) return;
        }
        tc_fence_after_sync();
        // S (fp32) -> bf16 operand tile: dv halves as regions, row t.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[64];
            tmem_ld64f(tmem + lane_base + COL_S + 64u * half, x);
            store_row64_bf16(sm.sb() + (uint32_t)half * 16384u, t, x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(kBar);
        // D1 = [PT; Tm] V + [Q'; -W] S once the chunk group has handed its chunk over.
        bool ok = true;
        if (t == 0) {
            ok = ctl.wait(B_QW_READY + g, (uint32_t)(c >> 1)) && ctl.wait(B_V_FULL, (uint32_t)c);
            if (ok) {
                tc_fence_after_sync();
                const uint32_t tp = sm.tp(g), qw = tmem + COL_GRP + 128u * (uint32_t)g;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + COL_D1, sw128_desc(tp + 32u * kk, 16, 1024),
                                sw128_desc(sm.v() + 2048u * kk, 8192, 1024), IDESC_KB, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + COL_D1, qw + 8u * kk,
                                sw128_desc(sm.sb() + 2048u * kk, 16384, 1024), IDESC_KB, 1);
                mma_commit(ctl.bar(B_D1_FULL));
                mma_commit(ctl.bar(B_V_EMPTY));
                mma_commit(ctl.bar(B_FREE + g));
                ok = ctl.wait(B_D1_FULL, (uint32_t)c);
            }
        }
        if (wg_sync_or(kBar, !ok)) return;
        tc_fence_after_sync();
        // The S operand is spent: rows 0-63 (o) into its upper 16 KB as the o
        // tile, rows 64-127 (U') into its lower 16 KB.
        {
            const uint32_t dst = sm.sb() + (t < 64 ? 16384u : 0u);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[64];
                tmem_ld64f(tmem + lane_base + COL_D1 + 64u * half, x);
                store_row64_bf16(dst + (uint32_t)half * 8192u, t & 63, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(kBar);
        if (t == 0) {
            // o tile out (rows past the end of the sequence are clipped)
            tma_store_3d(tm_o, sm.sb() + 16384u, 0, c * kC, bh);
            tma_store_3d(tm_o, sm.sb() + 24576u, 64, c * kC, bh);
            bulk_commit_group();
            // S += K^T U'
            const uint32_t kq = sm.kq(c % kStages);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + COL_S, sw128_desc(kq + 2048u * kk, kRegKQ, 1024),
                            sw128_desc(sm.sb() + 2048u * kk, 8192, 1024), IDESC_MM, 1);
            mma_commit(ctl.bar(B_S_READY));
            mma_commit(ctl.bar(B_KQ_EMPTY + c % kStages));
        }
    }
    if (nchunks > 0 && !wg_wait(ctl, B_S_READY, (uint32_t)(nchunks - 1), t, kBar)) return;
    tc_fence_after_sync();
    if (S_T) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[64];
            tmem_ld64f(tmem + lane_base + COL_S + 64u * half, x);
            float4* dst = reinterpret_cast<float4*>(S_T + ((size_t)bh * kD + t) * kD + 64 * half);
#pragma unroll
            for (int v4 = 0; v4 < 16; ++v4)
                dst[v4] = make_float4(x[4 * v4], x[4 * v4 + 1], x[4 * v4 + 2], x[4 * v4 + 3]);
        }
    }
}

__device__ void state_role(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t,
                           const float* __restrict__ S0, float* __restrict__ S_T,
                           const CUtensorMap* tm_o, int bh, int nchunks) {
    state_role_body(ctl, sm, tmem, t, S0, S_T, tm_o, bh, nchunks);
    if (t == 0) {
        drain_mmas(ctl, B_DRAIN + 0);
        bulk_wait_group0();  // o tiles written
    }
}

// One quarter (32 dk columns) of the [Q'; -W] operand, packed to bf16 pairs:
// rows 0-63 (t < 64) take Q - PT K with Q from the chunk's q tile, rows 64-127
// take -W.  `x` holds the fp32 DW values of the quarter for this row.
__device__ __forceinline__ void qw_quarter(const float (&x)[32], bool is_q, uint32_t q_region,
                                           int row, int ch0, uint32_t* pk) {
    if (is_q) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint4 qv = ld_shared_v4(q_region + sw128(64 + row, ch0 + cc));
            const float2 a0 = unpack_bf16(qv.x), a1 = unpack_bf16(qv.y), a2 = unpack_bf16(qv.z),
                         a3 = unpack_bf16(qv.w);
            const float* d = x + 8 * cc;
            pk[4 * cc + 0] = pack_bf16(a0.x - d[0], a0.y - d[1]);
            pk[4 * cc + 1] = pack_bf16(a1.x - d[2], a1.y - d[3]);
            pk[4 * cc + 2] = pack_bf16(a2.x - d[4], a2.y - d[5]);
            pk[4 * cc + 3] = pack_bf16(a3.x - d[6], a3.y - d[7]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(-x[2 * e], -x[2 * e + 1]);
    }
}

// Chunk group g (0: even chunks, warps 8-11; 1: odd chunks, warps 12-15);
// thread 0 issues the group's MMAs.  Iteration `it` handles chunk c = g + 2 it.
__device__ void chunk_role_body(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t, int g,
                                const __nv_bfloat16* __restrict__ beta, int bh, int T,
                                int nchunks) {
    const int barid = 2 + g;
    const uint32_t lane_base = (uint32_t)(32 * (t >> 5)) << 16;
    const uint32_t colQW = COL_GRP + 128u * (uint32_t)g, colG = colQW + 64u;
    float* const X = sm.x(g);
    float* const Ys = sm.y(g);
    float* const betas = sm.beta(g);
    const uint32_t tp = sm.tp(g);
    const int row = t & 63;
    const __nv_bfloat16* const beta_bh = beta + (size_t)bh * T;
    // Strengths of the group's next chunk, loaded one iteration ahead (0 past
    // T); the load is issued as volatile PTX so it stays where it is written.
    uint16_t bnext = 0;
    if (t < kC && g * kC + t < T) bnext = ld_nc_u16(beta_bh + g * kC + t);

    for (int c = g, it = 0; c < nchunks; c += 2, ++it) {
        const uint32_t kq = sm.kq(c % kStages);
        if (t < kC) {
            betas[t] = __bfloat162float(__ushort_as_bfloat16(bnext));
            const int nx = (c + 2) * kC + t;
            bnext = nx < T ? ld_nc_u16(beta_bh + nx) : (uint16_t)0;
        }
        // G = [K; Q] K^T
        bool ok = true;
        if (t == 0) {
            ok = ctl.wait(B_KQ_FULL + c % 6, (uint32_t)(c / 6));
            if (ok) {
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t a = kq + (uint32_t)(kk >> 2) * kRegKQ + (uint32_t)(kk & 3) * 32u;
                    mma_bf16_ss(tmem + colG, sw128_desc(a, 16, 1024), sw128_desc(a, 16, 1024),
                                IDESC_G, kk > 0);
                }
                mma_commit(ctl.bar(B_G_FULL + g));
                ok = ctl.wait(B_G_FULL + g, (uint32_t)it);
            }
        }
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        // A = beta_i (k_i . k_j) for j < i (TMEM rows 0-63) into the fp32 solve
        // array.  P (rows 64-127) stays in TMEM until the solve is done.
        if (t < 64) {
            float x[64];
            tmem_ld64f(tmem + lane_base + colG, x);
            const float bi = betas[row];
#pragma unroll
            for (int j = 0; j < 64; j += 4)
                sts4(X + row * kP + j,
                     make_float4(j + 0 < row ? bi * x[j + 0] : 0.f, j + 1 < row ? bi * x[j + 1] : 0.f,
                                 j + 2 < row ? bi * x[j + 2] : 0.f, j + 3 < row ? bi * x[j + 3] : 0.f));
        }
        tc_fence_before_sync();
        wg_sync(barid);
        solve_unit_lower64(X, Ys, t, barid);
        // [PT; Tm] and [Q'; -W] of chunk c - 2 must have been read by the state group.
        if (it > 0 && !wg_wait(ctl, B_FREE + g, (uint32_t)(it - 1), t, barid)) return;
        tc_fence_after_sync();
        {
            float x[64];
            if (t < 64) {  // Tm row t = X row t diag(beta) -> bf16 row 64 + t of [PT; Tm]
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    const float4 xv = lds4(X + t * kP + e), bv = lds4(betas + e);
                    x[e] = xv.x * bv.x;
                    x[e + 1] = xv.y * bv.y;
                    x[e + 2] = xv.z * bv.z;
                    x[e + 3] = xv.w * bv.w;
                }
                store_row64_bf16(tp, 64 + t, x);
            } else {  // P row: q_t . k_j for j <= t -> bf16 row t of [PT; Tm]
                tmem_ld64f(tmem + lane_base + colG, x);
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j > row) x[j] = 0.f;
                store_row64_bf16(tp, row, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(barid);
        // PT = P Tm into the group's columns
        ok = true;
        if (t == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + colG, sw128_desc(tp + 32u * kk, 16, 1024),
                            sw128_desc(tp + 8192u + 2048u * kk, 8192, 1024), IDESC_N64, kk > 0);
            mma_commit(ctl.bar(B_PT_FULL + g));
            ok = ctl.wait(B_PT_FULL + g, (uint32_t)it);
        }
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        if (t < 64) {  // PT -> bf16 over P
            float x[64];
            tmem_ld64f(tmem + lane_base + colG, x);
            store_row64_bf16(tp, t, x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        wg_sync(barid);
        // DW = [PT; Tm] K over the group's 128 columns
        ok = true;
        if (t == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + colQW, sw128_desc(tp + 32u * kk, 16, 1024),
                            sw128_desc(kq + 2048u * kk, kRegKQ, 1024), IDESC_KB, kk > 0);
            mma_commit(ctl.bar(B_DW_FULL + g));
            ok = ctl.wait(B_DW_FULL + g, (uint32_t)it);
        }
        if (wg_sync_or(barid, !ok)) return;
        tc_fence_after_sync();
        // [Q'; -W] as bf16 pairs into the group's first 64 columns; all of DW
        // is read before the packed operand overwrites its dk 0-63 half.
        {
            const bool is_q = t < 64;
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {  // dk quarter qd sits in columns colQW + 32 qd
                float x[32];
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + colQW + 32u * (uint32_t)qd, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
                qw_quarter(x, is_q, kq + (uint32_t)(qd >> 1) * kRegKQ, row, (qd & 1) * 4,
                           (qd < 2 ? lo : hi) + 16 * (qd & 1));
            }
            tmem_st32(tmem + lane_base + colQW, lo);
            tmem_st32(tmem + lane_base + colQW + 32u, hi);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        wg_sync(barid);
        if (t == 0) mbar_arrive(ctl.bar(B_QW_READY + g));
    }
}

__device__ void chunk_role(const Ctl& ctl, const Smem& sm, uint32_t tmem, int t, int g,
                           const __nv_bfloat16* __restrict__ beta, int bh, int T, int nchunks) {
    chunk_role_body(ctl, sm, tmem, t, g, beta, bh, T, nchunks);
    if (t == 0) drain_mmas(ctl, B_DRAIN + 1 + g);
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
    } else if (warp >= 4 && warp < 8) {
        state_role(ctl, sm, tmem, tid - 128, S0, S_T, &tm_o, bh, nchunks);
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
