// chunk_simt.cu -- chunkwise delta-rule forward on CUDA cores, fp32 throughout.
//
// This is the full-precision path (fp32 I/O is held to 1e-4 relative L2,
// which bf16 or tf32 tensor-core operands cannot meet) and the fallback for
// shapes the tensor-core kernel does not cover.
//
// Chunk algebra ("Chunkwise KDA : réorganiser la récurrence en
// multiplications matricielles", fr.news.hada.io/topic?id=31925, with the
// decay D = I; appendix B.2 "UT transform" of paperlayer.ai/abs/2406.06484v6).
// For a chunk of C tokens (rows of K, Q, V) and incoming state S ([dk][dv]):
//     A   = tril(diag(beta) K K^T, -1)            (strictly lower)
//     X   = (I + A)^{-1}                          (blocked forward substitution)
//     R'  = diag(beta) (V - K S)
//     U'  = X R'                                  (the true per-token errors)
//     O   = Q S + (Q K^T . M) U'                  (M: causal incl. diagonal)
//     S  <- S + K^T U'
// A CTA owns one (batch, head) and a slice of NV value channels; it walks the
// chunks in order with its slice of S resident in shared memory.  For the
// backward pass it can also record the state at the start of every chunk
// (S_chunks, [BH][chunk][dk][dv] fp32) and skip the outputs (o == nullptr).  Value
// channels are independent in every step above, so slices never exchange
// data; the key-side work (A, X, Q K^T) is recomputed per slice.
//
// Gated DeltaNet (a log keep rate g_t per token, alpha_t = exp(g_t); "Gated
// DeltaNet : oublier d'abord l'état entier", fr.news.hada.io/topic?id=31925,
// and "Gated DeltaNet", garden.houmin.site/infra/delta-net) runs through the
// same kernel.  With G_t the cumulative log decay from the chunk start
// (G = 0 without g, which makes every factor below exactly 1):
//     A   = tril(diag(beta) (K K^T . exp(G_i - G_j)), -1)
//     R'  = diag(beta) (V - diag(exp G) K S)
//     O   = diag(exp G) Q S + (Q K^T . M . exp(G_i - G_j)) U'
//     S  <- exp(G_C) S + K^T diag(exp(G_C - G_s)) U'
// (the state S / Gamma_t follows the plain rule on values v_t / Gamma_t; the
// ratios of Gamma within a chunk are at most 1).
//
// KDA (one keep rate per key channel, "Kimi Delta Attention : atténuation
// par canal", same page) is the kChan instance: G_t[d] per channel, and
//     A[i][j] = beta_i sum_d k_i[d] k_j[d] exp(G_i[d] - G_j[d])          (j < i)
//     P[i][j] = sum_d q_i[d] k_j[d] exp(G_i[d] - G_j[d])                 (j <= i)
//     R'  = diag(beta) (V - (K . exp G) S),   O = (Q . exp G) S + P U'
//     S  <- diag(exp G_C) S + (K . exp(G_C - G))^T U'
// The ratios sit inside the sums, so every exponent is <= 0 however strong
// the decay (no 1 / Gamma factors).
#include <type_traits>
#include "dn_common.cuh"
#include "dn_internal.h"
#include "simt_mm.cuh"
#include "tile_load.cuh"
#include "tri_inverse.cuh"

namespace dn {
namespace {

using simt::kThreads;
using simt::mm_acc;
using simt::zero;
constexpr int kC = 64;         // chunk length
constexpr int kLC = kC + 1;    // odd row pitches keep shared-memory reads conflict-free

template <int DK, int NV, bool kChan = false>
struct SimtSmem {
    static constexpr int LK = DK + 1, LV = NV + 1;
    static constexpr int kK = 0;                       // C x LK   keys
    static constexpr int kQ = kK + kC * LK;            // C x LK   queries
    static constexpr int kR = kQ + kC * LK;            // C x LV   values, then R'
    static constexpr int kU = kR + kC * LV;            // C x LV   U'
    static constexpr int kS = kU + kC * LV;            // DK x LV  state slice
    static constexpr int kA = kS + DK * LV;            // C x kLC  A
    static constexpr int kX = kA + kC * kLC;           // C x kLC  (I + A)^{-1}
    static constexpr int kP = kX + kC * kLC;           // C x kLC  Q K^T . M
    static constexpr int kY = kP + kC * kLC;           // 3 x 16 x 17 solve scratch
    static constexpr int kB = kY + 3 * 16 * 17;        // C        beta
    static constexpr int kG = kB + kC;                 // 3 x C    G, exp(G), exp(G_C - G)
    static constexpr int kGk = kG + 3 * kC;            // C x LK   per-channel G (KDA)
    static constexpr int kFloats = kGk + (kChan ? kC * LK : 0);
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// NMAX > 1: packed variable-length sequences (the CTA's state index is
// (sequence, head); tokens come from the packed [H][T] layout).
template <typename T, int DK, int DV, int NV, int NMAX, bool kChan = false>
__global__ void __launch_bounds__(kThreads, 1)
chunk_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                  const T* __restrict__ v, const T* __restrict__ beta,
                  const float* __restrict__ S0, T* __restrict__ o,
                  float* __restrict__ S_T, float* __restrict__ S_chunks,
                  const float* __restrict__ g, int Ttot, int H,
                  const __grid_constant__ SeqTable<NMAX> seqs, QkNorm nm) {
    using L = SimtSmem<DK, NV, kChan>;
    constexpr int LK = L::LK, LV = L::LV;
    constexpr int NSLICE = DV / NV;
    extern __shared__ float smem[];
    float* Ks = smem + L::kK;
    float* Qs = smem + L::kQ;
    float* Rs = smem + L::kR;
    float* Us = smem + L::kU;
    float* Ss = smem + L::kS;
    float* Am = smem + L::kA;
    float* Xm = smem + L::kX;
    float* Pm = smem + L::kP;
    float* Ys = smem + L::kY;
    float* bs = smem + L::kB;
    float* Gc = smem + L::kG;          // cumulative log decay within the chunk
    float* eG = Gc + kC;               // exp(G_t)
    float* dec = eG + kC;              // exp(G_C - G_t)
    float* Gk = smem + L::kGk;         // KDA: cumulative log decay per key channel
    float* eC = Gc;                    // KDA: exp(G_C) per key channel (DK <= 3 C floats)
    static_assert(!kChan || DK <= 3 * kC, "room for exp(G_C)");

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int bh = blockIdx.x / NSLICE;  // the state's index
    const int j0 = (blockIdx.x % NSLICE) * NV;
    size_t tok0 = (size_t)bh * Ttot;
    int Tlen = Ttot;
    if constexpr (NMAX > 1) {
        const int n = bh / H, h = bh % H;
        tok0 = (size_t)h * Ttot + seqs.start[n];
        Tlen = seqs.start[n + 1] - seqs.start[n];
    }

    for (int e = tid; e < DK * NV; e += kThreads) {
        const int i = e / NV, jj = e % NV;
        Ss[i * LV + jj] = S0 ? S0[((size_t)bh * DK + i) * DV + j0 + jj] : 0.f;
    }

    const int nchunks = (Tlen + kC - 1) / kC;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kC;
        const int n = min(kC, Tlen - t0);
        if (S_chunks) {  // the state this chunk starts from
            for (int e = tid; e < DK * NV; e += kThreads) {
                const int i = e / NV, jj = e % NV;
                S_chunks[(((size_t)bh * nchunks + c) * DK + i) * DV + j0 + jj] = Ss[i * LV + jj];
            }
        }
        // ---- load the chunk (padding rows: k = q = v = 0, beta = 0) ----
        load_tile<kThreads, kC, DK, LK, DK>(Ks, k, tok0 + t0, n, 0);
        load_tile<kThreads, kC, DK, LK, DK>(Qs, q, tok0 + t0, n, 0);
        load_tile<kThreads, kC, NV, LV, DV>(Rs, v, tok0 + t0, n, j0);
        if (tid < kC) bs[tid] = tid < n ? to_f32(beta[tok0 + t0 + tid]) : 0.f;
        if (norm_active(nm)) {  // q and k prepared in place: thread r owns row r of [K; Q]
            __syncthreads();
            static_assert(2 * kC <= kThreads, "a thread per row");
            const bool is_q = tid >= kC;
            if (tid < 2 * kC && (is_q || nm.l2norm)) {
                float* const row = is_q ? Qs + (tid - kC) * LK : Ks + tid * LK;
                float f = is_q ? nm.qscale : 1.f;
                if (nm.l2norm) {
                    float ss = 0.f;
                    for (int d = 0; d < DK; ++d) ss = fmaf(row[d], row[d], ss);
                    f *= rsqrtf(ss + nm.eps);
                }
                for (int d = 0; d < DK; ++d) row[d] *= f;
            }
        }
        // KDA: while the chunk's decay stays within exp(-80) on every key
        // channel (G is non-increasing, so G_C is each channel's lowest), the
        // ratio exp(G_i - G_j) is the product exp(G_i) exp(-G_j) of two normal
        // fp32 numbers: K and Q become K exp(G), Q exp(G) in place and Gk
        // becomes K exp(-G), so A, P, the state read and the update are plain
        // products.  Otherwise every ratio takes its own clamped exponential.
        bool sep = false;
        if constexpr (kChan) {  // per-channel rates, then prefix sums over the chunk
            load_tile<kThreads, kC, DK, LK, DK>(Gk, g, tok0 + t0, n, 0);
            __syncthreads();
            if (tid < DK)
                for (int t = 1; t < kC; ++t) Gk[t * LK + tid] += Gk[(t - 1) * LK + tid];
            __syncthreads();
            sep = __syncthreads_and(tid >= DK || Gk[(kC - 1) * LK + tid] >= -80.f);
            if (sep) {
                if (tid < DK) eC[tid] = __expf(Gk[(kC - 1) * LK + tid]);
                for (int e = tid; e < kC * DK; e += kThreads) {
                    const int t = e / DK, d = e % DK;
                    const float G = Gk[t * LK + d], kv = Ks[t * LK + d];
                    const float ep = __expf(G);
                    Ks[t * LK + d] = kv * ep;
                    Qs[t * LK + d] *= ep;
                    Gk[t * LK + d] = kv * __expf(-G);
                }
            }
        } else if (tid < 32) {  // prefix sums of the log keep rates (padding tokens keep everything)
            const int t = 2 * tid;
            const float a = (g && t < n) ? g[tok0 + t0 + t] : 0.f;
            const float b = (g && t + 1 < n) ? g[tok0 + t0 + t + 1] : 0.f;
            float incl = a + b;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += y;
            }
            const float last = __shfl_sync(0xffffffffu, incl, 31);
            const float g0 = incl - b;
            Gc[t] = g0;
            Gc[t + 1] = incl;
            eG[t] = expf(g0);
            eG[t + 1] = expf(incl);
            dec[t] = expf(last - g0);
            dec[t + 1] = expf(last - incl);
        }
        __syncthreads();

        // ---- A = tril(diag(beta) K K^T, -1) and P = tril(Q K^T) ----
        // (the KDA forms choose once per chunk, so every inner loop below is
        // compiled for one form and carries no per-element branch)
        auto form_ap = [&](auto per_entry) {
            constexpr bool kExp = decltype(per_entry)::value;
            const float* const Bk = (kChan && !kExp) ? Gk : Ks;  // KDA product form: K exp(-G)
            float aa[4][4], ap[4][4];
            zero<64, 64>(aa);
            zero<64, 64>(ap);
#pragma unroll 2
            for (int kk = 0; kk < DK; ++kk) {
                float ak[4], aq[4], bk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ak[i] = Ks[(ty + 16 * i) * LK + kk];
                    aq[i] = Qs[(ty + 16 * i) * LK + kk];
                    bk[i] = Bk[(tx + 16 * i) * LK + kk];
                }
                if constexpr (kExp) {  // the channel's decay ratio inside the sum
                    float gi[4], gj[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        gi[i] = Gk[(ty + 16 * i) * LK + kk];
                        gj[i] = Gk[(tx + 16 * i) * LK + kk];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {  // pairs past the diagonal are masked below
                            const float e = __expf(fminf(gi[i] - gj[j], 0.f));
                            aa[i][j] = fmaf(ak[i] * e, bk[j], aa[i][j]);
                            ap[i][j] = fmaf(aq[i] * e, bk[j], ap[i][j]);
                        }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            aa[i][j] = fmaf(ak[i], bk[j], aa[i][j]);
                            ap[i][j] = fmaf(aq[i], bk[j], ap[i][j]);
                        }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int m = ty + 16 * i, nn = tx + 16 * j;
                    const float r = kChan ? 1.f : (nn <= m ? expf(Gc[m] - Gc[nn]) : 0.f);
                    Am[m * kLC + nn] = nn < m ? bs[m] * (aa[i][j] * r) : 0.f;
                    Pm[m * kLC + nn] = nn <= m ? ap[i][j] * r : 0.f;
                }
        };
        if (kChan && !sep)
            form_ap(std::true_type{});
        else
            form_ap(std::false_type{});
        __syncthreads();

        // ---- R' = diag(beta) (V - diag(exp G) K S), in place over V ----
        {
            float acc[4][NV / 16];
            zero<64, NV>(acc);
            const auto state = [&](int kk, int nn) { return Ss[kk * LV + nn]; };
            if (kChan && !sep)
                mm_acc<64, NV, DK>(acc, [&](int m, int kk) {
                    return Ks[m * LK + kk] * __expf(Gk[m * LK + kk]);
                }, state);
            else
                mm_acc<64, NV, DK>(acc, [&](int m, int kk) { return Ks[m * LK + kk]; }, state);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < NV / 16; ++j) {
                    const int m = ty + 16 * i, nn = tx + 16 * j;
                    const float sc = kChan ? 1.f : eG[m];
                    Rs[m * LV + nn] = bs[m] * (Rs[m * LV + nn] - sc * acc[i][j]);
                }
        }
        // ---- X = (I + A)^{-1} (touches only Am, Xm, Ys; ends with a barrier) ----
        unit_lower_inverse64<kThreads>(Am, Xm, Ys);

        // ---- U' = X R' ----
        {
            float acc[4][NV / 16];
            zero<64, NV>(acc);
            mm_acc<64, NV, kC>(acc, [&](int m, int kk) { return Xm[m * kLC + kk]; },
                               [&](int kk, int nn) { return Rs[kk * LV + nn]; });
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < NV / 16; ++j)
                    Us[(ty + 16 * i) * LV + tx + 16 * j] = acc[i][j];
        }
        __syncthreads();

        // ---- O = diag(exp G) Q S + P U' ----
        if (o) {
            float acc[4][NV / 16];
            zero<64, NV>(acc);
            const auto state = [&](int kk, int nn) { return Ss[kk * LV + nn]; };
            if (kChan && !sep)
                mm_acc<64, NV, DK>(acc, [&](int m, int kk) {
                    return Qs[m * LK + kk] * __expf(Gk[m * LK + kk]);
                }, state);
            else
                mm_acc<64, NV, DK>(acc, [&](int m, int kk) { return Qs[m * LK + kk]; }, state);
            if constexpr (!kChan) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < NV / 16; ++j) acc[i][j] *= eG[ty + 16 * i];
            }
            mm_acc<64, NV, kC>(acc, [&](int m, int kk) { return Pm[m * kLC + kk]; },
                               [&](int kk, int nn) { return Us[kk * LV + nn]; });
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = ty + 16 * i;
                if (m < n) {
#pragma unroll
                    for (int j = 0; j < NV / 16; ++j)
                        o[(tok0 + t0 + m) * DV + j0 + tx + 16 * j] = from_f32<T>(acc[i][j]);
                }
            }
        }
        __syncthreads();

        // ---- S <- exp(G_C) S + K^T diag(exp(G_C - G)) U' ----
        {
            float acc[DK / 16][NV / 16];
            zero<DK, NV>(acc);
            const auto upd = [&](int kk, int nn) { return Us[kk * LV + nn]; };
            if constexpr (kChan) {
                if (sep)
                    mm_acc<DK, NV, kC>(acc, [&](int m, int kk) { return Gk[kk * LK + m] * eC[m]; },
                                       upd);
                else
                    mm_acc<DK, NV, kC>(acc, [&](int m, int kk) {
                        return Ks[kk * LK + m] * __expf(Gk[(kC - 1) * LK + m] - Gk[kk * LK + m]);
                    }, upd);
            } else {
                mm_acc<DK, NV, kC>(acc, [&](int m, int kk) { return Ks[kk * LK + m] * dec[kk]; },
                                   upd);
            }
#pragma unroll
            for (int i = 0; i < DK / 16; ++i) {
                const int row = ty + 16 * i;
                const float keep = kChan ? (sep ? eC[row] : __expf(Gk[(kC - 1) * LK + row]))
                                         : eG[kC - 1];
#pragma unroll
                for (int j = 0; j < NV / 16; ++j) {
                    float* const sp = Ss + row * LV + tx + 16 * j;
                    *sp = fmaf(keep, *sp, acc[i][j]);
                }
            }
        }
        __syncthreads();
    }

    if (S_T) {
        for (int e = tid; e < DK * NV; e += kThreads) {
            const int i = e / NV, jj = e % NV;
            S_T[((size_t)bh * DK + i) * DV + j0 + jj] = Ss[i * LV + jj];
        }
    }
}

template <typename T, int DK, int DV, int NMAX = 1, bool kChan = false>
cudaError_t launch_typed(const void* q, const void* k, const void* v,
                         const void* beta, const float* S0, void* o, float* S_T,
                         float* S_chunks, const float* g, int BH, int Tlen, cudaStream_t stream,
                         int H = 1, const SeqTable<NMAX>* seqs = nullptr,
                         const QkNorm& nm = kNoNorm) {
    constexpr int NV = DV < 64 ? DV : 64;
    using L = SimtSmem<DK, NV, kChan>;
    auto kern = chunk_simt_kernel<T, DK, DV, NV, NMAX, kChan>;
    cudaError_t err = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
    if (err != cudaSuccess) return err;
    const long long grid = (long long)BH * (DV / NV);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kThreads, L::kBytes, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k),
        static_cast<const T*>(v), static_cast<const T*>(beta), S0,
        static_cast<T*>(o), S_T, S_chunks, g, Tlen, H, seqs ? *seqs : SeqTable<NMAX>{}, nm);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dims(const void* q, const void* k, const void* v,
                        const void* beta, const float* S0, void* o, float* S_T,
                        float* Sc, const float* g, int BH, int Tlen, int dk, int dv,
                        cudaStream_t st, const QkNorm& nm) {
#define DN_SIMT_CASE(DK_, DV_)                                                             \
    if (dk == DK_ && dv == DV_)                                                            \
        return launch_typed<T, DK_, DV_>(q, k, v, beta, S0, o, S_T, Sc, g, BH, Tlen, st, 1, \
                                         static_cast<const SeqTable<1>*>(nullptr), nm);
    DN_SIMT_CASE(128, 128)
    DN_SIMT_CASE(128, 64)
    DN_SIMT_CASE(64, 128)
    DN_SIMT_CASE(64, 64)
#undef DN_SIMT_CASE
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v,
                              const void* beta, const float* S0, void* o,
                              float* S_T, int BH, int T, int dk, int dv, int dt,
                              cudaStream_t stream, float* S_chunks, const float* g,
                              const QkNorm& norm) {
    if (BH <= 0 || T <= 0) return cudaSuccess;
    if (dt == 0)
        return launch_dims<float>(q, k, v, beta, S0, o, S_T, S_chunks, g, BH, T, dk, dv, stream,
                                  norm);
    return launch_dims<__nv_bfloat16>(q, k, v, beta, S0, o, S_T, S_chunks, g, BH, T, dk, dv,
                                      stream, norm);
}

cudaError_t launch_chunk_simt_varlen(const void* q, const void* k, const void* v,
                                     const void* beta, const float* S0, void* o, float* S_T,
                                     const VarlenTable& seqs, int H, int T, int dk, int dv,
                                     int dt, cudaStream_t st, const QkNorm& norm) {
    const long long ctas = (long long)seqs.n * H;
    if (ctas <= 0) return cudaSuccess;
    if (ctas > 0x3fffffffLL) return cudaErrorInvalidValue;
#define DN_SIMT_VARLEN(T_, DK_, DV_)                                                           \
    if (dk == DK_ && dv == DV_)                                                                \
        return launch_typed<T_, DK_, DV_, kMaxVarlenSeqs>(q, k, v, beta, S0, o, S_T, nullptr,  \
                                                          nullptr, (int)ctas, T, st, H, &seqs,  \
                                                          norm);
    if (dt == 0) {
        DN_SIMT_VARLEN(float, 128, 128)
        DN_SIMT_VARLEN(float, 128, 64)
        DN_SIMT_VARLEN(float, 64, 128)
        DN_SIMT_VARLEN(float, 64, 64)
    } else {
        DN_SIMT_VARLEN(__nv_bfloat16, 128, 128)
        DN_SIMT_VARLEN(__nv_bfloat16, 128, 64)
        DN_SIMT_VARLEN(__nv_bfloat16, 64, 128)
        DN_SIMT_VARLEN(__nv_bfloat16, 64, 64)
    }
#undef DN_SIMT_VARLEN
    return cudaErrorNotSupported;
}

cudaError_t launch_chunk_simt_kda(const void* q, const void* k, const void* v, const void* beta,
                                  const float* g, const float* S0, void* o, float* S_T, int BH,
                                  int T, int dk, int dv, int dt, cudaStream_t st,
                                  const QkNorm& norm, float* S_chunks) {
    if (BH <= 0 || T <= 0) return cudaSuccess;
#define DN_SIMT_KDA(T_, DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_)                                                                \
        return launch_typed<T_, DK_, DV_, 1, true>(q, k, v, beta, S0, o, S_T, S_chunks, g, BH,   \
                                                   T, st, 1, nullptr, norm);
    if (dt == 0) {
        DN_SIMT_KDA(float, 128, 128)
        DN_SIMT_KDA(float, 128, 64)
        DN_SIMT_KDA(float, 64, 128)
        DN_SIMT_KDA(float, 64, 64)
    } else {
        DN_SIMT_KDA(__nv_bfloat16, 128, 128)
        DN_SIMT_KDA(__nv_bfloat16, 128, 64)
        DN_SIMT_KDA(__nv_bfloat16, 64, 128)
        DN_SIMT_KDA(__nv_bfloat16, 64, 64)
    }
#undef DN_SIMT_KDA
    return cudaErrorNotSupported;
}

}  // namespace dn
