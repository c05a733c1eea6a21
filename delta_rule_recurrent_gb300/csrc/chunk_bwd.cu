// chunk_bwd.cu -- chunkwise delta-rule backward (fp32 accumulation throughout).
//
// The training pass that follows the chunkwise forward ("Hardware-efficient
// implementation", section 3 of paperlayer.ai/abs/2406.06484v6, which
// recomputes the chunk states during backpropagation instead of storing
// them).  It returns the gradients of L = <d_o, o> + <d_S_T, S_T>.
//
// Forward per chunk (rows K, Q, V, strengths beta, incoming state S, stored
// [dk][dv]; the algebra of chunk_simt.cu):
//     A = tril(diag(beta) K K^T, -1),  X = (I + A)^{-1},  Tm = X diag(beta)
//     R = V - K S,  U' = Tm R,  P = tril(Q K^T),  O = Q S + P U',
//     S_next = S + K^T U'
// Backward per chunk, last to first, with G = dL/dS_next:
//     dU' = P^T dO + K G,   dV = Tm^T dU',   dL/dS = G + Q^T dO - K^T dV
//     dP = tril(dO U'^T),   dTm = dU' R^T
//     dQ = dO S^T + dP K
//     dK = dP^T Q + U' G^T - dV S^T + Z K
//     dA = strict_tril(-X^T (dTm diag(beta)) X^T),   Z = diag(beta) dA + (diag(beta) dA)^T
//     dbeta_j = sum_i X_ij dTm_ij + sum_l dA_jl (K K^T)_jl
// Value channels are independent in the chain (dU', dV and dL/dS column by
// column), so it runs per (batch, head, value slice); dQ, dK and dbeta sum
// over all value channels, and every chunk's share needs only S and G at its
// ends, so they run in parallel over all chunks.  Three launches:
//   1. the forward without outputs, recording S at every chunk start (the
//      tensor-core two-pass forward where it covers the shape, else the
//      CUDA-core one);
//   2. chunk_bwd_chain_kernel: per (b, h, value slice), chunks last to first:
//      G at every chunk end, d_v, d_S0;
//   3. chunk_bwd_grads_kernel: one CTA per (b, h, chunk): d_q, d_k, d_beta.
// The products run as fp32 FMA for fp32 I/O (held to 1e-4) and as warp-level
// tf32 tensor-core MMAs for bf16 I/O (simt_mm.cuh); the triangular solve is
// fp32 on CUDA cores in both.
#include <algorithm>
#include <type_traits>

#include "dn_common.cuh"
#include "dn_internal.h"
#include "simt_mm.cuh"
#include "tile_load.cuh"
#include "tri_inverse.cuh"

namespace dn {
namespace {

constexpr int kC = 64;  // chunk length
// Row pitches are the operand width plus the policy's padding (Ops::kPad).

// Chunk rows [t0, t0 + 64) of a [T][D] tensor of head bh (tok0 = bh * T),
// zeros past the end of the sequence.
template <int NT, int W, int LD, int D, typename T>
__device__ __forceinline__ void load_rows(float* dst, const T* __restrict__ src, size_t tok0,
                                          int t0, int n, int c0) {
    load_tile<NT, kC, W, LD, D>(dst, src, tok0 + t0, n, c0);
}

// A = tril(diag(beta) K K^T, -1) and P = tril(Q K^T) (diagonal included);
// K K^T itself too when KK is given.
template <class Ops, int DK>
__device__ __forceinline__ void form_a_p(const float* Ks, const float* Qs, const float* bs,
                                         float* Am, float* Pm, float* KK) {
    constexpr int LK = DK + Ops::kPad, kLC = kC + Ops::kPad;
    typename Ops::template Acc<64, 64> aa, ap;
    Ops::zero(aa);
    Ops::zero(ap);
    Ops::template mm<64, 64, DK>(aa, [&](int m, int i) { return Ks[m * LK + i]; },
                                 [&](int i, int nn) { return Ks[nn * LK + i]; });
    Ops::template mm<64, 64, DK>(ap, [&](int m, int i) { return Qs[m * LK + i]; },
                                 [&](int i, int nn) { return Ks[nn * LK + i]; });
    Ops::for_each(aa, [&](int m, int nn, float x) {
        Am[m * kLC + nn] = nn < m ? bs[m] * x : 0.f;
        if (KK) KK[m * kLC + nn] = x;
    });
    Ops::for_each(ap, [&](int m, int nn, float x) { Pm[m * kLC + nn] = nn <= m ? x : 0.f; });
}

// Gated DeltaNet: the chunk's decay from its log keep rates g (fp32, 0 past
// the end): Gl[t] = sum_{u <= t} g_u (thread t < 64 sums its own prefix),
// gam[t] = exp Gl[t] and rg[t] = Gamma / gam[t], Gamma = gam[63] (the padded
// tokens keep everything, so it is the decay through the last real token).
// Ends without a barrier.
__device__ __forceinline__ void chunk_decay(const float* __restrict__ g, size_t tok, int n,
                                            float* gs, float* Gl, float* gam, float* rg, int tid) {
    if (tid < kC) gs[tid] = tid < n ? g[tok + tid] : 0.f;
    __syncthreads();
    if (tid < kC) {
        float s = 0.f;
        for (int u = 0; u <= tid; ++u) s += gs[u];
        Gl[tid] = s;
    }
    __syncthreads();
    if (tid < kC) {
        gam[tid] = expf(Gl[tid]);
        rg[tid] = expf(Gl[kC - 1] - Gl[tid]);
    }
}
// exp(G_i - G_j) for j <= i (at most 1), 0 above the diagonal
__device__ __forceinline__ float decay_ratio(const float* Gl, int i, int j) {
    return j <= i ? expf(Gl[i] - Gl[j]) : 0.f;
}

// A = tril(diag(beta) (K K^T o D), -1) and P = tril(Q K^T o D) with the
// decay ratios D_ij = exp(G_i - G_j); (K K^T o D) itself too when KK is given.
template <class Ops, int DK>
__device__ __forceinline__ void form_a_p_gated(const float* Ks, const float* Qs, const float* bs,
                                               const float* Gl, float* Am, float* Pm, float* KK) {
    constexpr int LK = DK + Ops::kPad, kLC = kC + Ops::kPad;
    typename Ops::template Acc<64, 64> aa, ap;
    Ops::zero(aa);
    Ops::zero(ap);
    Ops::template mm<64, 64, DK>(aa, [&](int m, int i) { return Ks[m * LK + i]; },
                                 [&](int i, int nn) { return Ks[nn * LK + i]; });
    Ops::template mm<64, 64, DK>(ap, [&](int m, int i) { return Qs[m * LK + i]; },
                                 [&](int i, int nn) { return Ks[nn * LK + i]; });
    Ops::for_each(aa, [&](int m, int nn, float x) {
        const float y = x * decay_ratio(Gl, m, nn);
        Am[m * kLC + nn] = nn < m ? bs[m] * y : 0.f;
        if (KK) KK[m * kLC + nn] = y;
    });
    Ops::for_each(ap, [&](int m, int nn, float x) { Pm[m * kLC + nn] = x * decay_ratio(Gl, m, nn); });
}

// ------------------------------------------------------------------ chain
template <int DK, int NV, int PAD>
struct ChainSmem {
    static constexpr int LK = DK + PAD, LV = NV + PAD, kLC = kC + PAD;
    static constexpr int kK = 0;                  // C x LK   keys
    static constexpr int kQ = kK + kC * LK;       // C x LK   queries
    static constexpr int kD = kQ + kC * LK;       // C x LV   output gradient slice
    static constexpr int kU = kD + kC * LV;       // C x LV   dU'
    static constexpr int kV = kU + kC * LV;       // C x LV   dV
    static constexpr int kG = kV + kC * LV;       // DK x LV  state gradient slice
    static constexpr int kA = kG + DK * LV;       // C x kLC  A
    static constexpr int kX = kA + kC * kLC;      // C x kLC  (I + A)^{-1}
    static constexpr int kP = kX + kC * kLC;      // C x kLC  tril(Q K^T)
    static constexpr int kY = kP + kC * kLC;      // solve scratch
    static constexpr int kB = kY + 3 * 16 * 17;   // C        beta
    static constexpr int kGd = kB + kC;           // 4 x C    gated: g, G, gamma, Gamma / gamma
    static constexpr int kFloats = kGd + 4 * kC;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    static_assert(kBytes <= 232448, "one CTA's shared memory");
};

// One CTA per (batch, head, slice of NV value channels): G = dL/dS from the
// last chunk to the first.  Writes G at the end of every chunk (G_chunks,
// [BH][chunk][dk][dv] fp32), d_v, and d_S0 (if given).
// kGate (Gated DeltaNet, g the fp32 [BH][T] log keep rates): per chunk
//     dU' = P^T dO + diag(Gamma / gamma) K G,  dV = Tm^T dU',
//     G <- Gamma G + (diag(gamma) Q)^T dO - (diag(gamma) K)^T dV
// with P and A carrying the decay ratios.
template <class Ops, typename T, int DK, int DV, int NV, bool kGate = false>
__global__ void __launch_bounds__(Ops::kThreads, 1)
chunk_bwd_chain_kernel(const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ beta, const T* __restrict__ d_o,
                       const float* __restrict__ d_S_T, T* __restrict__ d_v,
                       float* __restrict__ d_S0, float* __restrict__ G_chunks, int Tlen,
                       const float* __restrict__ gate) {
    using L = ChainSmem<DK, NV, Ops::kPad>;
    constexpr int LK = L::LK, LV = L::LV, kLC = L::kLC, NSLICE = DV / NV, NT = Ops::kThreads;
    extern __shared__ float smem[];
    float* Ks = smem + L::kK;
    float* Qs = smem + L::kQ;
    float* Ds = smem + L::kD;
    float* Us = smem + L::kU;
    float* Vs = smem + L::kV;
    float* Gs = smem + L::kG;
    float* Am = smem + L::kA;
    float* Xm = smem + L::kX;
    float* Pm = smem + L::kP;
    float* Ys = smem + L::kY;
    float* bs = smem + L::kB;
    float* gs = smem + L::kGd;
    float* Gl = gs + kC;
    float* gam = Gl + kC;
    float* rg = gam + kC;
    const int tid = threadIdx.x;
    const int bh = blockIdx.x / NSLICE, j0 = (blockIdx.x % NSLICE) * NV;
    const size_t tok0 = (size_t)bh * Tlen;
    const int nchunks = (Tlen + kC - 1) / kC;

    for (int e = tid; e < DK * NV; e += NT) {
        const int i = e / NV, jj = e % NV;
        Gs[i * LV + jj] = d_S_T ? d_S_T[((size_t)bh * DK + i) * DV + j0 + jj] : 0.f;
    }
    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * kC, n = min(kC, Tlen - t0);
        for (int e = tid; e < DK * NV; e += NT) {  // G at the end of chunk c
            const int i = e / NV, jj = e % NV;
            G_chunks[(((size_t)bh * nchunks + c) * DK + i) * DV + j0 + jj] = Gs[i * LV + jj];
        }
        load_rows<NT, DK, LK, DK>(Ks, k, tok0, t0, n, 0);
        load_rows<NT, DK, LK, DK>(Qs, q, tok0, t0, n, 0);
        load_rows<NT, NV, LV, DV>(Ds, d_o, tok0, t0, n, j0);
        if (tid < kC) bs[tid] = tid < n ? to_f32(beta[tok0 + t0 + tid]) : 0.f;
        if constexpr (kGate) chunk_decay(gate, tok0 + t0, n, gs, Gl, gam, rg, tid);
        __syncthreads();
        if constexpr (kGate)
            form_a_p_gated<Ops, DK>(Ks, Qs, bs, Gl, Am, Pm, nullptr);
        else
            form_a_p<Ops, DK>(Ks, Qs, bs, Am, Pm, nullptr);
        __syncthreads();
        {   // dU' = P^T dO + K G  (gated: K's rows times Gamma / gamma)
            typename Ops::template Acc<64, NV> acc;
            Ops::zero(acc);
            Ops::template mm<64, NV, kC>(acc, [&](int m, int s) { return Pm[s * kLC + m]; },
                               [&](int s, int nn) { return Ds[s * LV + nn]; });
            Ops::template mm<64, NV, DK>(acc, [&](int m, int i) {
                return kGate ? Ks[m * LK + i] * rg[m] : Ks[m * LK + i];
            }, [&](int i, int nn) { return Gs[i * LV + nn]; });
            Ops::for_each(acc, [&](int m, int nn, float x) { Us[m * LV + nn] = x; });
        }
        unit_lower_inverse64<NT, kLC>(Am, Xm, Ys);  // ends with a barrier
        {   // dV = Tm^T dU' = diag(beta) X^T dU'
            typename Ops::template Acc<64, NV> acc;
            Ops::zero(acc);
            Ops::template mm<64, NV, kC>(acc, [&](int m, int s) { return Xm[s * kLC + m]; },
                               [&](int s, int nn) { return Us[s * LV + nn]; });
            Ops::for_each(acc, [&](int m, int nn, float x) {
                const float y = bs[m] * x;
                Vs[m * LV + nn] = y;
                if (m < n) d_v[(tok0 + t0 + m) * DV + j0 + nn] = from_f32<T>(y);
            });
        }
        __syncthreads();
        {   // G <- G + Q^T dO - K^T dV  (the gradient of the state chunk c starts from;
            // gated: Gamma G and the rows of Q and K times gamma)
            typename Ops::template Acc<DK, NV> acc;
            Ops::zero(acc);
            Ops::template mm<DK, NV, kC>(acc, [&](int i, int s) {
                return kGate ? Qs[s * LK + i] * gam[s] : Qs[s * LK + i];
            }, [&](int s, int nn) { return Ds[s * LV + nn]; });
            Ops::template mm<DK, NV, kC>(acc, [&](int i, int s) {
                return kGate ? -Ks[s * LK + i] * gam[s] : -Ks[s * LK + i];
            }, [&](int s, int nn) { return Vs[s * LV + nn]; });
            const float keep = kGate ? gam[kC - 1] : 1.f;
            Ops::for_each(acc, [&](int i, int nn, float x) {
                Gs[i * LV + nn] = kGate ? keep * Gs[i * LV + nn] + x : Gs[i * LV + nn] + x;
            });
        }
        __syncthreads();
    }
    if (d_S0) {
        for (int e = tid; e < DK * NV; e += NT) {
            const int i = e / NV, jj = e % NV;
            d_S0[((size_t)bh * DK + i) * DV + j0 + jj] = Gs[i * LV + jj];
        }
    }
}

// ------------------------------------------------------------------ grads
template <int DK, int NS, int PAD>
struct GradSmem {
    static constexpr int LK = DK + PAD, LS = NS + PAD, kLC = kC + PAD;
    static constexpr int kK = 0;                  // C x LK   keys
    static constexpr int kQ = kK + kC * LK;       // C x LK   queries
    static constexpr int kX = kQ + kC * LK;       // C x kLC  (I + A)^{-1}
    static constexpr int kP = kX + kC * kLC;      // C x kLC  tril(Q K^T)
    static constexpr int kKK = kP + kC * kLC;     // C x kLC  K K^T
    static constexpr int kB = kKK + kC * kLC;     // C        beta
    // gated: g (then dG), G, gamma, Gamma / gamma, and the per-token sums
    // t1 = gamma dO . (Q S), t2 = gamma dV . (K S), t3 = (Gamma / gamma) (K G) . U',
    // then <G, S> in one float
    static constexpr int kGd = kB + kC;           // 7 x C + 4
    static constexpr int kRs = kGd + 7 * kC + 4;  // 3 x 2 x C  gated: row-sum parts of t1, t2, t3
    // The work area: A and the solve scratch until X is formed, then the
    // value-slice operands, then C x C matrices once the slices are done.
    static constexpr int kW = kRs + 6 * kC;
    static constexpr int kA = kW;                 // C x kLC  A
    static constexpr int kY = kA + kC * kLC;      // solve scratch
    static constexpr int kV = kW;                 // C x LS   V
    static constexpr int kD = kV + kC * LS;       // C x LS   dO
    static constexpr int kR = kD + kC * LS;       // C x LS   R = V - K S
    static constexpr int kU = kR + kC * LS;       // C x LS   U'
    static constexpr int kE = kU + kC * LS;       // C x LS   dU'
    static constexpr int kF = kE + kC * LS;       // C x LS   dV
    static constexpr int kS = kF + kC * LS;       // DK x LS  S slice
    static constexpr int kG = kS + DK * LS;       // DK x LS  G slice
    static constexpr int kFloats = kG + DK * LS;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    static_assert(kFloats - kW >= 4 * kC * kLC, "room for dP, dTm, M1, dA");
    static_assert(kFloats - kW >= kC * kLC + 3 * 16 * 17, "room for A and the solve scratch");
    static_assert(kBytes <= 232448, "one CTA's shared memory");
};

// One CTA per (batch, head, chunk): the chunk's d_q, d_k and d_beta from S at
// its start (S_chunks) and G at its end (G_chunks), over all value channels
// in slices of NS.
// kGate (Gated DeltaNet): the chunk algebra with the decay ratios in A and P,
// gamma on K S in R and on Q S in O, Gamma / gamma on K in the state update,
// and d_g: per token dG_i (the decay ratios' terms, gamma's and Gamma's) summed
// from each token to the chunk's end.
template <class Ops, typename T, int DK, int DV, bool kGate = false>
__global__ void __launch_bounds__(Ops::kThreads, 1)
chunk_bwd_grads_kernel(const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ v, const T* __restrict__ beta,
                       const T* __restrict__ d_o, const float* __restrict__ S_chunks,
                       const float* __restrict__ G_chunks, T* __restrict__ d_q,
                       T* __restrict__ d_k, T* __restrict__ d_beta, int Tlen, int nchunks,
                       const float* __restrict__ gate, float* __restrict__ d_g) {
    constexpr int NS = 32;
    using L = GradSmem<DK, NS, Ops::kPad>;
    constexpr int LK = L::LK, LS = L::LS, kLC = L::kLC, NT = Ops::kThreads;
    extern __shared__ float smem[];
    float* Ks = smem + L::kK;
    float* Qs = smem + L::kQ;
    float* Am = smem + L::kA;
    float* Xm = smem + L::kX;
    float* Pm = smem + L::kP;
    float* KK = smem + L::kKK;
    float* Ys = smem + L::kY;
    float* bs = smem + L::kB;
    float* Vs = smem + L::kV;
    float* Ds = smem + L::kD;
    float* Rs = smem + L::kR;
    float* Us = smem + L::kU;
    float* Es = smem + L::kE;
    float* Fs = smem + L::kF;
    float* Ss = smem + L::kS;
    float* Gs = smem + L::kG;
    float* gs = smem + L::kGd;  // g, then dG
    float* Gl = gs + kC;
    float* gam = Gl + kC;
    float* rg = gam + kC;
    float* t1 = rg + kC;
    float* t2 = t1 + kC;
    float* t3 = t2 + kC;
    float* t4 = t3 + kC;
    // gated: each slice's row sums of t1, t2, t3 by column part (Ops::row_sums),
    // added to t1, t2, t3 in a fixed order so that d_g is reproducible
    float* rs1 = smem + L::kRs;
    float* rs2 = rs1 + 2 * kC;
    float* rs3 = rs2 + 2 * kC;
    static_assert(Ops::kRowParts <= 2, "two column parts at most");
    const int tid = threadIdx.x;
    const int bh = blockIdx.x / nchunks, c = blockIdx.x % nchunks;
    const int t0 = c * kC, n = min(kC, Tlen - t0);
    const size_t tok0 = (size_t)bh * Tlen;
    const size_t st0 = ((size_t)bh * nchunks + c) * DK * DV;

    load_rows<NT, DK, LK, DK>(Ks, k, tok0, t0, n, 0);
    load_rows<NT, DK, LK, DK>(Qs, q, tok0, t0, n, 0);
    if (tid < kC) bs[tid] = tid < n ? to_f32(beta[tok0 + t0 + tid]) : 0.f;
    if constexpr (kGate) {
        if (tid < 3 * kC + 1) t1[tid] = 0.f;  // t1, t2, t3 and <G, S>
        chunk_decay(gate, tok0 + t0, n, gs, Gl, gam, rg, tid);
    }
    __syncthreads();
    if constexpr (kGate)
        form_a_p_gated<Ops, DK>(Ks, Qs, bs, Gl, Am, Pm, KK);
    else
        form_a_p<Ops, DK>(Ks, Qs, bs, Am, Pm, KK);
    __syncthreads();
    unit_lower_inverse64<NT, kLC>(Am, Xm, Ys);  // ends with a barrier

    typename Ops::template Acc<64, DK> aQ, aK;
    typename Ops::template Acc<64, 64> aP, aT;
    Ops::zero(aQ);
    Ops::zero(aK);
    Ops::zero(aP);
    Ops::zero(aT);
    float t4p = 0.f;  // gated: this thread's part of <G, S>
    for (int js = 0; js < DV; js += NS) {
        load_rows<NT, NS, LS, DV>(Vs, v, tok0, t0, n, js);
        load_rows<NT, NS, LS, DV>(Ds, d_o, tok0, t0, n, js);
        load_tile<NT, DK, NS, LS, DV>(Ss, S_chunks + st0, 0, DK, js);
        load_tile<NT, DK, NS, LS, DV>(Gs, G_chunks + st0, 0, DK, js);
        __syncthreads();
        if constexpr (kGate)
            for (int e = tid; e < DK * NS; e += NT) {
                const int i = e / NS, jj = e % NS;
                t4p = fmaf(Gs[i * LS + jj], Ss[i * LS + jj], t4p);
            }
        {   // R = V - K S and dU' = P^T dO + K G.  Gated: Rs holds W = diag(gamma) K S
            // (R = V - W), Us the term diag(Gamma / gamma) K G until U' replaces it,
            // and t1 gathers gamma dO . (Q S)
            typename Ops::template Acc<64, NS> r, e;
            Ops::zero(r);
            Ops::zero(e);
            Ops::template mm<64, NS, DK>(r, [&](int m, int i) { return Ks[m * LK + i]; },
                               [&](int i, int nn) { return Ss[i * LS + nn]; });
            Ops::template mm<64, NS, kC>(e, [&](int m, int s) { return Pm[s * kLC + m]; },
                               [&](int s, int nn) { return Ds[s * LS + nn]; });
            if constexpr (kGate) {
                typename Ops::template Acc<64, NS> kg, qs;
                Ops::zero(kg);
                Ops::zero(qs);
                Ops::template mm<64, NS, DK>(kg, [&](int m, int i) { return Ks[m * LK + i]; },
                                   [&](int i, int nn) { return Gs[i * LS + nn]; });
                Ops::template mm<64, NS, DK>(qs, [&](int m, int i) { return Qs[m * LK + i]; },
                                   [&](int i, int nn) { return Ss[i * LS + nn]; });
                Ops::for_each(r, [&](int m, int nn, float x) { Rs[m * LS + nn] = gam[m] * x; });
                Ops::for_each(e, [&](int m, int nn, float x) { Es[m * LS + nn] = x; });
                Ops::for_each(kg, [&](int m, int nn, float x) {
                    const float y = rg[m] * x;
                    Es[m * LS + nn] += y;
                    Us[m * LS + nn] = y;
                });
                Ops::row_sums(qs, [&](int m, int nn, float x) {
                    return gam[m] * Ds[m * LS + nn] * x;
                }, rs1);
            } else {
                Ops::template mm<64, NS, DK>(e, [&](int m, int i) { return Ks[m * LK + i]; },
                                   [&](int i, int nn) { return Gs[i * LS + nn]; });
                Ops::for_each(r, [&](int m, int nn, float x) { Rs[m * LS + nn] = Vs[m * LS + nn] - x; });
                Ops::for_each(e, [&](int m, int nn, float x) { Es[m * LS + nn] = x; });
            }
        }
        __syncthreads();
        // R as stored, or V - W in the gated form
        auto Rv = [&](int s, int nn) {
            return kGate ? Vs[s * LS + nn] - Rs[s * LS + nn] : Rs[s * LS + nn];
        };
        {   // U' = X diag(beta) R and dV = diag(beta) X^T dU' (gated: t3 and t2 too)
            typename Ops::template Acc<64, NS> u, f;
            Ops::zero(u);
            Ops::zero(f);
            Ops::template mm<64, NS, kC>(u, [&](int m, int s) { return Xm[m * kLC + s] * bs[s]; },
                               [&](int s, int nn) { return Rv(s, nn); });
            Ops::template mm<64, NS, kC>(f, [&](int m, int s) { return Xm[s * kLC + m]; },
                               [&](int s, int nn) { return Es[s * LS + nn]; });
            if constexpr (kGate) {  // each thread reads only the elements it then overwrites
                Ops::row_sums(u, [&](int m, int nn, float x) { return Us[m * LS + nn] * x; }, rs3);
                Ops::row_sums(f, [&](int m, int nn, float x) {
                    return bs[m] * x * Rs[m * LS + nn];
                }, rs2);
            }
            Ops::for_each(u, [&](int m, int nn, float x) { Us[m * LS + nn] = x; });
            Ops::for_each(f, [&](int m, int nn, float x) { Fs[m * LS + nn] = bs[m] * x; });
        }
        __syncthreads();
        if constexpr (kGate) {  // the slice's row sums, parts in order
            if (tid < kC) {
                float a1 = rs1[tid], a2 = rs2[tid], a3 = rs3[tid];
                if (Ops::kRowParts == 2) {
                    a1 += rs1[kC + tid];
                    a2 += rs2[kC + tid];
                    a3 += rs3[kC + tid];
                }
                t1[tid] += a1;
                t2[tid] += a2;
                t3[tid] += a3;
            }
        }
        // dP += dO U'^T, dTm += dU' R^T, dQ += dO S^T, dK += U' G^T - dV S^T
        // (gated: dQ's rows times gamma, U' G^T's times Gamma / gamma, dV S^T's times gamma)
        Ops::template mm<64, 64, NS>(aP, [&](int m, int j) { return Ds[m * LS + j]; },
                           [&](int j, int nn) { return Us[nn * LS + j]; });
        Ops::template mm<64, 64, NS>(aT, [&](int m, int j) { return Es[m * LS + j]; },
                           [&](int j, int nn) { return Rv(nn, j); });
        Ops::template mm<64, DK, NS>(aQ, [&](int m, int j) {
            return kGate ? Ds[m * LS + j] * gam[m] : Ds[m * LS + j];
        }, [&](int j, int i) { return Ss[i * LS + j]; });
        Ops::template mm<64, DK, NS>(aK, [&](int m, int j) {
            return kGate ? Us[m * LS + j] * rg[m] : Us[m * LS + j];
        }, [&](int j, int i) { return Gs[i * LS + j]; });
        Ops::template mm<64, DK, NS>(aK, [&](int m, int j) {
            return kGate ? -Fs[m * LS + j] * gam[m] : -Fs[m * LS + j];
        }, [&](int j, int i) { return Ss[i * LS + j]; });
        __syncthreads();
    }
    if constexpr (kGate) {  // <G, S>: warp sums, then the warps in order
        const float wsum = warp_sum(t4p);
        if ((tid & 31) == 0) rs1[tid >> 5] = wsum;
        __syncthreads();
        if (tid == 0) {
            float s4 = 0.f;
            for (int w = 0; w < NT / 32; ++w) s4 += rs1[w];
            t4[0] = s4;
        }
    }

    // The work area now holds C x C matrices.
    float* dPm = smem + L::kW;
    float* dTs = dPm + kC * kLC;
    float* M1 = dTs + kC * kLC;
    float* dAm = M1 + kC * kLC;
    Ops::for_each(aP, [&](int m, int nn, float x) { dPm[m * kLC + nn] = nn <= m ? x : 0.f; });
    Ops::for_each(aT, [&](int m, int nn, float x) { dTs[m * kLC + nn] = x; });
    __syncthreads();
    // dQ += dP K, dK += dP^T Q (gated: dP times the decay ratios)
    Ops::template mm<64, DK, kC>(aQ, [&](int m, int s) {
        return kGate ? dPm[m * kLC + s] * decay_ratio(Gl, m, s) : dPm[m * kLC + s];
    }, [&](int s, int i) { return Ks[s * LK + i]; });
    Ops::template mm<64, DK, kC>(aK, [&](int m, int s) {
        return kGate ? dPm[s * kLC + m] * decay_ratio(Gl, s, m) : dPm[s * kLC + m];
    }, [&](int s, int i) { return Qs[s * LK + i]; });
    {   // M1 = (dTm diag(beta)) X^T
        typename Ops::template Acc<64, 64> acc;
        Ops::zero(acc);
        Ops::template mm<64, 64, kC>(acc, [&](int m, int s) { return dTs[m * kLC + s] * bs[s]; },
                           [&](int s, int nn) { return Xm[nn * kLC + s]; });
        Ops::for_each(acc, [&](int m, int nn, float x) { M1[m * kLC + nn] = x; });
    }
    float db = 0.f;  // thread j < 64: dbeta_j
    if (tid < kC)
        for (int i = 0; i < kC; ++i) db = fmaf(Xm[i * kLC + tid], dTs[i * kLC + tid], db);
    __syncthreads();
    {   // dA = strict_tril(-X^T M1)
        typename Ops::template Acc<64, 64> acc;
        Ops::zero(acc);
        Ops::template mm<64, 64, kC>(acc, [&](int m, int s) { return Xm[s * kLC + m]; },
                           [&](int s, int nn) { return M1[s * kLC + nn]; });
        Ops::for_each(acc, [&](int m, int nn, float x) { dAm[m * kLC + nn] = nn < m ? -x : 0.f; });
    }
    __syncthreads();
    if (tid < kC)
        for (int l = 0; l < kC; ++l) db = fmaf(dAm[tid * kLC + l], KK[tid * kLC + l], db);
    // dK += Z K with Z = diag(beta) dA + (diag(beta) dA)^T (gated: dA times the decay ratios)
    Ops::template mm<64, DK, kC>(aK, [&](int m, int s) {
        return kGate ? bs[m] * dAm[m * kLC + s] * decay_ratio(Gl, m, s) +
                           bs[s] * dAm[s * kLC + m] * decay_ratio(Gl, s, m)
                     : bs[m] * dAm[m * kLC + s] + bs[s] * dAm[s * kLC + m];
    }, [&](int s, int i) { return Ks[s * LK + i]; });
    if constexpr (kGate) {  // dG per token, then d_g = its sums from each token to the chunk's end
        if (tid < kC) {
            const int i = tid;
            float dG = t1[i] - t2[i] - t3[i];
            for (int j = 0; j < kC; ++j) {
                // A_ij = beta_i (K K^T o D)_ij (j < i) and P (with the ratios) as formed
                const float aij = j < i ? bs[i] * KK[i * kLC + j] : 0.f;
                const float aji = i < j ? bs[j] * KK[j * kLC + i] : 0.f;
                dG += dAm[i * kLC + j] * aij - dAm[j * kLC + i] * aji;
                dG += dPm[i * kLC + j] * Pm[i * kLC + j] - dPm[j * kLC + i] * Pm[j * kLC + i];
            }
            if (i == n - 1) {  // <G, S_next> = Gamma <G, S> + sum_j t3_j
                float s3 = 0.f;
                for (int j = 0; j < kC; ++j) s3 += t3[j];
                dG += gam[kC - 1] * t4[0] + s3;
            }
            gs[i] = dG;
        }
        __syncthreads();
        if (tid < n) {
            float s = 0.f;
            for (int i = tid; i < n; ++i) s += gs[i];
            d_g[tok0 + t0 + tid] = s;
        }
    }

    Ops::for_each(aQ, [&](int m, int i, float x) {
        if (m < n) d_q[(tok0 + t0 + m) * DK + i] = from_f32<T>(x);
    });
    Ops::for_each(aK, [&](int m, int i, float x) {
        if (m < n) d_k[(tok0 + t0 + m) * DK + i] = from_f32<T>(x);
    });
    if (tid < n) d_beta[tok0 + t0 + tid] = from_f32<T>(db);
}

// ------------------------------------------------------------------ KDA
// KDA ("Kimi Delta Attention : atténuation par canal", fr.news.hada.io/topic?id=31925):
// one log keep rate per key channel, G_t[c] its sum from the chunk start
// through token t (padding tokens keep everything), G_L[c] that of the
// chunk's last token.  Per chunk, with gamma = exp(G), f = exp(G_L - G) and
// the ratios D[t][s][c] = exp(G_t[c] - G_s[c]) inside the channel sums:
//     A2[t][s] = sum_c k_t[c] k_s[c] D[t][s][c],  A = tril(diag(beta) A2, -1)
//     P[t][s]  = sum_c q_t[c] k_s[c] D[t][s][c]   (s <= t)
//     R = V - (K o gamma) S,  U' = X diag(beta) R,
//     S_next = diag(exp G_L) S + (K o f)^T U'
// The chain (per value slice), last chunk first, with G = dL/dS_next:
//     dU' = P^T dO + (K o f) G,  dV = diag(beta) X^T dU',
//     G <- diag(exp G_L) G + (Q o gamma)^T dO - (K o gamma)^T dV
// The per-chunk gradients (all value channels), dP and dA as in the plain
// backward and dA2 = diag(beta) dA:
//     dQ = gamma o (dO S^T) + dQ_P
//     dK = [gamma o (-dV S^T) + dK_r] + [f o (U' G^T) + dK_P + dK_c]
//     dQ_P[t][c] = sum_s dP[t][s] k_s[c] D[t][s][c],  dK_P[s][c] = sum_t dP[t][s] q_t[c] D[t][s][c]
//     dK_r[t][c] = sum_s dA2[t][s] k_s[c] D[t][s][c], dK_c[s][c] = sum_t dA2[t][s] k_t[c] D[t][s][c]
//     dG = q o dQ + k o [first bracket] - k o [second bracket], plus, on the
//          last token, sum_j G[c][j] S_next[c][j] = exp(G_L[c]) <G, S>_c + sum_s k_s[c] f_s[c] (U' G^T)[s][c]
//     d_g = dG summed from each token to the chunk's end
// While every channel's decay over the chunk stays within exp(-60), each ratio
// is the product exp(G_t) exp(-G_s) of two normal fp32 numbers, so the ratio
// sums are plain products of scaled operands; otherwise every ratio takes its
// own exponential, clamped at 1.
constexpr float kKdaSepLimit = -60.f;

// The chunk's per-channel cumulative log decay into Gk (C x LK, padding rows
// 0) and G_L into GL, from the rates g ([token][DK] fp32) of tokens tok ..
// tok + n - 1.  Returns, to every thread, whether every channel's decay over
// the chunk stays within exp(kKdaSepLimit).  Ends with a barrier, which also
// completes the caller's earlier tile loads.
template <int NT, int DK, int LK>
__device__ __forceinline__ bool chunk_decay_kda(const float* __restrict__ g, size_t tok, int n,
                                                float* Gk, float* GL) {
    load_tile<NT, kC, DK, LK, DK>(Gk, g, tok, n, 0);
    __syncthreads();
    const int tid = threadIdx.x;
    if (tid < DK) {
        float s = Gk[tid];
        for (int t = 1; t < kC; ++t) {
            s += Gk[t * LK + tid];
            Gk[t * LK + tid] = s;
        }
        GL[tid] = s;
    }
    return __syncthreads_and(tid >= DK || GL[tid] >= kKdaSepLimit);
}

// A = tril(diag(beta) A2, -1), P (diagonal included) and, with KK, A2 below
// the diagonal, one clamped exponential per ratio: 256 threads, thread
// (tid / 16, tid % 16) forms rows ty + 16 i and columns tx + 16 j.
template <int DK, int LK, int kLC>
__device__ __forceinline__ void form_a_p_kda_exact(const float* Ks, const float* Qs,
                                                   const float* Gk, const float* bs, float* Am,
                                                   float* Pm, float* KK) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float aa[4][4], ap[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) aa[i][j] = ap[i][j] = 0.f;
#pragma unroll 2
    for (int c = 0; c < DK; ++c) {
        float ak[4], aq[4], gi[4], bk[4], gj[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ak[i] = Ks[(ty + 16 * i) * LK + c];
            aq[i] = Qs[(ty + 16 * i) * LK + c];
            gi[i] = Gk[(ty + 16 * i) * LK + c];
            bk[i] = Ks[(tx + 16 * i) * LK + c];
            gj[i] = Gk[(tx + 16 * i) * LK + c];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // pairs past the diagonal are masked below
                const float e = __expf(fminf(gi[i] - gj[j], 0.f)) * bk[j];
                aa[i][j] = fmaf(ak[i], e, aa[i][j]);
                ap[i][j] = fmaf(aq[i], e, ap[i][j]);
            }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = ty + 16 * i, nn = tx + 16 * j;
            Am[m * kLC + nn] = nn < m ? bs[m] * aa[i][j] : 0.f;
            Pm[m * kLC + nn] = nn <= m ? ap[i][j] : 0.f;
            if (KK) KK[m * kLC + nn] = nn < m ? aa[i][j] : 0.f;
        }
}

// The same from scaled operands, (K o exp G)(K o exp(-G))^T and
// (Q o exp G)(K o exp(-G))^T, when the chunk's decay allows it.
template <class Ops, int DK>
__device__ __forceinline__ void form_a_p_kda_sep(const float* Ks, const float* Qs,
                                                 const float* Gk, const float* bs, float* Am,
                                                 float* Pm, float* KK) {
    constexpr int LK = DK + Ops::kPad, kLC = kC + Ops::kPad;
    typename Ops::template Acc<64, 64> aa, ap;
    Ops::zero(aa);
    Ops::zero(ap);
    const auto km = [&](int c, int nn) { return Ks[nn * LK + c] * __expf(-Gk[nn * LK + c]); };
    Ops::template mm<64, 64, DK>(aa, [&](int m, int c) {
        return Ks[m * LK + c] * __expf(Gk[m * LK + c]);
    }, km);
    Ops::template mm<64, 64, DK>(ap, [&](int m, int c) {
        return Qs[m * LK + c] * __expf(Gk[m * LK + c]);
    }, km);
    Ops::for_each(aa, [&](int m, int nn, float x) {
        Am[m * kLC + nn] = nn < m ? bs[m] * x : 0.f;
        if (KK) KK[m * kLC + nn] = nn < m ? x : 0.f;
    });
    Ops::for_each(ap, [&](int m, int nn, float x) { Pm[m * kLC + nn] = nn <= m ? x : 0.f; });
}

// The same from operands already scaled in shared memory: A2 = Kp Km^T and
// P = Qp Km^T (Kp = K o exp G, Qp = Q o exp G, Km = K o exp(-G)).
template <class Ops, int DK>
__device__ __forceinline__ void form_a_p_scaled(const float* Kp, const float* Qp, const float* Km,
                                                const float* bs, float* Am, float* Pm) {
    constexpr int LK = DK + Ops::kPad, kLC = kC + Ops::kPad;
    typename Ops::template Acc<64, 64> aa, ap;
    Ops::zero(aa);
    Ops::zero(ap);
    const auto km = [&](int c, int nn) { return Km[nn * LK + c]; };
    Ops::template mm<64, 64, DK>(aa, [&](int m, int c) { return Kp[m * LK + c]; }, km);
    Ops::template mm<64, 64, DK>(ap, [&](int m, int c) { return Qp[m * LK + c]; }, km);
    Ops::for_each(aa, [&](int m, int nn, float x) { Am[m * kLC + nn] = nn < m ? bs[m] * x : 0.f; });
    Ops::for_each(ap, [&](int m, int nn, float x) { Pm[m * kLC + nn] = nn <= m ? x : 0.f; });
}

template <int DK, int NV, int PAD>
struct ChainKdaSmem {
    static constexpr int LK = DK + PAD, LV = NV + PAD, kLC = kC + PAD;
    static constexpr int kK = 0;                  // C x LK   keys, then K o gamma
    static constexpr int kQ = kK + kC * LK;       // C x LK   queries, then Q o gamma
    static constexpr int kGk = kQ + kC * LK;      // C x LK   cumulative log decay, then K o f
    static constexpr int kD = kGk + kC * LK;      // C x LV   output gradient slice
    static constexpr int kU = kD + kC * LV;       // C x LV   A until X is formed, then dU'
    static constexpr int kV = kU + kC * LV;       // C x LV   dV
    static constexpr int kG = kV + kC * LV;       // DK x LV  state gradient slice
    static constexpr int kA = kU;
    static constexpr int kX = kG + DK * LV;       // C x kLC  (I + A)^{-1}
    static constexpr int kP = kX + kC * kLC;      // C x kLC  P
    static constexpr int kY = kP + kC * kLC;      // solve scratch
    static constexpr int kB = kY + 3 * 16 * 17;   // C        beta
    static constexpr int kGL = kB + kC;           // DK       G_L
    static constexpr int kFloats = kGL + DK;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    static_assert(LV >= kLC, "A fits dU's region");
    static_assert(kBytes <= 232448, "one CTA's shared memory");
};

// KDA's chain: one CTA per (batch, head, slice of NV value channels), chunks
// last to first; writes G at every chunk end (G_chunks, fp32 [BH][chunk][dk][dv]),
// d_v and d_S0.  g: fp32 [BH][T][DK] log keep rates.
template <class Ops, typename T, int DK, int DV, int NV>
__global__ void __launch_bounds__(Ops::kThreads, 1)
chunk_bwd_chain_kda_kernel(const T* __restrict__ q, const T* __restrict__ k,
                           const T* __restrict__ beta, const T* __restrict__ d_o,
                           const float* __restrict__ d_S_T, T* __restrict__ d_v,
                           float* __restrict__ d_S0, float* __restrict__ G_chunks, int Tlen,
                           const float* __restrict__ gate) {
    using L = ChainKdaSmem<DK, NV, Ops::kPad>;
    constexpr int LK = L::LK, LV = L::LV, kLC = L::kLC, NSLICE = DV / NV, NT = Ops::kThreads;
    static_assert(NT == 256 && DK <= NT, "the exact form's thread grid; a thread per channel");
    extern __shared__ float smem[];
    float* Ks = smem + L::kK;
    float* Qs = smem + L::kQ;
    float* Gk = smem + L::kGk;
    float* Ds = smem + L::kD;
    float* Us = smem + L::kU;
    float* Vs = smem + L::kV;
    float* Gs = smem + L::kG;
    float* Am = smem + L::kA;
    float* Xm = smem + L::kX;
    float* Pm = smem + L::kP;
    float* Ys = smem + L::kY;
    float* bs = smem + L::kB;
    float* GL = smem + L::kGL;
    const int tid = threadIdx.x;
    const int bh = blockIdx.x / NSLICE, j0 = (blockIdx.x % NSLICE) * NV;
    const size_t tok0 = (size_t)bh * Tlen;
    const int nchunks = (Tlen + kC - 1) / kC;

    for (int e = tid; e < DK * NV; e += NT) {
        const int i = e / NV, jj = e % NV;
        Gs[i * LV + jj] = d_S_T ? d_S_T[((size_t)bh * DK + i) * DV + j0 + jj] : 0.f;
    }
    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * kC, n = min(kC, Tlen - t0);
        for (int e = tid; e < DK * NV; e += NT) {  // G at the end of chunk c
            const int i = e / NV, jj = e % NV;
            G_chunks[(((size_t)bh * nchunks + c) * DK + i) * DV + j0 + jj] = Gs[i * LV + jj];
        }
        load_rows<NT, DK, LK, DK>(Ks, k, tok0, t0, n, 0);
        load_rows<NT, DK, LK, DK>(Qs, q, tok0, t0, n, 0);
        load_rows<NT, NV, LV, DV>(Ds, d_o, tok0, t0, n, j0);
        if (tid < kC) bs[tid] = tid < n ? to_f32(beta[tok0 + t0 + tid]) : 0.f;
        const bool sep = chunk_decay_kda<NT, DK, LK>(gate, tok0 + t0, n, Gk, GL);
        // Both forms leave K o gamma, Q o gamma and K o f in place of K, Q and G
        // (the solve's barriers order these writes before the products below).
        if (sep) {  // K o exp(-G) over G, the products plain, then exp G_L per channel
            for (int e = tid; e < kC * DK; e += NT) {
                const int t = e / DK, i = e % DK;
                const float G = Gk[t * LK + i], kv = Ks[t * LK + i], ga = __expf(G);
                Ks[t * LK + i] = kv * ga;
                Qs[t * LK + i] *= ga;
                Gk[t * LK + i] = kv * __expf(-G);
            }
            __syncthreads();
            form_a_p_scaled<Ops, DK>(Ks, Qs, Gk, bs, Am, Pm);
            __syncthreads();
            for (int e = tid; e < kC * DK; e += NT) {
                const int t = e / DK, i = e % DK;
                Gk[t * LK + i] *= __expf(GL[i]);
            }
        } else {
            form_a_p_kda_exact<DK, LK, kLC>(Ks, Qs, Gk, bs, Am, Pm, nullptr);
            __syncthreads();
            for (int e = tid; e < kC * DK; e += NT) {
                const int t = e / DK, i = e % DK;
                const float G = Gk[t * LK + i], kv = Ks[t * LK + i], ga = __expf(G);
                Ks[t * LK + i] = kv * ga;
                Qs[t * LK + i] *= ga;
                Gk[t * LK + i] = kv * __expf(GL[i] - G);
            }
        }
        unit_lower_inverse64<NT, kLC>(Am, Xm, Ys);  // ends with a barrier; A is dead
        {   // dU' = P^T dO + (K o f) G, over A's region
            typename Ops::template Acc<64, NV> acc;
            Ops::zero(acc);
            Ops::template mm<64, NV, kC>(acc, [&](int m, int s) { return Pm[s * kLC + m]; },
                               [&](int s, int nn) { return Ds[s * LV + nn]; });
            Ops::template mm<64, NV, DK>(acc, [&](int m, int i) { return Gk[m * LK + i]; },
                               [&](int i, int nn) { return Gs[i * LV + nn]; });
            Ops::for_each(acc, [&](int m, int nn, float x) { Us[m * LV + nn] = x; });
        }
        __syncthreads();
        {   // dV = diag(beta) X^T dU'
            typename Ops::template Acc<64, NV> acc;
            Ops::zero(acc);
            Ops::template mm<64, NV, kC>(acc, [&](int m, int s) { return Xm[s * kLC + m]; },
                               [&](int s, int nn) { return Us[s * LV + nn]; });
            Ops::for_each(acc, [&](int m, int nn, float x) {
                const float y = bs[m] * x;
                Vs[m * LV + nn] = y;
                if (m < n) d_v[(tok0 + t0 + m) * DV + j0 + nn] = from_f32<T>(y);
            });
        }
        __syncthreads();
        {   // G <- diag(exp G_L) G + (Q o gamma)^T dO - (K o gamma)^T dV
            typename Ops::template Acc<DK, NV> acc;
            Ops::zero(acc);
            Ops::template mm<DK, NV, kC>(acc, [&](int i, int s) { return Qs[s * LK + i]; },
                               [&](int s, int nn) { return Ds[s * LV + nn]; });
            Ops::template mm<DK, NV, kC>(acc, [&](int i, int s) { return -Ks[s * LK + i]; },
                               [&](int s, int nn) { return Vs[s * LV + nn]; });
            Ops::for_each(acc, [&](int i, int nn, float x) {
                Gs[i * LV + nn] = fmaf(__expf(GL[i]), Gs[i * LV + nn], x);
            });
        }
        __syncthreads();
    }
    if (d_S0) {
        for (int e = tid; e < DK * NV; e += NT) {
            const int i = e / NV, jj = e % NV;
            d_S0[((size_t)bh * DK + i) * DV + j0 + jj] = Gs[i * LV + jj];
        }
    }
}

template <int DK, int NS, int PAD>
struct GradKdaSmem {
    static constexpr int LK = DK + PAD, LS = NS + PAD, kLC = kC + PAD;
    static constexpr int kK = 0;                  // C x LK   keys
    static constexpr int kQ = kK + kC * LK;       // C x LK   queries
    static constexpr int kGk = kQ + kC * LK;      // C x LK   cumulative log decay, then dG
    static constexpr int kX = kGk + kC * LK;      // C x kLC  (I + A)^{-1}
    static constexpr int kP = kX + kC * kLC;      // C x kLC  P
    static constexpr int kKK = kP + kC * kLC;     // C x kLC  A2 below the diagonal
    static constexpr int kB = kKK + kC * kLC;     // C        beta
    static constexpr int kGL = kB + kC;           // DK       G_L
    static constexpr int kT3 = kGL + DK;          // DK       sum_s k_s f_s (U' G^T)[s]
    static constexpr int kT4 = kT3 + DK;          // DK       <G, S> per key channel
    // The work area: A and the solve scratch until X is formed, then the
    // value-slice operands, then C x C matrices once the slices are done.
    static constexpr int kW = kT4 + DK;
    static constexpr int kA = kW;                 // C x kLC  A
    static constexpr int kY = kA + kC * kLC;      // solve scratch
    static constexpr int kV = kW;                 // C x LS   V
    static constexpr int kD = kV + kC * LS;       // C x LS   dO
    static constexpr int kR = kD + kC * LS;       // C x LS   R
    static constexpr int kU = kR + kC * LS;       // C x LS   U'
    static constexpr int kE = kU + kC * LS;       // C x LS   dU'
    static constexpr int kF = kE + kC * LS;       // C x LS   dV
    static constexpr int kS = kF + kC * LS;       // DK x LS  S slice
    static constexpr int kG = kS + DK * LS;       // DK x LS  G slice
    static constexpr int kEnd0 = kG + DK * LS, kEnd1 = kW + 4 * kC * kLC,
                         kEnd2 = kY + 3 * 16 * 17;
    static constexpr int kFloats = kEnd0 > kEnd1 ? (kEnd0 > kEnd2 ? kEnd0 : kEnd2)
                                                 : (kEnd1 > kEnd2 ? kEnd1 : kEnd2);
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    static_assert(kBytes <= 232448, "one CTA's shared memory");
    static_assert(kFloats - kW >= kC * LK, "room for the t3 terms");
};

// KDA's per-chunk gradients: one CTA per (batch, head, chunk), d_q, d_k,
// d_beta and d_g (fp32 [BH][T][DK]) from S at the chunk's start (S_chunks)
// and G at its end (G_chunks), over the value channels in slices of NS.
template <class Ops, typename T, int DK, int DV>
__global__ void __launch_bounds__(Ops::kThreads, 1)
chunk_bwd_grads_kda_kernel(const T* __restrict__ q, const T* __restrict__ k,
                           const T* __restrict__ v, const T* __restrict__ beta,
                           const T* __restrict__ d_o, const float* __restrict__ S_chunks,
                           const float* __restrict__ G_chunks, T* __restrict__ d_q,
                           T* __restrict__ d_k, T* __restrict__ d_beta, int Tlen, int nchunks,
                           const float* __restrict__ gate, float* __restrict__ d_g) {
    constexpr int NS = 16;
    using L = GradKdaSmem<DK, NS, Ops::kPad>;
    constexpr int LK = L::LK, LS = L::LS, kLC = L::kLC, NT = Ops::kThreads;
    static_assert(NT == 256 && DK <= NT, "thread layout: a thread per key channel");
    extern __shared__ float smem[];
    float* Ks = smem + L::kK;
    float* Qs = smem + L::kQ;
    float* Gk = smem + L::kGk;
    float* Am = smem + L::kA;
    float* Xm = smem + L::kX;
    float* Pm = smem + L::kP;
    float* KK = smem + L::kKK;
    float* Ys = smem + L::kY;
    float* bs = smem + L::kB;
    float* GL = smem + L::kGL;
    float* t3 = smem + L::kT3;
    float* t4 = smem + L::kT4;
    float* Vs = smem + L::kV;
    float* Ds = smem + L::kD;
    float* Rs = smem + L::kR;
    float* Us = smem + L::kU;
    float* Es = smem + L::kE;
    float* Fs = smem + L::kF;
    float* Ss = smem + L::kS;
    float* Gs = smem + L::kG;
    const int tid = threadIdx.x;
    const int bh = blockIdx.x / nchunks, c = blockIdx.x % nchunks;
    const int t0 = c * kC, n = min(kC, Tlen - t0);
    const size_t tok0 = (size_t)bh * Tlen;
    const size_t st0 = ((size_t)bh * nchunks + c) * DK * DV;

    load_rows<NT, DK, LK, DK>(Ks, k, tok0, t0, n, 0);
    load_rows<NT, DK, LK, DK>(Qs, q, tok0, t0, n, 0);
    if (tid < kC) bs[tid] = tid < n ? to_f32(beta[tok0 + t0 + tid]) : 0.f;
    const bool sep = chunk_decay_kda<NT, DK, LK>(gate, tok0 + t0, n, Gk, GL);
    if (sep)
        form_a_p_kda_sep<Ops, DK>(Ks, Qs, Gk, bs, Am, Pm, KK);
    else
        form_a_p_kda_exact<DK, LK, kLC>(Ks, Qs, Gk, bs, Am, Pm, KK);
    __syncthreads();
    unit_lower_inverse64<NT, kLC>(Am, Xm, Ys);  // ends with a barrier

    const auto gam = [&](int t, int i) { return __expf(Gk[t * LK + i]); };
    const auto fdec = [&](int t, int i) { return __expf(GL[i] - Gk[t * LK + i]); };
    // aQ: dO S^T (then times gamma); aKs: -dV S^T (then times gamma), plus dK_r;
    // aKg: U' G^T (then times f), plus dK_P and dK_c
    typename Ops::template Acc<64, DK> aQ, aKs, aKg;
    typename Ops::template Acc<64, 64> aP, aT;
    Ops::zero(aQ);
    Ops::zero(aKs);
    Ops::zero(aKg);
    Ops::zero(aP);
    Ops::zero(aT);
    float t4c = 0.f;  // thread i < DK: <G, S> over key channel i
    for (int js = 0; js < DV; js += NS) {
        load_rows<NT, NS, LS, DV>(Vs, v, tok0, t0, n, js);
        load_rows<NT, NS, LS, DV>(Ds, d_o, tok0, t0, n, js);
        load_tile<NT, DK, NS, LS, DV>(Ss, S_chunks + st0, 0, DK, js);
        load_tile<NT, DK, NS, LS, DV>(Gs, G_chunks + st0, 0, DK, js);
        __syncthreads();
        if (tid < DK)
            for (int jj = 0; jj < NS; ++jj) t4c = fmaf(Gs[tid * LS + jj], Ss[tid * LS + jj], t4c);
        {   // R = V - (K o gamma) S and dU' = P^T dO + (K o f) G
            typename Ops::template Acc<64, NS> r, e;
            Ops::zero(r);
            Ops::zero(e);
            Ops::template mm<64, NS, DK>(r, [&](int m, int i) { return Ks[m * LK + i] * gam(m, i); },
                               [&](int i, int nn) { return Ss[i * LS + nn]; });
            Ops::template mm<64, NS, kC>(e, [&](int m, int s) { return Pm[s * kLC + m]; },
                               [&](int s, int nn) { return Ds[s * LS + nn]; });
            Ops::template mm<64, NS, DK>(e, [&](int m, int i) { return Ks[m * LK + i] * fdec(m, i); },
                               [&](int i, int nn) { return Gs[i * LS + nn]; });
            Ops::for_each(r, [&](int m, int nn, float x) { Rs[m * LS + nn] = Vs[m * LS + nn] - x; });
            Ops::for_each(e, [&](int m, int nn, float x) { Es[m * LS + nn] = x; });
        }
        __syncthreads();
        {   // U' = X diag(beta) R and dV = diag(beta) X^T dU'
            typename Ops::template Acc<64, NS> u, f;
            Ops::zero(u);
            Ops::zero(f);
            Ops::template mm<64, NS, kC>(u, [&](int m, int s) { return Xm[m * kLC + s] * bs[s]; },
                               [&](int s, int nn) { return Rs[s * LS + nn]; });
            Ops::template mm<64, NS, kC>(f, [&](int m, int s) { return Xm[s * kLC + m]; },
                               [&](int s, int nn) { return Es[s * LS + nn]; });
            Ops::for_each(u, [&](int m, int nn, float x) { Us[m * LS + nn] = x; });
            Ops::for_each(f, [&](int m, int nn, float x) { Fs[m * LS + nn] = bs[m] * x; });
        }
        __syncthreads();
        // dP += dO U'^T, dTm += dU' R^T, and the value sums of aQ, aKs, aKg
        Ops::template mm<64, 64, NS>(aP, [&](int m, int j) { return Ds[m * LS + j]; },
                           [&](int j, int nn) { return Us[nn * LS + j]; });
        Ops::template mm<64, 64, NS>(aT, [&](int m, int j) { return Es[m * LS + j]; },
                           [&](int j, int nn) { return Rs[nn * LS + j]; });
        Ops::template mm<64, DK, NS>(aQ, [&](int m, int j) { return Ds[m * LS + j]; },
                           [&](int j, int i) { return Ss[i * LS + j]; });
        Ops::template mm<64, DK, NS>(aKs, [&](int m, int j) { return -Fs[m * LS + j]; },
                           [&](int j, int i) { return Ss[i * LS + j]; });
        Ops::template mm<64, DK, NS>(aKg, [&](int m, int j) { return Us[m * LS + j]; },
                           [&](int j, int i) { return Gs[i * LS + j]; });
        __syncthreads();
    }
    {   // t3 = sum_s k_s f_s (U' G^T)[s] per key channel, through the work area so
        // that its order (and that of t4) is fixed: d_g is reproducible bit for bit
        float* kfu = smem + L::kW;  // C x LK
        Ops::for_each(aKg, [&](int s, int i, float x) {
            kfu[s * LK + i] = Ks[s * LK + i] * fdec(s, i) * x;
        });
        __syncthreads();
        if (tid < DK) {
            float acc = 0.f;
            for (int s = 0; s < n; ++s) acc += kfu[s * LK + tid];
            t3[tid] = acc;
            t4[tid] = t4c;
        }
        __syncthreads();
    }

    // The work area now holds C x C matrices.
    float* dPm = smem + L::kW;
    float* dTs = dPm + kC * kLC;
    float* M1 = dTs + kC * kLC;
    float* dAm = M1 + kC * kLC;
    Ops::for_each(aP, [&](int m, int nn, float x) { dPm[m * kLC + nn] = nn <= m ? x : 0.f; });
    Ops::for_each(aT, [&](int m, int nn, float x) { dTs[m * kLC + nn] = x; });
    __syncthreads();
    {   // M1 = (dTm diag(beta)) X^T
        typename Ops::template Acc<64, 64> acc;
        Ops::zero(acc);
        Ops::template mm<64, 64, kC>(acc, [&](int m, int s) { return dTs[m * kLC + s] * bs[s]; },
                           [&](int s, int nn) { return Xm[nn * kLC + s]; });
        Ops::for_each(acc, [&](int m, int nn, float x) { M1[m * kLC + nn] = x; });
    }
    float db = 0.f;  // thread j < 64: dbeta_j
    if (tid < kC)
        for (int i = 0; i < kC; ++i) db = fmaf(Xm[i * kLC + tid], dTs[i * kLC + tid], db);
    __syncthreads();
    {   // dA = strict_tril(-X^T M1)
        typename Ops::template Acc<64, 64> acc;
        Ops::zero(acc);
        Ops::template mm<64, 64, kC>(acc, [&](int m, int s) { return Xm[s * kLC + m]; },
                           [&](int s, int nn) { return M1[s * kLC + nn]; });
        Ops::for_each(acc, [&](int m, int nn, float x) { dAm[m * kLC + nn] = nn < m ? -x : 0.f; });
    }
    __syncthreads();
    if (tid < kC)
        for (int l = 0; l < kC; ++l) db = fmaf(dAm[tid * kLC + l], KK[tid * kLC + l], db);

    if (sep) {
        // the ratio sums as products of scaled operands, added before the
        // gamma / f factors: K o exp(-G) on the right of dP and dA2, and
        // (Q, K) o exp(G - G_L) on the right of their transposes
        const auto km = [&](int s, int i) { return Ks[s * LK + i] * __expf(-Gk[s * LK + i]); };
        Ops::template mm<64, DK, kC>(aQ, [&](int m, int s) { return dPm[m * kLC + s]; }, km);
        Ops::template mm<64, DK, kC>(aKs, [&](int m, int s) { return bs[m] * dAm[m * kLC + s]; },
                                     km);
        Ops::template mm<64, DK, kC>(aKg, [&](int m, int t) { return dPm[t * kLC + m]; },
                                     [&](int t, int i) {
                                         return Qs[t * LK + i] * __expf(Gk[t * LK + i] - GL[i]);
                                     });
        Ops::template mm<64, DK, kC>(aKg, [&](int m, int t) { return bs[t] * dAm[t * kLC + m]; },
                                     [&](int t, int i) {
                                         return Ks[t * LK + i] * __expf(Gk[t * LK + i] - GL[i]);
                                     });
        Ops::update2(aQ, aKs, [&](int t, int i, float& xq, float& xk) {
            const float ga = gam(t, i);
            xq *= ga;
            xk *= ga;
        });
        Ops::update2(aKg, aKg, [&](int s, int i, float& x, float&) { x *= fdec(s, i); });
    } else {
        // the factors first, then every ratio with its own exponential
        Ops::update2(aQ, aKs, [&](int t, int i, float& xq, float& xk) {
            const float Gt = Gk[t * LK + i];
            float sq = 0.f, sk = 0.f;
            for (int s = 0; s <= t; ++s) {
                const float e = __expf(fminf(Gt - Gk[s * LK + i], 0.f)) * Ks[s * LK + i];
                sq = fmaf(dPm[t * kLC + s], e, sq);
                sk = fmaf(dAm[t * kLC + s], e, sk);
            }
            const float ga = __expf(Gt);
            xq = fmaf(xq, ga, sq);
            xk = fmaf(xk, ga, bs[t] * sk);
        });
        Ops::update2(aKg, aKg, [&](int s, int i, float& x, float&) {
            const float Gs_ = Gk[s * LK + i];
            float acc = 0.f;
            for (int t = s; t < kC; ++t) {
                const float w = fmaf(dPm[t * kLC + s], Qs[t * LK + i],
                                     bs[t] * dAm[t * kLC + s] * Ks[t * LK + i]);
                acc = fmaf(w, __expf(fminf(Gk[t * LK + i] - Gs_, 0.f)), acc);
            }
            x = fmaf(x, __expf(GL[i] - Gs_), acc);
        });
    }
    __syncthreads();  // every read of the decay is done: Gk takes dG
    Ops::for_each(aQ, [&](int m, int i, float x) {
        Gk[m * LK + i] = Qs[m * LK + i] * x;
        if (m < n) d_q[(tok0 + t0 + m) * DK + i] = from_f32<T>(x);
    });
    Ops::update2(aKs, aKg, [&](int m, int i, float& xs, float& xg) {
        Gk[m * LK + i] += Ks[m * LK + i] * (xs - xg);
        if (m < n) d_k[(tok0 + t0 + m) * DK + i] = from_f32<T>(xs + xg);
    });
    __syncthreads();
    if (tid < DK) {  // d_g: dG summed from each token to the chunk's end
        float s = __expf(GL[tid]) * t4[tid] + t3[tid];  // the last token's share of <G, S_next>
        for (int t = n - 1; t >= 0; --t) {
            s += Gk[t * LK + tid];
            d_g[(tok0 + t0 + t) * DK + tid] = s;
        }
    }
    if (tid < n) d_beta[tok0 + t0 + tid] = from_f32<T>(db);
}

// With `tiles` (the tensor-core state recompute's [PT; Tm] workspace), the
// chain runs on tcgen05 (chunk_tc.cu) instead of chunk_bwd_chain_kernel.
template <typename T, int DK, int DV>
cudaError_t launch_bwd_typed(const void* q, const void* k, const void* v, const void* beta,
                             const void* d_o, const float* d_S_T, void* d_q, void* d_k, void* d_v,
                             void* d_beta, float* d_S0, float* Sc, float* Gc, int BH, int Tlen,
                             const void* tiles, cudaStream_t stream) {
    constexpr int NV = DV < 64 ? DV : 64;
    // fp32 I/O keeps fp32 products; bf16 I/O runs them on tf32 tensor cores.
    using Ops = std::conditional_t<std::is_same_v<T, float>, simt::Fp32Ops, simt::Tf32Ops<8>>;
    using LC = ChainSmem<DK, NV, Ops::kPad>;
    using LG = GradSmem<DK, 32, Ops::kPad>;
    const int nchunks = (Tlen + kC - 1) / kC;
    auto chain = chunk_bwd_chain_kernel<Ops, T, DK, DV, NV>;
    auto grads = chunk_bwd_grads_kernel<Ops, T, DK, DV>;
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LC::kBytes)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grads, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LG::kBytes)) != cudaSuccess)
        return err;
    const long long g_chain = (long long)BH * (DV / NV), g_grads = (long long)BH * nchunks;
    if (g_chain > 0x7fffffffLL || g_grads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (tiles)
        err = launch_chunk_bwd_chain_tc(q, k, d_o, d_S_T, d_v, d_S0, Gc, tiles, BH, Tlen, stream);
    else {
        chain<<<(unsigned)g_chain, Ops::kThreads, LC::kBytes, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(beta),
            static_cast<const T*>(d_o), d_S_T, static_cast<T*>(d_v), d_S0, Gc, Tlen, nullptr);
        err = cudaGetLastError();
    }
    if (err != cudaSuccess) return err;
    grads<<<(unsigned)g_grads, Ops::kThreads, LG::kBytes, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(beta), static_cast<const T*>(d_o), Sc, Gc, static_cast<T*>(d_q),
        static_cast<T*>(d_k), static_cast<T*>(d_beta), Tlen, nchunks, nullptr, nullptr);
    return cudaGetLastError();
}

// Gated DeltaNet's backward: the chain and the per-chunk gradients with the
// decay; fp32 products on the CUDA cores for fp32 I/O, tf32 tensor-core
// products (fp32 accumulation) for bf16 I/O, as the plain backward.
// chain_done: the tcgen05 chain has already written Gc, d_v and d_S0.
template <typename T, int DK, int DV>
cudaError_t launch_bwd_gated_typed(const void* q, const void* k, const void* v, const void* beta,
                                   const float* g, const void* d_o, const float* d_S_T, void* d_q,
                                   void* d_k, void* d_v, void* d_beta, float* d_g, float* d_S0,
                                   float* Sc, float* Gc, int BH, int Tlen, cudaStream_t stream,
                                   bool chain_done) {
    constexpr int NV = DV < 64 ? DV : 64;
    using Ops = std::conditional_t<std::is_same_v<T, float>, simt::Fp32Ops, simt::Tf32Ops<8>>;
    using LC = ChainSmem<DK, NV, Ops::kPad>;
    using LG = GradSmem<DK, 32, Ops::kPad>;
    const int nchunks = (Tlen + kC - 1) / kC;
    auto chain = chunk_bwd_chain_kernel<Ops, T, DK, DV, NV, true>;
    auto grads = chunk_bwd_grads_kernel<Ops, T, DK, DV, true>;
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LC::kBytes)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grads, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LG::kBytes)) != cudaSuccess)
        return err;
    const long long g_chain = (long long)BH * (DV / NV), g_grads = (long long)BH * nchunks;
    if (g_chain > 0x7fffffffLL || g_grads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (!chain_done) {
        chain<<<(unsigned)g_chain, Ops::kThreads, LC::kBytes, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(beta),
            static_cast<const T*>(d_o), d_S_T, static_cast<T*>(d_v), d_S0, Gc, Tlen, g);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    grads<<<(unsigned)g_grads, Ops::kThreads, LG::kBytes, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(beta), static_cast<const T*>(d_o), Sc, Gc, static_cast<T*>(d_q),
        static_cast<T*>(d_k), static_cast<T*>(d_beta), Tlen, nchunks, g, d_g);
    return cudaGetLastError();
}

// KDA's backward: its chain and per-chunk gradients, fp32 products on the
// CUDA cores for fp32 I/O and tf32 tensor-core products for bf16 I/O.
// chain_done: the tcgen05 chain has already written Gc, d_v and d_S0.
template <typename T, int DK, int DV>
cudaError_t launch_bwd_kda_typed(const void* q, const void* k, const void* v, const void* beta,
                                 const float* g, const void* d_o, const float* d_S_T, void* d_q,
                                 void* d_k, void* d_v, void* d_beta, float* d_g, float* d_S0,
                                 float* Sc, float* Gc, int BH, int Tlen, cudaStream_t stream,
                                 bool chain_done) {
    constexpr int NV = 64;
    using Ops = std::conditional_t<std::is_same_v<T, float>, simt::Fp32Ops, simt::Tf32Ops<8>>;
    using LC = ChainKdaSmem<DK, NV, Ops::kPad>;
    using LG = GradKdaSmem<DK, 16, Ops::kPad>;
    const int nchunks = (Tlen + kC - 1) / kC;
    auto chain = chunk_bwd_chain_kda_kernel<Ops, T, DK, DV, NV>;
    auto grads = chunk_bwd_grads_kda_kernel<Ops, T, DK, DV>;
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LC::kBytes)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grads, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)LG::kBytes)) != cudaSuccess)
        return err;
    const long long g_chain = (long long)BH * (DV / NV), g_grads = (long long)BH * nchunks;
    if (g_chain > 0x7fffffffLL || g_grads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (!chain_done) {
        chain<<<(unsigned)g_chain, Ops::kThreads, LC::kBytes, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(beta),
            static_cast<const T*>(d_o), d_S_T, static_cast<T*>(d_v), d_S0, Gc, Tlen, g);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    grads<<<(unsigned)g_grads, Ops::kThreads, LG::kBytes, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(beta), static_cast<const T*>(d_o), Sc, Gc, static_cast<T*>(d_q),
        static_cast<T*>(d_k), static_cast<T*>(d_beta), Tlen, nchunks, g, d_g);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_dims(const void* q, const void* k, const void* v, const void* beta,
                            const void* d_o, const float* d_S_T, void* d_q, void* d_k, void* d_v,
                            void* d_beta, float* d_S0, float* Sc, float* Gc, int BH, int Tlen,
                            int dk, int dv, const void* tiles, cudaStream_t st) {
#define DN_BWD_CASE(DK_, DV_)                                                                   \
    if (dk == DK_ && dv == DV_)                                                                 \
        return launch_bwd_typed<T, DK_, DV_>(q, k, v, beta, d_o, d_S_T, d_q, d_k, d_v, d_beta,  \
                                             d_S0, Sc, Gc, BH, Tlen, tiles, st);
    DN_BWD_CASE(128, 128)
    DN_BWD_CASE(128, 64)
    DN_BWD_CASE(64, 128)
    DN_BWD_CASE(64, 64)
#undef DN_BWD_CASE
    return cudaErrorNotSupported;
}

}  // namespace

namespace {
// Gated DeltaNet's rate on every key channel: gk[bh][t][c] = g[bh][t] (the
// KDA form with equal channels is Gated DeltaNet).
__global__ void broadcast_gate_kernel(const float* __restrict__ g, float4* __restrict__ gk,
                                      size_t n4, int per_tok4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float x = g[i / per_tok4];
        gk[i] = make_float4(x, x, x, x);
    }
}
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

// Workspace.  The fp32 S and G of every chunk; for bf16 with d = 128 also the
// tensor-core KDA forward's scratch and the broadcast rates it reads.
size_t chunk_bwd_gated_workspace_bytes(int BH, int T, int dk, int dv, int dt) {
    if (BH <= 0 || T <= 0) return 0;
    const size_t items = (size_t)BH * (size_t)((T + kC - 1) / kC);
    const size_t states = 2 * items * (size_t)dk * (size_t)dv * sizeof(float);
    if (!chunk_tc_supports(dk, dv, dt)) return states;
    return states + align256(chunk_tc_kda_workspace_bytes(BH, T)) +
           (size_t)BH * (size_t)T * (size_t)dk * sizeof(float);
}

cudaError_t launch_chunk_bwd_gated(const void* q, const void* k, const void* v, const void* beta,
                                   const float* g, const float* S0, const void* d_o,
                                   const float* d_S_T, void* d_q, void* d_k, void* d_v,
                                   void* d_beta, float* d_g, float* d_S0, int BH, int T, int dk,
                                   int dv, int dt, void* workspace, cudaStream_t stream,
                                   const char** stage) {
    if (BH <= 0 || T <= 0) return cudaSuccess;
    *stage = "state recompute";
    const size_t per = (size_t)BH * ((T + kC - 1) / kC) * (size_t)dk * dv;
    float* const Sc = static_cast<float*>(workspace);
    float* const Gc = Sc + per;
    const bool tc = chunk_tc_supports(dk, dv, dt);
    cudaError_t err;
    if (tc) {
        // bf16, d = 128: Gated DeltaNet as KDA with the rate on every key
        // channel, so the states come from the tcgen05 KDA forward and the
        // chain runs on tcgen05 from the decayed operands that forward leaves
        uint8_t* const kws = reinterpret_cast<uint8_t*>(Gc + per);
        float* const gk = reinterpret_cast<float*>(kws + align256(chunk_tc_kda_workspace_bytes(BH, T)));
        *stage = "rates on every key channel";
        const size_t n4 = (size_t)BH * (size_t)T * (size_t)(dk / 4);
        broadcast_gate_kernel<<<1216, 256, 0, stream>>>(g, reinterpret_cast<float4*>(gk), n4, dk / 4);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        *stage = "state recompute";
        err = launch_chunk_tc_kda(q, k, v, beta, gk, S0, nullptr, nullptr, BH, T, dk, dv, dt, kws,
                                  stream, kNoNorm, Sc);
        if (err != cudaSuccess) return err;
        *stage = "state-gradient chain";
        err = launch_chunk_bwd_chain_tc_kda(d_o, d_S_T, d_v, d_S0, Gc, kws, BH, T, stream);
    } else {
        err = launch_chunk_simt(q, k, v, beta, S0, nullptr, nullptr, BH, T, dk, dv, dt, stream,
                                Sc, g);
    }
    if (err != cudaSuccess) return err;
    *stage = "gated chain and gradients";
#define DN_GBWD_CASE(T_, DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_)                                                                 \
        return launch_bwd_gated_typed<T_, DK_, DV_>(q, k, v, beta, g, d_o, d_S_T, d_q, d_k, d_v,\
                                                     d_beta, d_g, d_S0, Sc, Gc, BH, T, stream, tc);
    if (dt == 0) {
        DN_GBWD_CASE(float, 128, 128)
        DN_GBWD_CASE(float, 128, 64)
        DN_GBWD_CASE(float, 64, 128)
        DN_GBWD_CASE(float, 64, 64)
    } else {
        DN_GBWD_CASE(__nv_bfloat16, 128, 128)
        DN_GBWD_CASE(__nv_bfloat16, 128, 64)
        DN_GBWD_CASE(__nv_bfloat16, 64, 128)
        DN_GBWD_CASE(__nv_bfloat16, 64, 64)
    }
#undef DN_GBWD_CASE
    return cudaErrorNotSupported;
}

size_t chunk_bwd_kda_workspace_bytes(int BH, int T, int dk, int dv, int dt) {
    if (BH <= 0 || T <= 0) return 0;
    const size_t items = (size_t)BH * (size_t)((T + kC - 1) / kC);
    const size_t states = 2 * items * (size_t)dk * (size_t)dv * sizeof(float);
    return states + (chunk_tc_supports(dk, dv, dt) ? chunk_tc_kda_workspace_bytes(BH, T) : 0);
}

cudaError_t launch_chunk_bwd_kda(const void* q, const void* k, const void* v, const void* beta,
                                 const float* g, const float* S0, const void* d_o,
                                 const float* d_S_T, void* d_q, void* d_k, void* d_v,
                                 void* d_beta, float* d_g, float* d_S0, int BH, int T, int dk,
                                 int dv, int dt, void* workspace, cudaStream_t stream,
                                 const char** stage) {
    if (BH <= 0 || T <= 0) return cudaSuccess;
    *stage = "state recompute";
    const size_t per = (size_t)BH * ((T + kC - 1) / kC) * (size_t)dk * dv;
    float* const Sc = static_cast<float*>(workspace);
    float* const Gc = Sc + per;
    const bool tc = chunk_tc_supports(dk, dv, dt);
    cudaError_t err =
        tc ? launch_chunk_tc_kda(q, k, v, beta, g, S0, nullptr, nullptr, BH, T, dk, dv, dt,
                                 Gc + per, stream, kNoNorm, Sc)
           : launch_chunk_simt_kda(q, k, v, beta, g, S0, nullptr, nullptr, BH, T, dk, dv, dt,
                                   stream, kNoNorm, Sc);
    if (err != cudaSuccess) return err;
    if (tc) {  // the chain on tcgen05, from the forward's decayed operands and tiles
        *stage = "KDA state-gradient chain";
        err = launch_chunk_bwd_chain_tc_kda(d_o, d_S_T, d_v, d_S0, Gc, Gc + per, BH, T, stream);
        if (err != cudaSuccess) return err;
    }
    *stage = "KDA chain and gradients";
#define DN_KBWD_CASE(T_, DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_)                                                                 \
        return launch_bwd_kda_typed<T_, DK_, DV_>(q, k, v, beta, g, d_o, d_S_T, d_q, d_k, d_v,  \
                                                   d_beta, d_g, d_S0, Sc, Gc, BH, T, stream, tc);
    if (dt == 0) {
        DN_KBWD_CASE(float, 128, 128)
        DN_KBWD_CASE(float, 128, 64)
        DN_KBWD_CASE(float, 64, 128)
        DN_KBWD_CASE(float, 64, 64)
    } else {
        DN_KBWD_CASE(__nv_bfloat16, 128, 128)
        DN_KBWD_CASE(__nv_bfloat16, 128, 64)
        DN_KBWD_CASE(__nv_bfloat16, 64, 128)
        DN_KBWD_CASE(__nv_bfloat16, 64, 64)
    }
#undef DN_KBWD_CASE
    return cudaErrorNotSupported;
}

// Workspace.  Tensor-core path (bf16, dk = dv = 128): S at every chunk start
// and G at every chunk end as bf16, the forward's [PT; Tm] tiles and every
// chunk's (I + A)^{-1} (bf16 64 x 64).  Otherwise S and G in fp32.
size_t chunk_bwd_workspace_bytes(int BH, int T, int dk, int dv, int dt) {
    if (BH <= 0 || T <= 0) return 0;
    const size_t items = (size_t)BH * (size_t)((T + kC - 1) / kC);
    if (chunk_tc_supports(dk, dv, dt))
        return items * (4 * (size_t)dk * dv * 2 + 64 * 64 * 2) + chunk_tc_workspace_bytes(BH, T);
    return 2 * items * (size_t)dk * (size_t)dv * sizeof(float);
}

cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const void* beta,
                             const float* S0, const void* d_o, const float* d_S_T, void* d_q,
                             void* d_k, void* d_v, void* d_beta, float* d_S0, int BH, int T,
                             int dk, int dv, int dt, void* workspace, cudaStream_t stream,
                             const char** stage) {
    if (BH <= 0 || T <= 0) return cudaSuccess;
    *stage = "state recompute";
    const size_t items = (size_t)BH * ((T + kC - 1) / kC);
    const size_t per = items * (size_t)dk * dv;
    if (chunk_tc_supports(dk, dv, dt)) {
        // The tensor-core path: the two-pass forward records S (a bf16 hi
        // and lo tile per chunk) and X, the tcgen05 chain G (likewise) and
        // d_v, the tcgen05 gradient kernel d_q, d_k and d_beta.
        __nv_bfloat16* const Sb = static_cast<__nv_bfloat16*>(workspace);
        __nv_bfloat16* const Gb = Sb + 2 * per;
        __nv_bfloat16* const Xb = Gb + 2 * per;
        void* const tiles = Xb + items * 64 * 64;
        cudaError_t err = launch_chunk_tc(q, k, v, beta, S0, nullptr, nullptr, BH, T, dk, dv, dt,
                                          tiles, stream, Sb, kNoNorm, Xb);
        if (err != cudaSuccess) return err;
        *stage = "state-gradient chain";
        err = launch_chunk_bwd_chain_tc(q, k, d_o, d_S_T, d_v, d_S0, Gb, tiles, BH, T, stream);
        if (err != cudaSuccess) return err;
        *stage = "gradient kernel";
        return launch_chunk_bwd_grads_tc(q, k, v, beta, d_o, Sb, Gb, Xb, tiles, d_q, d_k, d_beta,
                                         BH, T, stream);
    }
    float* const Sc = static_cast<float*>(workspace);
    float* const Gc = Sc + per;
    cudaError_t err =
        launch_chunk_simt(q, k, v, beta, S0, nullptr, nullptr, BH, T, dk, dv, dt, stream, Sc);
    if (err != cudaSuccess) return err;
    *stage = "gradient kernels";
    if (dt == 0)
        return launch_bwd_dims<float>(q, k, v, beta, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_S0, Sc,
                                      Gc, BH, T, dk, dv, nullptr, stream);
    return launch_bwd_dims<__nv_bfloat16>(q, k, v, beta, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_S0,
                                          Sc, Gc, BH, T, dk, dv, nullptr, stream);
}

// ------------------------------------------------- packed variable-length sequences
// The backward of dn_chunk_fwd_varlen: sequence n is tokens cu[n] .. cu[n+1]-1
// of the packed [H][T][d] tensors.  Each sequence runs as its own batched
// backward (B = 1, H heads, its length) on contiguous copies: its rows of q,
// k, v, beta and d_o are gathered with one strided copy per tensor (H rows of
// len * d elements, T * d apart), and its gradients scattered back the same
// way.  The copies and the launches of one sequence queue on the stream
// behind the previous sequence's, so one set of scratch buffers serves all.
namespace {
struct VarlenBwdScratch {
    size_t ws, q, v, b;  // bytes: the batched backward's workspace, a dk tensor, a dv tensor, beta
};
VarlenBwdScratch varlen_bwd_scratch(int H, int lmax, int dk, int dv, int dt) {
    const size_t es = dt ? 2 : 4, rows = (size_t)H * (size_t)lmax;
    return {align256(chunk_bwd_workspace_bytes(H, lmax, dk, dv, dt)), align256(rows * dk * es),
            align256(rows * dv * es), align256(rows * es)};
}
int varlen_max_len(const int* cu, int N) {
    int lmax = 0;
    for (int n = 0; n < N; ++n) lmax = std::max(lmax, cu[n + 1] - cu[n]);
    return lmax;
}
}  // namespace

size_t chunk_bwd_varlen_workspace_bytes(const int* cu, int N, int H, int dk, int dv, int dt) {
    if (!cu || N <= 0 || H <= 0) return 0;
    const int lmax = varlen_max_len(cu, N);
    if (lmax <= 0) return 0;
    const VarlenBwdScratch s = varlen_bwd_scratch(H, lmax, dk, dv, dt);
    // inputs q, k, v, d_o, beta; gradients d_q, d_k, d_v, d_beta
    return s.ws + 4 * s.q + 3 * s.v + 2 * s.b;
}

cudaError_t launch_chunk_bwd_varlen(const void* q, const void* k, const void* v, const void* beta,
                                    const float* S0, const void* d_o, const float* d_S_T,
                                    void* d_q, void* d_k, void* d_v, void* d_beta, float* d_S0,
                                    const int* cu, int N, int H, int T, int dk, int dv, int dt,
                                    void* workspace, cudaStream_t stream, const char** stage) {
    const int lmax = varlen_max_len(cu, N);
    const VarlenBwdScratch s = varlen_bwd_scratch(H, std::max(lmax, 1), dk, dv, dt);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    void* const ws = p;
    p += s.ws;
    uint8_t *tq = p, *tk = p + s.q, *tdq = p + 2 * s.q, *tdk = p + 3 * s.q;
    p += 4 * s.q;
    uint8_t *tv = p, *tdo = p + s.v, *tdv = p + 2 * s.v;
    p += 3 * s.v;
    uint8_t *tb = p, *tdb = p + s.b;
    const size_t es = dt ? 2 : 4, state = (size_t)H * dk * dv;
    cudaError_t e = cudaSuccess;
    // H rows of `width` bytes, `pitch` bytes apart on the packed side
    auto gather = [&](void* dst, const void* src, size_t tok0, int len, int d) {
        const size_t w = (size_t)len * d * es;
        return cudaMemcpy2DAsync(dst, w, static_cast<const uint8_t*>(src) + tok0 * d * es,
                                 (size_t)T * d * es, w, (size_t)H, cudaMemcpyDeviceToDevice, stream);
    };
    auto scatter = [&](void* dst, const void* src, size_t tok0, int len, int d) {
        const size_t w = (size_t)len * d * es;
        return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + tok0 * d * es, (size_t)T * d * es,
                                 src, w, w, (size_t)H, cudaMemcpyDeviceToDevice, stream);
    };
    for (int n = 0; n < N && e == cudaSuccess; ++n) {
        const int a = cu[n], len = cu[n + 1] - cu[n];
        const float* const s0 = S0 ? S0 + (size_t)n * state : nullptr;
        const float* const dst = d_S_T ? d_S_T + (size_t)n * state : nullptr;
        float* const ds0 = d_S0 ? d_S0 + (size_t)n * state : nullptr;
        if (len == 0) {  // the state gradient passes through
            *stage = "empty sequence";
            if (ds0)
                e = dst ? cudaMemcpyAsync(ds0, dst, state * sizeof(float), cudaMemcpyDeviceToDevice,
                                          stream)
                        : cudaMemsetAsync(ds0, 0, state * sizeof(float), stream);
            continue;
        }
        *stage = "gathering a sequence";
        if ((e = gather(tq, q, a, len, dk)) != cudaSuccess || (e = gather(tk, k, a, len, dk)) != cudaSuccess ||
            (e = gather(tv, v, a, len, dv)) != cudaSuccess || (e = gather(tdo, d_o, a, len, dv)) != cudaSuccess ||
            (e = gather(tb, beta, a, len, 1)) != cudaSuccess)
            break;
        if ((e = launch_chunk_bwd(tq, tk, tv, tb, s0, tdo, dst, tdq, tdk, tdv, tdb, ds0, H, len, dk,
                                  dv, dt, ws, stream, stage)) != cudaSuccess)
            break;
        *stage = "scattering a sequence";
        if ((e = scatter(d_q, tdq, a, len, dk)) != cudaSuccess ||
            (e = scatter(d_k, tdk, a, len, dk)) != cudaSuccess ||
            (e = scatter(d_v, tdv, a, len, dv)) != cudaSuccess ||
            (e = scatter(d_beta, tdb, a, len, 1)) != cudaSuccess)
            break;
    }
    return e;
}

}  // namespace dn
