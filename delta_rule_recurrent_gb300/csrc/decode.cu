// decode.cu -- fused single-token delta-rule step (dn_recurrent_step).
//
// Per (batch, head) the state S ([dk][dv] fp32, value channel contiguous) is
// streamed from HBM once and written back once:
//     p = S^T k,  r = S^T q            (reductions over the key channel)
//     u = beta (v - p)                 (the error of "DeltaNet : écrire
//                                       l'erreur de prédiction plutôt que la
//                                       valeur", fr.news.hada.io/topic?id=31925)
//     S <- S + k u^T,  o = r + (k . q) u   (= S_new^T q, read after write)
// With a log keep rate g (Gated DeltaNet, "Gated DeltaNet : oublier d'abord
// l'état entier", same page) the state is first decayed by alpha = exp(g):
// p and r are taken from alpha S and the write is S <- alpha S + k u^T.  With
// one rate per key channel (KDA, "Kimi Delta Attention : atténuation par
// canal") row i of the stored state decays by alpha[i] instead.
//
// With a dn_qk_norm, q and k are L2-normalised (and q scaled) in fp32 after
// they are loaded, before any product uses them.
//
// Consecutive steps overlap their launches: each is launched with
// programmatic stream serialization, lets the next launch be scheduled once
// all of its CTAs have started, and waits (griddepcontrol.wait) for the grid
// before it in the stream to finish and flush before reading anything.
//
// Work split: one CTA per head.  A thread owns one float4 column group of
// the value channel and DK / RG rows of the key channel, so a warp's loads
// and stores cover 512 contiguous bytes, and the whole head's state sits in
// registers between the read and the write (one HBM round trip).  The
// column sums over the key channel are per-thread partials combined through
// shared memory; k . q is a warp-shuffle reduction.
#include "dn_common.cuh"
#include "dn_internal.h"

namespace dn {
namespace {

// kMode: 0 no decay, 1 one log keep rate per head (Gated DeltaNet), 2 one
// per key channel (KDA).
template <typename T, int DK, int DV, int NT, int kMode>
__global__ void __launch_bounds__(NT)
recurrent_step_kernel(const T* __restrict__ q, const T* __restrict__ k,
                      const T* __restrict__ v, const T* __restrict__ beta,
                      const float* __restrict__ g, float* __restrict__ S,
                      T* __restrict__ o, QkNorm nm) {
    constexpr int CG = DV / 4;    // float4 column groups per state row
    constexpr int RG = NT / CG;   // row groups (threads sharing a column group)
    constexpr int RPT = DK / RG;  // state rows per thread
    static_assert(NT % CG == 0 && DK % RG == 0, "bad decode tiling");

    __shared__ float ks[DK], qs[DK], vs[DV];
    __shared__ float4 red_p[RG][CG], red_r[RG][CG];
    __shared__ float kq_s, beta_s;

    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    float4* Sh = reinterpret_cast<float4*>(S + (size_t)head * DK * DV);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous step's state is written

    // Issue every state load first: RPT independent 16-byte loads per thread.
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = Sh[(size_t)(rg + r * RG) * CG + cg];
    // ... and the log keep rates with them, ahead of the barrier below.
    float graw[kMode == 2 ? RPT : 1];
    if constexpr (kMode == 2) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) graw[r] = g[(size_t)head * DK + rg + r * RG];
    } else if constexpr (kMode == 1) {
        graw[0] = g[head];
    }

    for (int i = tid; i < DK; i += NT) {
        ks[i] = to_f32(k[(size_t)head * DK + i]);
        qs[i] = to_f32(q[(size_t)head * DK + i]);
    }
    for (int j = tid; j < DV; j += NT) vs[j] = to_f32(v[(size_t)head * DV + j]);
    if (tid == 0) beta_s = to_f32(beta[head]);
    __syncthreads();
    if (norm_active(nm)) {  // k prepared by warp 0, q by warp 1, in fp32
        if (tid < 64) {
            const bool is_q = tid >= 32;
            float* const x = is_q ? qs : ks;
            float f = is_q ? nm.qscale : 1.f;
            if (nm.l2norm) {
                float ss = 0.f;
                for (int i = tid & 31; i < DK; i += 32) ss = fmaf(x[i], x[i], ss);
                f *= rsqrtf(warp_sum(ss) + nm.eps);
            }
            if (is_q || nm.l2norm)
                for (int i = tid & 31; i < DK; i += 32) x[i] *= f;
        }
        __syncthreads();
    }

    if (tid < 32) {
        float a = 0.f;
        for (int i = tid; i < DK; i += 32) a = fmaf(ks[i], qs[i], a);
        a = warp_sum(a);
        if (tid == 0) kq_s = a;
    }

    // keep rate of each of this thread's state rows (1 without decay)
    float a[RPT];
    if constexpr (kMode == 2) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) a[r] = __expf(graw[r]);
    } else {
        const float ah = kMode == 1 ? expf(graw[0]) : 1.f;
#pragma unroll
        for (int r = 0; r < RPT; ++r) a[r] = ah;
    }

    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {  // forget before predicting and reading
        const float kr = a[r] * ks[rg + r * RG], qr = a[r] * qs[rg + r * RG];
        pk.x = fmaf(s[r].x, kr, pk.x); pk.y = fmaf(s[r].y, kr, pk.y);
        pk.z = fmaf(s[r].z, kr, pk.z); pk.w = fmaf(s[r].w, kr, pk.w);
        pq.x = fmaf(s[r].x, qr, pq.x); pq.y = fmaf(s[r].y, qr, pq.y);
        pq.z = fmaf(s[r].z, qr, pq.z); pq.w = fmaf(s[r].w, qr, pq.w);
    }
    red_p[rg][cg] = pk;
    red_r[rg][cg] = pq;
    __syncthreads();

    float4 P = red_p[0][cg], R = red_r[0][cg];
#pragma unroll
    for (int g = 1; g < RG; ++g) {
        const float4 a = red_p[g][cg], b = red_r[g][cg];
        P.x += a.x; P.y += a.y; P.z += a.z; P.w += a.w;
        R.x += b.x; R.y += b.y; R.z += b.z; R.w += b.w;
    }
    const float bt = beta_s;
    const int j = cg * 4;
    float4 u;
    u.x = bt * (vs[j + 0] - P.x);
    u.y = bt * (vs[j + 1] - P.y);
    u.z = bt * (vs[j + 2] - P.z);
    u.w = bt * (vs[j + 3] - P.w);

    if (rg == 0) {
        const float kq = kq_s;
        T* oh = o + (size_t)head * DV + j;
        oh[0] = from_f32<T>(fmaf(kq, u.x, R.x));
        oh[1] = from_f32<T>(fmaf(kq, u.y, R.y));
        oh[2] = from_f32<T>(fmaf(kq, u.z, R.z));
        oh[3] = from_f32<T>(fmaf(kq, u.w, R.w));
    }

#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kr = ks[rg + r * RG];
        float4 x = s[r];
        x.x = fmaf(kr, u.x, a[r] * x.x); x.y = fmaf(kr, u.y, a[r] * x.y);
        x.z = fmaf(kr, u.z, a[r] * x.z); x.w = fmaf(kr, u.w, a[r] * x.w);
        Sh[(size_t)(rg + r * RG) * CG + cg] = x;
    }
}

template <typename T, int DK, int DV>
cudaError_t launch_typed(const void* q, const void* k, const void* v,
                         const void* beta, const float* g, int gpc, float* S, void* o, int BH,
                         cudaStream_t stream, const QkNorm& nm) {
    constexpr int NT = 256;
    const T* const qt = static_cast<const T*>(q);
    const T* const kt = static_cast<const T*>(k);
    const T* const vt = static_cast<const T*>(v);
    const T* const bt = static_cast<const T*>(beta);
    T* const ot = static_cast<T*>(o);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)BH);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!g)
        return cudaLaunchKernelEx(&cfg, recurrent_step_kernel<T, DK, DV, NT, 0>, qt, kt, vt, bt, g,
                                  S, ot, nm);
    if (gpc)
        return cudaLaunchKernelEx(&cfg, recurrent_step_kernel<T, DK, DV, NT, 2>, qt, kt, vt, bt, g,
                                  S, ot, nm);
    return cudaLaunchKernelEx(&cfg, recurrent_step_kernel<T, DK, DV, NT, 1>, qt, kt, vt, bt, g, S,
                              ot, nm);
}

template <typename T>
cudaError_t launch_dims(const void* q, const void* k, const void* v,
                        const void* beta, const float* g, int gpc, float* S, void* o, int BH,
                        int dk, int dv, cudaStream_t st, const QkNorm& nm) {
    if (dk == 128 && dv == 128)
        return launch_typed<T, 128, 128>(q, k, v, beta, g, gpc, S, o, BH, st, nm);
    if (dk == 128 && dv == 64)
        return launch_typed<T, 128, 64>(q, k, v, beta, g, gpc, S, o, BH, st, nm);
    if (dk == 64 && dv == 128)
        return launch_typed<T, 64, 128>(q, k, v, beta, g, gpc, S, o, BH, st, nm);
    if (dk == 64 && dv == 64) return launch_typed<T, 64, 64>(q, k, v, beta, g, gpc, S, o, BH, st, nm);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_recurrent_step(const void* q, const void* k, const void* v,
                                  const void* beta, float* S, void* o, int BH,
                                  int dk, int dv, int dt, cudaStream_t stream, const float* g,
                                  int g_per_channel, const QkNorm& norm) {
    if (BH <= 0) return cudaSuccess;
    if (dt == 0)
        return launch_dims<float>(q, k, v, beta, g, g_per_channel, S, o, BH, dk, dv, stream, norm);
    return launch_dims<__nv_bfloat16>(q, k, v, beta, g, g_per_channel, S, o, BH, dk, dv, stream,
                                      norm);
}

}  // namespace dn
