// api.cu -- the C ABI declared in include/deltanet.h: argument checks and
// dispatch.  Every check runs on the host before anything is enqueued.
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/deltanet.h"
#include "dn_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

int ok() {
    g_last_error[0] = '\0';
    return DN_OK;
}

struct Span {
    const char* name;
    const void* p;
    size_t bytes;
};

bool overlaps(const Span& a, const Span& b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// The pointer must be device (or managed) memory of the current device and
// aligned to `align` bytes.
int check_device_ptr(const Span& s, size_t align, int device) {
    if (!s.p) return fail(DN_ERR_INVALID_ARG, "%s is NULL", s.name);
    if ((uintptr_t)s.p % align != 0)
        return fail(DN_ERR_INVALID_ARG, "%s is not %zu-byte aligned", s.name, align);
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, s.p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DN_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes failed (%s)", s.name,
                    cudaGetErrorString(e));
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(DN_ERR_INVALID_ARG, "%s is not device memory", s.name);
    if (attr.type == cudaMemoryTypeDevice && attr.device != device)
        return fail(DN_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", s.name,
                    attr.device, device);
    return DN_OK;
}

// The calling thread's device, with its primary context made current: the
// tensor maps are encoded through the driver, which needs a current context,
// and a thread that has made no runtime call yet (an autograd worker, say)
// has none.
int current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e == cudaSuccess) e = cudaSetDevice(*dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DN_ERR_CUDA, "cudaGetDevice/cudaSetDevice: %s", cudaGetErrorString(e));
    }
    return DN_OK;
}

int cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(DN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool supported_dim(int d) { return d == 64 || d == 128; }

size_t elem_size(int dt) { return dt == DN_F32 ? 4 : 2; }

}  // namespace

extern "C" {

const char* dn_status_string(int status) {
    switch (status) {
        case DN_OK: return "DN_OK";
        case DN_ERR_INVALID_ARG: return "DN_ERR_INVALID_ARG";
        case DN_ERR_UNSUPPORTED: return "DN_ERR_UNSUPPORTED";
        case DN_ERR_CUDA: return "DN_ERR_CUDA";
        default: return "DN_UNKNOWN_STATUS";
    }
}

const char* dn_last_error(void) { return g_last_error; }

int dn_abi_version(void) { return DN_ABI_VERSION; }

int dn_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    const unsigned int e = dn::chunk_tc_take_device_error();
    return e == ~0u ? -1 : (int)e;
}

int dn_debug_first_wait_ns(unsigned long long ns) {
    const cudaError_t e = dn::set_first_wait_limit(ns);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DN_ERR_CUDA, "setting the wait limit: %s", cudaGetErrorString(e));
    }
    return DN_OK;
}

size_t dn_chunk_fwd_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || !dn::chunk_tc_fwd_supports(dk, dv, dt)) return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    const size_t chunks = (size_t)BH * (size_t)((T + 63) / 64);
    return dn::chunk_tc_workspace_bytes((int)BH, T) + chunks * dn::chunk_tc_side_bytes_per_chunk();
}

// The optional in-kernel preparation of q and k (NULL: none).
static int norm_options(const dn_qk_norm* norm, dn::QkNorm* out) {
    *out = dn::kNoNorm;
    if (!norm) return DN_OK;
    if (!isfinite(norm->scale)) return fail(DN_ERR_INVALID_ARG, "dn_qk_norm.scale must be finite");
    if (norm->l2norm && (!isfinite(norm->eps) || norm->eps < 0.0f))
        return fail(DN_ERR_INVALID_ARG, "dn_qk_norm.eps must be finite and >= 0");
    out->l2norm = norm->l2norm ? 1 : 0;
    out->qscale = norm->scale;
    out->eps = norm->l2norm ? norm->eps : 0.0f;
    return DN_OK;
}

// The checks every chunkwise forward shares: sizes, dtype, supported shape.
static int check_chunk_sizes(long long nseq, int H, int T, int dk, int dv, int C, int dt,
                             const char* nname) {
    if (nseq < 0 || H < 0 || T < 0)
        return fail(DN_ERR_INVALID_ARG, "negative size (%s=%lld H=%d T=%d)", nname, nseq, H, T);
    if (dt != DN_F32 && dt != DN_BF16) return fail(DN_ERR_INVALID_ARG, "unknown dtype %d", dt);
    if (dk <= 0 || dv <= 0 || C <= 0)
        return fail(DN_ERR_INVALID_ARG, "dk, dv and C must be positive");
    if (!supported_dim(dk) || !supported_dim(dv))
        return fail(DN_ERR_UNSUPPORTED, "dk=%d dv=%d: this library supports 64 and 128", dk, dv);
    if (C != 64) return fail(DN_ERR_UNSUPPORTED, "chunk length C=%d: this library supports 64", C);
    return DN_OK;
}

// The tensors of one chunkwise forward (g: the log keep rates of the
// decayed forms, g_align its required alignment, 0 when the form has none).
struct ChunkSpans {
    Span q, k, v, beta, g, o, S0, S_T;
    size_t beta_align, g_align, state_bytes;
};

static ChunkSpans chunk_spans(const void* q, const void* k, const void* v, const void* beta,
                              const float* g, size_t g_per_token, size_t g_align,
                              const float* S0, void* o, float* S_T, size_t ntok, long long nstate,
                              int dk, int dv, int dt) {
    const size_t es = elem_size(dt);
    const size_t state_bytes = (size_t)nstate * dk * dv * sizeof(float);
    return ChunkSpans{Span{"q", q, ntok * dk * es},
                      Span{"k", k, ntok * dk * es},
                      Span{"v", v, ntok * dv * es},
                      Span{"beta", beta, ntok * es},
                      Span{"g", g, ntok * g_per_token * sizeof(float)},
                      Span{"o", o, ntok * dv * es},
                      Span{"S0", S0, state_bytes},
                      Span{"S_T", S_T, state_bytes},
                      es, g_align, state_bytes};
}

// Device, alignment and overlap checks of a chunkwise forward's tensors;
// with_tokens is false for T = 0 (only the states are touched then).
static int check_chunk_spans(const ChunkSpans& c, bool with_tokens, int dev) {
    if (with_tokens) {
        for (const Span* s : {&c.q, &c.k, &c.v, &c.o})
            if (int st = check_device_ptr(*s, 16, dev)) return st;
        if (int st = check_device_ptr(c.beta, c.beta_align, dev)) return st;
        if (c.g_align)
            if (int st = check_device_ptr(c.g, c.g_align, dev)) return st;
    }
    if (c.S0.p)
        if (int st = check_device_ptr(c.S0, 16, dev)) return st;
    if (c.S_T.p)
        if (int st = check_device_ptr(c.S_T, 16, dev)) return st;
    if (with_tokens) {
        for (const Span* s : {&c.q, &c.k, &c.v, &c.beta, &c.g, &c.S0, &c.S_T})
            if (overlaps(c.o, *s)) return fail(DN_ERR_INVALID_ARG, "o overlaps %s", s->name);
        for (const Span* s : {&c.q, &c.k, &c.v, &c.beta, &c.g})
            if (overlaps(c.S_T, *s)) return fail(DN_ERR_INVALID_ARG, "S_T overlaps %s", s->name);
    }
    if (c.S_T.p && c.S0.p && c.S_T.p != c.S0.p && overlaps(c.S_T, c.S0))
        return fail(DN_ERR_INVALID_ARG, "S_T partly overlaps S0");
    return DN_OK;
}

// A workspace of `need` bytes: device memory of this device, 16-byte
// aligned, overlapping none of the call's tensors.
static int check_workspace(const ChunkSpans& c, void* workspace, size_t need, int dev) {
    const Span sw{"workspace", workspace, need};
    if (int st = check_device_ptr(sw, 16, dev)) return st;
    for (const Span* s : {&c.q, &c.k, &c.v, &c.beta, &c.g, &c.o, &c.S0, &c.S_T})
        if (overlaps(sw, *s)) return fail(DN_ERR_INVALID_ARG, "workspace overlaps %s", s->name);
    return DN_OK;
}

// T = 0: no token, so S_T is S0 (or zeros without S0).
static int pass_state_through(const float* S0, float* S_T, size_t state_bytes, cudaStream_t st) {
    if (!S_T || S_T == S0) return ok();
    if (S0)
        return cuda_status(cudaMemcpyAsync(S_T, S0, state_bytes, cudaMemcpyDeviceToDevice, st),
                           "cudaMemcpyAsync(S_T <- S0)");
    return cuda_status(cudaMemsetAsync(S_T, 0, state_bytes, st), "cudaMemsetAsync(S_T)");
}

int dn_chunk_fwd_qk(const void* q, const void* k, const void* v, const void* beta,
                    const float* S0, void* o, float* S_T, int B, int H, int T, int dk, int dv,
                    int C, int dt, void* workspace, size_t workspace_bytes, void* stream,
                    int algo, const dn_qk_norm* norm) {
    if (int st = check_chunk_sizes(B, H, T, dk, dv, C, dt, "B")) return st;
    if (algo != DN_ALGO_AUTO && algo != DN_ALGO_SIMT && algo != DN_ALGO_TCGEN05)
        return fail(DN_ERR_INVALID_ARG, "unknown algo %d", algo);
    dn::QkNorm nm;
    if (int st = norm_options(norm, &nm)) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    const size_t need_ws = dn_chunk_fwd_workspace_bytes(B, H, T, dk, dv, C, dt);
    if (workspace && workspace_bytes < need_ws)
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed (or pass NULL)",
                    workspace_bytes, need_ws);
    if (algo == DN_ALGO_TCGEN05 && !dn::chunk_tc_fwd_supports(dk, dv, dt))
        return fail(DN_ERR_UNSUPPORTED, "tcgen05 path does not cover dk=%d dv=%d dtype=%d", dk,
                    dv, dt);
    // the fused tensor-core kernel (no workspace) covers 128-wide heads only
    const bool fused_ok = dn::chunk_tc_supports(dk, dv, dt);
    if (algo == DN_ALGO_TCGEN05 && !workspace && !fused_ok && B > 0 && H > 0 && T > 0)
        return fail(DN_ERR_UNSUPPORTED, "tcgen05 without a workspace covers dk = dv = 128 only");
    if (BH == 0) return ok();
    const ChunkSpans c = chunk_spans(q, k, v, beta, nullptr, 0, 0, S0, o, S_T,
                                     (size_t)BH * (size_t)T, BH, dk, dv, dt);
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (int st = check_chunk_spans(c, T > 0, dev)) return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return pass_state_through(S0, S_T, c.state_bytes, st);
    const bool use_tc = algo == DN_ALGO_TCGEN05 ||
                        (algo == DN_ALGO_AUTO && dn::chunk_tc_fwd_supports(dk, dv, dt) &&
                         (workspace || fused_ok));
    void* const ws = (use_tc && workspace && need_ws > 0) ? workspace : nullptr;
    if (ws)
        if (int st2 = check_workspace(c, ws, need_ws, dev)) return st2;
    cudaError_t e = use_tc
        ? dn::launch_chunk_tc(q, k, v, beta, S0, o, S_T, (int)BH, T, dk, dv, dt, ws, st, nullptr,
                              nm)
        : dn::launch_chunk_simt(q, k, v, beta, S0, o, S_T, (int)BH, T, dk, dv, dt, st, nullptr,
                                nullptr, nm);
    return cuda_status(e, use_tc ? "chunk forward (tcgen05) launch" : "chunk forward (SIMT) launch");
}

int dn_chunk_fwd_algo(const void* q, const void* k, const void* v, const void* beta,
                      const float* S0, void* o, float* S_T, int B, int H, int T, int dk,
                      int dv, int C, int dt, void* workspace, size_t workspace_bytes,
                      void* stream, int algo) {
    return dn_chunk_fwd_qk(q, k, v, beta, S0, o, S_T, B, H, T, dk, dv, C, dt, workspace,
                           workspace_bytes, stream, algo, nullptr);
}

int dn_chunk_fwd(const void* q, const void* k, const void* v, const void* beta, const float* S0,
                 void* o, float* S_T, int B, int H, int T, int dk, int dv, int C, int dt,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return dn_chunk_fwd_qk(q, k, v, beta, S0, o, S_T, B, H, T, dk, dv, C, dt, workspace,
                           workspace_bytes, stream, DN_ALGO_AUTO, nullptr);
}

static int split_segments(long long BH, int T, int segments) {
    return segments > 0 ? segments : dn::chunk_tc_split_segments((int)BH, T);
}

size_t dn_chunk_fwd_split_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt,
                                          int segments) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || segments < 0 ||
        segments > dn::kMaxVarlenSeqs || !dn::chunk_tc_supports(dk, dv, dt))
        return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_tc_split_workspace_bytes((int)BH, T, split_segments(BH, T, segments));
}

int dn_chunk_fwd_split(const void* q, const void* k, const void* v, const void* beta,
                       const float* S0, void* o, float* S_T, int B, int H, int T, int dk, int dv,
                       int C, int dt, int segments, void* workspace, size_t workspace_bytes,
                       void* stream) {
    if (int st = check_chunk_sizes(B, H, T, dk, dv, C, dt, "B")) return st;
    if (!dn::chunk_tc_supports(dk, dv, dt))
        return fail(DN_ERR_UNSUPPORTED, "the split runs on tensor cores: dk=%d dv=%d dtype=%d", dk,
                    dv, dt);
    if (segments < 0 || segments > dn::kMaxVarlenSeqs)
        return fail(DN_ERR_INVALID_ARG, "segments %d outside 0 .. %d", segments,
                    dn::kMaxVarlenSeqs);
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    if (BH == 0) return ok();
    const ChunkSpans c = chunk_spans(q, k, v, beta, nullptr, 0, 0, S0, o, S_T,
                                     (size_t)BH * (size_t)T, BH, dk, dv, dt);
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (int st = check_chunk_spans(c, T > 0, dev)) return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return pass_state_through(S0, S_T, c.state_bytes, st);
    const int nseg = split_segments(BH, T, segments);
    const size_t need = dn::chunk_tc_split_workspace_bytes((int)BH, T, nseg);
    if (!workspace || workspace_bytes < need)
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need);
    if (int st2 = check_workspace(c, workspace, need, dev)) return st2;
    return cuda_status(dn::launch_chunk_tc_split(q, k, v, beta, S0, o, S_T, (int)BH, T, nseg,
                                                 workspace, st),
                       "chunk forward (sequence split) launch");
}

int dn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* beta,
                         const float* S0, void* o, float* S_T, int B, int H, int T, int dk,
                         int dv, int C, int dt, void* stream) {
    if (B < 0 || H < 0 || T < 0)
        return fail(DN_ERR_INVALID_ARG, "negative size (B=%d H=%d T=%d)", B, H, T);
    if (dt != DN_F32 && dt != DN_BF16) return fail(DN_ERR_INVALID_ARG, "unknown dtype %d", dt);
    if (C != 64 || !dn::chunk_tc_supports(dk, dv, dt))
        return fail(DN_ERR_UNSUPPORTED,
                    "the no-alloc entry point covers bf16, dk = dv = 128, C = 64 (got dk=%d dv=%d "
                    "C=%d dtype=%d)", dk, dv, C, dt);
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    const long long tiles = BH * (((long long)T + 63) / 64);
    if (tiles > (long long)dn::noalloc_max_tiles())
        return fail(DN_ERR_INVALID_ARG,
                    "B*H*ceil(T/64) = %lld chunk tiles; the no-alloc entry point holds %zu",
                    tiles, dn::noalloc_max_tiles());
    if (BH == 0) return ok();
    const ChunkSpans c = chunk_spans(q, k, v, beta, nullptr, 0, 0, S0, o, S_T,
                                     (size_t)BH * (size_t)T, BH, dk, dv, dt);
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (int st = check_chunk_spans(c, T > 0, dev)) return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return pass_state_through(S0, S_T, c.state_bytes, st);
    return cuda_status(
        dn::launch_chunk_tc_noalloc(q, k, v, beta, S0, o, S_T, (int)BH, T, dk, dv, dt, st),
        "chunk forward (tcgen05, static scratch) launch");
}

// Checks cu_seqlens (host) and fills the kernels' sequence table.
static int varlen_table(const int* cu, int N, int T, dn::VarlenTable* tab) {
    if (N < 0 || N > dn::kMaxVarlenSeqs)
        return fail(DN_ERR_INVALID_ARG, "%d sequences; 0 to %d are supported", N,
                    dn::kMaxVarlenSeqs);
    if (!cu) return fail(DN_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (cu[0] != 0 || cu[N] != T)
        return fail(DN_ERR_INVALID_ARG, "cu_seqlens must run from 0 to T=%d (got %d .. %d)", T,
                    cu[0], cu[N]);
    tab->n = N;
    tab->start[0] = 0;
    tab->chunk[0] = 0;
    for (int i = 0; i < N; ++i) {
        if (cu[i + 1] < cu[i]) return fail(DN_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
        tab->start[i + 1] = cu[i + 1];
        tab->chunk[i + 1] = tab->chunk[i] + (cu[i + 1] - cu[i] + 63) / 64;
    }
    return DN_OK;
}

size_t dn_chunk_fwd_varlen_workspace_bytes(const int* cu_seqlens, int N, int H, int dk, int dv,
                                           int C, int dt) {
    if (!cu_seqlens || N <= 0 || N > dn::kMaxVarlenSeqs || H <= 0 || C != 64 ||
        !dn::chunk_tc_supports(dk, dv, dt))
        return 0;
    long long chunks = 0;
    for (int i = 0; i < N; ++i) {
        const long long len = (long long)cu_seqlens[i + 1] - cu_seqlens[i];
        if (len < 0) return 0;
        chunks += (len + 63) / 64;
    }
    return (size_t)H * (size_t)chunks * (16384 + dn::chunk_tc_side_bytes_per_chunk());
}

int dn_chunk_fwd_varlen_qk(const void* q, const void* k, const void* v, const void* beta,
                           const float* S0, void* o, float* S_T, const int* cu_seqlens, int N,
                           int H, int T, int dk, int dv, int C, int dt, void* workspace,
                           size_t workspace_bytes, void* stream, const dn_qk_norm* norm) {
    if (int st = check_chunk_sizes(N, H, T, dk, dv, C, dt, "N")) return st;
    dn::QkNorm nm;
    if (int st = norm_options(norm, &nm)) return st;
    static thread_local dn::VarlenTable tab;
    if (int st = varlen_table(cu_seqlens, N, T, &tab)) return st;
    const size_t need_ws = dn_chunk_fwd_varlen_workspace_bytes(cu_seqlens, N, H, dk, dv, C, dt);
    if (workspace && workspace_bytes < need_ws)
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed (or pass NULL)",
                    workspace_bytes, need_ws);
    if ((long long)N * H == 0) return ok();
    const ChunkSpans c = chunk_spans(q, k, v, beta, nullptr, 0, 0, S0, o, S_T,
                                     (size_t)H * (size_t)T, (long long)N * H, dk, dv, dt);
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (int st = check_chunk_spans(c, T > 0, dev)) return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return pass_state_through(S0, S_T, c.state_bytes, st);  // every sequence is empty
    const bool use_tc = workspace && need_ws > 0;
    if (use_tc)
        if (int st2 = check_workspace(c, workspace, need_ws, dev)) return st2;
    const cudaError_t e = use_tc
        ? dn::launch_chunk_tc_varlen(q, k, v, beta, S0, o, S_T, tab, H, T, workspace, st, nm)
        : dn::launch_chunk_simt_varlen(q, k, v, beta, S0, o, S_T, tab, H, T, dk, dv, dt, st, nm);
    return cuda_status(e, use_tc ? "varlen chunk forward (tcgen05) launch"
                                 : "varlen chunk forward (SIMT) launch");
}

int dn_chunk_fwd_varlen(const void* q, const void* k, const void* v, const void* beta,
                        const float* S0, void* o, float* S_T, const int* cu_seqlens, int N, int H,
                        int T, int dk, int dv, int C, int dt, void* workspace,
                        size_t workspace_bytes, void* stream) {
    return dn_chunk_fwd_varlen_qk(q, k, v, beta, S0, o, S_T, cu_seqlens, N, H, T, dk, dv, C, dt,
                                  workspace, workspace_bytes, stream, nullptr);
}

size_t dn_chunk_fwd_gated_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || !dn::chunk_tc_supports(dk, dv, dt)) return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_tc_gated_workspace_bytes((int)BH, T);
}

size_t dn_chunk_fwd_kda_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || !dn::chunk_tc_supports(dk, dv, dt)) return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_tc_kda_workspace_bytes((int)BH, T);
}

// The decayed chunkwise forms: Gated DeltaNet (one log keep rate per token,
// per_channel = 0) and KDA (one per token and key channel, per_channel = 1).
// A workspace of the form's size selects its two-pass tensor-core path where
// that size is non-zero.
static int chunk_fwd_decayed(const void* q, const void* k, const void* v, const void* beta,
                             const float* g, int per_channel, const float* S0, void* o,
                             float* S_T, int B, int H, int T, int dk, int dv, int C, int dt,
                             void* workspace, size_t workspace_bytes, void* stream,
                             const dn_qk_norm* norm) {
    if (int st = check_chunk_sizes(B, H, T, dk, dv, C, dt, "B")) return st;
    dn::QkNorm nm;
    if (int st = norm_options(norm, &nm)) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    const size_t need_ws = per_channel
        ? dn_chunk_fwd_kda_workspace_bytes(B, H, T, dk, dv, C, dt)
        : dn_chunk_fwd_gated_workspace_bytes(B, H, T, dk, dv, C, dt);
    if (workspace && workspace_bytes < need_ws)
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed (or pass NULL)",
                    workspace_bytes, need_ws);
    if (BH == 0) return ok();
    // the KDA kernel reads its [T][dk] g tile in 16-byte groups
    const ChunkSpans c = chunk_spans(q, k, v, beta, g, per_channel ? (size_t)dk : 1,
                                     per_channel ? 16 : sizeof(float), S0, o, S_T,
                                     (size_t)BH * (size_t)T, BH, dk, dv, dt);
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (int st = check_chunk_spans(c, T > 0, dev)) return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return pass_state_through(S0, S_T, c.state_bytes, st);
    const bool use_tc = workspace && need_ws > 0;
    if (use_tc)
        if (int st2 = check_workspace(c, workspace, need_ws, dev)) return st2;
    if (per_channel && use_tc)
        return cuda_status(dn::launch_chunk_tc_kda(q, k, v, beta, g, S0, o, S_T, (int)BH, T, dk,
                                                   dv, dt, workspace, st, nm),
                           "KDA chunk forward (tcgen05) launch");
    if (per_channel)
        return cuda_status(dn::launch_chunk_simt_kda(q, k, v, beta, g, S0, o, S_T, (int)BH, T,
                                                     dk, dv, dt, st, nm),
                           "KDA chunk forward launch");
    if (use_tc)
        return cuda_status(dn::launch_chunk_tc_gated(q, k, v, beta, g, S0, o, S_T, (int)BH, T, dk,
                                                     dv, dt, workspace, st, nm),
                           "gated chunk forward (tcgen05) launch");
    return cuda_status(dn::launch_chunk_simt(q, k, v, beta, S0, o, S_T, (int)BH, T, dk, dv, dt, st,
                                             nullptr, g, nm),
                       "gated chunk forward launch");
}

int dn_chunk_fwd_gated_qk(const void* q, const void* k, const void* v, const void* beta,
                          const float* g, const float* S0, void* o, float* S_T, int B, int H,
                          int T, int dk, int dv, int C, int dt, void* workspace,
                          size_t workspace_bytes, void* stream, const dn_qk_norm* norm) {
    return chunk_fwd_decayed(q, k, v, beta, g, 0, S0, o, S_T, B, H, T, dk, dv, C, dt, workspace,
                             workspace_bytes, stream, norm);
}

int dn_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* beta,
                       const float* g, const float* S0, void* o, float* S_T, int B, int H,
                       int T, int dk, int dv, int C, int dt, void* workspace,
                       size_t workspace_bytes, void* stream) {
    return chunk_fwd_decayed(q, k, v, beta, g, 0, S0, o, S_T, B, H, T, dk, dv, C, dt, workspace,
                             workspace_bytes, stream, nullptr);
}

int dn_chunk_fwd_kda_qk(const void* q, const void* k, const void* v, const void* beta,
                        const float* g, const float* S0, void* o, float* S_T, int B, int H, int T,
                        int dk, int dv, int C, int dt, void* workspace, size_t workspace_bytes,
                        void* stream, const dn_qk_norm* norm) {
    return chunk_fwd_decayed(q, k, v, beta, g, 1, S0, o, S_T, B, H, T, dk, dv, C, dt, workspace,
                             workspace_bytes, stream, norm);
}

int dn_chunk_fwd_kda(const void* q, const void* k, const void* v, const void* beta,
                     const float* g, const float* S0, void* o, float* S_T, int B, int H, int T,
                     int dk, int dv, int C, int dt, void* stream) {
    return chunk_fwd_decayed(q, k, v, beta, g, 1, S0, o, S_T, B, H, T, dk, dv, C, dt, nullptr, 0,
                             stream, nullptr);
}

// One decoding step of any form: g_mode 0 (none), 1 (per head), 2 (per key
// channel).
static int recurrent_step_any(const void* q, const void* k, const void* v, const void* beta,
                              const float* g, int g_mode, float* S, void* o, int B, int H, int dk,
                              int dv, int dt, void* stream, const dn_qk_norm* norm) {
    if (B < 0 || H < 0) return fail(DN_ERR_INVALID_ARG, "negative size (B=%d H=%d)", B, H);
    if (dt != DN_F32 && dt != DN_BF16) return fail(DN_ERR_INVALID_ARG, "unknown dtype %d", dt);
    if (dk <= 0 || dv <= 0) return fail(DN_ERR_INVALID_ARG, "dk and dv must be positive");
    if (!supported_dim(dk) || !supported_dim(dv))
        return fail(DN_ERR_UNSUPPORTED, "dk=%d dv=%d: this library supports 64 and 128", dk, dv);
    dn::QkNorm nm;
    if (int st = norm_options(norm, &nm)) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    if (BH == 0) return ok();
    const size_t es = elem_size(dt);
    const Span sq{"q", q, (size_t)BH * dk * es}, sk{"k", k, (size_t)BH * dk * es},
        sv{"v", v, (size_t)BH * dv * es}, sb{"beta", beta, (size_t)BH * es},
        sg{"g", g, (size_t)BH * (g_mode == 2 ? dk : 1) * sizeof(float)},
        so{"o", o, (size_t)BH * dv * es},
        sS{"S", S, (size_t)BH * dk * dv * sizeof(float)};
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    for (const Span* s : {&sq, &sk, &sv, &so, &sS})
        if (int st = check_device_ptr(*s, 16, dev)) return st;
    if (int st = check_device_ptr(sb, es, dev)) return st;
    if (g_mode)
        if (int st = check_device_ptr(sg, sizeof(float), dev)) return st;
    for (const Span* s : {&sq, &sk, &sv, &sb, &sg, &sS})
        if (overlaps(so, *s)) return fail(DN_ERR_INVALID_ARG, "o overlaps %s", s->name);
    for (const Span* s : {&sq, &sk, &sv, &sb, &sg})
        if (overlaps(sS, *s)) return fail(DN_ERR_INVALID_ARG, "S overlaps %s", s->name);
    static const char* const what[3] = {"recurrent step launch", "gated recurrent step launch",
                                        "KDA recurrent step launch"};
    return cuda_status(dn::launch_recurrent_step(q, k, v, beta, S, o, (int)BH, dk, dv, dt,
                                                 static_cast<cudaStream_t>(stream),
                                                 g_mode ? g : nullptr, g_mode == 2 ? 1 : 0, nm),
                       what[g_mode]);
}

int dn_recurrent_step_qk(const void* q, const void* k, const void* v, const void* beta, float* S,
                         void* o, int B, int H, int dk, int dv, int dt, void* stream,
                         const dn_qk_norm* norm) {
    return recurrent_step_any(q, k, v, beta, nullptr, 0, S, o, B, H, dk, dv, dt, stream, norm);
}

int dn_recurrent_step(const void* q, const void* k, const void* v, const void* beta, float* S,
                      void* o, int B, int H, int dk, int dv, int dt, void* stream) {
    return recurrent_step_any(q, k, v, beta, nullptr, 0, S, o, B, H, dk, dv, dt, stream, nullptr);
}

int dn_recurrent_step_gated_qk(const void* q, const void* k, const void* v, const void* beta,
                               const float* g, float* S, void* o, int B, int H, int dk, int dv,
                               int dt, void* stream, const dn_qk_norm* norm) {
    return recurrent_step_any(q, k, v, beta, g, 1, S, o, B, H, dk, dv, dt, stream, norm);
}

int dn_recurrent_step_gated(const void* q, const void* k, const void* v, const void* beta,
                            const float* g, float* S, void* o, int B, int H, int dk, int dv,
                            int dt, void* stream) {
    return recurrent_step_any(q, k, v, beta, g, 1, S, o, B, H, dk, dv, dt, stream, nullptr);
}

int dn_recurrent_step_kda_qk(const void* q, const void* k, const void* v, const void* beta,
                             const float* g, float* S, void* o, int B, int H, int dk, int dv,
                             int dt, void* stream, const dn_qk_norm* norm) {
    return recurrent_step_any(q, k, v, beta, g, 2, S, o, B, H, dk, dv, dt, stream, norm);
}

int dn_recurrent_step_kda(const void* q, const void* k, const void* v, const void* beta,
                          const float* g, float* S, void* o, int B, int H, int dk, int dv,
                          int dt, void* stream) {
    return recurrent_step_any(q, k, v, beta, g, 2, S, o, B, H, dk, dv, dt, stream, nullptr);
}

// Row count, dtype, d and the options of the preparation and its gradient.
static int check_prepare_args(long long rows, int d, float scale, float eps, int dt) {
    if (rows < 0) return fail(DN_ERR_INVALID_ARG, "negative row count %lld", rows);
    if (rows > (1LL << 40)) return fail(DN_ERR_INVALID_ARG, "row count %lld too large", rows);
    if (dt != DN_F32 && dt != DN_BF16) return fail(DN_ERR_INVALID_ARG, "unknown dtype %d", dt);
    if (d <= 0) return fail(DN_ERR_INVALID_ARG, "d must be positive");
    if (!supported_dim(d))
        return fail(DN_ERR_UNSUPPORTED, "d=%d: this library supports 64 and 128", d);
    if (!isfinite(scale)) return fail(DN_ERR_INVALID_ARG, "scale must be finite");
    if (!isfinite(eps) || eps < 0.0f)
        return fail(DN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    return DN_OK;
}

int dn_qk_prepare(const void* q, const void* k, void* q_out, void* k_out, long long rows,
                  int d, int normalize, float scale, float eps, int dt, void* stream) {
    if (int st = check_prepare_args(rows, d, scale, eps, dt)) return st;
    if (rows == 0) return ok();
    const size_t bytes = (size_t)rows * d * elem_size(dt);
    const Span sq{"q", q, bytes}, sqo{"q_out", q_out, bytes}, sk{"k", k, bytes},
        sko{"k_out", k_out, bytes};
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    for (const Span* s : {&sq, &sqo})
        if (int st = check_device_ptr(*s, 16, dev)) return st;
    if (q_out != q && overlaps(sqo, sq)) return fail(DN_ERR_INVALID_ARG, "q_out overlaps q");
    if (normalize) {
        for (const Span* s : {&sk, &sko})
            if (int st = check_device_ptr(*s, 16, dev)) return st;
        if (k_out != k && overlaps(sko, sk)) return fail(DN_ERR_INVALID_ARG, "k_out overlaps k");
        if (overlaps(sqo, sk)) return fail(DN_ERR_INVALID_ARG, "q_out overlaps k");
        if (overlaps(sko, sq)) return fail(DN_ERR_INVALID_ARG, "k_out overlaps q");
        if (overlaps(sqo, sko)) return fail(DN_ERR_INVALID_ARG, "q_out overlaps k_out");
    }
    return cuda_status(dn::launch_qk_prepare(q, k, q_out, k_out, rows, d, normalize ? 1 : 0,
                                             scale, eps, dt, static_cast<cudaStream_t>(stream)),
                       "q/k preparation launch");
}

int dn_qk_prepare_bwd(const void* q, const void* k, const void* d_q_out, const void* d_k_out,
                      void* d_q, void* d_k, long long rows, int d, int normalize, float scale,
                      float eps, int dt, void* stream) {
    if (int st = check_prepare_args(rows, d, scale, eps, dt)) return st;
    if (rows == 0) return ok();
    const size_t bytes = (size_t)rows * d * elem_size(dt);
    const Span sq{"q", q, bytes}, sk{"k", k, bytes}, sgq{"d_q_out", d_q_out, bytes},
        sgk{"d_k_out", d_k_out, bytes}, sdq{"d_q", d_q, bytes}, sdk{"d_k", d_k, bytes};
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    for (const Span* s : {&sgq, &sdq})
        if (int st = check_device_ptr(*s, 16, dev)) return st;
    if (normalize)
        for (const Span* s : {&sq, &sk, &sgk, &sdk})
            if (int st = check_device_ptr(*s, 16, dev)) return st;
    // Each output may be its own incoming gradient (in place); otherwise
    // outputs overlap no input and not each other.
    const Span* ins[] = {&sq, &sk, &sgq, &sgk};
    const Span* outs[] = {&sdq, &sdk};
    for (const Span* o : outs) {
        if (o == &sdk && !normalize) continue;
        for (const Span* i : ins) {
            if (!normalize && (i == &sq || i == &sk || i == &sgk)) continue;
            const bool self = (o == &sdq && i == &sgq) || (o == &sdk && i == &sgk);
            if (self && o->p == i->p) continue;
            if (overlaps(*o, *i)) return fail(DN_ERR_INVALID_ARG, "%s overlaps %s", o->name, i->name);
        }
    }
    if (normalize && overlaps(sdq, sdk)) return fail(DN_ERR_INVALID_ARG, "d_q overlaps d_k");
    return cuda_status(dn::launch_qk_prepare_bwd(q, k, d_q_out, d_k_out, d_q, d_k, rows, d,
                                                 normalize ? 1 : 0, scale, eps, dt,
                                                 static_cast<cudaStream_t>(stream)),
                       "q/k preparation gradient launch");
}

size_t dn_chunk_bwd_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || (dt != DN_F32 && dt != DN_BF16) ||
        !supported_dim(dk) || !supported_dim(dv))
        return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_bwd_workspace_bytes((int)BH, T, dk, dv, dt);
}

// The backward's pointer checks: ntok tokens of q, k, v, beta, d_o and their
// gradients, nstate states of S0, d_S_T, d_S0, and the workspace; outputs
// overlap no input and no other output.  T == 0 checks the states alone.
static int check_bwd_spans(const void* q, const void* k, const void* v, const void* beta,
                           const float* S0, const void* d_o, const float* d_S_T, void* d_q,
                           void* d_k, void* d_v, void* d_beta, float* d_S0, size_t ntok,
                           long long nstate, int T, int dk, int dv, int dt, void* workspace,
                           size_t need_ws) {
    const size_t es = elem_size(dt);
    const size_t state_bytes = (size_t)nstate * dk * dv * sizeof(float);
    const Span sq{"q", q, ntok * dk * es}, sk{"k", k, ntok * dk * es}, sv{"v", v, ntok * dv * es},
        sb{"beta", beta, ntok * es}, s0{"S0", S0, state_bytes}, sdo{"d_o", d_o, ntok * dv * es},
        sdT{"d_S_T", d_S_T, state_bytes}, sdq{"d_q", d_q, ntok * dk * es},
        sdk{"d_k", d_k, ntok * dk * es}, sdv{"d_v", d_v, ntok * dv * es},
        sdb{"d_beta", d_beta, ntok * es}, sd0{"d_S0", d_S0, state_bytes},
        sw{"workspace", workspace, need_ws};
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    if (T > 0) {
        for (const Span* s : {&sq, &sk, &sv, &sdo, &sdq, &sdk, &sdv, &sw})
            if (int st = check_device_ptr(*s, 16, dev)) return st;
        for (const Span* s : {&sb, &sdb})
            if (int st = check_device_ptr(*s, es, dev)) return st;
    }
    for (const Span* s : {&s0, &sdT, &sd0})
        if (s->p)
            if (int st = check_device_ptr(*s, 16, dev)) return st;
    // Outputs (and the workspace) overlap no input and no other output.
    const Span* ins[] = {&sq, &sk, &sv, &sb, &s0, &sdo, &sdT};
    const Span* outs[] = {&sdq, &sdk, &sdv, &sdb, &sd0, &sw};
    for (const Span* o : outs) {
        if (T == 0 && o != &sd0) continue;
        for (const Span* i : ins)
            if ((T > 0 || i == &sdT) && overlaps(*o, *i))
                return fail(DN_ERR_INVALID_ARG, "%s overlaps %s", o->name, i->name);
        for (const Span* o2 : outs)
            if (o2 != o && (T > 0 || o2 == &sd0) && overlaps(*o, *o2))
                return fail(DN_ERR_INVALID_ARG, "%s overlaps %s", o->name, o2->name);
    }
    return DN_OK;
}

// Shape and dtype checks shared by the backward entry points (n: B or N).
static int check_bwd_sizes(int n, int H, int T, int dk, int dv, int C, int dt, const char* nn) {
    if (n < 0 || H < 0 || T < 0)
        return fail(DN_ERR_INVALID_ARG, "negative size (%s=%d H=%d T=%d)", nn, n, H, T);
    if (dt != DN_F32 && dt != DN_BF16) return fail(DN_ERR_INVALID_ARG, "unknown dtype %d", dt);
    if (dk <= 0 || dv <= 0 || C <= 0)
        return fail(DN_ERR_INVALID_ARG, "dk, dv and C must be positive");
    if (!supported_dim(dk) || !supported_dim(dv))
        return fail(DN_ERR_UNSUPPORTED, "dk=%d dv=%d: this library supports 64 and 128", dk, dv);
    if (C != 64) return fail(DN_ERR_UNSUPPORTED, "chunk length C=%d: this library supports 64", C);
    return DN_OK;
}

int dn_chunk_bwd(const void* q, const void* k, const void* v, const void* beta, const float* S0,
                 const void* d_o, const float* d_S_T, void* d_q, void* d_k, void* d_v,
                 void* d_beta, float* d_S0, int B, int H, int T, int dk, int dv, int C, int dt,
                 void* workspace, size_t workspace_bytes, void* stream) {
    if (int st = check_bwd_sizes(B, H, T, dk, dv, C, dt, "B")) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    const size_t need_ws = dn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, C, dt);
    if (workspace_bytes < need_ws || (need_ws > 0 && !workspace))
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need_ws);
    if (BH == 0) return ok();
    if (int st = check_bwd_spans(q, k, v, beta, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_S0,
                                 (size_t)BH * (size_t)T, BH, T, dk, dv, dt, workspace, need_ws))
        return st;
    const size_t state_bytes = (size_t)BH * dk * dv * sizeof(float);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // the state passes through unchanged
        if (!d_S0) return ok();
        if (d_S_T)
            return cuda_status(
                cudaMemcpyAsync(d_S0, d_S_T, state_bytes, cudaMemcpyDeviceToDevice, st),
                "cudaMemcpyAsync(d_S0 <- d_S_T)");
        return cuda_status(cudaMemsetAsync(d_S0, 0, state_bytes, st), "cudaMemsetAsync(d_S0)");
    }
    const char* stage = "launch";
    const cudaError_t e = dn::launch_chunk_bwd(q, k, v, beta, S0, d_o, d_S_T, d_q, d_k, d_v,
                                               d_beta, d_S0, (int)BH, T, dk, dv, dt, workspace,
                                               st, &stage);
    if (e == cudaSuccess) return ok();
    return fail(DN_ERR_CUDA, "chunk backward (%s): %s", stage, cudaGetErrorString(e));
}

size_t dn_chunk_bwd_gated_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || !supported_dim(dk) || !supported_dim(dv) ||
        (dt != DN_F32 && dt != DN_BF16))
        return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_bwd_gated_workspace_bytes((int)BH, T, dk, dv, dt);
}

// The gated and KDA backwards: g and d_g are fp32 with one rate per token
// (gated) or per token and key channel (KDA).
static int chunk_bwd_decayed(const void* q, const void* k, const void* v, const void* beta,
                             const float* g, const float* S0, const void* d_o,
                             const float* d_S_T, void* d_q, void* d_k, void* d_v, void* d_beta,
                             float* d_g, float* d_S0, int B, int H, int T, int dk, int dv, int C,
                             int dt, void* workspace, size_t workspace_bytes, void* stream,
                             bool per_channel) {
    if (int st = check_bwd_sizes(B, H, T, dk, dv, C, dt, "B")) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return fail(DN_ERR_INVALID_ARG, "B*H too large");
    const size_t need_ws = per_channel
                               ? dn_chunk_bwd_kda_workspace_bytes(B, H, T, dk, dv, C, dt)
                               : dn_chunk_bwd_gated_workspace_bytes(B, H, T, dk, dv, C, dt);
    if (workspace_bytes < need_ws || (need_ws > 0 && !workspace))
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need_ws);
    if (BH == 0) return ok();
    const size_t ntok = (size_t)BH * (size_t)T;
    if (int st = check_bwd_spans(q, k, v, beta, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_S0,
                                 ntok, BH, T, dk, dv, dt, workspace, need_ws))
        return st;
    if (T > 0) {  // the log keep rates and their gradient
        int dev = 0;
        if (int st = current_device(&dev)) return st;
        const size_t gb = ntok * (per_channel ? (size_t)dk : 1) * sizeof(float);
        const int galign = per_channel ? 16 : 4;  // KDA's rates load as 16-byte rows
        const Span sg{"g", g, gb}, sdg{"d_g", d_g, gb};
        if (int st = check_device_ptr(sg, galign, dev)) return st;
        if (int st = check_device_ptr(sdg, 4, dev)) return st;
        const size_t es = elem_size(dt), sb = (size_t)BH * dk * dv * sizeof(float);
        const Span others[] = {{"q", q, ntok * dk * es},     {"k", k, ntok * dk * es},
                               {"v", v, ntok * dv * es},     {"beta", beta, ntok * es},
                               {"S0", S0, sb},               {"d_o", d_o, ntok * dv * es},
                               {"d_S_T", d_S_T, sb},         {"d_q", d_q, ntok * dk * es},
                               {"d_k", d_k, ntok * dk * es}, {"d_v", d_v, ntok * dv * es},
                               {"d_beta", d_beta, ntok * es}, {"d_S0", d_S0, sb},
                               {"workspace", workspace, need_ws}, sg};
        for (const Span& s : others)
            if (overlaps(sdg, s)) return fail(DN_ERR_INVALID_ARG, "d_g overlaps %s", s.name);
        for (int i = 7; i < 13; ++i)  // the outputs and the workspace against g
            if (overlaps(others[i], sg))
                return fail(DN_ERR_INVALID_ARG, "%s overlaps g", others[i].name);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // the state gradient passes through
        const size_t sb = (size_t)BH * dk * dv * sizeof(float);
        if (!d_S0) return ok();
        if (d_S_T)
            return cuda_status(cudaMemcpyAsync(d_S0, d_S_T, sb, cudaMemcpyDeviceToDevice, st),
                               "cudaMemcpyAsync(d_S0 <- d_S_T)");
        return cuda_status(cudaMemsetAsync(d_S0, 0, sb, st), "cudaMemsetAsync(d_S0)");
    }
    const char* stage = "launch";
    const cudaError_t e =
        per_channel
            ? dn::launch_chunk_bwd_kda(q, k, v, beta, g, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta,
                                       d_g, d_S0, (int)BH, T, dk, dv, dt, workspace, st, &stage)
            : dn::launch_chunk_bwd_gated(q, k, v, beta, g, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta,
                                         d_g, d_S0, (int)BH, T, dk, dv, dt, workspace, st,
                                         &stage);
    if (e == cudaSuccess) return ok();
    return fail(DN_ERR_CUDA, "%s chunk backward (%s): %s", per_channel ? "KDA" : "gated", stage,
                cudaGetErrorString(e));
}

int dn_chunk_bwd_gated(const void* q, const void* k, const void* v, const void* beta,
                       const float* g, const float* S0, const void* d_o, const float* d_S_T,
                       void* d_q, void* d_k, void* d_v, void* d_beta, float* d_g, float* d_S0,
                       int B, int H, int T, int dk, int dv, int C, int dt, void* workspace,
                       size_t workspace_bytes, void* stream) {
    return chunk_bwd_decayed(q, k, v, beta, g, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_g, d_S0,
                             B, H, T, dk, dv, C, dt, workspace, workspace_bytes, stream, false);
}

size_t dn_chunk_bwd_kda_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int dt) {
    if (B <= 0 || H <= 0 || T <= 0 || C != 64 || !supported_dim(dk) || !supported_dim(dv) ||
        (dt != DN_F32 && dt != DN_BF16))
        return 0;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return 0;
    return dn::chunk_bwd_kda_workspace_bytes((int)BH, T, dk, dv, dt);
}

int dn_chunk_bwd_kda(const void* q, const void* k, const void* v, const void* beta,
                     const float* g, const float* S0, const void* d_o, const float* d_S_T,
                     void* d_q, void* d_k, void* d_v, void* d_beta, float* d_g, float* d_S0,
                     int B, int H, int T, int dk, int dv, int C, int dt, void* workspace,
                     size_t workspace_bytes, void* stream) {
    return chunk_bwd_decayed(q, k, v, beta, g, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_g, d_S0,
                             B, H, T, dk, dv, C, dt, workspace, workspace_bytes, stream, true);
}

size_t dn_chunk_bwd_varlen_workspace_bytes(const int* cu_seqlens, int N, int H, int dk, int dv,
                                           int C, int dt) {
    if (!cu_seqlens || N <= 0 || N > dn::kMaxVarlenSeqs || H <= 0 || C != 64 ||
        !supported_dim(dk) || !supported_dim(dv) || (dt != DN_F32 && dt != DN_BF16))
        return 0;
    for (int i = 0; i < N; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return 0;
    return dn::chunk_bwd_varlen_workspace_bytes(cu_seqlens, N, H, dk, dv, dt);
}

int dn_chunk_bwd_varlen(const void* q, const void* k, const void* v, const void* beta,
                        const float* S0, const void* d_o, const float* d_S_T, void* d_q,
                        void* d_k, void* d_v, void* d_beta, float* d_S0, const int* cu_seqlens,
                        int N, int H, int T, int dk, int dv, int C, int dt, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (int st = check_bwd_sizes(N, H, T, dk, dv, C, dt, "N")) return st;
    static thread_local dn::VarlenTable tab;
    if (int st = varlen_table(cu_seqlens, N, T, &tab)) return st;
    if ((long long)N * H == 0) return ok();
    const size_t need_ws =
        dn_chunk_bwd_varlen_workspace_bytes(cu_seqlens, N, H, dk, dv, C, dt);
    if (workspace_bytes < need_ws || (need_ws > 0 && !workspace))
        return fail(DN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need_ws);
    if (int st = check_bwd_spans(q, k, v, beta, S0, d_o, d_S_T, d_q, d_k, d_v, d_beta, d_S0,
                                 (size_t)H * (size_t)T, (long long)N * H, T, dk, dv, dt,
                                 workspace, need_ws))
        return st;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t state_bytes = (size_t)N * H * dk * dv * sizeof(float);
    if (T == 0) {  // every sequence is empty: the state gradient passes through
        if (!d_S0) return ok();
        if (d_S_T)
            return cuda_status(
                cudaMemcpyAsync(d_S0, d_S_T, state_bytes, cudaMemcpyDeviceToDevice, st),
                "cudaMemcpyAsync(d_S0 <- d_S_T)");
        return cuda_status(cudaMemsetAsync(d_S0, 0, state_bytes, st), "cudaMemsetAsync(d_S0)");
    }
    const char* stage = "launch";
    const cudaError_t e = dn::launch_chunk_bwd_varlen(q, k, v, beta, S0, d_o, d_S_T, d_q, d_k, d_v,
                                                      d_beta, d_S0, cu_seqlens, N, H, T, dk, dv,
                                                      dt, workspace, st, &stage);
    if (e == cudaSuccess) return ok();
    return fail(DN_ERR_CUDA, "varlen chunk backward (%s): %s", stage, cudaGetErrorString(e));
}

}  // extern "C"
