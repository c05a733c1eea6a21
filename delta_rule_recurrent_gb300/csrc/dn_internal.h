// dn_internal.h -- launchers behind the C ABI (host side, no validation).
//
// Each launcher assumes the ABI layer has already checked pointers, sizes and
// the (dtype, dk, dv) combination, and returns the cudaError_t of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace dn {

// Optional preparation of q and k inside the kernels that read them (the
// ABI's dn_qk_norm): with l2norm every row of q and k (the head dimension)
// becomes x / sqrt(sum x^2 + eps); q is then multiplied by qscale.  Each
// kernel applies it to the rows it loads, before any product uses them.
struct QkNorm {
    int l2norm;
    float qscale;
    float eps;
};
constexpr QkNorm kNoNorm{0, 1.0f, 0.0f};
__host__ __device__ inline bool norm_active(const QkNorm& n) {
    return n.l2norm != 0 || n.qscale != 1.0f;
}

// Packed variable-length sequences: sequence n is tokens start[n] ..
// start[n+1] - 1 of an [H][T][d] tensor, and chunk[n] counts the 64-token
// chunks of the sequences before it.  Kernels take the table by value (a
// kernel parameter), so varlen calls need no device memory for it.
constexpr int kMaxVarlenSeqs = 1024;
template <int NMAX>
struct SeqTable {
    int n;
    int start[NMAX + 1];
    int chunk[NMAX + 1];
};
using VarlenTable = SeqTable<kMaxVarlenSeqs>;

// One decoding step over B*H heads (see dn_recurrent_step); with g (fp32
// log keep rates, [BH], or [BH][dk] when g_per_channel) the gated or KDA step.
cudaError_t launch_recurrent_step(const void* q, const void* k, const void* v,
                                  const void* beta, float* S, void* o, int BH,
                                  int dk, int dv, int dt, cudaStream_t stream,
                                  const float* g = nullptr, int g_per_channel = 0,
                                  const QkNorm& norm = kNoNorm);

// Optional input preparation (see dn_qk_prepare): rows of d (64 or 128)
// elements; q rows scaled by `scale` (after the L2 normalisation when
// normalize != 0), k rows normalised (only when normalize != 0).
cudaError_t launch_qk_prepare(const void* q, const void* k, void* q_out, void* k_out,
                              long long rows, int d, int normalize, float scale, float eps,
                              int dt, cudaStream_t stream);
// Its gradient (see dn_qk_prepare_bwd): dq, dk from the raw rows q, k and
// the gradients dq_out, dk_out of the prepared ones (dk untouched when
// normalize == 0).
cudaError_t launch_qk_prepare_bwd(const void* q, const void* k, const void* dq_out,
                                  const void* dk_out, void* dq, void* dk, long long rows, int d,
                                  int normalize, float scale, float eps, int dt,
                                  cudaStream_t stream);

// Chunkwise forward with fp32 CUDA-core arithmetic (any T >= 1).  o may be
// nullptr (no outputs); S_chunks, if given, receives the state at the start
// of every chunk ([BH][ceil(T/64)][dk][dv] fp32), for the backward pass; g,
// if given, is the fp32 [BH][T] log keep rate of Gated DeltaNet.
cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v,
                              const void* beta, const float* S0, void* o,
                              float* S_T, int BH, int T, int dk, int dv, int dt,
                              cudaStream_t stream, float* S_chunks = nullptr,
                              const float* g = nullptr, const QkNorm& norm = kNoNorm);

// Chunkwise backward (fp32 CUDA-core arithmetic): the gradients of
// L = <d_o, o> + <d_S_T, S_T> for dn_chunk_fwd's outputs.  The workspace
// holds chunk_bwd_workspace_bytes(BH, T, dk, dv, dt) bytes: the state at the
// start of every chunk, the gradient of the state at its end, and the
// tensor-core forward's scratch when that path recomputes the states.  d_S_T, S0 and
// d_S0 may be nullptr.
size_t chunk_bwd_workspace_bytes(int BH, int T, int dk, int dv, int dt);
cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const void* beta,
                             const float* S0, const void* d_o, const float* d_S_T, void* d_q,
                             void* d_k, void* d_v, void* d_beta, float* d_S0, int BH, int T,
                             int dk, int dv, int dt, void* workspace, cudaStream_t stream,
                             const char** stage);

// Gated DeltaNet's backward (g the fp32 [BH][T] log keep rates; d_g its
// gradient, fp32 [BH][T]): the forward records every chunk's start state
// (the two-pass tensor-core form for bf16, d = 128, whose tiles then follow
// in the workspace; else the CUDA-core form), then the chain and the
// per-chunk gradients run with the decay on the CUDA cores.  The workspace
// holds the fp32 S and G of every chunk.
size_t chunk_bwd_gated_workspace_bytes(int BH, int T, int dk, int dv, int dt);
cudaError_t launch_chunk_bwd_gated(const void* q, const void* k, const void* v, const void* beta,
                                   const float* g, const float* S0, const void* d_o,
                                   const float* d_S_T, void* d_q, void* d_k, void* d_v,
                                   void* d_beta, float* d_g, float* d_S0, int BH, int T, int dk,
                                   int dv, int dt, void* workspace, cudaStream_t stream,
                                   const char** stage);

// KDA's backward chain on tcgen05 (bf16, dk = dv = 128): the state gradient
// from the last chunk to the first with the decayed operands, tiles and keep
// factors the tensor-core KDA forward left in its workspace (kda_workspace,
// as launch_chunk_tc_kda lays it out); writes d_v, d_S0 and G at every chunk
// end in fp32 (G_chunks, [BH][chunk][dk][dv]).
cudaError_t launch_chunk_bwd_chain_tc_kda(const void* d_o, const float* d_S_T, void* d_v,
                                          float* d_S0, float* G_chunks, const void* kda_workspace,
                                          int BH, int T, cudaStream_t stream);
// KDA's backward (g, d_g: fp32 [BH][T][dk]): the states recomputed by the
// KDA forward (on tcgen05 for bf16 with dk = dv = 128, else on the CUDA
// cores), then its chain and per-chunk gradients with the per-channel decay.
// The workspace holds the fp32 S and G of every chunk, plus the tensor-core
// forward's scratch where it runs.
size_t chunk_bwd_kda_workspace_bytes(int BH, int T, int dk, int dv, int dt);
cudaError_t launch_chunk_bwd_kda(const void* q, const void* k, const void* v, const void* beta,
                                 const float* g, const float* S0, const void* d_o,
                                 const float* d_S_T, void* d_q, void* d_k, void* d_v,
                                 void* d_beta, float* d_g, float* d_S0, int BH, int T, int dk,
                                 int dv, int dt, void* workspace, cudaStream_t stream,
                                 const char** stage);

// The backward of the packed-sequence forward (cu: N + 1 host offsets into
// the [H][T][d] tensors; states [N][H][dk][dv]): one batched backward per
// sequence on gathered copies, in the scratch this many bytes hold.
size_t chunk_bwd_varlen_workspace_bytes(const int* cu, int N, int H, int dk, int dv, int dt);
cudaError_t launch_chunk_bwd_varlen(const void* q, const void* k, const void* v, const void* beta,
                                    const float* S0, const void* d_o, const float* d_S_T,
                                    void* d_q, void* d_k, void* d_v, void* d_beta, float* d_S0,
                                    const int* cu, int N, int H, int T, int dk, int dv, int dt,
                                    void* workspace, cudaStream_t stream, const char** stage);

// Chunkwise forward on tcgen05 tensor cores.  Returns cudaErrorNotSupported
// (without launching) for shapes or dtypes it does not cover.  With a
// workspace of chunk_tc_workspace_bytes(BH, T) bytes (16-byte aligned) it runs
// in two passes: every chunk's [PT; Tm] in parallel, then the sequences;
// with workspace == nullptr one fused kernel does both.  On the two-pass path
// o may be nullptr (no outputs) and S_rec, if given, receives the fp32
// state at the start of every chunk as two bf16 tiles, hi = bf16(S) and
// lo = bf16(S - hi) ([BH][ceil(T/64)][2][dk][dv]), and X_rec, if given, every
// chunk's (I + A)^{-1} ([BH][ceil(T/64)][64][64] bf16), for the backward.
bool chunk_tc_supports(int dk, int dv, int dt);
// The plain forward's tensor-core path also covers 64-wide heads (bf16,
// dk = dv = 64) in its two-pass form: the tiles keep 128 columns, the second
// half zero.
bool chunk_tc_fwd_supports(int dk, int dv, int dt);
size_t chunk_tc_workspace_bytes(int BH, int T);
// With prepared inputs (a QkNorm) the two-pass forms also keep the row
// factors of every chunk after the tiles: this many bytes per chunk.
size_t chunk_tc_side_bytes_per_chunk();
cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v,
                            const void* beta, const float* S0, void* o,
                            float* S_T, int BH, int T, int dk, int dv, int dt,
                            void* workspace, cudaStream_t stream, void* S_rec = nullptr,
                            const QkNorm& norm = kNoNorm, void* X_rec = nullptr);

// Varlen forms: q, k, v, beta, o are [H][T][.] (T the packed length), the
// states [seqs.n][H][dk][dv].  The tensor-core form runs in two passes and
// needs H * seqs.chunk[seqs.n] tiles of workspace.
cudaError_t launch_chunk_tc_varlen(const void* q, const void* k, const void* v,
                                   const void* beta, const float* S0, void* o, float* S_T,
                                   const VarlenTable& seqs, int H, int T, void* workspace,
                                   cudaStream_t stream, const QkNorm& norm = kNoNorm);
// Few long sequences on tensor cores (bf16, dk = dv = 128): each sequence
// cut into segments of whole chunks that run in parallel, their start states
// joined through the segments' transitions.  chunk_tc_split_segments is the
// segment count that fills the GPU once; the workspace holds the tiles and
// three [nseg][BH][dk][dv] fp32 state arrays.  o is required.
int chunk_tc_split_segments(int BH, int T);
size_t chunk_tc_split_workspace_bytes(int BH, int T, int nseg);
cudaError_t launch_chunk_tc_split(const void* q, const void* k, const void* v, const void* beta,
                                  const float* S0, void* o, float* S_T, int BH, int T, int nseg,
                                  void* workspace, cudaStream_t stream);
// The backward's chain on tcgen05 (bf16, dk = dv = 128): G = dL/dS from the
// last chunk to the first, with the forward's [PT; Tm] tiles (`tiles`, the
// workspace the state recompute used) read transposed.  Writes G at every
// chunk end (G_chunks, [BH][chunk][2][dk][dv] bf16: hi and lo tiles as for
// S_rec), d_v and d_S0 (if given).
cudaError_t launch_chunk_bwd_chain_tc(const void* q, const void* k, const void* d_o,
                                      const float* d_S_T, void* d_v, float* d_S0,
                                      void* G_chunks, const void* tiles, int BH, int T,
                                      cudaStream_t stream);
// The backward's per-chunk gradients on tcgen05 (bf16, dk = dv = 128): d_q,
// d_k and d_beta of every chunk from its inputs, the state at its start
// (S_rec), the state gradient at its end (G_rec), its (I + A)^{-1} (X_rec)
// and its [PT; Tm] tile, all as the recompute and the chain recorded them.
cudaError_t launch_chunk_bwd_grads_tc(const void* q, const void* k, const void* v,
                                      const void* beta, const void* d_o, const void* S_rec,
                                      const void* G_rec, const void* X_rec, const void* tiles,
                                      void* d_q, void* d_k, void* d_beta, int BH, int T,
                                      cudaStream_t stream);
// Gated DeltaNet on tensor cores (two passes; g the fp32 [BH][T] log keep
// rate): the workspace holds the [PT; Tm] tiles and then kSideFloats fp32
// decay values per chunk, chunk_tc_gated_workspace_bytes(BH, T) in all.
size_t chunk_tc_gated_workspace_bytes(int BH, int T);
// With S_rec32 it records every chunk's start state in fp32 ([BH][chunk][dk][dv],
// the gated backward's recompute) and o may be nullptr.
cudaError_t launch_chunk_tc_gated(const void* q, const void* k, const void* v, const void* beta,
                                  const float* g, const float* S0, void* o, float* S_T, int BH,
                                  int T, int dk, int dv, int dt, void* workspace,
                                  cudaStream_t stream, const QkNorm& norm = kNoNorm,
                                  float* S_rec32 = nullptr);
// KDA on tensor cores (bf16, dk = dv = 128; g the fp32 [BH][T][dk] per-key-
// channel log keep rate), with a workspace of chunk_tc_kda_workspace_bytes.
// With S_rec32 (fp32 [BH][chunk][dk][dv]) the scan records the state at every
// chunk start (for the backward's recompute) and o may be nullptr.
size_t chunk_tc_kda_workspace_bytes(int BH, int T);
cudaError_t launch_chunk_tc_kda(const void* q, const void* k, const void* v, const void* beta,
                                const float* g, const float* S0, void* o, float* S_T, int BH,
                                int T, int dk, int dv, int dt, void* workspace,
                                cudaStream_t stream, const QkNorm& norm = kNoNorm,
                                float* S_rec32 = nullptr);
// Its CUDA-core parts (kda_tc.cu): the decayed operands of every chunk
// (qt, kt, kh, kb: [BH][T][128] bf16; side: 256 fp32 per chunk) with the list
// of chunks beyond the separable range (fix: a count, then chunk indices;
// 1 + BH * nchunks ints), and the exact [PT; Tm] tiles of those chunks.
cudaError_t launch_kda_decay(const void* q, const void* k, const float* g, void* qt, void* kt,
                             void* kh, void* kb, float* side, int* fix, int BH, int T,
                             const QkNorm& nm, cudaStream_t stream);
cudaError_t launch_kda_fix(const void* q, const void* k, const void* beta, const float* g,
                           const int* fix, void* tiles, int BH, int T, const QkNorm& nm,
                           cudaStream_t stream);
// KDA: g is the fp32 [BH][T][dk] per-key-channel log keep rate.  With
// S_chunks (fp32 [BH][chunk][dk][dv]) it records the state at every chunk
// start; o may then be null.
cudaError_t launch_chunk_simt_kda(const void* q, const void* k, const void* v, const void* beta,
                                  const float* g, const float* S0, void* o, float* S_T, int BH,
                                  int T, int dk, int dv, int dt, cudaStream_t stream,
                                  const QkNorm& norm = kNoNorm, float* S_chunks = nullptr);
cudaError_t launch_chunk_simt_varlen(const void* q, const void* k, const void* v,
                                     const void* beta, const float* S0, void* o, float* S_T,
                                     const VarlenTable& seqs, int H, int T, int dk, int dv,
                                     int dt, cudaStream_t stream, const QkNorm& norm = kNoNorm);

// As launch_chunk_tc with the workspace in a static device array of
// noalloc_max_tiles tiles (the caller has checked the size).  The array's
// address is looked up once per device, on the first call with that device
// current; no memory is allocated.
size_t noalloc_max_tiles();
cudaError_t launch_chunk_tc_noalloc(const void* q, const void* k, const void* v,
                                    const void* beta, const float* S0, void* o,
                                    float* S_T, int BH, int T, int dk, int dv,
                                    int dt, cudaStream_t stream);

// Returns and clears the error word the tensor-core kernel sets when one of
// its bounded waits runs out (0 = none, ~0u = could not read it).  Synchronous.
unsigned int chunk_tc_take_device_error();
// Sets the limit of the tensor-core gradient kernel's first bounded wait
// (0: it gives up at once) on the current device.
cudaError_t set_first_wait_limit(unsigned long long ns);

}  // namespace dn
