/*
 * deltanet.h -- C ABI of the GB300 (sm_103a) DeltaNet delta-rule operator.
 *
 * The operator is the delta-rule recurrence of "DeltaNet 引入 Delta Rule"
 * (garden.houmin.site/infra/delta-net) and of "DeltaNet : écrire l'erreur de
 * prédiction plutôt que la valeur" / "Transition d'état structurée"
 * (fr.news.hada.io/topic?id=31925), per batch b and head h:
 *
 *     S_t = S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
 *
 * i.e. u_t = beta_t (v_t - S_{t-1} k_t), S_t = S_{t-1} + u_t k_t^T, and the
 * output is read after the token's own write.  The pages' state S is
 * dv x dk (key space -> value space); this library stores it transposed,
 * as [dk][dv] fp32 with the value channel contiguous.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers (cudaMalloc, or managed
 *     memory), contiguous, row-major, 16-byte aligned (beta: aligned to its
 *     element).  Host pointers are rejected with DN_ERR_INVALID_ARG.
 *   - The caller owns all memory.  The library allocates nothing, never
 *     synchronises, and enqueues its kernels on `stream` (a cudaStream_t;
 *     NULL means the legacy default stream).  Results are ready when the
 *     stream reaches them.
 *   - q and k are used as given: the caller L2-normalises them and applies
 *     any query scale, runs dn_qk_prepare first, or calls the *_qk entry
 *     points, whose kernels prepare them as they load them.  beta is used as given
 *     (0..1, or 0..2 for the negative-eigenvalue variant), with no clamping.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     rejected call enqueues nothing.  Kernels have no device traps and no
 *     unbounded waits.  Launch failures are reported as DN_ERR_CUDA.
 *   - Global state: a thread-local error message (dn_last_error); per device,
 *     one word where a tensor-core kernel records the first of its bounded
 *     waits that ran out (read and cleared by dn_device_error), and the
 *     testing hook's limit of the gradient kernel's first wait
 *     (dn_debug_first_wait_ns); and the static scratch array of
 *     dn_chunk_fwd_noalloc with its looked-up device address.  Calls from
 *     several threads are safe, except that
 *     dn_chunk_fwd_noalloc calls whose kernels overlap on one device race on
 *     that array.
 */
#ifndef DELTANET_H
#define DELTANET_H

#include <stddef.h>

#if defined(__GNUC__)
#define DN_API __attribute__((visibility("default")))
#else
#define DN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
    DN_OK = 0,
    DN_ERR_INVALID_ARG = 1, /* NULL / host / misaligned / aliasing pointer, bad size */
    DN_ERR_UNSUPPORTED = 2, /* valid request this library does not implement   */
    DN_ERR_CUDA = 3         /* the CUDA runtime reported an error              */
} dn_status;

/* Element type of q, k, v, beta and o.  The state is always fp32. */
typedef enum { DN_F32 = 0, DN_BF16 = 1 } dn_dtype;

/* Which kernel evaluates the chunkwise forward. */
typedef enum {
    DN_ALGO_AUTO = 0,  /* tensor cores when the shape and dtype allow, else SIMT  */
    DN_ALGO_SIMT = 1,  /* fp32 CUDA-core arithmetic throughout                    */
    DN_ALGO_TCGEN05 = 2 /* tcgen05 tensor cores (bf16 operands, fp32 accumulate)  */
} dn_algo;

/*
 * dn_chunk_fwd -- chunkwise-parallel forward over whole sequences (training
 * and prefill).
 *
 * Computes, for every (b, h), the recurrence above over t = 0..T-1 starting
 * from S0, evaluated chunk by chunk in the UT / WY form ("Chunkwise KDA :
 * réorganiser la récurrence en multiplications matricielles",
 * fr.news.hada.io/topic?id=31925, with no decay; "Chunkwise parallelization"
 * and appendix B.2 of paperlayer.ai/abs/2406.06484v6).  Per chunk of C
 * tokens with incoming state S:
 *     A = tril(diag(beta) K K^T, -1),  T = (I + A)^{-1} diag(beta),
 *     U' = T (V - K S),  O = Q S + (Q K^T . M) U',  S <- S + K^T U'
 * where M is the causal mask including the diagonal.  The result equals the
 * token-by-token recurrence up to rounding.
 *
 * Arguments:
 *   q, k    [B, H, T, dk]   dtype `dt`
 *   v       [B, H, T, dv]   dtype `dt`
 *   beta    [B, H, T]       dtype `dt`
 *   S0      [B, H, dk, dv]  fp32 initial state, or NULL for zeros
 *   o       [B, H, T, dv]   dtype `dt`, written; must not overlap any input
 *   S_T     [B, H, dk, dv]  fp32 final state, or NULL to skip; may equal S0
 *                           (updated in place) but must not partly overlap it
 *   B, H, T >= 0 (T = 0 only copies S0, or zeros, to S_T)
 *   dk, dv  64 or 128;  C (chunk length) 64
 *   dt      DN_F32 or DN_BF16
 *   workspace, workspace_bytes: device scratch, 16-byte aligned, of at least
 *           dn_chunk_fwd_workspace_bytes(...) bytes, not overlapping any other
 *           argument; or NULL.  With it the tensor-core path runs in two
 *           passes (every chunk's [PT; Tm] = [P T; T] with P = (Q K^T . M),
 *           in parallel over all chunks, then the sequential scan); with NULL
 *           one fused kernel does both (slower).  Other paths ignore it.  The
 *           contents need no initialisation and are undefined afterwards.
 *   stream  cudaStream_t
 * A last chunk shorter than C is handled exactly (as if padded with beta = 0
 * and k = 0 tokens, whose outputs are dropped).
 * Errors: DN_ERR_INVALID_ARG (including a non-NULL workspace that is too
 * small, misaligned, not device memory or overlapping), DN_ERR_UNSUPPORTED
 * (other dk, dv, C), DN_ERR_CUDA.
 */
DN_API int dn_chunk_fwd(const void *q, const void *k, const void *v, const void *beta,
                 const float *S0, void *o, float *S_T,
                 int B, int H, int T, int dk, int dv, int C,
                 int dt, void *workspace, size_t workspace_bytes,
                 void *stream);

/* As dn_chunk_fwd, choosing the kernel explicitly.  DN_ALGO_TCGEN05 returns
 * DN_ERR_UNSUPPORTED for shapes or dtypes it does not cover. */
DN_API int dn_chunk_fwd_algo(const void *q, const void *k, const void *v,
                      const void *beta, const float *S0, void *o, float *S_T,
                      int B, int H, int T, int dk, int dv, int C,
                      int dt, void *workspace, size_t workspace_bytes,
                      void *stream, int algo);

/* Scratch bytes the fastest dn_chunk_fwd path uses for this problem: one
 * 16 KB bf16 [PT; T] tile (128 x 64) and 1 KB of fp32 side vectors (the q
 * and k row factors when dn_chunk_fwd_qk prepares q and k) per (batch, head,
 * chunk) on the tensor-core path (bf16, dk = dv = 128, C = 64), else 0.
 * Host-only. */
DN_API size_t dn_chunk_fwd_workspace_bytes(int B, int H, int T, int dk, int dv,
                                    int C, int dt);

/*
 * dn_recurrent_step -- one decoding step, fused: for every (b, h) it reads
 * the state once, forms p = S k and r = S q (reductions over dk), sets
 * u = beta (v - p), writes S <- S + u k^T back in place and returns
 * o = S_new q = r + (k . q) u.  This is the error-correcting update of
 * "DeltaNet : écrire l'erreur de prédiction plutôt que la valeur" followed
 * by the read, as the fused recurrent kernel of "Kernel Triton récurrent
 * fusionné pour le décodage" (fr.news.hada.io/topic?id=31925) performs it.
 *
 * Arguments:
 *   q, k  [B, H, dk]      dtype `dt`
 *   v     [B, H, dv]      dtype `dt`
 *   beta  [B, H]          dtype `dt`
 *   S     [B, H, dk, dv]  fp32 state, updated in place
 *   o     [B, H, dv]      dtype `dt`, written; must not overlap any input
 *   B, H >= 0; dk, dv 64 or 128; dt DN_F32 or DN_BF16; stream cudaStream_t.
 * Errors: DN_ERR_INVALID_ARG, DN_ERR_UNSUPPORTED (other dk, dv), DN_ERR_CUDA.
 */
DN_API int dn_recurrent_step(const void *q, const void *k, const void *v,
                      const void *beta, float *S, void *o,
                      int B, int H, int dk, int dv, int dt, void *stream);

/*
 * dn_device_error -- returns the first error code a kernel recorded on the
 * device since the previous call (0 if none) and clears it.  Kernels whose
 * internal waits are bounded record a code instead of hanging when a wait
 * runs out (1: a TMA load or a tensor-core operation did not complete within
 * its limit); such a kernel then waits (bounded) for what it started, frees
 * its tensor memory and returns, and the outputs of the call are undefined.
 * This call synchronises the current device.  Returns -1 if the word could
 * not be read.
 */
DN_API int dn_device_error(void);

/*
 * dn_chunk_fwd_split -- dn_chunk_fwd for a few long sequences (bf16,
 * dk = dv = 128, C = 64): each sequence is cut into `segments` runs of whole
 * chunks that are scanned in parallel.  The state is linear in its start
 * value, S_end = A S_start + B per run, where A is the product of the runs'
 * chunk transitions (I - K^T T K) and B its end state from zero ("Chunkwise
 * parallelization", paperlayer.ai/abs/2406.06484v6: the chunk states are the
 * only thing carried from chunk to chunk).  The call scans every run but the
 * last from zero (B) and from the identity with zero values (A), joins the
 * start states in fp32, then scans every run from its own start writing o and
 * the final state.  Results agree with dn_chunk_fwd within bf16 rounding; the
 * chunk arithmetic is the same, only the start states of the runs are formed
 * differently.
 *   arguments as for dn_chunk_fwd; o is required;
 *   segments  number of runs, 1 .. 1024, or 0 to fill the current device's
 *             SMs once (SMs / (B * H), at least 1); capped at the chunk count;
 *   workspace device scratch of dn_chunk_fwd_split_workspace_bytes(...) bytes
 *             (required), 16-byte aligned.
 * S0 == S_T is allowed.  Errors: as dn_chunk_fwd; DN_ERR_UNSUPPORTED outside
 * bf16 with dk = dv = 128.
 */
DN_API int dn_chunk_fwd_split(const void *q, const void *k, const void *v, const void *beta,
                              const float *S0, void *o, float *S_T, int B, int H, int T, int dk,
                              int dv, int C, int dt, int segments, void *workspace,
                              size_t workspace_bytes, void *stream);
/* Scratch bytes dn_chunk_fwd_split needs (0 for unsupported arguments): the
 * tiles of every chunk and three fp32 states per run and head.
 * With segments = 0 it queries the current device.  Host-only. */
DN_API size_t dn_chunk_fwd_split_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                                 int dt, int segments);

/*
 * dn_debug_first_wait_ns -- a testing hook for the failure path above, with
 * no counterpart in the method: sets, for the current device, the limit in
 * nanoseconds of the first bounded wait of the tensor-core gradient kernel
 * (the dn_chunk_bwd path for bf16, dk = dv = 128).  0 makes that wait give up
 * at once, so the kernel records code 1 and returns without results; the
 * default is 2e9 (every other wait keeps it).  Process-wide state: set it
 * only while no dn_chunk_bwd call is in flight.  Returns DN_OK or
 * DN_ERR_CUDA.
 */
DN_API int dn_debug_first_wait_ns(unsigned long long ns);

/* Static text for a dn_status value. */
DN_API const char *dn_status_string(int status);

/* Detail of the last non-OK return on the calling thread ("" if none).  The
 * pointer stays valid until the next call into the library on this thread. */
DN_API const char *dn_last_error(void);

/*
 * dn_chunk_fwd_noalloc -- dn_chunk_fwd on the two-pass tensor-core path,
 * using no memory the caller provides and allocating none.  The paper has no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc.  The per-chunk [PT; T] tiles go to a static device array inside
 * the library that holds DN_NOALLOC_MAX_TILES tiles of 16 KB (8 MiB).
 *
 *   - Covers bf16 with dk = dv = 128 and C = 64 only; other shapes and dtypes
 *     return DN_ERR_UNSUPPORTED.
 *   - Needs B * H * ceil(T / 64) <= DN_NOALLOC_MAX_TILES; larger problems
 *     return DN_ERR_INVALID_ARG before anything is launched.
 *   - Nothing in the array has to start at zero: within a call every tile is
 *     written before it is read.
 *   - Every call on a device shares the array, so calls whose kernels overlap
 *     on the GPU (on different streams, say) race; serialise them.
 *   - The first call on each device looks the array's address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after cudaDeviceReset (which unloads the library's device
 *     code) do not call this entry point again on that device.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments, layouts and the remaining errors are those of dn_chunk_fwd.
 */
#define DN_NOALLOC_MAX_TILES 512
DN_API int dn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                         const void *beta, const float *S0, void *o, float *S_T,
                         int B, int H, int T, int dk, int dv, int C, int dt,
                         void *stream);

/*
 * dn_chunk_bwd -- gradients of the chunkwise forward, for training: given
 * the gradient d_o of the outputs and d_S_T of the final state, returns the
 * gradients of L = <d_o, o> + <d_S_T, S_T> with respect to q, k, v, beta and
 * S0.  The pages run this pass after the forward and recompute the chunk
 * states instead of storing them ("Hardware-efficient implementation",
 * section 3 of paperlayer.ai/abs/2406.06484v6); the result is the exact
 * gradient of the recurrence up to rounding.  Where the tensor-core forward
 * covers the shape (bf16, dk = dv = 128) it recomputes the states and the
 * chain of state gradients (last chunk to first) runs on tcgen05 with fp32
 * accumulation; the per-chunk gradients run as fp32 CUDA-core products for
 * fp32 I/O and as tf32 tensor-core products (fp32 accumulation) for bf16.
 *
 * Arguments:
 *   q, k, v, beta, S0   as for dn_chunk_fwd (S0 may be NULL: zeros)
 *   d_o     [B, H, T, dv]   dtype `dt`
 *   d_S_T   [B, H, dk, dv]  fp32, or NULL (zeros)
 *   d_q, d_k [B, H, T, dk], d_v [B, H, T, dv], d_beta [B, H, T]   dtype `dt`,
 *           written
 *   d_S0    [B, H, dk, dv]  fp32, written, or NULL to skip
 *   B, H, T, dk, dv, C, dt  as for dn_chunk_fwd
 *   workspace, workspace_bytes: device scratch, 16-byte aligned, of at least
 *           dn_chunk_bwd_workspace_bytes(...) bytes (required when
 *           B * H * T > 0); the contents need no initialisation and are
 *           undefined afterwards.
 *   stream  cudaStream_t
 * No output may overlap an input, another output or the workspace.  With
 * T = 0 only d_S0 is written (a copy of d_S_T, or zeros).
 * Errors: DN_ERR_INVALID_ARG (including a missing or short workspace),
 * DN_ERR_UNSUPPORTED (other dk, dv, C), DN_ERR_CUDA.
 */
DN_API int dn_chunk_bwd(const void *q, const void *k, const void *v, const void *beta,
                 const float *S0, const void *d_o, const float *d_S_T,
                 void *d_q, void *d_k, void *d_v, void *d_beta, float *d_S0,
                 int B, int H, int T, int dk, int dv, int C, int dt,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Scratch bytes dn_chunk_bwd needs: the fp32 state at the start of every
 * chunk and the gradient of the state at its end, 2 * B * H * ceil(T / 64) *
 * dk * dv * 4 bytes, plus dn_chunk_fwd_workspace_bytes(...) where the
 * tensor-core forward recomputes the states (0 for unsupported arguments).
 * Host-only. */
DN_API size_t dn_chunk_bwd_workspace_bytes(int B, int H, int T, int dk, int dv,
                                    int C, int dt);

/*
 * dn_chunk_fwd_gated -- Gated DeltaNet, chunkwise: a scalar keep rate
 * alpha_t = exp(g_t) per token decays the whole state before the delta rule
 * ("Gated DeltaNet", garden.houmin.site/infra/delta-net; "Gated DeltaNet :
 * oublier d'abord l'état entier", fr.news.hada.io/topic?id=31925):
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
 * i.e. forget (alpha S), predict, correct, write, read, in that order.
 *   g       [B, H, T] fp32 log keep rates, g <= 0 (keep rates alpha in
 *           (0, 1], as the method defines them); 4-byte aligned device
 *           memory.  Not checked: the chunk kernels clamp every in-chunk
 *           decay ratio exp(G_i - G_j) at 1, so a positive g gives results
 *           the recurrence does not define.
 *   workspace, workspace_bytes
 *           NULL: one fp32 CUDA-core kernel (any supported shape and dtype).
 *           Otherwise device scratch of at least
 *           dn_chunk_fwd_gated_workspace_bytes(...) bytes, 16-byte aligned,
 *           owned by the caller and disjoint from every other argument; where
 *           that size is non-zero (dk = dv = 128, bf16) the call runs in two
 *           tcgen05 passes like dn_chunk_fwd: per chunk, the decay ratios
 *           exp(G_i - G_j) (G the in-chunk cumulative log keep rate) enter A
 *           and P before the solve, and the state is carried as
 *           S <- exp(G_C) S + K^T diag(exp(G_C - G_s)) U'.  Its contents on
 *           return are unspecified.  A smaller workspace is DN_ERR_INVALID_ARG.
 * Every other argument, layout and error as for dn_chunk_fwd.
 */
DN_API int dn_chunk_fwd_gated(const void *q, const void *k, const void *v,
                       const void *beta, const float *g, const float *S0, void *o,
                       float *S_T, int B, int H, int T, int dk, int dv, int C, int dt,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Scratch bytes of the tensor-core form of dn_chunk_fwd_gated: two 16 KB
 * tiles ([PT; Tm] and [PT; Tm] diag(exp G)) and 1 KB of fp32 decay factors
 * per (batch, head, chunk), B * H * ceil(T / 64) * 33792 bytes; 0 where
 * that form does not apply (dk or dv != 128, fp32 I/O, C != 64, an empty
 * problem).  Host-only. */
DN_API size_t dn_chunk_fwd_gated_workspace_bytes(int B, int H, int T, int dk, int dv,
                                          int C, int dt);

/*
 * dn_recurrent_step_gated -- one Gated DeltaNet decoding step: with
 * alpha = exp(g) per (b, h), p = alpha S k, u = beta (v - p),
 * S <- alpha S + u k^T (stored layout: S += k u^T after the decay) and
 * o = S_new q.  g is [B, H] fp32; everything else as for dn_recurrent_step.
 */
DN_API int dn_recurrent_step_gated(const void *q, const void *k, const void *v,
                            const void *beta, const float *g, float *S, void *o,
                            int B, int H, int dk, int dv, int dt, void *stream);

/*
 * dn_chunk_fwd_varlen -- dn_chunk_fwd over packed variable-length sequences
 * (no padding): N sequences of one batch element lie back to back along T,
 * sequence n being tokens cu_seqlens[n] .. cu_seqlens[n+1] - 1.  Each runs
 * the recurrence from its own initial state.  The pages' layer takes such
 * cu_seqlens offsets for variable-length batches (fla/layers/delta_net.py,
 * DeltaNet.forward); the result per sequence is that of dn_chunk_fwd on it.
 *
 *   q, k [H, T, dk], v, o [H, T, dv], beta [H, T]   dtype `dt` (T = packed length)
 *   S0, S_T [N, H, dk, dv] fp32 (S0 may be NULL: zeros; S_T may be NULL)
 *   cu_seqlens  HOST array of N + 1 ints, 0 = cu_seqlens[0] <= ... <=
 *               cu_seqlens[N] = T (empty sequences allowed);
 *               1 <= N <= DN_MAX_VARLEN_SEQS
 *   workspace   as for dn_chunk_fwd, of dn_chunk_fwd_varlen_workspace_bytes
 *               bytes (one tile per head and chunk of every sequence); with it
 *               the two-pass tensor-core path runs (bf16, dk = dv = 128), with
 *               NULL (or for other shapes) the fp32 CUDA-core path
 * Errors: as for dn_chunk_fwd, plus DN_ERR_INVALID_ARG for a bad cu_seqlens.
 */
#define DN_MAX_VARLEN_SEQS 1024
DN_API int dn_chunk_fwd_varlen(const void *q, const void *k, const void *v,
                        const void *beta, const float *S0, void *o, float *S_T,
                        const int *cu_seqlens, int N, int H, int T, int dk, int dv,
                        int C, int dt, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Scratch bytes for dn_chunk_fwd_varlen's tensor-core path (0 where it does
 * not apply).  Host-only; reads cu_seqlens (host, N + 1 ints). */
DN_API size_t dn_chunk_fwd_varlen_workspace_bytes(const int *cu_seqlens, int N, int H,
                                           int dk, int dv, int C, int dt);

/*
 * dn_chunk_bwd_gated -- the gradients of dn_chunk_fwd_gated's outputs: for
 * L = <d_o, o> + <d_S_T, S_T>, the gradients with respect to q, k, v, beta,
 * the log keep rates g and S0 ("Gated DeltaNet", garden.houmin.site/infra/
 * delta-net; "Gated DeltaNet : oublier d'abord l'état entier",
 * fr.news.hada.io/topic?id=31925; the states recomputed as in
 * "Hardware-efficient implementation", paperlayer.ai/abs/2406.06484v6).
 *   g, d_g  [B, H, T] fp32 (4-byte aligned); the rest as dn_chunk_bwd.
 *   workspace  device scratch of dn_chunk_bwd_gated_workspace_bytes(...) bytes.
 * For bf16 with dk = dv = 128 the states are recomputed and the state
 * gradient carried on tcgen05, through the KDA form with the rate on every
 * key channel (Gated DeltaNet is KDA with equal channels); otherwise both run
 * on the CUDA cores.  The per-chunk gradients are formed on the CUDA cores
 * (fp32 products for fp32 I/O, tf32 tensor-core products with fp32
 * accumulation for bf16).  d_g is
 * the gradient of each token's log keep rate, through every later ratio
 * exp(G_i - G_j), keep factor and state carried out of its chunk.  Errors and
 * overlap rules as dn_chunk_bwd; d_g may overlap nothing else.
 */
DN_API int dn_chunk_bwd_gated(const void *q, const void *k, const void *v, const void *beta,
                              const float *g, const float *S0, const void *d_o,
                              const float *d_S_T, void *d_q, void *d_k, void *d_v, void *d_beta,
                              float *d_g, float *d_S0, int B, int H, int T, int dk, int dv, int C,
                              int dt, void *workspace, size_t workspace_bytes, void *stream);
/* Its scratch: the fp32 state and state gradient of every chunk,
 * 2 * B * H * ceil(T / 64) * dk * dv * 4 bytes, plus, for bf16 with
 * dk = dv = 128, the tensor-core KDA forward's scratch (as
 * dn_chunk_fwd_kda_workspace_bytes, rounded up to 256 bytes) and the rates
 * broadcast over the key channels (B * H * T * dk * 4 bytes); 0 for invalid
 * arguments.  Host-only. */
DN_API size_t dn_chunk_bwd_gated_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                                 int dt);

/*
 * dn_chunk_bwd_kda -- the gradients of dn_chunk_fwd_kda's outputs: for
 * L = <d_o, o> + <d_S_T, S_T>, the gradients with respect to q, k, v, beta,
 * the per-key-channel log keep rates g and S0 ("Kimi Delta Attention :
 * atténuation par canal" and "Transition diagonale-bas rang",
 * fr.news.hada.io/topic?id=31925; the states recomputed as in
 * "Hardware-efficient implementation", paperlayer.ai/abs/2406.06484v6).
 *   g, d_g  [B, H, T, dk] fp32 (g 16-byte aligned); the rest as dn_chunk_bwd.
 *   workspace  device scratch of dn_chunk_bwd_kda_workspace_bytes(...) bytes.
 * For bf16 with dk = dv = 128 the states are recomputed and the state
 * gradient carried on tcgen05 (the tensor-core KDA forward, then a chain
 * that reads the decayed operands it leaves); otherwise both run on the CUDA
 * cores.  The per-chunk gradients are formed on the CUDA cores (fp32
 * products for fp32 I/O, tf32 tensor-core products with fp32 accumulation
 * for bf16).  The decay ratios
 * exp(G_t[c] - G_s[c]) sit inside the channel sums: as products of
 * exp(G) and exp(-G) scaled operands while a chunk's decay stays within
 * exp(-60) on every channel, else one exponential per ratio.  d_g[t][c] is
 * the gradient of token t's log keep rate on key channel c.  Errors and
 * overlap rules as dn_chunk_bwd; d_g may overlap nothing else.
 */
DN_API int dn_chunk_bwd_kda(const void *q, const void *k, const void *v, const void *beta,
                            const float *g, const float *S0, const void *d_o,
                            const float *d_S_T, void *d_q, void *d_k, void *d_v, void *d_beta,
                            float *d_g, float *d_S0, int B, int H, int T, int dk, int dv, int C,
                            int dt, void *workspace, size_t workspace_bytes, void *stream);
/* Its scratch: the fp32 state and state gradient of every chunk,
 * 2 * B * H * ceil(T / 64) * dk * dv * 4 bytes, plus, for bf16 with
 * dk = dv = 128, the tensor-core forward's scratch (as
 * dn_chunk_fwd_kda_workspace_bytes); 0 for invalid arguments.  Host-only. */
DN_API size_t dn_chunk_bwd_kda_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                               int dt);

/*
 * dn_chunk_bwd_varlen -- the gradients of dn_chunk_fwd_varlen's outputs, as
 * dn_chunk_bwd gives them for the batched forward (the pages' backward with
 * the states recomputed: "Hardware-efficient implementation",
 * paperlayer.ai/abs/2406.06484v6), for N sequences packed along T.
 *   q, k, d_q, d_k  [H, T, dk];  v, d_o, d_v  [H, T, dv];  beta, d_beta [H, T]
 *   S0, d_S_T, d_S0 [N, H, dk, dv] fp32 (NULL: zero / not wanted)
 *   cu_seqlens      host array of N + 1 ints, 0 = cu[0] <= ... <= cu[N] = T
 *   workspace       device scratch of dn_chunk_bwd_varlen_workspace_bytes(...)
 *                   bytes, 16-byte aligned.
 * Each sequence runs as its own batched backward on copies of its rows
 * gathered into the workspace, its gradients scattered back; an empty
 * sequence passes d_S_T through to d_S0.  Errors and overlap rules as
 * dn_chunk_bwd.
 */
DN_API int dn_chunk_bwd_varlen(const void *q, const void *k, const void *v, const void *beta,
                               const float *S0, const void *d_o, const float *d_S_T, void *d_q,
                               void *d_k, void *d_v, void *d_beta, float *d_S0,
                               const int *cu_seqlens, int N, int H, int T, int dk, int dv, int C,
                               int dt, void *workspace, size_t workspace_bytes, void *stream);
/* Its scratch: the batched backward's for the longest sequence plus the
 * gathered rows and gradients of one sequence (0 for invalid arguments).
 * Host-only. */
DN_API size_t dn_chunk_bwd_varlen_workspace_bytes(const int *cu_seqlens, int N, int H, int dk,
                                                  int dv, int C, int dt);

/*
 * dn_chunk_fwd_kda / dn_recurrent_step_kda -- Kimi Delta Attention: one keep
 * rate per key channel, D_t = Diag(exp(g_t)), decays the state's key
 * channels before the delta rule ("Kimi Delta Attention : atténuation par
 * canal" and "Transition diagonale-bas rang", fr.news.hada.io/topic?id=31925):
 *     S_t = S_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
 * (in the stored [dk][dv] layout, row i of S is scaled by exp(g_t[i])).  The
 * page's read uses d_k^{-1/2} q_t; as everywhere in this library the caller
 * applies any query scale.
 *   g   [B, H, T, dk] fp32 for the chunkwise form (16-byte aligned: the
 *       kernel reads it in 16-byte rows), [B, H, dk] for a step (4-byte
 *       aligned)
 * Every other argument, layout and error as for dn_chunk_fwd_gated (with no
 * workspace) / dn_recurrent_step_gated.  fp32 arithmetic on CUDA cores.
 */
DN_API int dn_chunk_fwd_kda(const void *q, const void *k, const void *v,
                     const void *beta, const float *g, const float *S0, void *o,
                     float *S_T, int B, int H, int T, int dk, int dv, int C, int dt,
                     void *stream);
DN_API int dn_recurrent_step_kda(const void *q, const void *k, const void *v,
                          const void *beta, const float *g, float *S, void *o,
                          int B, int H, int dk, int dv, int dt, void *stream);

/*
 * dn_qk_prepare -- optional input preparation for every entry point above:
 * the query/key L2 normalisation and query scale that the pages apply
 * before the recurrence.  Per row of d elements (the head dimension):
 *     q_out = scale * q / sqrt(sum q^2 + eps)     (normalize != 0)
 *     k_out =         k / sqrt(sum k^2 + eps)     (normalize != 0)
 *     q_out = scale * q                           (normalize == 0; k, k_out unused)
 * This is the l2norm helper and the 1/sqrt(head_dim) query factor of the
 * Gated DeltaNet PyTorch code on "DeltaNet 引入 Delta Rule"
 * (garden.houmin.site/infra/delta-net), which the DeltaNet layer of
 * "fla/layers/delta_net.py" asks its kernels for (use_qk_l2norm_in_kernel),
 * and the d_k^{-1/2} read of "Kimi Delta Attention"
 * (fr.news.hada.io/topic?id=31925); the pages use eps = 1e-6.  The keys are
 * never scaled: the read o_t = S_t q_t is linear in q, so the scale
 * multiplies the outputs and leaves the state as it is.
 *
 * Arithmetic in fp32 (sum of squares, reciprocal square root, products),
 * rounded once to `dt` on the store.  One kernel over all rows; it runs as
 * its own pass (reads q and k once, writes them once) ahead of the
 * recurrence.
 *
 * Arguments:
 *   q, q_out   [rows, d]  dtype `dt`; q_out may be q itself (in place) but
 *                         must not partially overlap it
 *   k, k_out   [rows, d]  dtype `dt`; read and written only when
 *                         normalize != 0 (k_out may be k)
 *   rows >= 0 (B * H * T for the chunkwise forms, B * H for a step,
 *   H * T for packed sequences); d 64 or 128; scale finite; eps finite,
 *   >= 0 (with eps = 0 a zero row gives NaN); dt DN_F32 or DN_BF16.
 * Errors: DN_ERR_INVALID_ARG (pointers, sizes, overlaps, non-finite scale or
 * eps), DN_ERR_UNSUPPORTED (other d), DN_ERR_CUDA.
 */
DN_API int dn_qk_prepare(const void *q, const void *k, void *q_out, void *k_out,
                  long long rows, int d, int normalize, float scale, float eps,
                  int dt, void *stream);

/*
 * dn_qk_prepare_bwd -- gradient of dn_qk_prepare with respect to its raw
 * inputs, for training through the preparation.  Given the raw rows q, k and
 * the gradients d_q_out, d_k_out of the prepared rows, per row x with
 * n = sqrt(sum x^2 + eps) and f = scale / n (scale = 1 for k):
 *     d_x = f (d_out - x (x . d_out) / n^2)      (normalize != 0)
 *     d_q = scale d_q_out                        (normalize == 0; k unused)
 * the chain rule through y = f x with dn/dx_i = x_i / n.  fp32 arithmetic,
 * rounded once to `dt`.
 *   q, k, d_q_out, d_k_out  [rows, d] dtype `dt` (k, d_k_out, d_k are read /
 *                           written only when normalize != 0; q only then)
 *   d_q, d_k                [rows, d] written; each may be its own incoming
 *                           gradient (d_q == d_q_out, in place) but must
 *                           not otherwise overlap an input or each other
 *   rows, d, normalize, scale, eps, dt, stream  as for dn_qk_prepare
 * Errors as for dn_qk_prepare.
 */
DN_API int dn_qk_prepare_bwd(const void *q, const void *k, const void *d_q_out,
                             const void *d_k_out, void *d_q, void *d_k, long long rows,
                             int d, int normalize, float scale, float eps, int dt,
                             void *stream);

/*
 * In-kernel preparation of q and k.  The pages' layer asks its kernels to
 * L2-normalise q and k themselves (use_qk_l2norm_in_kernel, DeltaNet.forward
 * of fla/layers/delta_net.py) and scales the query by 1/sqrt(d_head) ("DeltaNet
 * 引入 Delta Rule", garden.houmin.site/infra/delta-net; the d_k^{-1/2} read of
 * "Kimi Delta Attention", fr.news.hada.io/topic?id=31925).  The *_qk entry
 * points below take a dn_qk_norm (NULL: q and k used as given) and apply
 *     q <- scale * q / sqrt(sum q^2 + eps),  k <- k / sqrt(sum k^2 + eps)
 * (with l2norm == 0: q <- scale * q, k as given) to every row of the head
 * dimension as the kernels load it, before any product uses it; q and k in
 * memory are not modified.  The arithmetic is fp32 (sum of squares,
 * reciprocal square root, products); the tensor-core kernels round the
 * prepared rows to bf16 as their MMA operands, the CUDA-core kernels keep
 * them in fp32.  This is dn_qk_prepare's arithmetic without its separate
 * pass over q and k.  scale must be finite; with l2norm, eps finite and >= 0.
 */
typedef struct {
    int l2norm;   /* nonzero: L2-normalise every row of q and k */
    float scale;  /* multiplies q after the normalisation (1.0f: none) */
    float eps;    /* added to the sum of squares (the pages use 1e-6) */
} dn_qk_norm;

/* dn_chunk_fwd_algo with an optional dn_qk_norm. */
DN_API int dn_chunk_fwd_qk(const void *q, const void *k, const void *v, const void *beta,
                           const float *S0, void *o, float *S_T, int B, int H, int T,
                           int dk, int dv, int C, int dt, void *workspace,
                           size_t workspace_bytes, void *stream, int algo,
                           const dn_qk_norm *norm);
/* dn_chunk_fwd_gated with an optional dn_qk_norm. */
DN_API int dn_chunk_fwd_gated_qk(const void *q, const void *k, const void *v,
                                 const void *beta, const float *g, const float *S0, void *o,
                                 float *S_T, int B, int H, int T, int dk, int dv, int C,
                                 int dt, void *workspace, size_t workspace_bytes,
                                 void *stream, const dn_qk_norm *norm);
/* dn_chunk_fwd_varlen with an optional dn_qk_norm. */
DN_API int dn_chunk_fwd_varlen_qk(const void *q, const void *k, const void *v,
                                  const void *beta, const float *S0, void *o, float *S_T,
                                  const int *cu_seqlens, int N, int H, int T, int dk, int dv,
                                  int C, int dt, void *workspace, size_t workspace_bytes,
                                  void *stream, const dn_qk_norm *norm);
/* dn_chunk_fwd_kda with a workspace (dn_chunk_fwd_kda_workspace_bytes; where
 * that size is non-zero it selects the tensor-core form, NULL the CUDA-core
 * kernel) and an optional dn_qk_norm. */
DN_API int dn_chunk_fwd_kda_qk(const void *q, const void *k, const void *v,
                               const void *beta, const float *g, const float *S0, void *o,
                               float *S_T, int B, int H, int T, int dk, int dv, int C, int dt,
                               void *workspace, size_t workspace_bytes, void *stream,
                               const dn_qk_norm *norm);
DN_API size_t dn_chunk_fwd_kda_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                               int dt);
/* The decoding steps with an optional dn_qk_norm. */
DN_API int dn_recurrent_step_qk(const void *q, const void *k, const void *v,
                                const void *beta, float *S, void *o, int B, int H, int dk,
                                int dv, int dt, void *stream, const dn_qk_norm *norm);
DN_API int dn_recurrent_step_gated_qk(const void *q, const void *k, const void *v,
                                      const void *beta, const float *g, float *S, void *o,
                                      int B, int H, int dk, int dv, int dt, void *stream,
                                      const dn_qk_norm *norm);
DN_API int dn_recurrent_step_kda_qk(const void *q, const void *k, const void *v,
                                    const void *beta, const float *g, float *S, void *o,
                                    int B, int H, int dk, int dv, int dt, void *stream,
                                    const dn_qk_norm *norm);

/* ABI version of this header (bumped on incompatible changes). */
DN_API int dn_abi_version(void);

#define DN_ABI_VERSION 9

#ifdef __cplusplus
}
#endif

#endif /* DELTANET_H */
