/*
 * kda.h - C ABI of libkda.so: Kimi Delta Attention (KDA) chunked prefill and
 * decode step on one GB300 (sm_103a).
 *
 * Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
 * (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
 *
 * The operation ([K3-notes §2.2, KDA state recurrence]), per sequence n and
 * head h, over that sequence's tokens t in order:
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t,            alpha_t = exp(log_alpha_t)  (per channel)
 * with S in R^{dk x dv}.  The library does not scale or normalise q or k.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    keeps no pointer after the call returns.  Alignment (KDA_ERR_ALIGN
 *    otherwise): kda_chunk_fwd needs q, k, v, log_alpha and out 16-byte
 *    aligned and the other pointers 4-byte aligned; kda_decode_step needs
 *    state_inout 16-byte aligned and the other pointers aligned to their
 *    element size.  Tensors are dense and row-major in the shapes written
 *    below (last index contiguous).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without waiting, except in validate mode.
 *  - Argument errors are reported synchronously, before anything is launched,
 *    as a negative kda_status.  A launch failure returns KDA_ERR_CUDA.
 *    Asynchronous device faults surface at the caller's next synchronisation.
 *  - Preconditions on values ([K3-notes §2.2, Eq. 5] bounds the log-decay
 *    below by g_min = -5): log_alpha in [-5, 0], beta in [0, 1], cu_seqlens
 *    non-decreasing from 0 to T.  The kernels rely on the log-decay floor for
 *    their range guard.  They are checked only in validate mode (desc.validate
 *    = 1), which runs a check kernel first, synchronises the stream and
 *    returns KDA_ERR_RANGE without computing anything if a value is outside.
 *  - Results are deterministic: the same inputs give bitwise the same outputs.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *kda_stream_t; /* the same type as cudaStream_t */

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_NULL = -1,        /* a required pointer (or the descriptor) is NULL      */
  KDA_ERR_SHAPE = -2,       /* a size is out of the supported set                  */
  KDA_ERR_DTYPE = -3,       /* unsupported dtype combination                       */
  KDA_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned                    */
  KDA_ERR_RANGE = -5,       /* validate mode found a value outside its range       */
  KDA_ERR_CUDA = -6,        /* a CUDA call or kernel launch failed                 */
  KDA_ERR_UNSUPPORTED = -7, /* a kernel choice that does not cover these arguments */
  KDA_ERR_ALIAS = -8,       /* forbidden aliasing between arguments                */
  KDA_ERR_SCRATCH_LIMIT = -9 /* kda_chunk_fwd_noalloc: the call needs more scratch
                                than KDA_STATIC_WORKSPACE_BYTES                      */
} kda_status;

/* Which prefill kernel runs.  AUTO picks the tensor-core kernel when it covers
 * the arguments (bf16 q/k/v, bf16 out, dk = dv = 128, chunk = 64) and the
 * CUDA-core kernel otherwise.  Asking for TC on arguments it does not cover
 * returns KDA_ERR_UNSUPPORTED. */
typedef enum { KDA_KERNEL_AUTO = 0, KDA_KERNEL_SIMT = 1, KDA_KERNEL_TC = 2 } kda_kernel;

typedef struct {
  int B;          /* batch; must be 1 when cu_seqlens is given                */
  int T;          /* tokens per sequence, or total tokens when varlen          */
  int H;          /* heads                                                    */
  int dk, dv;     /* key and value head dims: each one of 16, 32, 64, 128      */
  int chunk;      /* chunk length C: 16, 32 or 64 (outputs do not depend on it
                     beyond rounding)                                          */
  int num_seqs;   /* varlen: number of sequences N (cu_seqlens has N+1 entries);
                     0 when cu_seqlens is NULL                                 */
  kda_dtype qkv_dtype;  /* q, k, v                                             */
  kda_dtype out_dtype;  /* out                                                 */
  kda_dtype gate_dtype; /* log_alpha and beta                                  */
  int validate;   /* 1: range-check inputs first (synchronises the stream)     */
  kda_kernel kernel;
  int segments;   /* long sequences: split each sequence into this many
                     segments that run in parallel and are joined through
                     their affine pairs; 0 = choose automatically, 1 = never  */
} kda_chunk_desc;

/*
 * kda_chunk_fwd - chunked prefill ([K3-notes §2.2, chunkwise form];
 * initial/final state for prefix-cache resume, [K3-notes §2.5, Fig. 12]).
 *
 *   q, k        [B*T, H, dk]  qkv_dtype   (token-major; B sequences of T
 *                                          tokens, or N packed sequences)
 *   v           [B*T, H, dv]  qkv_dtype
 *   log_alpha   [B*T, H, dk]  gate_dtype  (g = ln alpha, per channel)
 *   beta        [B*T, H]      gate_dtype
 *   initial_state [Nseq, H, dk, dv] fp32, or NULL for zeros
 *   cu_seqlens  [N+1] int32 (varlen: sequence n is tokens
 *               [cu_seqlens[n], cu_seqlens[n+1]) ), or NULL for B x T
 *   out         [B*T, H, dv]  out_dtype   (written)
 *   final_state [Nseq, H, dk, dv] fp32, or NULL (written)
 * Nseq = num_seqs when varlen, else B.  An empty sequence leaves its
 * final state equal to its initial state.  initial_state may equal
 * final_state (in-place resume); out may not alias any input.
 * When the planner splits long sequences into segments it allocates a
 * stream-ordered workspace (cudaMallocAsync/cudaFreeAsync on `stream`); use
 * kda_chunk_fwd_ex to pass one instead.
 */
kda_status kda_chunk_fwd(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta, const float *initial_state,
                         const int32_t *cu_seqlens, void *out, float *final_state,
                         kda_stream_t stream);

/* Bytes of device workspace kda_chunk_fwd_ex needs for these arguments (0 when
 * no sequence is split).  Host-only; launches nothing. */
kda_status kda_chunk_fwd_workspace_size(const kda_chunk_desc *desc, size_t *bytes);

/* kda_chunk_fwd with a caller-owned device workspace of at least
 * kda_chunk_fwd_workspace_size bytes (16-byte aligned; NULL allowed when that
 * size is 0).  The workspace must not be in use by another call in flight. */
kda_status kda_chunk_fwd_ex(const kda_chunk_desc *desc, const void *q, const void *k,
                            const void *v, const void *log_alpha, const void *beta,
                            const float *initial_state, const int32_t *cu_seqlens, void *out,
                            float *final_state, void *workspace, size_t workspace_bytes,
                            kda_stream_t stream);

/*
 * kda_chunk_fwd_ckpt - kda_chunk_fwd that also stores the state at fixed
 * intervals along each sequence, for prefix-cache reuse ([K3-notes §2.5,
 * Fig. 12]: a request that shares a cached prefix resumes from the state at
 * the prefix's end; a cache that keeps a state every `every` tokens can
 * resume at any multiple of it).
 *
 *   every     checkpoint interval in tokens, a positive multiple of
 *             desc->chunk (KDA_ERR_SHAPE otherwise)
 *   cu_ckpt   [N+1] int32 device, required with cu_seqlens: sequence n's
 *             checkpoints go to slots cu_ckpt[n] .. cu_ckpt[n+1]-1, and
 *             cu_ckpt[n+1] - cu_ckpt[n] must be floor(len_n / every)
 *             (checked in validate mode); NULL for a B x T batch, whose
 *             sequence n uses slots n*floor(T/every) .. (n+1)*floor(T/every)-1
 *   ckpt      [slots, H, dk, dv] fp32 device, written: the j-th slot of a
 *             sequence (j = 1, 2, ...) holds its state after its first
 *             j*every tokens, exactly what kda_chunk_fwd on that prefix
 *             alone would return as final_state (up to rounding)
 *   workspace as in kda_chunk_fwd_ex; NULL makes a split plan allocate its
 *             workspace stream-ordered, as kda_chunk_fwd does
 * Other arguments and conventions as kda_chunk_fwd.  ckpt may alias no other
 * argument (KDA_ERR_ALIAS; for packed sequences only its first slot's extent
 * is known on the host and checked).
 */
kda_status kda_chunk_fwd_ckpt(const kda_chunk_desc *desc, const void *q, const void *k,
                              const void *v, const void *log_alpha, const void *beta,
                              const float *initial_state, const int32_t *cu_seqlens, void *out,
                              float *final_state, int every, const int32_t *cu_ckpt, float *ckpt,
                              void *workspace, size_t workspace_bytes, kda_stream_t stream);

typedef struct {
  int N;          /* independent sequences, one token each                    */
  int H;          /* heads                                                    */
  int dk, dv;     /* each one of 16, 32, 64, 128                              */
  kda_dtype qkv_dtype, out_dtype, gate_dtype;
  int validate;   /* 1: range-check inputs first (synchronises the stream)     */
} kda_decode_desc;

/*
 * kda_decode_step - one token of the recurrence for N sequences, updating
 * their states in place ([K3-notes §2.2, KDA state recurrence]; the decode
 * regime of [K3-notes §2.5]).
 *
 *   q, k        [N, H, dk]  qkv_dtype
 *   v           [N, H, dv]  qkv_dtype
 *   log_alpha   [N, H, dk]  gate_dtype
 *   beta        [N, H]      gate_dtype
 *   state_inout [N, H, dk, dv] fp32, read and overwritten
 *   out         [N, H, dv]  out_dtype, written
 * state_inout may not alias out or any input.
 */
kda_status kda_decode_step(const kda_decode_desc *desc, const void *q, const void *k,
                           const void *v, const void *log_alpha, const void *beta,
                           float *state_inout, void *out, kda_stream_t stream);

/*
 * The KDA layer's gates around the recurrence ([K3-notes §2.2]):
 *   decay gate (Eq. 5):  log_alpha = g_min * Sigmoid(exp(A_h) * z)
 *       z the decay logits [tokens, H, dk] (from the layer's low-rank decay
 *       projection), A_h a per-head log scale, Sigmoid(x) = 1 / (1 + e^-x);
 *   output (the KDA output equation, before W_o):
 *       y = Sigmoid(out_gate) * RMSNorm(o),   per token and head over dv,
 *       RMSNorm(o)_j = o_j * norm_weight_j / sqrt(mean_j o_j^2 + norm_eps),
 *       out_gate = W_g x [tokens, H, dv].
 * The page names the RMSNorm without its weight or epsilon; here the weight
 * is one learned value per channel, shared by the heads, and eps is given.
 * The projections W_g x, W_o y and the one that makes z are plain GEMMs
 * outside these calls.
 */
typedef struct {
  const float *A_log;       /* [H] fp32 device, required                         */
  float g_min;              /* log-decay floor, in [-5, 0) (-5 on the page: the
                               kernels' range guard needs g_min >= -5)           */
  const void *out_gate;     /* [tokens, H, dv] qkv_dtype device, or NULL: out is
                               o itself (no norm, no gate)                       */
  const float *norm_weight; /* [dv] fp32 device, or NULL for ones               */
  float norm_eps;           /* >= 0 (used only with out_gate)                   */
} kda_layer_gates;

/*
 * kda_layer_fwd - kda_chunk_fwd_ex with the layer's gates: the log-decay is
 * computed in the kernels from z (so log_alpha is never materialised) and,
 * when gates->out_gate is given, each output row is normalised and gated
 * before it is stored.
 *
 *   z         [B*T, H, dk] qkv_dtype (takes log_alpha's place; desc->gate_dtype
 *             now describes beta alone)
 *   out       [B*T, H, dv] out_dtype: y, or o when out_gate is NULL
 * Other arguments and conventions as kda_chunk_fwd_ex (workspace NULL: a
 * split plan allocates its workspace stream-ordered).  z, out_gate and out are
 * 16-byte aligned, A_log and norm_weight 4-byte aligned.  Validate mode checks
 * that z has no NaN, A_log is finite and beta is in [0, 1]; g_min outside
 * [-5, 0) or a negative (or NaN) norm_eps is KDA_ERR_RANGE without validate.
 * On the tensor-core kernel the norm reads the bf16-rounded o, the value an
 * unfused norm would read from out.
 */
kda_status kda_layer_fwd(const kda_chunk_desc *desc, const kda_layer_gates *gates, const void *q,
                         const void *k, const void *v, const void *z, const void *beta,
                         const float *initial_state, const int32_t *cu_seqlens, void *out,
                         float *final_state, void *workspace, size_t workspace_bytes,
                         kda_stream_t stream);

/*
 * kda_layer_decode_step - kda_decode_step with the layer's gates:
 *   z        [N, H, dk] qkv_dtype (in log_alpha's place)
 *   out      [N, H, dv] out_dtype: y, or o when gates->out_gate is NULL
 *   gates->out_gate, when given, [N, H, dv] qkv_dtype
 * Other arguments as kda_decode_step; alignment as kda_decode_step for z and
 * out_gate, 4 bytes for A_log and norm_weight.
 */
kda_status kda_layer_decode_step(const kda_decode_desc *desc, const kda_layer_gates *gates,
                                 const void *q, const void *k, const void *v, const void *z,
                                 const void *beta, float *state_inout, void *out,
                                 kda_stream_t stream);

/*
 * Context parallelism across GPUs ([K3-notes §2.5, context-parallel affine
 * pair]): a segment of a sequence maps any entry state to
 *     S_out = S~ + M S_in,
 * S~ its final state from S_in = 0 and M (dk x dk) the product of its
 * per-token transitions (I - beta k k^T) Diag(alpha); the pairs compose.  A
 * sequence split over R GPUs runs on each rank r: kda_chunk_affine_pair on
 * its segment, an all-gather of the R pairs (fixed size, independent of the
 * segment length), kda_affine_compose for the entry states, and
 * kda_chunk_fwd on its segment from entry state r.
 *
 * kda_chunk_affine_pair - the pair of each sequence of the call (each whole
 * sequence is one segment).  Arguments as kda_chunk_fwd (no states, no out);
 *   pairs  [2][Nseq][H][dk][dv] fp32 device, written: [0] = S~, [1] = M.
 * Tensor-core arguments only (bf16 q/k/v, fp32 gates, dk = dv = 128, chunk
 * 64); KDA_ERR_UNSUPPORTED otherwise or with desc->kernel = KDA_KERNEL_SIMT.
 */
kda_status kda_chunk_affine_pair(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                                 const void *log_alpha, const void *beta, const int32_t *cu_seqlens,
                                 float *pairs, kda_stream_t stream);

/*
 * kda_affine_compose - entry states of P consecutive segments:
 *   E_0 = initial_state (NULL: zero),  E_{p+1} = S~_p + M_p E_p   (fp32)
 *   pairs         [2][N][P-1][H][dk][dv] fp32 device (S~ block, then M block;
 *                 may be NULL when P = 1)
 *   entry_states  [N][P][H][dk][dv] fp32 device, written
 * dk = dv = 128; pointers 16-byte aligned; entry_states may alias nothing.
 */
kda_status kda_affine_compose(int N, int H, int dk, int dv, int P, const float *initial_state, const float *pairs,
                              float *entry_states, kda_stream_t stream);

/*
 * kda_chunk_bwd - gradients of kda_chunk_fwd, for training (the chunkwise form
 * of [K3-notes §2.2] is the training form; the page prints no backward, and
 * this one is the exact derivative of the forward's mathematics).  For the
 * scalar L = sum_t <d_out_t, o_t> + sum_n <d_final_state_n, S_T(n)> it writes
 *
 *   dq, dk       [B*T, H, dk] fp32    dL/dq, dL/dk
 *   dv           [B*T, H, dv] fp32    dL/dv
 *   dlog_alpha   [B*T, H, dk] fp32    dL/dlog_alpha
 *   dbeta        [B*T, H]     fp32    dL/dbeta
 *   d_initial_state [Nseq, H, dk, dv] fp32, or NULL   dL/dinitial_state
 *
 * from the forward's inputs (same arguments and conventions as kda_chunk_fwd;
 * initial_state NULL = zeros) and
 *   d_out          [B*T, H, dv] out_dtype   (gradient of out)
 *   d_final_state  [Nseq, H, dk, dv] fp32, or NULL for zero.
 * The forward is recomputed inside; nothing of it needs to be kept.  The
 * gradients do not depend on desc->chunk (the backward works on 16-token
 * chunks, the tile within which the decay floor keeps every factor in fp32
 * range); desc->segments is ignored and desc->kernel = KDA_KERNEL_TC returns
 * KDA_ERR_UNSUPPORTED (the backward runs on CUDA cores, in fp32).
 *
 *   workspace  device buffer of kda_chunk_bwd_workspace_size bytes, 16-byte
 *              aligned, or NULL: then the call allocates it stream-ordered
 *              (cudaMallocAsync / cudaFreeAsync on `stream`).  It holds, per
 *              16-token chunk and head, the state before the chunk and the
 *              state gradient after it (2 dk dv floats) and 3 C dk + 2 C^2 + dk
 *              floats of chunk matrices: about 130 KB per 16 tokens per head at
 *              dk = dv = 128.
 * Gradients may alias no input and no other gradient (KDA_ERR_ALIAS); all
 * pointers 4-byte aligned except q, k, v, log_alpha, d_out (16 bytes, as the
 * forward's q/k/v/log_alpha/out).
 */
kda_status kda_chunk_bwd_workspace_size(const kda_chunk_desc *desc, size_t *bytes);
kda_status kda_chunk_bwd(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta, const float *initial_state,
                         const int32_t *cu_seqlens, const void *d_out, const float *d_final_state,
                         float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta,
                         float *d_initial_state, void *workspace, size_t workspace_bytes,
                         kda_stream_t stream);

/* Static description of a status code (never NULL). */
const char *kda_status_string(kda_status status);

/* The last CUDA error string seen by this thread's most recent failing call,
 * or "" (never NULL). */
const char *kda_last_cuda_error(void);

/* The tensor-core prefill bounds every wait on its internal barriers (2 s).
 * A wait that runs out makes the kernel abandon its work, release what it
 * holds and OR a bit into a per-device word; the outputs of that call are
 * then undefined.  This call waits for the current device to go idle
 * (cudaDeviceSynchronize), stores that word in *flags (0 = no time-out since
 * it was last cleared) and clears it when `clear` is non-zero. */
kda_status kda_device_watchdog(unsigned int *flags, int clear);

/* Size of the library's built-in scratch array used by kda_chunk_fwd_noalloc:
 * 32 MiB of device memory on every GPU that loads libkda.so, held until the
 * process exits. */
#define KDA_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * kda_chunk_fwd_noalloc - kda_chunk_fwd for callers that cannot allocate.
 * The paper has no counterpart: this is a property of the library, not of the
 * method.
 *
 * Some callers own every byte of device memory through their own allocator
 * (for example a serving process that reserves the GPU's memory in fixed pools
 * at start-up), or run in code paths where a device allocation could block on
 * or fail against memory pressure they do not control.  For them kda_chunk_fwd
 * is unusable whenever its planner splits long sequences, because it then
 * allocates a stream-ordered workspace, and kda_chunk_fwd_ex needs a buffer they
 * may have no way to provide.  This entry point takes the same arguments as
 * kda_chunk_fwd (with desc->validate = 0) and computes the same results, but
 * takes its workspace from a fixed array inside the library
 * (KDA_STATIC_WORKSPACE_BYTES); it never calls cudaMalloc, cudaMallocAsync,
 * cudaFree or any other allocating routine.  The caller still passes every
 * input and output buffer.
 *
 * - A call whose plan needs more scratch than KDA_STATIC_WORKSPACE_BYTES (see
 *   kda_chunk_fwd_workspace_size) returns KDA_ERR_SCRATCH_LIMIT before launching
 *   anything.  Validate mode needs an allocation and is refused with
 *   KDA_ERR_UNSUPPORTED.
 * - Every call looks up the array's address in the current device's context
 *   (cudaGetSymbolAddress, which allocates nothing), so the address stays
 *   right after that context is destroyed and created again.  The first call
 *   in a context may load the library's device code into it; make that first
 *   call before any stream capture.
 * - All calls in the process share the one array, and it keeps whatever the
 *   previous call left in it (every call writes all the scratch it reads, so
 *   nothing has to start at zero).  Calls whose work overlaps on the GPU (on
 *   different streams, or from different threads without ordering between
 *   them) race on that array and may return wrong results: order them.
 */
kda_status kda_chunk_fwd_noalloc(const kda_chunk_desc *desc, const void *q, const void *k,
                                 const void *v, const void *log_alpha, const void *beta,
                                 const float *initial_state, const int32_t *cu_seqlens, void *out,
                                 float *final_state, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
