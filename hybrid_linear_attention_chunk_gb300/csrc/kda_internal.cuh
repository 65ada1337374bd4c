// Internal declarations shared by the libkda.so translation units.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Log-decay floor of [K3-notes §2.2, Eq. 5] (g_min = -5).  The kernels'
// range guard relies on it: 16 tokens at the floor sum to -80, and e^80 is
// still a finite fp32/bf16 value.
constexpr float kLogDecayFloor = -5.0f;
// A chunk whose per-channel cumulative log-decay stays at or above this uses
// one decay reference for the whole chunk; below it the Gram products are
// factored per 16-token tile ([K3-notes §2.2, Fig. 3]).
constexpr float kSingleRefBound = -80.0f;

struct PrefillArgs {
  int N;        // sequences
  int T_total;  // tokens in the packed buffer
  int T_seq;    // tokens per sequence when cu_seqlens == nullptr
  int H, dk, dv, chunk;
  kda_dtype qkv, out, gate;
  const void *q, *k, *v, *g, *beta;
  const float *s0;           // nullable
  const int32_t *cu;         // nullable
  void *o;                   // nullable only for the segment passes of the long-sequence plan
  float *sT;                 // nullable
  // Long-sequence plan (tensor-core kernel only; the defaults mean one work
  // item per (sequence, head)).  Sequence n is cut into segments of
  // seg_tokens tokens (a multiple of the chunk); this launch covers segments
  // [0, nseg).  With kinds == 2 every (n, segment, h) runs twice: kind 0
  // from a zero state with v as given, kind 1 from the identity with v = 0,
  // giving the segment's affine pair (S~, M); their final states go to
  // sT[kind][n][segment][h].  With kinds == 1 segment j starts from
  // s0[n][j][h] and only the last segment writes sT[n][h].
  int seg_tokens = 0;        // 0: the whole sequence is one segment
  int nseg = 1;
  int kinds = 1;
  // Passes of the long-sequence plan (tensor-core kernel, B x T batches
  // only); plan 0 is the layout above.  Sequence n is cut into P segments:
  // segment 0 of seg0 tokens, then segments of seg_tokens.
  //   plan 1 (pass 1): one work item per (n, h) runs segment 0 from s0 with
  //     outputs and writes its final state to E[n][0][h]; then every segment
  //     1 .. P-2 runs as kind 0 (zero state, v) and kind 1 (identity, v = 0)
  //     into pairs[kind][n][segment - 1][h], without outputs.
  //   plan 2 (pass 3): segment p = 1 .. P-1 runs from E[n][p - 1][h] with
  //     outputs; the last one writes sT[n][h].
  int plan = 0;
  int P = 1;
  int seg0 = 0;
  float *pairs = nullptr;    // [2][N][P-2][H][dk][dv]
  float *E = nullptr;        // [N][P-1][H][dk][dv]: entry states of segments 1 .. P-1
  // State checkpoints (nullable ck): the state after every ck_every tokens of
  // a sequence (a multiple of the chunk) goes to slot first + j - 1 of ck
  // [slots][H][dk][dv], first = ck_cu[n] when ck_cu is given, else
  // n * (T_seq / ck_every).
  int ck_every = 0;
  const int32_t *ck_cu = nullptr;
  float *ck = nullptr;
  // KDA layer gates ([K3-notes §2.2]).  With A_log set, g holds the decay
  // logits z (dtype qkv) and the log-decay is g_min Sigmoid(exp(A_log[h]) z)
  // (Eq. 5).  With og set, every output row is Sigmoid(og) o RMSNorm(o) over
  // its dv channels, RMSNorm(x)_j = x_j nw_j / sqrt(mean x^2 + eps) (nw
  // nullable: ones).
  const float *A_log = nullptr;
  float g_min = 0.f;
  const void *og = nullptr;
  const float *nw = nullptr;
  float eps = 0.f;
  __host__ __device__ kda_dtype gdt() const { return A_log ? qkv : gate; }  // dtype of the g array
};

// Where the state of (sequence n, head h) goes once `done` tokens of the
// sequence have been processed, or nullptr when no checkpoint falls there.
__device__ __forceinline__ float *ckpt_ptr(const PrefillArgs &a, int n, int h, int done) {
  if (!a.ck || done <= 0 || done % a.ck_every != 0) return nullptr;
  const long long first = a.ck_cu ? (long long)a.ck_cu[n] : (long long)n * (a.T_seq / a.ck_every);
  return a.ck + ((size_t)(first + done / a.ck_every - 1) * a.H + h) * a.dk * a.dv;
}

struct DecodeArgs {
  int N, H, dk, dv;
  kda_dtype qkv, out, gate;
  const void *q, *k, *v, *g, *beta;
  float *state;
  void *o;
  // layer gates, as in PrefillArgs
  const float *A_log = nullptr;
  float g_min = 0.f;
  const void *og = nullptr;
  const float *nw = nullptr;
  float eps = 0.f;
  __host__ __device__ kda_dtype gdt() const { return A_log ? qkv : gate; }
};

// Eq. 5 of [K3-notes §2.2] for one element: the log-decay from its logit z,
// with scale = exp(A_h) (fp32 library exponentials).
__device__ __forceinline__ float decay_from_logit(float z, float scale, float g_min) {
  return g_min / (1.f + expf(-scale * z));
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
// In place on a.o: every (token, head) row -> Sigmoid(og) o RMSNorm(row).
cudaError_t launch_norm_gate(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_chunk_simt(const PrefillArgs &a, cudaStream_t s);
bool chunk_tc_supports(const PrefillArgs &a);
cudaError_t launch_chunk_tc(const PrefillArgs &a, cudaStream_t s);
cudaError_t read_tc_watchdog(unsigned int *flags, bool clear);

// Backward of the chunked prefill (kda_bwd.cu).  dO in the forward's out
// dtype; dST and ds0 nullable; every gradient fp32.
struct BwdIo {
  const void *dO;
  const float *dST;
  float *dq, *dk, *dv, *dg, *dbeta, *ds0;
};
int bwd_slots(const PrefillArgs &p);
size_t bwd_workspace_bytes(const PrefillArgs &p);
cudaError_t launch_chunk_bwd(const PrefillArgs &p, const BwdIo &io, void *ws, cudaStream_t s);

// Segment plan for long sequences (kda_cp.cu).
struct SegPlan {
  int P;              // segments per sequence (1: no split)
  int seg_tokens;     // tokens of segments 1 .. P-1 (a multiple of the chunk; the last may be shorter)
  size_t ws_bytes;    // device workspace: (3P - 5) x N x H fp32 dk x dv states
  int seg0;           // tokens of segment 0 (a multiple of the chunk)
};
SegPlan plan_segments(const PrefillArgs &a, int requested);
cudaError_t launch_chunk_tc_segmented(const PrefillArgs &a, const SegPlan &pl, void *ws, cudaStream_t s);
cudaError_t launch_affine_pair(const PrefillArgs &a, float *pairs, cudaStream_t s);
cudaError_t launch_affine_compose(int N, int H, int P, const float *s0, const float *pairs, float *E,
                                  cudaStream_t s);
cudaError_t launch_validate_prefill(const PrefillArgs &a, int *d_flag, cudaStream_t s);
cudaError_t launch_validate_decode(const DecodeArgs &a, int *d_flag, cudaStream_t s);

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ float ld_elem(const void *p, size_t i, kda_dtype t) {
  if (t == KDA_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  return reinterpret_cast<const float *>(p)[i];
}

// Four consecutive elements from index i (a multiple of 4; base 16-byte aligned).
__device__ __forceinline__ float4 ld4_elem(const void *p, size_t i, kda_dtype t) {
  if (t == KDA_BF16) {
    const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p) + i);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  return *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i);
}

__device__ __forceinline__ void st_elem(void *p, size_t i, float x, kda_dtype t) {
  if (t == KDA_BF16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else reinterpret_cast<float *>(p)[i] = x;
}

// Token range of sequence n.
__device__ __forceinline__ void seq_range(const PrefillArgs &a, int n, int &bos, int &eos) {
  if (a.cu) {
    bos = a.cu[n];
    eos = a.cu[n + 1];
  } else {
    bos = n * a.T_seq;
    eos = bos + a.T_seq;
  }
}

}  // namespace kda
