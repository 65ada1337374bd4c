// Host side of the C ABI declared in include/kda.h: argument checks, kernel
// choice, launch.  Every compute step runs in the kernels of the other
// translation units; nothing here touches tensor data.
#include <stdio.h>
#include <string.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

thread_local char g_last_cuda_error[256] = "";

kda_status cuda_fail(cudaError_t e) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return KDA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool aligned_to(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool dtype_ok(kda_dtype t) { return t == KDA_F32 || t == KDA_BF16; }

size_t esize(kda_dtype t) { return t == KDA_BF16 ? 2 : 4; }

struct Range {
  uintptr_t lo, hi;
};

Range span(const void *p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

// --------------------------------------------------------------- validation

// The log-decay must lie in [g_min = -5, 0]; decay logits (layer form) may be
// any number but NaN, and A_h must be finite.
template <class Args>
__device__ int check_decay(const Args &a, size_t nk, size_t stride) {
  int bad = 0;
  const kda_dtype gdt = a.gdt();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nk; i += stride) {
    const float g = ld_elem(a.g, i, gdt);
    if (a.A_log ? isnan(g) : !(g >= kLogDecayFloor && g <= 0.f)) bad |= 1;
  }
  if (a.A_log && blockIdx.x == 2)
    for (int h = threadIdx.x; h < a.H; h += blockDim.x)
      if (!isfinite(a.A_log[h])) bad |= 16;
  return bad;
}

__global__ void validate_prefill_kernel(PrefillArgs a, int *flag) {
  const size_t nk = (size_t)a.T_total * a.H * a.dk;
  const size_t nb = (size_t)a.T_total * a.H;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  int bad = check_decay(a, nk, stride);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += stride) {
    float b = ld_elem(a.beta, i, a.gate);
    if (!(b >= 0.f && b <= 1.f)) bad |= 2;
  }
  if (a.cu && blockIdx.x == 0) {
    for (int n = threadIdx.x; n <= a.N; n += blockDim.x) {
      int c = a.cu[n];
      if (n == 0 && c != 0) bad |= 4;
      if (n == a.N && c != a.T_total) bad |= 4;
      if (n > 0 && c < a.cu[n - 1]) bad |= 4;
    }
  }
  if (a.ck && a.ck_cu && blockIdx.x == 1) {  // checkpoint slots: floor(len / every) per sequence
    for (int n = threadIdx.x; n <= a.N; n += blockDim.x) {
      const int c = a.ck_cu[n];
      if (n == 0 && c != 0) bad |= 8;
      if (n > 0) {
        const int len = a.cu ? a.cu[n] - a.cu[n - 1] : a.T_seq;
        if (len >= 0 && c - a.ck_cu[n - 1] != len / a.ck_every) bad |= 8;
      }
    }
  }
  if (bad) atomicOr(flag, bad);
}

__global__ void validate_decode_kernel(DecodeArgs a, int *flag) {
  const size_t nk = (size_t)a.N * a.H * a.dk;
  const size_t nb = (size_t)a.N * a.H;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  int bad = check_decay(a, nk, stride);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += stride) {
    float b = ld_elem(a.beta, i, a.gate);
    if (!(b >= 0.f && b <= 1.f)) bad |= 2;
  }
  if (bad) atomicOr(flag, bad);
}

// Runs a check kernel, waits for it and reports KDA_ERR_RANGE on a bad value.
template <class Launch>
kda_status run_validation(cudaStream_t s, Launch launch) {
  int *d_flag = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&d_flag), sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e);
  int h_flag = 0;
  e = cudaMemsetAsync(d_flag, 0, sizeof(int), s);
  if (e == cudaSuccess) e = launch(d_flag);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h_flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost, s);
  cudaError_t ef = cudaFreeAsync(d_flag, s);
  if (e == cudaSuccess) e = ef;
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  return h_flag ? KDA_ERR_RANGE : KDA_OK;
}

// Host checks of the layer gates shared by the prefill and decode entries.
kda_status check_gates(const kda_layer_gates *lg) {
  if (!lg || !lg->A_log) return KDA_ERR_NULL;
  if (!(lg->g_min >= kLogDecayFloor && lg->g_min < 0.f)) return KDA_ERR_RANGE;
  if (lg->out_gate && !(lg->norm_eps >= 0.f)) return KDA_ERR_RANGE;
  if (lg->out_gate && !aligned16(lg->out_gate)) return KDA_ERR_ALIGN;
  if (!aligned_to(lg->A_log, 4) || (lg->norm_weight && !aligned_to(lg->norm_weight, 4))) return KDA_ERR_ALIGN;
  return KDA_OK;
}

// Spans of the gate tensors: out_gate [rows, H, dv] in qkv dtype, A_log [H],
// norm_weight [dv].
void gate_spans(const kda_layer_gates *lg, size_t rows, int H, int dv, kda_dtype qkv, Range r[3]) {
  r[0] = span(lg->out_gate, lg->out_gate ? rows * H * dv * esize(qkv) : 0);
  r[1] = span(lg->A_log, (size_t)H * 4);
  r[2] = span(lg->norm_weight, lg->norm_weight ? (size_t)dv * 4 : 0);
}

// out may be NULL only with has_out = false (calls that write no output).
kda_status check_prefill(const kda_chunk_desc *d, const void *q, const void *k, const void *v,
                         const void *g, const void *beta, const float *s0, const int32_t *cu,
                         void *out, float *sT, PrefillArgs *a, const kda_layer_gates *lg = nullptr,
                         bool has_out = true) {
  if (!d || !q || !k || !v || !g || !beta || (has_out && !out)) return KDA_ERR_NULL;
  if (!dtype_ok(d->qkv_dtype) || !dtype_ok(d->out_dtype) || !dtype_ok(d->gate_dtype))
    return KDA_ERR_DTYPE;
  if (d->H <= 0 || !dim_ok(d->dk) || !dim_ok(d->dv) || d->T < 0 || d->B <= 0) return KDA_ERR_SHAPE;
  if (!(d->chunk == 16 || d->chunk == 32 || d->chunk == 64)) return KDA_ERR_SHAPE;
  if (d->segments < 0) return KDA_ERR_SHAPE;
  if (cu) {
    if (d->B != 1 || d->num_seqs <= 0) return KDA_ERR_SHAPE;
  } else if (d->num_seqs != 0) {
    return KDA_ERR_SHAPE;
  }
  const long long T_total = cu ? (long long)d->T : (long long)d->B * d->T;
  if (T_total * d->H * (d->dk > d->dv ? d->dk : d->dv) >= (1LL << 40)) return KDA_ERR_SHAPE;
  // q, k, v, log_alpha and out are tiled with bulk copies / 16-byte vectors;
  // beta, the states and cu_seqlens only need their element alignment.
  const void *ptrs16[] = {q, k, v, g, out};
  for (const void *p : ptrs16)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  const void *ptrs4[] = {beta, s0, cu, sT};
  for (const void *p : ptrs4)
    if (p && !aligned_to(p, 4)) return KDA_ERR_ALIGN;
  const int Nseq = cu ? d->num_seqs : d->B;
  const size_t th = (size_t)T_total * d->H;
  const kda_dtype gdt = lg ? d->qkv_dtype : d->gate_dtype;  // decay logits or log-decay
  Range r_out = span(out, has_out ? th * d->dv * esize(d->out_dtype) : 0);
  if (lg) {
    kda_status st = check_gates(lg);
    if (st != KDA_OK) return st;
    Range rg[3];
    gate_spans(lg, (size_t)T_total, d->H, d->dv, d->qkv_dtype, rg);
    const Range r_sT = span(sT, sT ? (size_t)Nseq * d->H * d->dk * d->dv * 4 : 0);
    for (const Range &r : rg)
      if (overlap(r_out, r) || overlap(r_sT, r)) return KDA_ERR_ALIAS;
  }
  Range ins[] = {span(q, th * d->dk * esize(d->qkv_dtype)), span(k, th * d->dk * esize(d->qkv_dtype)),
                 span(v, th * d->dv * esize(d->qkv_dtype)), span(g, th * d->dk * esize(gdt)),
                 span(beta, th * esize(d->gate_dtype)),
                 span(s0, s0 ? (size_t)Nseq * d->H * d->dk * d->dv * 4 : 0),
                 span(cu, cu ? (size_t)(Nseq + 1) * 4 : 0),
                 span(sT, sT ? (size_t)Nseq * d->H * d->dk * d->dv * 4 : 0)};
  for (const Range &r : ins)
    if (overlap(r_out, r)) return KDA_ERR_ALIAS;
  if (sT) {
    Range r_sT = span(sT, (size_t)Nseq * d->H * d->dk * d->dv * 4);
    for (int i = 0; i < 5; ++i)
      if (overlap(r_sT, ins[i])) return KDA_ERR_ALIAS;
    if (s0 && s0 != sT && overlap(r_sT, ins[5])) return KDA_ERR_ALIAS;
  }
  a->N = Nseq;
  a->T_total = (int)T_total;
  a->T_seq = cu ? 0 : d->T;
  a->H = d->H;
  a->dk = d->dk;
  a->dv = d->dv;
  a->chunk = d->chunk;
  a->qkv = d->qkv_dtype;
  a->out = d->out_dtype;
  a->gate = d->gate_dtype;
  a->q = q; a->k = k; a->v = v; a->g = g; a->beta = beta;
  a->s0 = s0; a->cu = cu; a->o = out; a->sT = sT;
  if (lg) {
    a->A_log = lg->A_log;
    a->g_min = lg->g_min;
    a->og = lg->out_gate;
    a->nw = lg->norm_weight;
    a->eps = lg->norm_eps;
  }
  return KDA_OK;
}

// ws_mode 0: a split plan allocates its workspace stream-ordered on s;
// ws_mode 1: the caller's (ws, ws_bytes) is used.
kda_status run_prefill(const kda_chunk_desc *d, const PrefillArgs &a, cudaStream_t s, int ws_mode, void *ws,
                       size_t ws_bytes) {
  const bool tc = chunk_tc_supports(a);
  if (d->kernel == KDA_KERNEL_TC && !tc) return KDA_ERR_UNSUPPORTED;
  const bool use_tc = d->kernel != KDA_KERNEL_SIMT && tc;
  if (d->segments > 1 && (!use_tc || a.cu)) return KDA_ERR_UNSUPPORTED;
  const SegPlan pl = use_tc ? plan_segments(a, d->segments) : SegPlan{1, 0, 0, 0};
  if (pl.P > 1 && ws_mode == 1) {
    if (!ws) return KDA_ERR_NULL;
    if (ws_bytes < pl.ws_bytes) return KDA_ERR_SHAPE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
  }
  if (d->validate) {
    kda_status st = run_validation(s, [&](int *flag) { return launch_validate_prefill(a, flag, s); });
    if (st != KDA_OK) return st;
  }
  cudaError_t e;
  if (pl.P <= 1) {
    e = use_tc ? launch_chunk_tc(a, s) : launch_chunk_simt(a, s);
    // the CUDA-core kernel leaves the output norm and gate to a row pass
    if (e == cudaSuccess && !use_tc && a.og) e = launch_norm_gate(a, s);
  } else if (ws_mode == 1) {
    e = launch_chunk_tc_segmented(a, pl, ws, s);
  } else {
    void *tmp = nullptr;
    e = cudaMallocAsync(&tmp, pl.ws_bytes, s);
    if (e == cudaSuccess) {
      e = launch_chunk_tc_segmented(a, pl, tmp, s);
      cudaError_t ef = cudaFreeAsync(tmp, s);
      if (e == cudaSuccess) e = ef;
    }
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

// Arguments as far as sizes go (for the workspace query, which has no pointers).
kda_status args_from_desc(const kda_chunk_desc *d, PrefillArgs *a) {
  if (!dtype_ok(d->qkv_dtype) || !dtype_ok(d->out_dtype) || !dtype_ok(d->gate_dtype)) return KDA_ERR_DTYPE;
  if (d->H <= 0 || !dim_ok(d->dk) || !dim_ok(d->dv) || d->T < 0 || d->B <= 0) return KDA_ERR_SHAPE;
  if (!(d->chunk == 16 || d->chunk == 32 || d->chunk == 64) || d->segments < 0) return KDA_ERR_SHAPE;
  const bool varlen = d->num_seqs > 0;
  if (varlen && d->B != 1) return KDA_ERR_SHAPE;
  a->N = varlen ? d->num_seqs : d->B;
  a->T_total = varlen ? d->T : d->B * d->T;
  a->T_seq = varlen ? 0 : d->T;
  a->H = d->H; a->dk = d->dk; a->dv = d->dv; a->chunk = d->chunk;
  a->qkv = d->qkv_dtype; a->out = d->out_dtype; a->gate = d->gate_dtype;
  a->q = a->k = a->v = a->g = a->beta = nullptr;
  a->s0 = nullptr; a->o = nullptr; a->sT = nullptr;
  static const int32_t dummy = 0;
  a->cu = varlen ? &dummy : nullptr;  // only its presence matters to the planner
  return KDA_OK;
}

kda_status run_decode(const kda_decode_desc *d, const kda_layer_gates *lg, const void *q, const void *k,
                      const void *v, const void *log_alpha, const void *beta, float *state_inout, void *out,
                      kda_stream_t stream) {
  if (!d || !q || !k || !v || !log_alpha || !beta || !state_inout || !out) return KDA_ERR_NULL;
  if (!dtype_ok(d->qkv_dtype) || !dtype_ok(d->out_dtype) || !dtype_ok(d->gate_dtype))
    return KDA_ERR_DTYPE;
  if (d->N <= 0 || d->H <= 0 || !dim_ok(d->dk) || !dim_ok(d->dv)) return KDA_ERR_SHAPE;
  if ((long long)d->N * d->H >= (1LL << 31)) return KDA_ERR_SHAPE;
  // the state is streamed as 16-byte vectors; the rest needs element alignment
  if (!aligned16(state_inout)) return KDA_ERR_ALIGN;
  if (!aligned_to(q, esize(d->qkv_dtype)) || !aligned_to(k, esize(d->qkv_dtype)) ||
      !aligned_to(v, esize(d->qkv_dtype)) || !aligned_to(out, esize(d->out_dtype)) ||
      !aligned_to(log_alpha, esize(lg ? d->qkv_dtype : d->gate_dtype)) || !aligned_to(beta, esize(d->gate_dtype)))
    return KDA_ERR_ALIGN;
  const size_t nh = (size_t)d->N * d->H;
  Range r_s = span(state_inout, nh * d->dk * d->dv * 4);
  Range r_o = span(out, nh * d->dv * esize(d->out_dtype));
  Range ins[] = {span(q, nh * d->dk * esize(d->qkv_dtype)), span(k, nh * d->dk * esize(d->qkv_dtype)),
                 span(v, nh * d->dv * esize(d->qkv_dtype)),
                 span(log_alpha, nh * d->dk * esize(lg ? d->qkv_dtype : d->gate_dtype)),
                 span(beta, nh * esize(d->gate_dtype))};
  if (overlap(r_s, r_o)) return KDA_ERR_ALIAS;
  for (const Range &r : ins)
    if (overlap(r_s, r) || overlap(r_o, r)) return KDA_ERR_ALIAS;
  if (lg) {
    kda_status st = check_gates(lg);
    if (st != KDA_OK) return st;
    if (lg->out_gate && !aligned_to(lg->out_gate, esize(d->qkv_dtype))) return KDA_ERR_ALIGN;
    Range rg[3];
    gate_spans(lg, (size_t)d->N, d->H, d->dv, d->qkv_dtype, rg);
    for (const Range &r : rg)
      if (overlap(r_s, r) || overlap(r_o, r)) return KDA_ERR_ALIAS;
  }
  DecodeArgs a;
  a.N = d->N; a.H = d->H; a.dk = d->dk; a.dv = d->dv;
  a.qkv = d->qkv_dtype; a.out = d->out_dtype; a.gate = d->gate_dtype;
  a.q = q; a.k = k; a.v = v; a.g = log_alpha; a.beta = beta;
  a.state = state_inout; a.o = out;
  if (lg) {
    a.A_log = lg->A_log;
    a.g_min = lg->g_min;
    a.og = lg->out_gate;
    a.nw = lg->norm_weight;
    a.eps = lg->norm_eps;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d->validate) {
    kda_status st = run_validation(s, [&](int *flag) { return launch_validate_decode(a, flag, s); });
    if (st != KDA_OK) return st;
  }
  cudaError_t e = launch_decode(a, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

}  // namespace

cudaError_t launch_validate_prefill(const PrefillArgs &a, int *d_flag, cudaStream_t s) {
  validate_prefill_kernel<<<1024, 256, 0, s>>>(a, d_flag);
  return cudaGetLastError();
}

cudaError_t launch_validate_decode(const DecodeArgs &a, int *d_flag, cudaStream_t s) {
  validate_decode_kernel<<<256, 256, 0, s>>>(a, d_flag);
  return cudaGetLastError();
}

}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_chunk_fwd(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta, const float *initial_state,
                         const int32_t *cu_seqlens, void *out, float *final_state,
                         kda_stream_t stream) {
  PrefillArgs a;
  kda_status st = check_prefill(desc, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                                final_state, &a);
  if (st != KDA_OK) return st;
  return run_prefill(desc, a, reinterpret_cast<cudaStream_t>(stream), 0, nullptr, 0);
}

kda_status kda_chunk_fwd_workspace_size(const kda_chunk_desc *desc, size_t *bytes) {
  if (!desc || !bytes) return KDA_ERR_NULL;
  *bytes = 0;
  PrefillArgs a;
  kda_status st = args_from_desc(desc, &a);
  if (st != KDA_OK) return st;
  const bool tc = chunk_tc_supports(a);
  if (desc->kernel == KDA_KERNEL_TC && !tc) return KDA_ERR_UNSUPPORTED;
  const bool use_tc = desc->kernel != KDA_KERNEL_SIMT && tc;
  if (desc->segments > 1 && (!use_tc || a.cu)) return KDA_ERR_UNSUPPORTED;
  if (use_tc) *bytes = plan_segments(a, desc->segments).ws_bytes;
  return KDA_OK;
}

kda_status kda_chunk_fwd_ex(const kda_chunk_desc *desc, const void *q, const void *k,
                            const void *v, const void *log_alpha, const void *beta,
                            const float *initial_state, const int32_t *cu_seqlens, void *out,
                            float *final_state, void *workspace, size_t workspace_bytes,
                            kda_stream_t stream) {
  PrefillArgs a;
  kda_status st = check_prefill(desc, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                                final_state, &a);
  if (st != KDA_OK) return st;
  return run_prefill(desc, a, reinterpret_cast<cudaStream_t>(stream), 1, workspace, workspace_bytes);
}

kda_status kda_chunk_fwd_ckpt(const kda_chunk_desc *desc, const void *q, const void *k,
                              const void *v, const void *log_alpha, const void *beta,
                              const float *initial_state, const int32_t *cu_seqlens, void *out,
                              float *final_state, int every, const int32_t *cu_ckpt, float *ckpt,
                              void *workspace, size_t workspace_bytes, kda_stream_t stream) {
  PrefillArgs a;
  kda_status st = check_prefill(desc, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                                final_state, &a);
  if (st != KDA_OK) return st;
  if (!ckpt || (cu_seqlens && !cu_ckpt)) return KDA_ERR_NULL;
  if (every <= 0 || every % desc->chunk != 0) return KDA_ERR_SHAPE;
  if (!aligned_to(ckpt, 4) || (cu_ckpt && !aligned_to(cu_ckpt, 4))) return KDA_ERR_ALIGN;
  // the checkpoints may alias nothing the call reads or writes (their count is
  // known on the host only for a B x T batch)
  const size_t state = (size_t)desc->H * desc->dk * desc->dv * 4;
  const size_t slots = cu_seqlens ? 1 : (size_t)a.N * (size_t)(desc->T / every);
  const size_t th = (size_t)a.T_total * desc->H;
  Range r_ck = span(ckpt, slots * state);
  Range others[] = {span(q, th * desc->dk * esize(desc->qkv_dtype)),
                    span(k, th * desc->dk * esize(desc->qkv_dtype)),
                    span(v, th * desc->dv * esize(desc->qkv_dtype)),
                    span(log_alpha, th * desc->dk * esize(desc->gate_dtype)),
                    span(beta, th * esize(desc->gate_dtype)),
                    span(out, th * desc->dv * esize(desc->out_dtype)),
                    span(initial_state, initial_state ? (size_t)a.N * state : 0),
                    span(final_state, final_state ? (size_t)a.N * state : 0),
                    span(cu_seqlens, cu_seqlens ? (size_t)(a.N + 1) * 4 : 0),
                    span(cu_ckpt, cu_ckpt ? (size_t)(a.N + 1) * 4 : 0)};
  for (const Range &r : others)
    if (overlap(r_ck, r)) return KDA_ERR_ALIAS;
  a.ck_every = every;
  a.ck_cu = cu_ckpt;
  a.ck = ckpt;
  return run_prefill(desc, a, reinterpret_cast<cudaStream_t>(stream), workspace ? 1 : 0, workspace,
                     workspace_bytes);
}


kda_status kda_decode_step(const kda_decode_desc *d, const void *q, const void *k, const void *v,
                           const void *log_alpha, const void *beta, float *state_inout, void *out,
                           kda_stream_t stream) {
  return run_decode(d, nullptr, q, k, v, log_alpha, beta, state_inout, out, stream);
}

kda_status kda_layer_decode_step(const kda_decode_desc *desc, const kda_layer_gates *gates,
                                 const void *q, const void *k, const void *v, const void *z,
                                 const void *beta, float *state_inout, void *out,
                                 kda_stream_t stream) {
  if (!gates) return KDA_ERR_NULL;
  return run_decode(desc, gates, q, k, v, z, beta, state_inout, out, stream);
}

kda_status kda_layer_fwd(const kda_chunk_desc *desc, const kda_layer_gates *gates, const void *q,
                         const void *k, const void *v, const void *z, const void *beta,
                         const float *initial_state, const int32_t *cu_seqlens, void *out,
                         float *final_state, void *workspace, size_t workspace_bytes,
                         kda_stream_t stream) {
  if (!gates) return KDA_ERR_NULL;
  PrefillArgs a;
  kda_status st = check_prefill(desc, q, k, v, z, beta, initial_state, cu_seqlens, out, final_state, &a, gates);
  if (st != KDA_OK) return st;
  return run_prefill(desc, a, reinterpret_cast<cudaStream_t>(stream), workspace ? 1 : 0, workspace,
                     workspace_bytes);
}

kda_status kda_chunk_affine_pair(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                                 const void *log_alpha, const void *beta, const int32_t *cu_seqlens,
                                 float *pairs, kda_stream_t stream) {
  PrefillArgs a;
  if (!pairs) return KDA_ERR_NULL;
  kda_status st = check_prefill(desc, q, k, v, log_alpha, beta, nullptr, cu_seqlens, nullptr, nullptr, &a,
                                nullptr, false);
  if (st != KDA_OK) return st;
  if (!chunk_tc_supports(a) || desc->kernel == KDA_KERNEL_SIMT) return KDA_ERR_UNSUPPORTED;
  const size_t bytes = (size_t)2 * a.N * a.H * a.dk * a.dv * 4;
  const Range r_p = span(pairs, bytes);
  const Range ins[] = {span(q, (size_t)a.T_total * a.H * a.dk * 2), span(k, (size_t)a.T_total * a.H * a.dk * 2),
                       span(v, (size_t)a.T_total * a.H * a.dv * 2), span(log_alpha, (size_t)a.T_total * a.H * a.dk * 4),
                       span(beta, (size_t)a.T_total * a.H * 4),
                       span(cu_seqlens, cu_seqlens ? (size_t)(a.N + 1) * 4 : 0)};
  for (const Range &r : ins)
    if (overlap(r_p, r)) return KDA_ERR_ALIAS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (desc->validate) {
    st = run_validation(s, [&](int *flag) { return launch_validate_prefill(a, flag, s); });
    if (st != KDA_OK) return st;
  }
  if (!aligned16(pairs)) return KDA_ERR_ALIGN;
  cudaError_t e = launch_affine_pair(a, pairs, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

kda_status kda_affine_compose(int N, int H, int dk, int dv, int P, const float *initial_state, const float *pairs,
                              float *entry_states, kda_stream_t stream) {
  if (!entry_states || (P > 1 && !pairs)) return KDA_ERR_NULL;
  if (N < 0 || H <= 0 || P <= 0 || dk != 128 || dv != 128) return KDA_ERR_SHAPE;
  const void *ptrs[] = {initial_state, pairs, entry_states};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  const size_t DD = (size_t)dk * dv * 4;
  const Range r_e = span(entry_states, (size_t)N * P * H * DD);
  if (overlap(r_e, span(pairs, pairs ? (size_t)2 * N * (P - 1) * H * DD : 0)) ||
      overlap(r_e, span(initial_state, initial_state ? (size_t)N * H * DD : 0)))
    return KDA_ERR_ALIAS;
  cudaError_t e = launch_affine_compose(N, H, P, initial_state, pairs, entry_states,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

kda_status kda_chunk_bwd_workspace_size(const kda_chunk_desc *desc, size_t *bytes) {
  if (!desc || !bytes) return KDA_ERR_NULL;
  *bytes = 0;
  PrefillArgs a;
  kda_status st = args_from_desc(desc, &a);
  if (st != KDA_OK) return st;
  *bytes = bwd_workspace_bytes(a);
  return KDA_OK;
}

kda_status kda_chunk_bwd(const kda_chunk_desc *desc, const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta, const float *initial_state,
                         const int32_t *cu_seqlens, const void *d_out, const float *d_final_state,
                         float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta,
                         float *d_initial_state, void *workspace, size_t workspace_bytes,
                         kda_stream_t stream) {
  PrefillArgs a;
  // the forward's checks, with d_out in out's place (same shape and dtype)
  kda_status st = check_prefill(desc, q, k, v, log_alpha, beta, initial_state, cu_seqlens,
                                const_cast<void *>(d_out), nullptr, &a);
  if (st != KDA_OK) return st;
  if (desc->kernel == KDA_KERNEL_TC) return KDA_ERR_UNSUPPORTED;  // one CUDA-core implementation
  if (!dq || !dk || !dv || !dlog_alpha || !dbeta) return KDA_ERR_NULL;
  float *outs[] = {dq, dk, dv, dlog_alpha, dbeta, d_initial_state};
  for (float *p : outs)
    if (p && !aligned_to(p, 4)) return KDA_ERR_ALIGN;
  if (d_final_state && !aligned_to(d_final_state, 4)) return KDA_ERR_ALIGN;
  const size_t th = (size_t)a.T_total * a.H, state = (size_t)a.N * a.H * a.dk * a.dv * 4;
  const Range r_out[] = {span(dq, th * a.dk * 4), span(dk, th * a.dk * 4), span(dv, th * a.dv * 4),
                         span(dlog_alpha, th * a.dk * 4), span(dbeta, th * 4),
                         span(d_initial_state, d_initial_state ? state : 0)};
  const Range r_in[] = {span(q, th * a.dk * esize(a.qkv)), span(k, th * a.dk * esize(a.qkv)),
                        span(v, th * a.dv * esize(a.qkv)), span(log_alpha, th * a.dk * esize(a.gate)),
                        span(beta, th * esize(a.gate)), span(initial_state, initial_state ? state : 0),
                        span(cu_seqlens, cu_seqlens ? (size_t)(a.N + 1) * 4 : 0),
                        span(d_out, th * a.dv * esize(a.out)), span(d_final_state, d_final_state ? state : 0)};
  for (int i = 0; i < 6; ++i) {
    for (const Range &r : r_in)
      if (overlap(r_out[i], r)) return KDA_ERR_ALIAS;
    for (int j = i + 1; j < 6; ++j)
      if (overlap(r_out[i], r_out[j])) return KDA_ERR_ALIAS;
  }
  const size_t need = bwd_workspace_bytes(a);
  if (workspace) {
    if (workspace_bytes < need) return KDA_ERR_SHAPE;
    if (!aligned16(workspace)) return KDA_ERR_ALIGN;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (desc->validate) {
    st = run_validation(s, [&](int *flag) { return launch_validate_prefill(a, flag, s); });
    if (st != KDA_OK) return st;
  }
  BwdIo io{d_out, d_final_state, dq, dk, dv, dlog_alpha, dbeta, d_initial_state};
  cudaError_t e;
  if (workspace || need == 0) {
    e = launch_chunk_bwd(a, io, workspace, s);
  } else {
    void *tmp = nullptr;
    e = cudaMallocAsync(&tmp, need, s);
    if (e == cudaSuccess) {
      e = launch_chunk_bwd(a, io, tmp, s);
      cudaError_t ef = cudaFreeAsync(tmp, s);
      if (e == cudaSuccess) e = ef;
    }
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "unsupported or inconsistent size";
    case KDA_ERR_DTYPE: return "unsupported dtype";
    case KDA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KDA_ERR_RANGE: return "input value outside its range (validate mode)";
    case KDA_ERR_CUDA: return "CUDA error (see kda_last_cuda_error)";
    case KDA_ERR_UNSUPPORTED: return "the requested kernel does not cover these arguments";
    case KDA_ERR_ALIAS: return "forbidden aliasing between arguments";
    case KDA_ERR_SCRATCH_LIMIT: return "the call needs more scratch than the library's static array";
  }
  return "unknown status";
}

const char *kda_last_cuda_error(void) { return g_last_cuda_error; }

kda_status kda_device_watchdog(unsigned int *flags, int clear) {
  if (!flags) return KDA_ERR_NULL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = read_tc_watchdog(flags, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e);
  return KDA_OK;
}

}  // extern "C"
