// Decode step: one token of the KDA recurrence per (sequence, head), state
// updated in place.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
//
// [K3-notes §2.2, KDA state recurrence] for one token, expanded so that the
// state is read once and written once:
//     a = exp(g),   x = S^T (a o k),   y = S^T (a o q)
//     u = beta (v - x)
//     S' = Diag(a) S + k u^T                (= (I - b k k^T) Diag(a) S + b k v^T)
//     o  = S'^T q = y + u (k . q)
// In the layer form ([K3-notes §2.2]) alpha comes from the decay logits z,
// g = g_min Sigmoid(exp(A_h) z) (Eq. 5), and the output row is normalised over
// dv and gated, Sigmoid(out_gate) o RMSNorm(o), before it is stored.
// The step is bound by HBM: 2 x dk x dv x 4 bytes of state per head against
// ~7 dk dv flops, so the kernel is a streaming read-modify-write with the
// state held in registers between the read and the write, column sums over
// dk reduced across warps through shared memory, and no tensor cores.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;  // 8 warps; warp w owns state rows [16w, 16w+16)

// dk = dv = 128: lane l owns columns [4l, 4l+4) as one float4 per row.
__global__ void __launch_bounds__(kDecThreads, 2)
decode_d128_kernel(DecodeArgs a) {
  constexpr int D = 128;
  const int nh = blockIdx.x;  // n * H + h
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float s_ak[D], s_aq[D], s_k[D], s_a[D];
  __shared__ float4 s_x[8][32], s_y[8][32];
  __shared__ float s_u[D];
  __shared__ float s_kq;
  __shared__ float s_ss[4];

  float4 *S = reinterpret_cast<float4 *>(a.state + (size_t)nh * D * D);
  float4 reg[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) reg[r] = __ldcs(S + (size_t)(16 * warp + r) * (D / 4) + lane);

  const size_t base = (size_t)nh * D;
  const float ogv = (a.og && tid < D) ? ld_elem(a.og, base + tid, a.qkv) : 0.f;
  if (tid < D) {
    float g = ld_elem(a.g, base + tid, a.gdt());
    if (a.A_log) g = decay_from_logit(g, expf(a.A_log[nh % a.H]), a.g_min);
    float al = expf(g);
    float kk = ld_elem(a.k, base + tid, a.qkv);
    float qq = ld_elem(a.q, base + tid, a.qkv);
    s_a[tid] = al;
    s_k[tid] = kk;
    s_ak[tid] = al * kk;
    s_aq[tid] = al * qq;
  }
  if (warp == 0) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int i = lane * 4 + c;
      acc += ld_elem(a.k, base + i, a.qkv) * ld_elem(a.q, base + i, a.qkv);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) s_kq = acc;
  }
  __syncthreads();

  float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int i = 16 * warp + r;
    const float ak = s_ak[i], aq = s_aq[i];
    x.x += reg[r].x * ak; x.y += reg[r].y * ak; x.z += reg[r].z * ak; x.w += reg[r].w * ak;
    y.x += reg[r].x * aq; y.y += reg[r].y * aq; y.z += reg[r].z * aq; y.w += reg[r].w * aq;
  }
  s_x[warp][lane] = x;
  s_y[warp][lane] = y;
  __syncthreads();

  float o_val = 0.f;
  if (tid < D) {
    const int l = tid >> 2, c = tid & 3;
    float X = 0.f, Y = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      X += reinterpret_cast<const float *>(&s_x[w][l])[c];
      Y += reinterpret_cast<const float *>(&s_y[w][l])[c];
    }
    const float b = ld_elem(a.beta, (size_t)nh, a.gate);
    const float u = b * (ld_elem(a.v, base + tid, a.qkv) - X);
    s_u[tid] = u;
    o_val = Y + u * s_kq;
    if (!a.og) st_elem(a.o, base + tid, o_val, a.out);
  }
  if (a.og) {  // the row's sum of squares: warps 0-3 hold its 128 channels
    float ss = o_val * o_val;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0 && warp < 4) s_ss[warp] = ss;
  }
  __syncthreads();
  if (a.og && tid < D) {
    const float r = rsqrtf((s_ss[0] + s_ss[1] + s_ss[2] + s_ss[3]) * (1.f / D) + a.eps);
    st_elem(a.o, base + tid, o_val * r * (a.nw ? a.nw[tid] : 1.f) * sigmoid_f(ogv), a.out);
  }

  const float4 u4 = reinterpret_cast<const float4 *>(s_u)[lane];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int i = 16 * warp + r;
    const float al = s_a[i], kk = s_k[i];
    float4 s = reg[r];
    s.x = al * s.x + kk * u4.x;
    s.y = al * s.y + kk * u4.y;
    s.z = al * s.z + kk * u4.z;
    s.w = al * s.w + kk * u4.w;
    __stcs(S + (size_t)i * (D / 4) + lane, s);
  }
}

// dk = dv = 128, no output gate: one CTA per (sequence, head, half of the
// state's columns).  The columns are independent in this update (x, y, u, o
// and the new column depend only on their own column and on k, q, alpha,
// beta), so a head splits into two CTAs of 128 threads that each stream
// 32 KB of state; four of them share an SM and overlap one another's load and
// store phases.  Warp w owns rows [32w, 32w+32), lane l columns
// [64 half + 2l, 64 half + 2l + 2).
constexpr int kHalfThreads = 128;

__global__ void __launch_bounds__(kHalfThreads, 4)
decode_d128_half_kernel(DecodeArgs a) {
  constexpr int D = 128;
  const int nh = blockIdx.x >> 1, c0 = 64 * (blockIdx.x & 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float s_ak[D], s_aq[D], s_k[D], s_a[D];
  __shared__ float2 s_x[4][32], s_y[4][32];
  __shared__ __align__(16) float s_u[64];
  __shared__ float s_kq[4];

  float2 *S = reinterpret_cast<float2 *>(a.state + (size_t)nh * D * D + c0);
  float2 reg[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) reg[r] = __ldcs(S + (size_t)(32 * warp + r) * (D / 2) + lane);

  const size_t base = (size_t)nh * D;
  float kk = 0.f, qq = 0.f;
  {  // thread t handles channel t
    float g = ld_elem(a.g, base + tid, a.gdt());
    if (a.A_log) g = decay_from_logit(g, expf(a.A_log[nh % a.H]), a.g_min);
    const float al = expf(g);
    kk = ld_elem(a.k, base + tid, a.qkv);
    qq = ld_elem(a.q, base + tid, a.qkv);
    s_a[tid] = al;
    s_k[tid] = kk;
    s_ak[tid] = al * kk;
    s_aq[tid] = al * qq;
  }
  float kq = kk * qq;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
  if (lane == 0) s_kq[warp] = kq;
  __syncthreads();

  float2 x = make_float2(0.f, 0.f), y = x;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int i = 32 * warp + r;
    const float ak = s_ak[i], aq = s_aq[i];
    x.x += reg[r].x * ak; x.y += reg[r].y * ak;
    y.x += reg[r].x * aq; y.y += reg[r].y * aq;
  }
  s_x[warp][lane] = x;
  s_y[warp][lane] = y;
  __syncthreads();

  if (tid < 64) {  // column c0 + tid
    const int l = tid >> 1, c = tid & 1;
    float X = 0.f, Y = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      X += c ? s_x[w][l].y : s_x[w][l].x;
      Y += c ? s_y[w][l].y : s_y[w][l].x;
    }
    const float b = ld_elem(a.beta, (size_t)nh, a.gate);
    const float u = b * (ld_elem(a.v, base + c0 + tid, a.qkv) - X);
    s_u[tid] = u;
    st_elem(a.o, base + c0 + tid, Y + u * (s_kq[0] + s_kq[1] + s_kq[2] + s_kq[3]), a.out);
  }
  __syncthreads();

  const float2 u2 = reinterpret_cast<const float2 *>(s_u)[lane];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int i = 32 * warp + r;
    const float al = s_a[i], kv = s_k[i];
    float2 sv = reg[r];
    sv.x = al * sv.x + kv * u2.x;
    sv.y = al * sv.y + kv * u2.y;
    __stcs(S + (size_t)i * (D / 2) + lane, sv);
  }
}

// Any supported dk, dv (<= 128): thread j owns state column j and walks the
// rows twice (the second read mostly hits L1/L2).
__global__ void __launch_bounds__(128)
decode_generic_kernel(DecodeArgs a) {
  const int nh = blockIdx.x;
  const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
  __shared__ float s_a[128], s_k[128], s_q[128];
  __shared__ float s_part[4], s_ss[4];
  const size_t bk = (size_t)nh * dk, bv = (size_t)nh * dv;
  float kq = 0.f;
  if (tid < dk) {
    float g = ld_elem(a.g, bk + tid, a.gdt());
    if (a.A_log) g = decay_from_logit(g, expf(a.A_log[nh % a.H]), a.g_min);
    float al = expf(g);
    float kk = ld_elem(a.k, bk + tid, a.qkv), qq = ld_elem(a.q, bk + tid, a.qkv);
    s_a[tid] = al;
    s_k[tid] = kk;
    s_q[tid] = qq;
    kq = kk * qq;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
  if ((tid & 31) == 0) s_part[tid >> 5] = kq;
  __syncthreads();
  kq = s_part[0] + s_part[1] + s_part[2] + s_part[3];
  const bool act = tid < dv;
  float *S = a.state + (size_t)nh * dk * dv;
  float u = 0.f, o_val = 0.f;
  if (act) {
    float x = 0.f, y = 0.f;
    for (int i = 0; i < dk; ++i) {
      float s = S[(size_t)i * dv + tid];
      x += s * s_a[i] * s_k[i];
      y += s * s_a[i] * s_q[i];
    }
    u = ld_elem(a.beta, (size_t)nh, a.gate) * (ld_elem(a.v, bv + tid, a.qkv) - x);
    o_val = y + u * kq;
    if (!a.og) st_elem(a.o, bv + tid, o_val, a.out);
  }
  if (a.og) {  // RMSNorm over the dv outputs, then the gate
    float ss = o_val * o_val;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) s_ss[tid >> 5] = ss;
    __syncthreads();
    if (act) {
      const float r = rsqrtf((s_ss[0] + s_ss[1] + s_ss[2] + s_ss[3]) / (float)dv + a.eps);
      st_elem(a.o, bv + tid, o_val * r * (a.nw ? a.nw[tid] : 1.f) * sigmoid_f(ld_elem(a.og, bv + tid, a.qkv)),
              a.out);
    }
  }
  if (!act) return;
  for (int i = 0; i < dk; ++i) {
    float *p = S + (size_t)i * dv + tid;
    *p = s_a[i] * *p + s_k[i] * u;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
  const int blocks = a.N * a.H;
  if (blocks == 0) return cudaSuccess;
  if (a.dk == 128 && a.dv == 128 && !a.og) {
    decode_d128_half_kernel<<<2 * blocks, kHalfThreads, 0, s>>>(a);
  } else if (a.dk == 128 && a.dv == 128) {
    decode_d128_kernel<<<blocks, kDecThreads, 0, s>>>(a);
  } else {
    decode_generic_kernel<<<blocks, 128, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kda
