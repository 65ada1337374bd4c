// Backward of the chunked KDA prefill: gradients of
//   L = sum_t <dO_t, o_t> + <dS_T, S_T>
// with respect to q, k, v, the log-decay, beta and the initial state.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.  [K3-notes §2.2]
// gives the chunkwise form and says it serves training; it prints no
// backward.  The one here differentiates the chunk form (per chunk of C
// tokens, G the within-chunk cumulative log-decay, Gamma = exp(G), gamma =
// exp(G_last)):
//   Qb = Q o Gamma, Kb = K / Gamma, GK = Gamma o K, Kh = K o gamma / Gamma
//   A = Tril_incl(Qb Kb^T),  M = GK Kb^T,  L = StrictTril(diag(beta) M),  T = (I + L)^-1
//   T_b = T diag(beta),  P = V - GK S,  V~ = T_b P  (= U - W S, W = T_b GK)
//   O = Qb S + A V~,  S' = diag(gamma) S + Kh^T V~
// in reverse, given dO and dS' (the gradient after the chunk):
//   dV~ = Kh dS' + A^T dO,  dV = T_b^T dV~,  dS = diag(gamma) dS' + Qb^T dO - W^T dV~
//   dQb = dO S^T + dA Kb,  dA = Tril_incl(dO V~^T),  dKh = V~ dS'^T,  dgamma = rowsum(dS' o S)
//   dT_b = dV~ P^T,  dbeta_s = sum_r dT_b[r,s] T[r,s] + sum_{s'<s} dL[s,s'] M[s,s']
//   dL = StrictTril(-T^T (dT_b diag(beta)) T^T),  dM = diag(beta) dL
//   dGK = -dV S^T + dM Kb,  dKb = dM^T GK + dA^T Qb
//   dq = dQb o Gamma,  dk = dKb / Gamma + dGK o Gamma + dKh o gamma / Gamma
//   dG = dQb o Qb - dKb o Kb + dGK o GK - dKh o Kh,  dG_last += colsum(dKh o Kh) + dgamma o gamma
//   dg = reverse cumulative sum of dG over the chunk's rows.
// The chunk is C = 16 tokens: by the decay floor of [K3-notes §2.2, Eq. 5]
// a 16-token tile sums to >= -80, so the chunk start serves as the one decay
// reference for every tile ([K3-notes §2.2, Fig. 3]) and all factors stay
// within e^{+-80} in fp32.
//
// Four launches, fp32 on CUDA cores:
//   bwd_prep   (every chunk in parallel)  Qb, Kh, W, A, T_b, gamma of each chunk
//   bwd_scan<forward>  (per sequence, head, 32 dv columns)  the entry state of every chunk
//   bwd_scan<reverse>  (same, last chunk first)  the state gradient after every chunk; dS_0
//   bwd_grads  (every chunk in parallel)  dq, dk, dv, dg, dbeta of the chunk's rows
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kBC = 16;       // tokens per backward chunk
constexpr int kBThreads = 256;
constexpr int kScanDvt = 32;  // state columns per scan CTA
constexpr int kGradDvt = 16;  // state columns per pass of the gradient kernel
static_assert(kBThreads == kBC * kBC && kBThreads == kBC * kGradDvt, "one thread per C x C and C x pass element");
static_assert(kBThreads == 2 * 128 && kBC == 16, "gradient tail: one channel and eight rows per thread");
static_assert(kBC * 128 / 4 <= 2 * kBThreads, "chunk loads: at most two 4-channel pieces per thread");

struct BwdArgs {
  int N, T_total, T_seq, H, dk, dv;
  kda_dtype qkv, out, gate;
  const void *q, *k, *v, *g, *beta;
  const float *s0;     // nullable
  const int32_t *cu;   // nullable: B x T batch
  const void *dO;      // out dtype
  const float *dST;    // nullable
  float *gq, *gk, *gv, *gg, *gbeta, *gs0;  // dq, dk, dv, dg, dbeta, dS_0 (gs0 nullable)
  int nslots;          // chunk slots (see slot_base)
  // workspace, per (slot, head)
  float *Qb, *Kh, *W;  // [nslots * H][C][dk]
  float *A, *Tb;       // [nslots * H][C][C]: A and T_b = T diag(beta)
  float *gam;          // [nslots * H][dk]
  float *Sent, *dSx;   // [nslots * H][dk][dv]: state before / state gradient after the chunk
};

__device__ __forceinline__ void bounds(const BwdArgs &a, int n, int &bos, int &eos) {
  if (a.cu) {
    bos = a.cu[n];
    eos = a.cu[n + 1];
  } else {
    bos = n * a.T_seq;
    eos = bos + a.T_seq;
  }
}

// First chunk slot of sequence n: floor(cu[n] / C) + n for packed sequences
// (strictly increasing, and sequence n's ceil(len / C) chunks fit before the
// next base), n * ceil(T / C) for a batch.
__device__ __forceinline__ int slot_base(const BwdArgs &a, int n) {
  return a.cu ? a.cu[n] / kBC + n : n * ((a.T_seq + kBC - 1) / kBC);
}

// (sequence, chunk) held by a slot; false for a slot between sequences.
__device__ bool locate(const BwdArgs &a, int slot, int &n, int &j) {
  if (a.N <= 0) return false;
  if (!a.cu) {
    const int per = (a.T_seq + kBC - 1) / kBC;
    if (per == 0) return false;
    n = slot / per;
    j = slot % per;
    return n < a.N;
  }
  int lo = 0, hi = a.N - 1;  // the last n with slot_base(n) <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(a, mid) <= slot) lo = mid;
    else hi = mid - 1;
  }
  n = lo;
  j = slot - slot_base(a, n);
  const int len = a.cu[n + 1] - a.cu[n];
  return j >= 0 && j < (len + kBC - 1) / kBC;
}

// 16-byte asynchronous global -> shared copies (zero-filled past src_bytes).
// Unlike a load into registers, a copy in flight does not hold up a barrier.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ------------------------------------------------------------- chunk setup

// Shared-memory arrays of one chunk (row stride ld = dk + 4 for [C][dk]).
struct ChunkSm {
  int ld;
  float *G, *Qb, *Kb, *GK, *Kh;  // [C][ld]
  float *A, *M, *T;              // [C][C]
  float *beta, *gam;             // [C], [dk]
};

__device__ __forceinline__ float *carve_chunk(ChunkSm &c, float *p, int dk) {
  c.ld = dk + 4;  // 16-byte rows
  c.G = p;  p += kBC * c.ld;
  c.Qb = p; p += kBC * c.ld;
  c.Kb = p; p += kBC * c.ld;
  c.GK = p; p += kBC * c.ld;
  c.Kh = p; p += kBC * c.ld;
  c.A = p;  p += kBC * kBC;
  c.M = p;  p += kBC * kBC;
  c.T = p;  p += kBC * kBC;
  c.beta = p; p += kBC;
  c.gam = p;  p += 128;
  return p;
}

// Loads the chunk's rows [t0, t0 + len) of head h (rows past len are the
// identity step: q = k = 0, g = 0, beta = 0) and forms G, Qb, Kb, GK, Kh,
// gamma, A, M and T = (I + L)^-1.  Ends with a barrier.
__device__ void setup_chunk(const BwdArgs &a, const ChunkSm &c, int t0, int len, int h) {
  const int dk = a.dk, H = a.H, ld = c.ld, tid = threadIdx.x;
  {  // q, k and the log-decay in 4-channel pieces (at most two per thread), all loads issued first
    const int q4 = dk / 4;
    float4 qv[2], kv[2], gv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = tid + u * kBThreads, r = e / q4;
      qv[u] = kv[u] = gv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < kBC * q4 && r < len) {
        const size_t idx = ((size_t)(t0 + r) * H + h) * dk + 4 * (e % q4);
        qv[u] = ld4_elem(a.q, idx, a.qkv);
        kv[u] = ld4_elem(a.k, idx, a.qkv);
        gv[u] = ld4_elem(a.g, idx, a.gate);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = tid + u * kBThreads;
      if (e < kBC * q4) {
        const int o = (e / q4) * ld + 4 * (e % q4);
        *reinterpret_cast<float4 *>(c.Qb + o) = qv[u];
        *reinterpret_cast<float4 *>(c.Kb + o) = kv[u];
        *reinterpret_cast<float4 *>(c.G + o) = gv[u];
      }
    }
  }
  if (tid < kBC) c.beta[tid] = tid < len ? ld_elem(a.beta, (size_t)(t0 + tid) * H + h, a.gate) : 0.f;
  __syncthreads();
  if (tid < dk) {  // within-chunk cumulative log-decay, per channel
    float acc = 0.f;
    for (int r = 0; r < kBC; ++r) {
      acc += c.G[r * ld + tid];
      c.G[r * ld + tid] = acc;
    }
    c.gam[tid] = expf(acc);
  }
  __syncthreads();
  for (int e = tid; e < kBC * dk; e += kBThreads) {
    const int r = e / dk, i = e % dk;
    const float G = c.G[r * ld + i], Gl = c.G[(kBC - 1) * ld + i];
    const float kv = c.Kb[r * ld + i];
    const float eg = expf(G);
    c.Qb[r * ld + i] *= eg;
    c.GK[r * ld + i] = kv * eg;
    c.Kb[r * ld + i] = kv * expf(-G);
    c.Kh[r * ld + i] = kv * expf(Gl - G);
  }
  __syncthreads();
  {  // one thread per (r, s): A and M, four channels per 128-bit load
    const int r = tid / kBC, s = tid % kBC;
    float accA = 0.f, accM = 0.f;
    if (s <= r) {
      const float *qr = c.Qb + r * ld, *gr = c.GK + r * ld, *ks = c.Kb + s * ld;
      for (int i = 0; i < dk; i += 4) {
        const float4 kb = *reinterpret_cast<const float4 *>(ks + i);
        const float4 qb = *reinterpret_cast<const float4 *>(qr + i);
        const float4 gk = *reinterpret_cast<const float4 *>(gr + i);
        accA = fmaf(qb.x, kb.x, fmaf(qb.y, kb.y, fmaf(qb.z, kb.z, fmaf(qb.w, kb.w, accA))));
        accM = fmaf(gk.x, kb.x, fmaf(gk.y, kb.y, fmaf(gk.z, kb.z, fmaf(gk.w, kb.w, accM))));
      }
    }
    c.A[tid] = accA;
    c.M[tid] = s < r ? accM : 0.f;
  }
  __syncthreads();
  if (tid < kBC) {  // T = (I + L)^-1, L = diag(beta) M: one column per thread, held in registers
    // (I + L) T = I row by row: T[r][s] = [r == s] - beta_r sum_{m<r} M[r][m] T[m][s]
    const int s = tid;
    float t[kBC];
#pragma unroll
    for (int r = 0; r < kBC; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m) acc += c.M[r * kBC + m] * t[m];
      t[r] = r == s ? 1.f : (r > s ? -c.beta[r] * acc : 0.f);
    }
#pragma unroll
    for (int r = 0; r < kBC; ++r) c.T[r * kBC + s] = t[r];
  }
  __syncthreads();
}

// ------------------------------------------------------------------ kernels

__global__ void __launch_bounds__(kBThreads) bwd_prep_kernel(BwdArgs a) {
  extern __shared__ float smem[];
  const int slot = blockIdx.x, h = blockIdx.y;
  int n, j;
  if (!locate(a, slot, n, j)) return;
  int bos, eos;
  bounds(a, n, bos, eos);
  const int t0 = bos + j * kBC, len = min(kBC, eos - t0);
  ChunkSm c;
  carve_chunk(c, smem, a.dk);
  setup_chunk(a, c, t0, len, h);
  const int dk = a.dk, ld = c.ld;
  const size_t sh = (size_t)slot * a.H + h;
  float *Qb = a.Qb + sh * kBC * dk, *Kh = a.Kh + sh * kBC * dk, *W = a.W + sh * kBC * dk;
  for (int e = threadIdx.x; e < kBC * dk; e += kBThreads) {
    const int r = e / dk, i = e % dk;
    float w = 0.f;  // W = T diag(beta) GK
    for (int s = 0; s <= r; ++s) w += c.T[r * kBC + s] * c.beta[s] * c.GK[s * ld + i];
    Qb[e] = c.Qb[r * ld + i];
    Kh[e] = c.Kh[r * ld + i];
    W[e] = w;
  }
  for (int e = threadIdx.x; e < kBC * kBC; e += kBThreads) {
    a.A[sh * kBC * kBC + e] = c.A[e];
    a.Tb[sh * kBC * kBC + e] = c.T[e] * c.beta[e % kBC];
  }
  for (int i = threadIdx.x; i < dk; i += kBThreads) a.gam[sh * dk + i] = c.gam[i];
}

// The state (kReverse false) or the state gradient (kReverse true) across the
// chunks of one sequence, for kScanDvt state columns.  Forward: records the
// entry state of each chunk, then S <- diag(gamma) S + Kh^T (T_b V - W S).
// Reverse: records the gradient after each chunk, then
// dS <- diag(gamma) dS + Qb^T dO - W^T (Kh dS + A^T dO).
// Products are register-tiled: the C x dvt product Y = (W or Kh) S is split
// over dk between thread groups (2 x 4 outputs per thread from 128-bit loads
// of four channels, partial sums meeting in shared memory), the dk x dvt
// update takes 4 x 4 outputs per thread from 128-bit shared loads.  The
// [C][dk] operands keep 16-byte-padded rows so that the row pairs a warp
// reads fall in distinct banks.
constexpr int kSP = kScanDvt + 4;  // row stride of the [.][dvt] arrays (16-byte rows)

template <bool kReverse>
__global__ void __launch_bounds__(kBThreads, 4) bwd_scan_kernel(BwdArgs a) {
  extern __shared__ __align__(16) float smem[];
  const int nh = blockIdx.x, n = nh / a.H, h = nh % a.H;
  const int c0g = blockIdx.y * kScanDvt;
  const int dk = a.dk, dv = a.dv, H = a.H, tid = threadIdx.x;
  const int dvt = min(kScanDvt, dv - c0g);   // 16 or 32
  const int ncb = dvt / 4;                   // 4-column blocks
  const int nblk = 8 * ncb;                  // (row pair, column block) tasks of the C x dvt product
  const int nsplit = kBThreads / nblk;       // dk split of that product
  const int ilen = dk / nsplit;
  float *S = smem;                     // [dk][kSP]
  float *X = S + dk * kSP;             // [C][kSP]: V or dO rows
  float *red = X + kBC * kSP;          // [nsplit][C][kSP]: partial sums
  float *Y = red;                      // [C][kSP]: V~ or dV~, over the first partial sums
  const int ldm = dk + 4;              // row stride of the [C][dk] operands
  float *Wm = red + nsplit * kBC * kSP;  // [C][ldm]
  float *Km = Wm + kBC * ldm;          // [C][ldm]: Kh
  float *Qm = Km + kBC * ldm;          // [C][ldm]: Qb (reverse only)
  float *Cm = Qm + (kReverse ? kBC * ldm : 0);  // [C][C]: T_b (forward) or A (reverse)
  float *gm = Cm + kBC * kBC;          // [dk]
  int bos, eos;
  bounds(a, n, bos, eos);
  const int nch = (eos - bos + kBC - 1) / kBC;
  const int base = slot_base(a, n);
  const size_t soff = ((size_t)n * H + h) * dk * dv;
  for (int e = tid; e < dk * dvt; e += kBThreads) {
    const int i = e / dvt, cc = e % dvt;
    const float *src = kReverse ? a.dST : a.s0;
    S[i * kSP + cc] = src ? src[soff + (size_t)i * dv + c0g + cc] : 0.f;
  }
  // tasks: the C x dvt product (row pair rp, column block cb, dk split sp) and
  // the dk x dvt update (rows i0..i0+3, columns c0..c0+3)
  const int blk = tid % nblk, sp = tid / nblk;
  const int r0 = 2 * (blk / ncb), cy = 4 * (blk % ncb);
  const int ib = tid / ncb, i0 = 4 * ib, cu0 = 4 * (tid % ncb);
  const bool upd = i0 < dk;
  for (int jj = 0; jj < nch; ++jj) {
    const int j = kReverse ? nch - 1 - jj : jj;
    const int t0 = bos + j * kBC, len = min(kBC, eos - t0);
    const size_t sh = (size_t)(base + j) * H + h;
    __syncthreads();  // S final for this chunk; the previous chunk's operands are consumed
    float *rec = (kReverse ? a.dSx : a.Sent) + sh * dk * dv;
    if (upd)
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4 *>(rec + (size_t)(i0 + r) * dv + c0g + cu0) =
            *reinterpret_cast<const float4 *>(S + (i0 + r) * kSP + cu0);
    for (int e = tid; e < kBC * dvt; e += kBThreads) {
      const int r = e / dvt, cc = e % dvt;
      float x = 0.f;
      if (r < len) {
        const size_t idx = ((size_t)(t0 + r) * H + h) * dv + c0g + cc;
        x = kReverse ? ld_elem(a.dO, idx, a.out) : ld_elem(a.v, idx, a.qkv);
      }
      X[r * kSP + cc] = x;
    }
    {
      const float4 *w4 = reinterpret_cast<const float4 *>(a.W + sh * kBC * dk);
      const float4 *k4 = reinterpret_cast<const float4 *>(a.Kh + sh * kBC * dk);
      const float4 *q4 = reinterpret_cast<const float4 *>(a.Qb + sh * kBC * dk);
      const int q4r = dk / 4;
      for (int e = tid; e < kBC * q4r; e += kBThreads) {
        const int o = (e / q4r) * ldm + 4 * (e % q4r);
        *reinterpret_cast<float4 *>(Wm + o) = w4[e];
        *reinterpret_cast<float4 *>(Km + o) = k4[e];
        if (kReverse) *reinterpret_cast<float4 *>(Qm + o) = q4[e];
      }
    }
    Cm[tid] = kReverse ? a.A[sh * kBC * kBC + tid] : a.Tb[sh * kBC * kBC + tid];  // kBThreads == C * C
    for (int i = tid; i < dk; i += kBThreads) gm[i] = a.gam[sh * dk + i];
    __syncthreads();
    {  // partial (W S) or (Kh S) over this thread's slice of dk
      const float *m0p = (kReverse ? Km : Wm) + r0 * ldm, *m1p = m0p + ldm;
      float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
      const int ia = sp * ilen, ie = ia + ilen;
      int i = ia;
#pragma unroll 2
      for (; i + 4 <= ie; i += 4) {  // (ilen is a multiple of 4 whenever this runs: ia is aligned)
        const float4 a4 = *reinterpret_cast<const float4 *>(m0p + i);
        const float4 b4 = *reinterpret_cast<const float4 *>(m1p + i);
        const float ma[4] = {a4.x, a4.y, a4.z, a4.w}, mb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 s4 = *reinterpret_cast<const float4 *>(S + (i + q) * kSP + cy);
          acc0.x += ma[q] * s4.x; acc0.y += ma[q] * s4.y; acc0.z += ma[q] * s4.z; acc0.w += ma[q] * s4.w;
          acc1.x += mb[q] * s4.x; acc1.y += mb[q] * s4.y; acc1.z += mb[q] * s4.z; acc1.w += mb[q] * s4.w;
        }
      }
      for (; i < ie; ++i) {  // slices of fewer than four channels (dk = 16 with 16 state columns)
        const float4 s4 = *reinterpret_cast<const float4 *>(S + i * kSP + cy);
        const float m0 = m0p[i], m1 = m1p[i];
        acc0.x += m0 * s4.x; acc0.y += m0 * s4.y; acc0.z += m0 * s4.z; acc0.w += m0 * s4.w;
        acc1.x += m1 * s4.x; acc1.y += m1 * s4.y; acc1.z += m1 * s4.z; acc1.w += m1 * s4.w;
      }
      *reinterpret_cast<float4 *>(red + (sp * kBC + r0) * kSP + cy) = acc0;
      *reinterpret_cast<float4 *>(red + (sp * kBC + r0 + 1) * kSP + cy) = acc1;
    }
    __syncthreads();
    for (int e = tid; e < kBC * dvt; e += kBThreads) {  // (each (r, cc) is read and then written by one thread)
      const int r = e / dvt, cc = e % dvt;
      float part = 0.f;
      for (int q = 0; q < nsplit; ++q) part += red[(q * kBC + r) * kSP + cc];
      float y = 0.f;
      if (!kReverse) {  // V~ = T_b V - W S
        for (int s = 0; s <= r; ++s) y += Cm[r * kBC + s] * X[s * kSP + cc];
        y -= part;
      } else {          // dV~ = A^T dO + Kh dS
        for (int s = r; s < kBC; ++s) y += Cm[s * kBC + r] * X[s * kSP + cc];
        y += part;
      }
      Y[r * kSP + cc] = y;
    }
    __syncthreads();
    if (upd) {  // rows i0..i0+3, columns cu0..cu0+3 of the new S
      float4 sv[4];
      float g4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sv[q] = *reinterpret_cast<const float4 *>(S + (i0 + q) * kSP + cu0);
        g4[q] = gm[i0 + q];
        sv[q].x *= g4[q]; sv[q].y *= g4[q]; sv[q].z *= g4[q]; sv[q].w *= g4[q];
      }
#pragma unroll 4
      for (int r = 0; r < kBC; ++r) {
        const float4 y4 = *reinterpret_cast<const float4 *>(Y + r * kSP + cu0);
        if (!kReverse) {
          const float4 k4 = *reinterpret_cast<const float4 *>(Km + r * ldm + i0);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sv[q].x += kk[q] * y4.x; sv[q].y += kk[q] * y4.y; sv[q].z += kk[q] * y4.z; sv[q].w += kk[q] * y4.w;
          }
        } else {
          const float4 o4 = *reinterpret_cast<const float4 *>(X + r * kSP + cu0);
          const float4 q4 = *reinterpret_cast<const float4 *>(Qm + r * ldm + i0);
          const float4 w4 = *reinterpret_cast<const float4 *>(Wm + r * ldm + i0);
          const float qq[4] = {q4.x, q4.y, q4.z, q4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sv[q].x += qq[q] * o4.x - ww[q] * y4.x; sv[q].y += qq[q] * o4.y - ww[q] * y4.y;
            sv[q].z += qq[q] * o4.z - ww[q] * y4.z; sv[q].w += qq[q] * o4.w - ww[q] * y4.w;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<float4 *>(S + (i0 + q) * kSP + cu0) = sv[q];
    }
  }
  if (kReverse && a.gs0) {
    __syncthreads();
    for (int e = tid; e < dk * dvt; e += kBThreads) {
      const int i = e / dvt, cc = e % dvt;
      a.gs0[soff + (size_t)i * dv + c0g + cc] = S[i * kSP + cc];
    }
  }
}

size_t scan_smem_bytes(bool reverse, int dk, int dv) {
  const int ncb = (dv < kScanDvt ? dv : kScanDvt) / 4, nsplit = kBThreads / (8 * ncb);
  return sizeof(float) * ((size_t)dk * kSP + kBC * kSP + (size_t)nsplit * kBC * kSP +
                          (reverse ? 3 : 2) * kBC * ((size_t)dk + 4) + kBC * kBC + dk);
}

// Gradients of one chunk's rows, from its entry state and the state gradient
// after it, streaming the state in kGradDvt-column passes.  Each pass keeps
// its state columns transposed ([column][dk], 16-byte rows) so that every
// product reads 128-bit operands; the C x dk gradient sums live in registers
// across the passes (4 rows x 2 channels of dQb, dKh and dGK per thread).
__global__ void __launch_bounds__(kBThreads, 2) bwd_grads_kernel(BwdArgs a) {
  extern __shared__ __align__(16) float smem[];
  const int slot = blockIdx.x, h = blockIdx.y;
  int n, j;
  if (!locate(a, slot, n, j)) return;
  int bos, eos;
  bounds(a, n, bos, eos);
  const int t0 = bos + j * kBC, len = min(kBC, eos - t0);
  const int dk = a.dk, dv = a.dv, H = a.H, tid = threadIdx.x;
  ChunkSm c;
  float *p = carve_chunk(c, smem, dk);
  const int ld = c.ld;
  constexpr int lw = kBC + 4;      // row stride of the [column][C] arrays
  float *dA = p;  p += kBC * kBC;
  float *dTb = p; p += kBC * kBC;
  float *X = p;   p += kBC * kBC;
  float *dgam = p; p += 128;
  // The rest is used twice: by the column passes, then by the tail's [C][dk] gradients.
  float *dQb = p, *dKb = p + kBC * ld, *dGK = p + 2 * kBC * ld, *dKh = p + 3 * kBC * ld;
  float *St = p;  p += kGradDvt * ld;   // S^T of this pass: [column][dk]
  float *dSt = p; p += kGradDvt * ld;   // dS'^T
  float *Pt = p;  p += kGradDvt * lw;   // V, then P = V - GK S: [column][row]
  float *dOt = p; p += kGradDvt * lw;
  float *Vtt = p; p += kGradDvt * lw;   // V~
  float *dVtt = p; p += kGradDvt * lw;  // dV~
  float *dVv = p; p += kGradDvt * lw;   // dV
  float *red = p; p += 4 * kBC * kBC;   // [product][dk half][row][column]
  float *Sst = p; p += dk * kGradDvt;   // staging of the next pass: S columns [dk][kGradDvt]
  float *dSst = p; p += dk * kGradDvt;  // dS' columns
  float *Vst = p; p += kBC * kGradDvt;  // V rows [C][kGradDvt], qkv dtype
  float *dOst = p;                      // dO rows, out dtype
  setup_chunk(a, c, t0, len, h);
  // register accumulators
  const int rb = 4 * (tid & 3), ip = 2 * (tid >> 2);  // rows rb..rb+3, channels ip, ip+1
  const bool own = ip < dk;
  float aQ[4][2] = {}, aH[4][2] = {}, aG[4][2] = {};
  const int rr = tid / kBC, ss = tid % kBC;  // (row, column) of the C x C sums
  float accTb = 0.f, accA = 0.f, accGam = 0.f;
  // tasks of the two C x w products over dk: Z = GK S, Y = Kh dS'
  const int zp = tid >> 7, zq = (tid >> 6) & 1, zb = tid & 63;
  const int zr = 2 * (zb >> 3), zc = 2 * (zb & 7);
  const size_t sh = (size_t)slot * H + h;
  const float *Sg = a.Sent + sh * dk * dv, *dSg = a.dSx + sh * dk * dv;
  // A pass's inputs are copied into the staging area one pass ahead, so that
  // their global-memory latency overlaps the previous pass: S and dS' columns
  // (64 bytes of each of dk rows) and the C rows of V and dO (kGradDvt
  // elements each, rows past the chunk's end zero-filled).
  static_assert(kGradDvt == 16, "a pass row is four 16-byte pieces of fp32, two or four of its V / dO row");
  const int vsz = a.qkv == KDA_BF16 ? 2 : 4, osz = a.out == KDA_BF16 ? 2 : 4;
  // This thread's V / dO piece: rows of 16 elements are 2 (bf16) or 4 (fp32) pieces.
  const int vsh = vsz == 2 ? 1 : 2, osh = osz == 2 ? 1 : 2;
  const bool vpiece = tid < (kBC << vsh), opiece = tid >= 128 && tid - 128 < (kBC << osh);
  const int vrow = vpiece ? tid >> vsh : opiece ? (tid - 128) >> osh : 0;
  const int vpc = vpiece ? tid & ((1 << vsh) - 1) : opiece ? (tid - 128) & ((1 << osh) - 1) : 0;
  const size_t vrow_off = ((size_t)(t0 + (vrow < len ? vrow : 0)) * H + h) * dv;  // (in range when zero-filled)
  auto fetch = [&](int c0) {
    for (int e = tid; e < dk * 4; e += kBThreads) {  // row e / 4, columns 4 (e % 4) .. + 3
      const size_t go = (size_t)(e >> 2) * dv + c0 + 4 * (e & 3);
      cp_async16(Sst + 4 * e, Sg + go, 16);
      cp_async16(dSst + 4 * e, dSg + go, 16);
    }
    if (vpiece)
      cp_async16(reinterpret_cast<char *>(Vst) + 16 * tid,
                 reinterpret_cast<const char *>(a.v) + (vrow_off + c0) * vsz + 16 * vpc, vrow < len ? 16 : 0);
    if (opiece)
      cp_async16(reinterpret_cast<char *>(dOst) + 16 * (tid - 128),
                 reinterpret_cast<const char *>(a.dO) + (vrow_off + c0) * osz + 16 * vpc, vrow < len ? 16 : 0);
    cp_async_commit();
  };
  const int vr = tid / kGradDvt, vc = tid % kGradDvt;  // kBThreads == C * kGradDvt
  fetch(0);
  for (int c0 = 0; c0 < dv; c0 += kGradDvt) {
    cp_async_wait_all();
    __syncthreads();  // this pass's staging has landed; the previous pass is done with the column buffers
    for (int e = tid; e < 2 * dk; e += kBThreads) {  // S, dS' columns, transposed in 4 x 4 blocks
      const int w = e >= dk, b = w ? e - dk : e;  // array, then block b < dk: rows 4 (b / 4).., columns 4 (b % 4)..
      const int i0 = 4 * (b >> 2), cq = 4 * (b & 3);
      const float *src = (w ? dSst : Sst) + i0 * kGradDvt + cq;
      float *dst = (w ? dSt : St) + cq * ld + i0;
      const float4 r0 = *reinterpret_cast<const float4 *>(src), r1 = *reinterpret_cast<const float4 *>(src + kGradDvt),
                   r2 = *reinterpret_cast<const float4 *>(src + 2 * kGradDvt),
                   r3 = *reinterpret_cast<const float4 *>(src + 3 * kGradDvt);
      *reinterpret_cast<float4 *>(dst) = make_float4(r0.x, r1.x, r2.x, r3.x);
      *reinterpret_cast<float4 *>(dst + ld) = make_float4(r0.y, r1.y, r2.y, r3.y);
      *reinterpret_cast<float4 *>(dst + 2 * ld) = make_float4(r0.z, r1.z, r2.z, r3.z);
      *reinterpret_cast<float4 *>(dst + 3 * ld) = make_float4(r0.w, r1.w, r2.w, r3.w);
    }
    {  // V rows (P = V - GK S after the next step) and dO rows, widened to fp32
      const int o = vr * kGradDvt + vc;
      Pt[vc * lw + vr] = vsz == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(Vst)[o]) : Vst[o];
      dOt[vc * lw + vr] = osz == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(dOst)[o]) : dOst[o];
    }
    __syncthreads();  // the staging area is free for the next pass
    if (c0 + kGradDvt < dv) fetch(c0 + kGradDvt);
    {  // partial Z = GK S (zp = 0) or Y = Kh dS' (zp = 1) over half of dk, 2 x 2 outputs
      const float *Mm = zp ? c.Kh : c.GK;
      const float *Vm = zp ? dSt : St;
      float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
      const int half = dk / 2, ia = zq * half;
#pragma unroll 2
      for (int i = ia; i < ia + half; i += 4) {
        const float4 m0 = *reinterpret_cast<const float4 *>(Mm + zr * ld + i);
        const float4 m1 = *reinterpret_cast<const float4 *>(Mm + (zr + 1) * ld + i);
        const float4 v0 = *reinterpret_cast<const float4 *>(Vm + zc * ld + i);
        const float4 v1 = *reinterpret_cast<const float4 *>(Vm + (zc + 1) * ld + i);
        a00 = fmaf(m0.x, v0.x, fmaf(m0.y, v0.y, fmaf(m0.z, v0.z, fmaf(m0.w, v0.w, a00))));
        a01 = fmaf(m0.x, v1.x, fmaf(m0.y, v1.y, fmaf(m0.z, v1.z, fmaf(m0.w, v1.w, a01))));
        a10 = fmaf(m1.x, v0.x, fmaf(m1.y, v0.y, fmaf(m1.z, v0.z, fmaf(m1.w, v0.w, a10))));
        a11 = fmaf(m1.x, v1.x, fmaf(m1.y, v1.y, fmaf(m1.z, v1.z, fmaf(m1.w, v1.w, a11))));
      }
      float *rd = red + (zp * 2 + zq) * kBC * kBC;
      rd[zr * kBC + zc] = a00;
      rd[zr * kBC + zc + 1] = a01;
      rd[(zr + 1) * kBC + zc] = a10;
      rd[(zr + 1) * kBC + zc + 1] = a11;
    }
    __syncthreads();
    {  // P = V - Z;  dV~ = Y + A^T dO   (thread = (row rr, column ss))
      const float z = red[rr * kBC + ss] + red[kBC * kBC + rr * kBC + ss];
      float y = red[2 * kBC * kBC + rr * kBC + ss] + red[3 * kBC * kBC + rr * kBC + ss];
      for (int s2 = rr; s2 < kBC; ++s2) y += c.A[s2 * kBC + rr] * dOt[ss * lw + s2];
      Pt[ss * lw + rr] -= z;
      dVtt[ss * lw + rr] = y;
    }
    __syncthreads();
    {  // V~ = T_b P;  dV = T_b^T dV~
      float y = 0.f, d = 0.f;
      for (int s2 = 0; s2 <= rr; ++s2) y += c.T[rr * kBC + s2] * c.beta[s2] * Pt[ss * lw + s2];
      for (int s2 = rr; s2 < kBC; ++s2) d += c.T[s2 * kBC + rr] * dVtt[ss * lw + s2];
      d *= c.beta[rr];
      Vtt[ss * lw + rr] = y;
      dVv[ss * lw + rr] = d;
      if (rr < len) a.gv[((size_t)(t0 + rr) * H + h) * dv + c0 + ss] = d;
    }
    __syncthreads();
    if (own) {  // dQb += dO S^T, dKh += V~ dS'^T, dGK -= dV S^T on this thread's 4 x 2 block
#pragma unroll 4
      for (int cc = 0; cc < kGradDvt; ++cc) {
        const float4 o4 = *reinterpret_cast<const float4 *>(dOt + cc * lw + rb);
        const float4 v4 = *reinterpret_cast<const float4 *>(Vtt + cc * lw + rb);
        const float4 d4 = *reinterpret_cast<const float4 *>(dVv + cc * lw + rb);
        const float2 s2 = *reinterpret_cast<const float2 *>(St + cc * ld + ip);
        const float2 ds2 = *reinterpret_cast<const float2 *>(dSt + cc * ld + ip);
        const float oo[4] = {o4.x, o4.y, o4.z, o4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w},
                    dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          aQ[q][0] += oo[q] * s2.x; aQ[q][1] += oo[q] * s2.y;
          aH[q][0] += vv[q] * ds2.x; aH[q][1] += vv[q] * ds2.y;
          aG[q][0] -= dd[q] * s2.x; aG[q][1] -= dd[q] * s2.y;
        }
      }
    }
    for (int cc = 0; cc < kGradDvt; ++cc) {  // dT_b += dV~ P^T, dA += dO V~^T
      accTb += dVtt[cc * lw + rr] * Pt[cc * lw + ss];
      accA += dOt[cc * lw + rr] * Vtt[cc * lw + ss];
    }
    if (tid < dk)
      for (int cc = 0; cc < kGradDvt; ++cc) accGam += dSt[cc * ld + tid] * St[cc * ld + tid];
  }
  __syncthreads();  // the pass buffers become dQb, dKb, dGK, dKh
  if (own)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dQb[(rb + q) * ld + ip] = aQ[q][0]; dQb[(rb + q) * ld + ip + 1] = aQ[q][1];
      dKh[(rb + q) * ld + ip] = aH[q][0]; dKh[(rb + q) * ld + ip + 1] = aH[q][1];
      dGK[(rb + q) * ld + ip] = aG[q][0]; dGK[(rb + q) * ld + ip + 1] = aG[q][1];
    }
  dTb[tid] = accTb;
  dA[tid] = accA;
  if (tid < dk) dgam[tid] = accGam;
  __syncthreads();
  // through T_b = T diag(beta) and T = (I + L)^-1:  X = T^T (dT_b diag(beta))
  {
    const int r = tid / kBC, s = tid % kBC;
    float x = 0.f;
    for (int m = 0; m < kBC; ++m) x += c.T[m * kBC + r] * dTb[m * kBC + s] * c.beta[s];
    X[tid] = x;
  }
  __syncthreads();
  {
    // dL[r][s] = -(X T^T)[r][s] below the diagonal, then in X's place
    const int r = tid / kBC, s = tid % kBC;
    float dl = 0.f;
    if (s < r)
      for (int m = 0; m < kBC; ++m) dl -= X[r * kBC + m] * c.T[s * kBC + m];
    __syncthreads();
    X[tid] = dl;
  }
  __syncthreads();
  if (tid < kBC) {  // dbeta_r = sum_s dT_b[s][r] T[s][r] + sum_{s<r} dL[r][s] M[r][s]
    const int r = tid;
    float acc = 0.f;
    for (int s = 0; s < kBC; ++s) acc += dTb[s * kBC + r] * c.T[s * kBC + r];
    for (int s = 0; s < r; ++s) acc += X[r * kBC + s] * c.M[r * kBC + s];
    if (r < len) a.gbeta[(size_t)(t0 + r) * H + h] = acc;
  }
  __syncthreads();
  {
    const int r = tid / kBC, s = tid % kBC;
    X[tid] *= c.beta[r];                   // dM = diag(beta) dL
    if (s > r) dA[tid] = 0.f;              // Tril_incl
  }
  __syncthreads();
  {  // dGK += dM Kb, dKb = dM^T GK + dA^T Qb, dQb += dA Kb: channel i, rows r0..r0+7 per thread
    const int i = tid & 127, r0 = 8 * (tid >> 7);
    if (i < dk) {
      float gk[8] = {}, kb[8] = {}, qb[8] = {};
#pragma unroll 1
      for (int s0 = 0; s0 < kBC; s0 += 4) {
        float kbs[4], gks[4], qbs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          kbs[u] = c.Kb[(s0 + u) * ld + i];
          gks[u] = c.GK[(s0 + u) * ld + i];
          qbs[u] = c.Qb[(s0 + u) * ld + i];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // row r0 + q of dM and dA, columns s0..s0+3
          const float4 x4 = *reinterpret_cast<const float4 *>(X + (r0 + q) * kBC + s0);
          const float4 a4 = *reinterpret_cast<const float4 *>(dA + (r0 + q) * kBC + s0);
          gk[q] += x4.x * kbs[0] + x4.y * kbs[1] + x4.z * kbs[2] + x4.w * kbs[3];
          qb[q] += a4.x * kbs[0] + a4.y * kbs[1] + a4.z * kbs[2] + a4.w * kbs[3];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // row s0 + u of dM and dA, columns r0..r0+7
          const float4 xa = *reinterpret_cast<const float4 *>(X + (s0 + u) * kBC + r0);
          const float4 xb = *reinterpret_cast<const float4 *>(X + (s0 + u) * kBC + r0 + 4);
          const float4 da = *reinterpret_cast<const float4 *>(dA + (s0 + u) * kBC + r0);
          const float4 db = *reinterpret_cast<const float4 *>(dA + (s0 + u) * kBC + r0 + 4);
          const float xm[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          const float dm[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) kb[q] += xm[q] * gks[u] + dm[q] * qbs[u];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dGK[(r0 + q) * ld + i] += gk[q];
        dKb[(r0 + q) * ld + i] = kb[q];
        dQb[(r0 + q) * ld + i] += qb[q];
      }
    }
  }
  __syncthreads();
  // elementwise to q, k and the cumulative log-decay G (dG in dKb's place)
  for (int e = tid; e < kBC * dk; e += kBThreads) {
    const int r = e / dk, i = e % dk;
    const float G = c.G[r * ld + i], Gl = c.G[(kBC - 1) * ld + i];
    const float eg = expf(G), ei = expf(-G), eh = expf(Gl - G);
    const float q = dQb[r * ld + i], kb = dKb[r * ld + i], gk = dGK[r * ld + i], kh = dKh[r * ld + i];
    if (r < len) {
      const size_t idx = ((size_t)(t0 + r) * H + h) * dk + i;
      a.gq[idx] = q * eg;
      a.gk[idx] = kb * ei + gk * eg + kh * eh;
    }
    dKb[r * ld + i] = q * c.Qb[r * ld + i] - kb * c.Kb[r * ld + i] + gk * c.GK[r * ld + i] - kh * c.Kh[r * ld + i];
  }
  __syncthreads();
  if (tid < dk) {  // G_last terms, then the reverse cumulative sum over rows
    const int i = tid;
    float last = dgam[i] * c.gam[i];
    for (int r = 0; r < kBC; ++r) last += dKh[r * ld + i] * c.Kh[r * ld + i];
    float acc = last;
    for (int r = kBC - 1; r >= 0; --r) {
      acc += dKb[r * ld + i];
      if (r < len) a.gg[((size_t)(t0 + r) * H + h) * dk + i] = acc;
    }
  }
}

size_t grads_smem_bytes(int dk) {
  const size_t ld = (size_t)dk + 4, lw = kBC + 4;
  const size_t pass = 2 * kGradDvt * ld + 5 * kGradDvt * lw + 4 * kBC * kBC + 2 * (size_t)dk * kGradDvt +
                      2 * kBC * kGradDvt;
  const size_t tail = 4 * kBC * ld;
  return sizeof(float) * (5 * kBC * ld + 6 * kBC * kBC + kBC + 2 * 128 + (pass > tail ? pass : tail));
}

size_t prep_smem_bytes(int dk) {
  const size_t ld = (size_t)dk + 4;
  return sizeof(float) * (5 * kBC * ld + 3 * kBC * kBC + kBC + 128);
}

}  // namespace

int bwd_slots(const PrefillArgs &p) {
  return p.cu ? p.T_total / kBC + p.N : p.N * ((p.T_seq + kBC - 1) / kBC);
}

size_t bwd_workspace_bytes(const PrefillArgs &p) {
  const size_t per = (size_t)3 * kBC * p.dk + 2 * kBC * kBC + p.dk + 2 * (size_t)p.dk * p.dv;
  return sizeof(float) * per * (size_t)bwd_slots(p) * p.H;
}

cudaError_t launch_chunk_bwd(const PrefillArgs &p, const BwdIo &io, void *ws, cudaStream_t s) {
  BwdArgs a;
  a.N = p.N; a.T_total = p.T_total; a.T_seq = p.T_seq; a.H = p.H; a.dk = p.dk; a.dv = p.dv;
  a.qkv = p.qkv; a.out = p.out; a.gate = p.gate;
  a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta; a.s0 = p.s0; a.cu = p.cu;
  a.dO = io.dO; a.dST = io.dST;
  a.gq = io.dq; a.gk = io.dk; a.gv = io.dv; a.gg = io.dg; a.gbeta = io.dbeta; a.gs0 = io.ds0;
  a.nslots = bwd_slots(p);
  const size_t sl = (size_t)a.nslots * p.H;
  float *w = reinterpret_cast<float *>(ws);
  a.Qb = w;  w += sl * kBC * p.dk;
  a.Kh = w;  w += sl * kBC * p.dk;
  a.W = w;   w += sl * kBC * p.dk;
  a.A = w;   w += sl * kBC * kBC;
  a.Tb = w;  w += sl * kBC * kBC;
  a.gam = w; w += sl * p.dk;
  a.Sent = w; w += sl * (size_t)p.dk * p.dv;
  a.dSx = w;
  if (a.N * a.H == 0) return cudaSuccess;
  cudaError_t e;
  if (a.nslots > 0) {
    const size_t sp = prep_smem_bytes(p.dk);
    e = cudaFuncSetAttribute(bwd_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e != cudaSuccess) return e;
    bwd_prep_kernel<<<dim3(a.nslots, p.H), kBThreads, sp, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t ssf = scan_smem_bytes(false, p.dk, p.dv), ssr = scan_smem_bytes(true, p.dk, p.dv);
  const dim3 sgrid(p.N * p.H, (p.dv + kScanDvt - 1) / kScanDvt);
  e = cudaFuncSetAttribute(bwd_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssf);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssr);
  if (e != cudaSuccess) return e;
  bwd_scan_kernel<false><<<sgrid, kBThreads, ssf, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_scan_kernel<true><<<sgrid, kBThreads, ssr, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.nslots > 0) {
    const size_t sg = grads_smem_bytes(p.dk);
    e = cudaFuncSetAttribute(bwd_grads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg);
    if (e != cudaSuccess) return e;
    bwd_grads_kernel<<<dim3(a.nslots, p.H), kBThreads, sg, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
