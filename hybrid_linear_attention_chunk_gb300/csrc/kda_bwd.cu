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
// Four launches, all in fp32 arithmetic:
//   bwd_prep   (every chunk in parallel)  Qb, Kh, W, A, T_b, gamma of each chunk
//   bwd_scan<forward>  (per sequence, head, 32 dv columns)  the entry state of every chunk
//   bwd_scan<reverse>  (same, last chunk first)  the state gradient after every chunk; dS_0
//   bwd_grads  (every chunk in parallel)  dq, dk, dv, dg, dbeta of the chunk's rows
// The prep kernel and the scans run on CUDA cores; the gradient kernel's
// products run on mma.sync with operands split into two tf32 parts (see
// mma_3xtf32), the rest of it on CUDA cores.
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
template <int kPending>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(kPending) : "memory");
}

// fp32 products on the tensor cores: mma.sync m16n8k8 with tf32 operands,
// each operand x split as hi = tf32(x), lo = tf32(x - hi) and the product
// taken as lo_a hi_b + hi_a lo_b + hi_a hi_b (the dropped lo_a lo_b term is
// below fp32 rounding).  Fragments per the PTX ISA for this shape, with
// g = lane / 4 and t = lane % 4: A (16 x 8, row) holds (g, t), (g + 8, t),
// (g, t + 4), (g + 8, t + 4); B (8 x 8, col) holds (t, g), (t + 4, g);
// D (16 x 8) holds (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void split_frag(uint32_t (&hi)[4], uint32_t (&lo)[4], float x0, float x1, float x2,
                                           float x3) {
  const float x[4] = {x0, x1, x2, x3};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hi[i] = to_tf32(x[i]);
    lo[i] = to_tf32(x[i] - __uint_as_float(hi[i]));
  }
}
__device__ __forceinline__ void split_frag(uint32_t (&hi)[2], uint32_t (&lo)[2], float x0, float x1) {
  hi[0] = to_tf32(x0);
  lo[0] = to_tf32(x0 - __uint_as_float(hi[0]));
  hi[1] = to_tf32(x1);
  lo[1] = to_tf32(x1 - __uint_as_float(hi[1]));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_3xtf32(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
  mma_tf32(d, al, bh);
  mma_tf32(d, ah, bl);
  mma_tf32(d, ah, bh);
}
__device__ __forceinline__ void mma_3xtf32(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
  split_frag(ah, al, a[0], a[1], a[2], a[3]);
  split_frag(bh, bl, b[0], b[1]);
  mma_3xtf32(d, ah, al, bh, bl);
}

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
  for (int e = tid; e < kBC * dk; e += kBThreads) {  // (Kh = K e^{G_C - G} = Kb gamma)
    const int r = e / dk, i = e % dk;
    const float G = c.G[r * ld + i];
    const float kv = c.Kb[r * ld + i];
    const float eg = expf(G), kb = kv * expf(-G);
    c.Qb[r * ld + i] *= eg;
    c.GK[r * ld + i] = kv * eg;
    c.Kb[r * ld + i] = kb;
    c.Kh[r * ld + i] = kb * c.gam[i];
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
  extern __shared__ __align__(16) float smem[];  // (the set-up stores 128-bit rows)
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
// A step's operands arrive by cp.async while the previous step runs, each as
// soon as its buffer is free: forward, W after the product, and X = V, T_b,
// Kh and gamma after the reduction (Kh and gamma into the buffer the update
// does not read); reverse, Kh after the product, and Qb, A, gamma and X = dO
// after the reduction, during which Qb^T dO is already added, so the last
// phase reads only W (fetched at the step's start) and V~-gradient rows.
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
  const int ldm = dk + 4;                    // row stride of the [C][dk] operands
  const kda_dtype xt = kReverse ? a.out : a.qkv;  // X rows: dO (reverse) or V (forward)
  const int xsz = xt == KDA_BF16 ? 2 : 4;
  float *S = smem;                       // [dk][kSP]
  float *red = S + dk * kSP;             // [nsplit][C][kSP]: partial sums
  float *Y = red;                        // [C][kSP]: V~ or dV~, over the first partial sums
  float *Xr = red + nsplit * kBC * kSP;  // [C][dvt] X rows in their dtype (2 KB)
  float *Wm = Xr + kBC * kScanDvt;       // [C][ldm]: W
  float *Km = Wm + kBC * ldm;            // [C][ldm]: Kh (forward: two buffers)
  float *Qm = Km + (kReverse ? 1 : 2) * kBC * ldm;  // [C][ldm]: Qb (reverse only)
  float *Cm = Qm + (kReverse ? kBC * ldm : 0);       // [C][C]: T_b (forward) or A (reverse)
  float *gm = Cm + kBC * kBC;            // [dk]: gamma (forward: two buffers)
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
  // asynchronous copies of chunk j's operands (all sizes powers of two)
  const int q4sh = __ffs(dk / 4) - 1;                    // log2 of the 16-byte pieces of a [dk] row
  const int xsh = __ffs(dvt * xsz / 16) - 1;             // log2 of the pieces of an X row
  auto chunk_at = [&](int j, int &t0, int &len, size_t &sh) {
    j = kReverse ? nch - 1 - j : j;
    t0 = bos + j * kBC;
    len = min(kBC, eos - t0);
    sh = (size_t)(base + j) * H + h;
  };
  auto fetch_rows = [&](float *dst, const float *src) {  // [C][dk] workspace rows -> [C][ldm]
    for (int e = tid; e < (kBC << q4sh); e += kBThreads)
      cp_async16(dst + (e >> q4sh) * ldm + 4 * (e & ((1 << q4sh) - 1)), src + 4 * e, 16);
  };
  auto fetch_small = [&](int jj, float *g_dst) {  // X rows, the C x C matrix and gamma of step jj
    int t0, len;
    size_t sh;
    chunk_at(jj, t0, len, sh);
    const char *xg = reinterpret_cast<const char *>(kReverse ? a.dO : a.v);
    for (int e = tid; e < (kBC << xsh); e += kBThreads) {
      const int r = e >> xsh, pc = e & ((1 << xsh) - 1);
      const size_t row = (size_t)(t0 + (r < len ? r : 0)) * H + h;  // (in range when zero-filled)
      cp_async16(reinterpret_cast<char *>(Xr) + r * dvt * xsz + 16 * pc, xg + (row * dv + c0g) * xsz + 16 * pc,
                 r < len ? 16 : 0);
    }
    if (tid < kBC * kBC / 4) cp_async16(Cm + 4 * tid, (kReverse ? a.A : a.Tb) + sh * kBC * kBC + 4 * tid, 16);
    if (tid < dk / 4) cp_async16(g_dst + 4 * tid, a.gam + sh * dk + 4 * tid, 16);
  };
  auto xval = [&](int r, int cc) -> float {
    return xsz == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(Xr)[r * dvt + cc])
                    : Xr[r * dvt + cc];
  };
  auto xval4 = [&](int r, int cc) -> float4 {
    if (xsz == 2) {
      const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(Xr) + r * dvt + cc);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
      return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    return *reinterpret_cast<const float4 *>(Xr + r * dvt + cc);
  };
  if (nch > 0) {  // the first step's operands (the reverse scan's W comes at each step's start)
    int t0, len;
    size_t sh;
    chunk_at(0, t0, len, sh);
    if (!kReverse) fetch_rows(Wm, a.W + sh * kBC * dk);
    fetch_rows(Km, a.Kh + sh * kBC * dk);
    if (kReverse) fetch_rows(Qm, a.Qb + sh * kBC * dk);
    fetch_small(0, gm);
    cp_async_commit();
  }
  // tasks: the C x dvt product (row pair rp, column block cb, dk split sp) and
  // the dk x dvt update (rows i0..i0+3, columns c0..c0+3)
  const int blk = tid % nblk, sp = tid / nblk;
  const int r0 = 2 * (blk / ncb), cy = 4 * (blk % ncb);
  const int ib = tid / ncb, i0 = 4 * ib, cu0 = 4 * (tid % ncb);
  const bool upd = i0 < dk;
  for (int jj = 0; jj < nch; ++jj) {
    int t0, len;
    size_t sh;
    chunk_at(jj, t0, len, sh);
    const bool more = jj + 1 < nch;
    const int buf = kReverse ? 0 : (jj & 1);  // forward: Kh and gamma buffers alternate
    const float *Kc = Km + buf * kBC * ldm, *gc = gm + buf * dk;
    cp_async_wait_all();
    __syncthreads();  // this step's operands have landed; S is final for this chunk
    if (kReverse) {   // W of this step, needed only by the last phase
      fetch_rows(Wm, a.W + sh * kBC * dk);
      cp_async_commit();
    }
    float *rec = (kReverse ? a.dSx : a.Sent) + sh * dk * dv;
    if (upd)
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4 *>(rec + (size_t)(i0 + r) * dv + c0g + cu0) =
            *reinterpret_cast<const float4 *>(S + (i0 + r) * kSP + cu0);
    {  // partial (W S) or (Kh S) over this thread's slice of dk
      const float *m0p = (kReverse ? Kc : Wm) + r0 * ldm, *m1p = m0p + ldm;
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
    __syncthreads();  // partial sums complete; the product's operand buffer is free
    if (more) {
      int t1, l1;
      size_t sh1;
      chunk_at(jj + 1, t1, l1, sh1);
      fetch_rows(kReverse ? Km : Wm, (kReverse ? a.Kh : a.W) + sh1 * kBC * dk);
      cp_async_commit();
    }
    for (int e = tid; e < kBC * dvt; e += kBThreads) {  // (each (r, cc) is read and then written by one thread)
      const int r = e / dvt, cc = e % dvt;
      float part = 0.f;
      for (int q = 0; q < nsplit; ++q) part += red[(q * kBC + r) * kSP + cc];
      float y = 0.f;
      if (!kReverse) {  // V~ = T_b V - W S
        for (int s = 0; s <= r; ++s) y += Cm[r * kBC + s] * xval(s, cc);
        y -= part;
      } else {          // dV~ = A^T dO + Kh dS
        for (int s = r; s < kBC; ++s) y += Cm[s * kBC + r] * xval(s, cc);
        y += part;
      }
      Y[r * kSP + cc] = y;
    }
    float4 sv[4];
    if (upd) {  // rows i0..i0+3, columns cu0..cu0+3 of the new S: diag(gamma) S (+ Qb^T dO, reverse)
      float g4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sv[q] = *reinterpret_cast<const float4 *>(S + (i0 + q) * kSP + cu0);
        g4[q] = gc[i0 + q];
        sv[q].x *= g4[q]; sv[q].y *= g4[q]; sv[q].z *= g4[q]; sv[q].w *= g4[q];
      }
      if (kReverse) {
#pragma unroll 4
        for (int r = 0; r < kBC; ++r) {
          const float4 o4 = xval4(r, cu0);
          const float4 q4 = *reinterpret_cast<const float4 *>(Qm + r * ldm + i0);
          const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sv[q].x += qq[q] * o4.x; sv[q].y += qq[q] * o4.y; sv[q].z += qq[q] * o4.z; sv[q].w += qq[q] * o4.w;
          }
        }
      }
    }
    if (kReverse) {
      if (more) cp_async_wait_group<1>();  // this step's W (the next step's Kh may stay in flight)
      else cp_async_wait_all();
    }
    __syncthreads();  // Y complete; X, the C x C matrix, gamma (and Qb) are free
    if (more) {
      fetch_small(jj + 1, kReverse ? gm : gm + (buf ^ 1) * dk);
      if (kReverse) {
        int t1, l1;
        size_t sh1;
        chunk_at(jj + 1, t1, l1, sh1);
        fetch_rows(Qm, a.Qb + sh1 * kBC * dk);
      } else {
        int t1, l1;
        size_t sh1;
        chunk_at(jj + 1, t1, l1, sh1);
        fetch_rows(Km + (buf ^ 1) * kBC * ldm, a.Kh + sh1 * kBC * dk);
      }
      cp_async_commit();
    }
    if (upd) {  // + Kh^T Y (forward) or - W^T dV~ (reverse)
      const float *Mu = kReverse ? Wm : Kc;
#pragma unroll 4
      for (int r = 0; r < kBC; ++r) {
        const float4 y4 = *reinterpret_cast<const float4 *>(Y + r * kSP + cu0);
        const float4 m4 = *reinterpret_cast<const float4 *>(Mu + r * ldm + i0);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (kReverse) {
            sv[q].x -= mm[q] * y4.x; sv[q].y -= mm[q] * y4.y; sv[q].z -= mm[q] * y4.z; sv[q].w -= mm[q] * y4.w;
          } else {
            sv[q].x += mm[q] * y4.x; sv[q].y += mm[q] * y4.y; sv[q].z += mm[q] * y4.z; sv[q].w += mm[q] * y4.w;
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
  return sizeof(float) * ((size_t)dk * kSP + (size_t)nsplit * kBC * kSP + kBC * kScanDvt +
                          3 * kBC * ((size_t)dk + 4) + kBC * kBC + (reverse ? 1 : 2) * (size_t)dk);
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
  constexpr int lr = kGradDvt + 4;  // row stride of the [row][column] pass arrays and of the staged rows
  float *dA = p;  p += kBC * kBC;
  float *dTb = p; p += kBC * kBC;
  float *X = p;   p += kBC * kBC;
  float *dgam = p; p += 128;
  // The rest is used twice: by the column passes, then by the tail's [C][dk] gradients.
  float *dQb = p, *dKb = p + kBC * ld, *dGK = p + 2 * kBC * ld, *dKh = p + 3 * kBC * ld;
  float *Pr = p;   p += kBC * lr;   // V, then P = V - GK S: [row][column]
  float *dOr = p;  p += kBC * lr;   // dO
  float *Vtr = p;  p += kBC * lr;   // V~
  float *dVtr = p; p += kBC * lr;   // dV~
  float *dVr = p;  p += kBC * lr;   // dV
  float *red = p;  p += 4 * kBC * kBC;  // [product][dk half][row][column]
  float *Sb = p;   p += 4 * dk * lr;    // two staging buffers, each the pass's S rows then dS' rows: [dk][lr]
  float *Vb = p;                        // two staging buffers of 2 KB: V rows, then dO rows at +1 KB, in their dtypes
  setup_chunk(a, c, t0, len, h);
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;  // mma fragment coordinates
  const int rr = tid / kBC, ss = tid % kBC;  // (row, column) of the C x C steps
  // accumulators over the passes: dQb, dKh, dGK (channels 16 warp .. + 15, two n-tiles), dT_b or dA (warps 4-7)
  float accQ[2][4] = {}, accH[2][4] = {}, accG[2][4] = {}, accTA[4] = {};
  float accGam = 0.f;
  const size_t sh = (size_t)slot * H + h;
  const float *Sg = a.Sent + sh * dk * dv, *dSg = a.dSx + sh * dk * dv;
  // A pass's inputs are copied into a staging buffer one pass ahead, so that
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
  auto fetch = [&](int c0, int bi) {
    float *sS = Sb + bi * 2 * dk * lr, *sD = sS + dk * lr;
    char *vb = reinterpret_cast<char *>(Vb + bi * 512);
    for (int e = tid; e < dk * 4; e += kBThreads) {  // row e / 4, columns 4 (e % 4) .. + 3
      const int i = e >> 2, q = 4 * (e & 3);
      const size_t go = (size_t)i * dv + c0 + q;
      cp_async16(sS + i * lr + q, Sg + go, 16);
      cp_async16(sD + i * lr + q, dSg + go, 16);
    }
    if (vpiece)
      cp_async16(vb + 16 * tid, reinterpret_cast<const char *>(a.v) + (vrow_off + c0) * vsz + 16 * vpc,
                 vrow < len ? 16 : 0);
    if (opiece)
      cp_async16(vb + 1024 + 16 * (tid - 128),
                 reinterpret_cast<const char *>(a.dO) + (vrow_off + c0) * osz + 16 * vpc, vrow < len ? 16 : 0);
    cp_async_commit();
  };
  fetch(0, 0);
  for (int c0 = 0, bi = 0; c0 < dv; c0 += kGradDvt, bi ^= 1) {
    const float *sS = Sb + bi * 2 * dk * lr, *sD = sS + dk * lr;
    const char *vb = reinterpret_cast<const char *>(Vb + bi * 512);
    cp_async_wait_all();
    __syncthreads();  // this pass's staging has landed; the previous pass is done with every pass array
    {  // V and dO rows, widened to fp32 (one element per thread: kBThreads == C * kGradDvt)
      const int o = rr * kGradDvt + ss;
      Pr[rr * lr + ss] = vsz == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(vb)[o])
                                  : reinterpret_cast<const float *>(vb)[o];
      dOr[rr * lr + ss] = osz == 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(vb + 1024)[o])
                                   : reinterpret_cast<const float *>(vb + 1024)[o];
    }
    if (c0 + kGradDvt < dv) fetch(c0 + kGradDvt, bi ^ 1);
    {  // partial Z = GK S (zp = 0) or Y = Kh dS' (zp = 1) over half of dk: warp (zp, column tile, half)
      const int zp = warp >> 2, n0 = 8 * ((warp >> 1) & 1), half = dk / 2, ka = (warp & 1) * half;
      const float *Am = zp ? c.Kh : c.GK, *Bm = zp ? sD : sS;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = ka; k0 < ka + half; k0 += 8) {
        const float av[4] = {Am[g * ld + k0 + t], Am[(g + 8) * ld + k0 + t], Am[g * ld + k0 + t + 4],
                             Am[(g + 8) * ld + k0 + t + 4]};
        const float bv[2] = {Bm[(k0 + t) * lr + n0 + g], Bm[(k0 + t + 4) * lr + n0 + g]};
        mma_3xtf32(d, av, bv);
      }
      float *rd = red + (zp * 2 + (warp & 1)) * kBC * kBC + n0 + 2 * t;
      *reinterpret_cast<float2 *>(rd + g * kBC) = make_float2(d[0], d[1]);
      *reinterpret_cast<float2 *>(rd + (g + 8) * kBC) = make_float2(d[2], d[3]);
    }
    __syncthreads();
    Pr[rr * lr + ss] -= red[rr * kBC + ss] + red[kBC * kBC + rr * kBC + ss];  // P = V - Z
    if (warp < 2) {  // dV~ = Y + A^T dO on the tensor cores: warp = 8-column tile
      const int n0 = 8 * warp, o = g * kBC + n0 + 2 * t, o8 = o + 8 * kBC;
      const float *ry = red + 2 * kBC * kBC;
      float d[4] = {ry[o] + ry[kBC * kBC + o], ry[o + 1] + ry[kBC * kBC + o + 1], ry[o8] + ry[kBC * kBC + o8],
                    ry[o8 + 1] + ry[kBC * kBC + o8 + 1]};
#pragma unroll
      for (int k0 = 0; k0 < kBC; k0 += 8) {  // A(r, s) = A^T[r][s] = A[s][r]; B(s, c) = dO[s][c]
        const float av[4] = {c.A[(k0 + t) * kBC + g], c.A[(k0 + t) * kBC + g + 8], c.A[(k0 + t + 4) * kBC + g],
                             c.A[(k0 + t + 4) * kBC + g + 8]};
        const float bv[2] = {dOr[(k0 + t) * lr + n0 + g], dOr[(k0 + t + 4) * lr + n0 + g]};
        mma_3xtf32(d, av, bv);
      }
      *reinterpret_cast<float2 *>(dVtr + g * lr + n0 + 2 * t) = make_float2(d[0], d[1]);
      *reinterpret_cast<float2 *>(dVtr + (g + 8) * lr + n0 + 2 * t) = make_float2(d[2], d[3]);
    }
    __syncthreads();
    if (warp < 4) {  // V~ = T_b P (warps 0, 1);  dV = T_b^T dV~ = diag(beta) T^T dV~ (warps 2, 3)
      const bool isD = warp >= 2;
      const int n0 = 8 * (warp & 1);
      const float *Bm = isD ? dVtr : Pr;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k0 = 0; k0 < kBC; k0 += 8) {
        const int s0 = k0 + t, s4 = k0 + t + 4;
        float av[4];
        if (isD) {  // A(r, s) = T[s][r]
          av[0] = c.T[s0 * kBC + g]; av[1] = c.T[s0 * kBC + g + 8];
          av[2] = c.T[s4 * kBC + g]; av[3] = c.T[s4 * kBC + g + 8];
        } else {    // A(r, s) = T[r][s] beta_s
          av[0] = c.T[g * kBC + s0] * c.beta[s0]; av[1] = c.T[(g + 8) * kBC + s0] * c.beta[s0];
          av[2] = c.T[g * kBC + s4] * c.beta[s4]; av[3] = c.T[(g + 8) * kBC + s4] * c.beta[s4];
        }
        const float bv[2] = {Bm[s0 * lr + n0 + g], Bm[s4 * lr + n0 + g]};
        mma_3xtf32(d, av, bv);
      }
      const int col = n0 + 2 * t;
      if (isD) {
        const float b0 = c.beta[g], b8 = c.beta[g + 8];
        d[0] *= b0; d[1] *= b0; d[2] *= b8; d[3] *= b8;
        *reinterpret_cast<float2 *>(dVr + g * lr + col) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(dVr + (g + 8) * lr + col) = make_float2(d[2], d[3]);
        // (the gradient outputs are only 4-byte aligned: scalar stores)
        if (g < len) {
          float *o = a.gv + ((size_t)(t0 + g) * H + h) * dv + c0 + col;
          o[0] = d[0];
          o[1] = d[1];
        }
        if (g + 8 < len) {
          float *o = a.gv + ((size_t)(t0 + g + 8) * H + h) * dv + c0 + col;
          o[0] = d[2];
          o[1] = d[3];
        }
      } else {
        *reinterpret_cast<float2 *>(Vtr + g * lr + col) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(Vtr + (g + 8) * lr + col) = make_float2(d[2], d[3]);
      }
    }
    __syncthreads();
    if (16 * warp < dk) {  // dQb += dO S^T, dKh += V~ dS'^T, dGK -= dV S^T on channels 16 warp .. + 15
#pragma unroll
      for (int k0 = 0; k0 < kGradDvt; k0 += 8) {
        const int ra = g * lr + k0 + t, rb = (g + 8) * lr + k0 + t;  // A fragment: rows g, g + 8
        uint32_t oh[4], ol[4], vh[4], vl[4], dh[4], dl[4];
        split_frag(oh, ol, dOr[ra], dOr[rb], dOr[ra + 4], dOr[rb + 4]);
        split_frag(vh, vl, Vtr[ra], Vtr[rb], Vtr[ra + 4], Vtr[rb + 4]);
        split_frag(dh, dl, -dVr[ra], -dVr[rb], -dVr[ra + 4], -dVr[rb + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // B(k = column, n = channel) = S[channel][column]
          const int cb = (16 * warp + 8 * nt + g) * lr + k0 + t;
          uint32_t sh2[2], sl2[2], dsh[2], dsl[2];
          split_frag(sh2, sl2, sS[cb], sS[cb + 4]);
          split_frag(dsh, dsl, sD[cb], sD[cb + 4]);
          mma_3xtf32(accQ[nt], oh, ol, sh2, sl2);
          mma_3xtf32(accH[nt], vh, vl, dsh, dsl);
          mma_3xtf32(accG[nt], dh, dl, sh2, sl2);
        }
      }
    }
    if (warp >= 4) {  // dT_b += dV~ P^T (warps 4, 5), dA += dO V~^T (warps 6, 7): one 8-column tile each
      const bool isA = warp >= 6;
      const float *Am = isA ? dOr : dVtr, *Bm = isA ? Vtr : Pr;
      const int n0 = 8 * (warp & 1);
#pragma unroll
      for (int k0 = 0; k0 < kGradDvt; k0 += 8) {
        const int ra = g * lr + k0 + t, rb = (g + 8) * lr + k0 + t, cb = (n0 + g) * lr + k0 + t;
        const float av[4] = {Am[ra], Am[rb], Am[ra + 4], Am[rb + 4]};
        const float bv[2] = {Bm[cb], Bm[cb + 4]};
        mma_3xtf32(accTA, av, bv);
      }
    } else if (tid < dk) {  // dgamma_i += sum over the pass's columns of dS'[i][c] S[i][c]
#pragma unroll
      for (int q = 0; q < kGradDvt; q += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(sS + tid * lr + q);
        const float4 y = *reinterpret_cast<const float4 *>(sD + tid * lr + q);
        accGam += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
      }
    }
  }
  __syncthreads();  // the pass buffers become dQb, dKb, dGK, dKh
  if (16 * warp < dk)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {  // D fragment: rows g, g + 8; columns 2t, 2t + 1 of the tile
      const int o = g * ld + 16 * warp + 8 * nt + 2 * t, o8 = o + 8 * ld;
      *reinterpret_cast<float2 *>(dQb + o) = make_float2(accQ[nt][0], accQ[nt][1]);
      *reinterpret_cast<float2 *>(dQb + o8) = make_float2(accQ[nt][2], accQ[nt][3]);
      *reinterpret_cast<float2 *>(dKh + o) = make_float2(accH[nt][0], accH[nt][1]);
      *reinterpret_cast<float2 *>(dKh + o8) = make_float2(accH[nt][2], accH[nt][3]);
      *reinterpret_cast<float2 *>(dGK + o) = make_float2(accG[nt][0], accG[nt][1]);
      *reinterpret_cast<float2 *>(dGK + o8) = make_float2(accG[nt][2], accG[nt][3]);
    }
  if (warp >= 4) {
    float *dst = (warp >= 6 ? dA : dTb) + g * kBC + 8 * (warp & 1) + 2 * t;
    *reinterpret_cast<float2 *>(dst) = make_float2(accTA[0], accTA[1]);
    *reinterpret_cast<float2 *>(dst + 8 * kBC) = make_float2(accTA[2], accTA[3]);
  }
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
    const float G = c.G[r * ld + i];
    const float eg = expf(G), ei = expf(-G), eh = ei * c.gam[i];  // e^{G_C - G}
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
  const size_t ld = (size_t)dk + 4, lr = kGradDvt + 4;
  const size_t pass = 5 * kBC * lr + 4 * kBC * kBC + 4 * (size_t)dk * lr + 2 * 512;
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
