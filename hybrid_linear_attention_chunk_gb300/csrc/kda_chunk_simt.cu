// Chunked prefill on CUDA cores, fp32 arithmetic throughout.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
//
// This kernel covers every supported shape and dtype (fp32 inputs included,
// where the tensor-core kernel's bf16 operands would not meet fp32 accuracy).
// Per (sequence, head, dv tile) one CTA walks the chunks in order.  Per chunk
// of C tokens, with G the within-chunk cumulative log-decay (row r includes
// token r), Gamma = exp(G), gamma_C = exp(G_C):
//   A   = Tril_incl[(Q o Gamma)(K / Gamma)^T]          [K3-notes §2.2, chunkwise form]
//   L   = StrictTril[diag(beta)(Gamma o K)(K / Gamma)^T]
//   T_b = (I + L)^{-1} diag(beta)                     (UT transform, forward substitution)
//   V~  = T_b (V - (Gamma o K) S)                     (= U - W S with U = T_b V, W = T_b (Gamma o K))
//   O   = (Gamma o Q) S + A V~
//   S  <- Diag(gamma_C) S + (K o gamma_C / Gamma)^T V~
// In the layer form the log-decay is formed on load from the decay logits z,
// g = g_min Sigmoid(exp(A_h) z) ([K3-notes §2.2, Eq. 5]); the output norm and
// gate run afterwards over whole rows (launch_norm_gate), since a CTA here
// holds only a dv tile.
// Range guard ([K3-notes §2.2, Eq. 5 and Fig. 3]): when every channel's
// G_C >= -80 the Gram products use the chunk start as the one decay reference
// (all factors within e^{+-80}); otherwise each entry uses exp(G_r - G_s) <= 1
// directly, which cannot overflow.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kSimtThreads = 256;

struct SimtSmem {
  int ld;      // padded row stride of the [C][dk] arrays
  int dvt;     // dv tile width
  float *Q, *K, *GK, *V, *Vt, *A, *L, *T, *S, *b, *gam, *gC;
};

__device__ __forceinline__ SimtSmem carve(float *base, int C, int dk, int dvt) {
  SimtSmem m;
  m.ld = dk + 1;
  m.dvt = dvt;
  float *p = base;
  m.Q = p;  p += C * m.ld;
  m.K = p;  p += C * m.ld;
  m.GK = p; p += C * m.ld;
  m.V = p;  p += C * dvt;
  m.Vt = p; p += C * dvt;
  m.A = p;  p += C * C;
  m.L = p;  p += C * C;
  m.T = p;  p += C * C;
  m.S = p;  p += dk * dvt;
  m.b = p;  p += C;
  m.gam = p; p += dk;
  m.gC = p; p += dk;
  return m;
}

size_t simt_smem_bytes(int C, int dk, int dvt) {
  return sizeof(float) * ((size_t)3 * C * (dk + 1) + 2 * C * dvt + 3 * C * C + (size_t)dk * dvt + C + 2 * dk);
}

__global__ void __launch_bounds__(kSimtThreads)
chunk_simt_kernel(PrefillArgs a, int dvt) {
  extern __shared__ float smem_raw[];
  const int C = a.chunk, dk = a.dk, dv = a.dv, H = a.H;
  const int nh = blockIdx.x, n = nh / H, h = nh % H;
  const int j0 = blockIdx.y * dvt;
  const int tid = threadIdx.x;
  SimtSmem m = carve(smem_raw, C, dk, dvt);
  const int ld = m.ld;

  int bos, eos;
  seq_range(a, n, bos, eos);
  const kda_dtype gdt = a.gdt();
  const float zscale = a.A_log ? expf(a.A_log[h]) : 0.f;

  // initial state tile S[i][j0 + j]
  const size_t sbase = (size_t)nh * dk * dv;
  for (int e = tid; e < dk * dvt; e += kSimtThreads) {
    int i = e / dvt, j = e % dvt;
    m.S[e] = a.s0 ? a.s0[sbase + (size_t)i * dv + j0 + j] : 0.f;
  }

  for (int t0 = bos; t0 < eos; t0 += C) {
    const int len = min(C, eos - t0);
    __syncthreads();  // previous chunk fully consumed
    // ---- load (rows past the sequence end are zero: an exact identity step)
    for (int e = tid; e < C * dk; e += kSimtThreads) {
      int r = e / dk, i = e % dk;
      float qv = 0.f, kv = 0.f, gv = 0.f;
      if (r < len) {
        size_t idx = ((size_t)(t0 + r) * H + h) * dk + i;
        qv = ld_elem(a.q, idx, a.qkv);
        kv = ld_elem(a.k, idx, a.qkv);
        gv = ld_elem(a.g, idx, gdt);
        if (a.A_log) gv = decay_from_logit(gv, zscale, a.g_min);
      }
      m.Q[r * ld + i] = qv;
      m.K[r * ld + i] = kv;
      m.GK[r * ld + i] = gv;
    }
    for (int e = tid; e < C * dvt; e += kSimtThreads) {
      int r = e / dvt, j = e % dvt;
      m.V[e] = r < len ? ld_elem(a.v, ((size_t)(t0 + r) * H + h) * dv + j0 + j, a.qkv) : 0.f;
    }
    for (int r = tid; r < C; r += kSimtThreads)
      m.b[r] = r < len ? ld_elem(a.beta, (size_t)(t0 + r) * H + h, a.gate) : 0.f;
    __syncthreads();

    // ---- within-chunk cumulative log-decay, in place in GK
    int slow = 0;
    if (tid < dk) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        acc += m.GK[r * ld + tid];
        m.GK[r * ld + tid] = acc;
      }
      m.gam[tid] = expf(acc);
      m.gC[tid] = acc;
      slow = acc < kSingleRefBound;
    }
    slow = __syncthreads_or(slow);

    if (!slow) {
      // one reference (chunk start): Q o Gamma, K / Gamma, Gamma o K
      for (int e = tid; e < C * dk; e += kSimtThreads) {
        int r = e / dk, i = e % dk;
        float G = m.GK[r * ld + i];
        float eg = expf(G), ei = expf(-G);
        float kv = m.K[r * ld + i];
        m.Q[r * ld + i] *= eg;
        m.K[r * ld + i] = kv * ei;
        m.GK[r * ld + i] = kv * eg;
      }
      __syncthreads();
      for (int e = tid; e < C * C; e += kSimtThreads) {
        int r = e / C, s = e % C;
        float accA = 0.f, accL = 0.f;
        if (s <= r) {
          for (int i = 0; i < dk; ++i) {
            float kb = m.K[s * ld + i];
            accA += m.Q[r * ld + i] * kb;
            accL += m.GK[r * ld + i] * kb;
          }
        }
        m.A[e] = accA;
        m.L[e] = (s < r) ? m.b[r] * accL : 0.f;
      }
      __syncthreads();
      // K / Gamma -> K o gamma_C / Gamma
      for (int e = tid; e < C * dk; e += kSimtThreads) {
        int r = e / dk, i = e % dk;
        m.K[r * ld + i] *= m.gam[i];
      }
    } else {
      // every pair with its own exponent exp(G_r - G_s) <= 1
      for (int e = tid; e < C * C; e += kSimtThreads) {
        int r = e / C, s = e % C;
        float accA = 0.f, accL = 0.f;
        if (s <= r) {
          for (int i = 0; i < dk; ++i) {
            float d = expf(m.GK[r * ld + i] - m.GK[s * ld + i]);
            float ks = m.K[s * ld + i];
            accA += m.Q[r * ld + i] * ks * d;
            accL += m.K[r * ld + i] * ks * d;
          }
        }
        m.A[e] = accA;
        m.L[e] = (s < r) ? m.b[r] * accL : 0.f;
      }
      __syncthreads();
      for (int e = tid; e < C * dk; e += kSimtThreads) {
        int r = e / dk, i = e % dk;
        float G = m.GK[r * ld + i];
        float GC = m.gC[i];
        float kv = m.K[r * ld + i];
        float eg = expf(G);
        m.Q[r * ld + i] *= eg;
        m.GK[r * ld + i] = kv * eg;
        m.K[r * ld + i] = kv * expf(GC - G);
      }
    }
    // ---- T = (I + L)^{-1} by forward substitution, one column per thread
    if (tid < C) {
      const int s = tid;
      for (int r = 0; r < C; ++r) m.T[r * C + s] = (r == s) ? 1.f : 0.f;
      for (int r = s + 1; r < C; ++r) {
        float acc = 0.f;
        for (int mm = s; mm < r; ++mm) acc += m.L[r * C + mm] * m.T[mm * C + s];
        m.T[r * C + s] = -acc;
      }
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += kSimtThreads) m.T[e] *= m.b[e % C];  // T diag(beta)
    // ---- P = V - (Gamma o K) S   (in place in V)
    for (int e = tid; e < C * dvt; e += kSimtThreads) {
      int r = e / dvt, j = e % dvt;
      float acc = m.V[e];
      for (int i = 0; i < dk; ++i) acc -= m.GK[r * ld + i] * m.S[i * dvt + j];
      m.V[e] = acc;
    }
    __syncthreads();
    // ---- V~ = T_b P
    for (int e = tid; e < C * dvt; e += kSimtThreads) {
      int r = e / dvt, j = e % dvt;
      float acc = 0.f;
      for (int s = 0; s <= r; ++s) acc += m.T[r * C + s] * m.V[s * dvt + j];
      m.Vt[e] = acc;
    }
    __syncthreads();
    // ---- O = (Gamma o Q) S + A V~
    for (int e = tid; e < C * dvt; e += kSimtThreads) {
      int r = e / dvt, j = e % dvt;
      if (r >= len) continue;
      float acc = 0.f;
      for (int i = 0; i < dk; ++i) acc += m.Q[r * ld + i] * m.S[i * dvt + j];
      for (int s = 0; s <= r; ++s) acc += m.A[r * C + s] * m.Vt[s * dvt + j];
      st_elem(a.o, ((size_t)(t0 + r) * H + h) * dv + j0 + j, acc, a.out);
    }
    __syncthreads();
    // ---- S <- Diag(gamma_C) S + K^T V~  (K now holds K o gamma_C / Gamma)
    for (int e = tid; e < dk * dvt; e += kSimtThreads) {
      int i = e / dvt, j = e % dvt;
      float acc = m.gam[i] * m.S[e];
      for (int r = 0; r < C; ++r) acc += m.K[r * ld + i] * m.Vt[r * dvt + j];
      m.S[e] = acc;
    }
    if (float *cp = ckpt_ptr(a, n, h, t0 + len - bos)) {  // a checkpoint ends this chunk
      __syncthreads();
      for (int e = tid; e < dk * dvt; e += kSimtThreads) {
        int i = e / dvt, j = e % dvt;
        cp[(size_t)i * dv + j0 + j] = m.S[e];
      }
    }
  }
  __syncthreads();
  if (a.sT) {
    for (int e = tid; e < dk * dvt; e += kSimtThreads) {
      int i = e / dvt, j = e % dvt;
      a.sT[sbase + (size_t)i * dv + j0 + j] = m.S[e];
    }
  }
}

}  // namespace

cudaError_t launch_chunk_simt(const PrefillArgs &a, cudaStream_t s) {
  const int dvt = a.dv >= 64 ? 64 : a.dv;
  const size_t smem = simt_smem_bytes(a.chunk, a.dk, dvt);
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.N * a.H, a.dv / dvt);
  if (grid.x == 0) return cudaSuccess;
  chunk_simt_kernel<<<grid, kSimtThreads, smem, s>>>(a, dvt);
  return cudaGetLastError();
}

}  // namespace kda
