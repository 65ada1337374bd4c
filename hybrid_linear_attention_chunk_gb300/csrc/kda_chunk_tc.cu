// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 MMA with
// TMEM accumulators, operands in 128-byte-swizzled shared memory, V tiles
// brought in by TMA).  bf16 q/k/v/out, fp32 log-decay and beta, fp32 state,
// dk = dv = 128, chunk C = 64.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
//
// One CTA walks the chunks of one (sequence, head) chain.  With Q, K, V the
// chunk's rows, G the within-chunk cumulative log-decay (row r includes token
// r), Gamma = exp(G) and gamma_C = exp(G_C) ([K3-notes §2.2, chunkwise form]):
//   M1  [A ; L''] = [Q o Gamma ; Gamma o K] (K / Gamma)^T      (M=128 N=64 K=128)
//   A  = Tril_incl(A), L = StrictTril(diag(beta) L'')
//   T_b = (I + L)^{-1} diag(beta)   blocked forward substitution on CUDA cores
//   M2  [0 | U^T] = V^T [0 ; T_b]^T                              (M=128 N=128 K=64)
//   M3  W^T = (Gamma o K)^T T_b^T                                (M=128 N=64 K=64)
//   M4  [O^T | V~^T] += S^T [Q o Gamma ; -W]^T                   (M=128 N=128 K=128)
//   M5  O^T += V~^T A^T                                          (M=128 N=64 K=64)
//   M6  D = V~^T (K o gamma_C / Gamma)                           (M=128 N=128 K=64)
//   S^T <- S^T Diag(gamma_C) + D     (fp32 master state kept in TMEM)
// Every product is computed transposed so that M = 128 (dv or dk) and the
// tensor core runs at full width; TMEM lane j holds row j of the result.
//
// Range guard ([K3-notes §2.2, Eq. 5 and Fig. 3]): with log-decay >= -5 a
// 16-token tile sums to >= -80.  If every channel's chunk total G_C is >= -80
// the chunk start serves as the single decay reference (all factors within
// e^{+-80}).  Otherwise M1 runs in four accumulating rounds, one per 16-token
// key tile b, with the cumulative decay at tile b's start as the reference:
// query-side factors are <= 1 (rows before the tile are zeroed) and key-side
// factors are <= e^{80}.
//
// Warp roles: warps 0-7 (256 threads) do the decay prologue, the solve and
// the TMEM epilogues; warp 8 allocates TMEM and issues the TMA loads of V;
// warp 9 issues the MMAs.  Hand-offs go through mbarriers; every wait is
// bounded (a 2 s watchdog), and on a time-out all roles leave their loops,
// drain outstanding copies and MMAs, free TMEM and return with an error bit
// set in a device word the host can read.
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

__device__ unsigned int g_tc_watchdog;  // OR of time-out codes since last cleared

namespace {
using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 320;
constexpr int kMathThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSingleRefBound2 = kSingleRefBound * kLog2e;  // the -80 bound in log2 units

// Shared-memory map (byte offsets from a 1024-aligned base).
constexpr uint32_t OFF_QG = 0;        // [Q o Gamma ; Gamma o K -> -W]: 128 rows x 128, 2 K-halves
constexpr uint32_t OFF_KB = 32768;    // K / Gamma: 64 rows x 128
constexpr uint32_t OFF_KH = 49152;    // K o gamma_C / Gamma: 64 rows x 128 (MN-major B of M6)
constexpr uint32_t OFF_ZT = 65536;    // [0 ; T_b]: 128 rows x 64
constexpr uint32_t OFF_ST = 81920;    // S^T bf16: 128 rows x 128
constexpr uint32_t OFF_VT = 114688;   // V~^T bf16: 128 rows x 64; also the output staging tile
constexpr uint32_t OFF_V0 = 131072;   // V tile stage 0 (TMA): 64 rows x 128
constexpr uint32_t OFF_V1 = 147456;   // V tile stage 1
constexpr uint32_t OFF_AM = 163840;   // A bf16: 64 rows x 64
constexpr uint32_t OFF_LF = 172032;   // L fp32 [64][65]
constexpr uint32_t OFF_TF = 188672;   // T fp32 [64][65]
constexpr uint32_t OFF_XF = 205312;   // solve scratch fp32 [3][16][17]
constexpr uint32_t OFF_CTL = 208640;  // control block (below)
constexpr uint32_t SMEM_USED = OFF_CTL + 4096;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
constexpr int LDF = 65;                            // fp32 row stride of L and T

// TMEM columns (512 allocated; lane = row of each transposed product).
constexpr uint32_t TM_D1 = 0;     // M1 result, later M3 (W^T)
constexpr uint32_t TM_O = 64;     // O^T accumulator (M2 zeroes it; M4, M5 add)
constexpr uint32_t TM_U = 128;    // U^T, then V~^T after M4
constexpr uint32_t TM_D6 = 192;   // M6 result
constexpr uint32_t TM_S = 320;    // fp32 master state S^T

enum Bar : int {
  B_PREP = 0, B_M1, B_SOLVE, B_M23, B_W, B_M4, B_E4, B_M56, B_VFULL0, B_VFULL1, B_VEMPTY0,
  B_VEMPTY1, B_TEARDOWN, B_COUNT
};

struct Ctl {
  uint64_t bar[16];
  float bs[64];          // beta of the chunk's rows (0 past the end)
  float gam[128];        // gamma_C per channel
  float tot[4][128];     // per-16-row-group log2-decay sums
  uint32_t tmem_slot;
  int abort;             // any role gave up
  int nb;                // M1 rounds for the current chunk (1 or 4)
  int slow[2];           // range-guard vote, double-buffered by chunk parity
  int go[2];             // math-group wait result, double-buffered
};
static_assert(sizeof(Ctl) <= 4096, "control block");

struct TcArgs {
  PrefillArgs a;
  unsigned int *err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
  return __bfloat1622float2(v);
}

// Named barrier 1 over the 256 math threads (warps reconverged first).
__device__ __forceinline__ void math_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// a[i] for a runtime i without spilling the array to local memory
__device__ __forceinline__ float pick4(const float (&a)[4], int i) {
  return i == 0 ? a[0] : (i == 1 ? a[1] : (i == 2 ? a[2] : a[3]));
}

__device__ __forceinline__ void st_shared_u32(uint8_t *p, uint32_t v) {
  *reinterpret_cast<uint32_t *>(p) = v;
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Stores 16 fp32 values as bf16 at columns [c0, c0+16) of row `row` of a
// 128-byte-swizzled tile (c0 a multiple of 8 within one 64-column half).
__device__ __forceinline__ void st_row16_bf16(uint8_t *tile, uint32_t row, uint32_t c0, const float (&v)[16]) {
  st_shared_v4(tile + sw128_offset(row, c0), pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
               pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  st_shared_v4(tile + sw128_offset(row, c0 + 8), pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]),
               pack_bf16(v[12], v[13]), pack_bf16(v[14], v[15]));
}

// Inputs of one chunk held in registers by a math thread: channel pair
// (2p, 2p+1), rows [16 rg, 16 rg + 16).
struct Prefetch {
  uint32_t q[16], k[16];
  float2 g[16];
  float beta;
};

__device__ __forceinline__ void prefetch_chunk(Prefetch &pf, const PrefillArgs &a, int h, int t0, int len,
                                               int p, int rg, int mtid) {
  const int H = a.H;
  const uint32_t *q = reinterpret_cast<const uint32_t *>(a.q);
  const uint32_t *k = reinterpret_cast<const uint32_t *>(a.k);
  const float2 *g = reinterpret_cast<const float2 *>(a.g);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = 16 * rg + r;
    if (row < len) {
      const size_t e = ((size_t)(t0 + row) * H + h) * (kD / 2) + p;  // in element pairs
      pf.q[r] = __ldg(q + e);
      pf.k[r] = __ldg(k + e);
      pf.g[r] = __ldg(g + e);
    } else {
      pf.q[r] = 0u;
      pf.k[r] = 0u;
      pf.g[r] = make_float2(0.f, 0.f);
    }
  }
  pf.beta = 0.f;
  if (mtid < kC && mtid < len) pf.beta = __ldg(reinterpret_cast<const float *>(a.beta) + (size_t)(t0 + mtid) * H + h);
}

// The math group's view of an mbarrier wait: thread 0 waits, the group
// synchronises, and everyone gets the same verdict (so that no thread can
// leave while others sit in a group barrier).
__device__ __forceinline__ bool math_wait(Ctl *ctl, int b, uint32_t &phase_bits, int mtid, int &seq,
                                          unsigned int *err) {
  const uint32_t parity = (phase_bits >> b) & 1u;
  if (mtid == 0) {
    const bool ok = mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, err, 1u << b);
    ctl->go[seq & 1] = ok && !ctl->abort;
  }
  phase_bits ^= 1u << b;
  math_bar();
  const bool go = ctl->go[seq & 1] != 0;
  ++seq;
  tc_fence_after();
  return go;
}

// Publish the group's shared-memory writes to the async proxy and signal.
__device__ __forceinline__ void math_signal(Ctl *ctl, int b, int mtid) {
  fence_proxy_async_smem();
  tc_fence_before();
  math_bar();
  if (mtid == 0) mbar_arrive(smem_u32(&ctl->bar[b]));
}

__device__ __forceinline__ bool one_wait(Ctl *ctl, int b, uint32_t &phase_bits, unsigned int *err) {
  const uint32_t parity = (phase_bits >> b) & 1u;
  phase_bits ^= 1u << b;
  const bool ok = mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, err, 1u << b);
  tc_fence_after();
  return ok;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_v, TcArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl *ctl = reinterpret_cast<Ctl *>(sm + OFF_CTL);
  const PrefillArgs &a = A.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  int bos, eos;
  seq_range(a, n, bos, eos);
  const int nchunks = (eos - bos + kC - 1) / kC;

  if (warp == kProducerWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(smem_u32(&ctl->bar[b]), 1);
    ctl->abort = 0;
    ctl->nb = 1;
    ctl->slow[0] = ctl->slow[1] = 0;
    ctl->go[0] = ctl->go[1] = 0;
    fence_mbar_init();
  }
  if (tid < kMathThreads) {
    // rows 0..63 of [0 ; T_b] stay zero for the whole kernel
    for (int e = tid; e < 8192 / 16; e += kMathThreads)
      reinterpret_cast<uint4 *>(sm + OFF_ZT)[e] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_v);
      uint32_t empty_phase = 0;
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int stage = c & 1, use = c >> 1;
        if (use > 0) {
          const int b = B_VEMPTY0 + stage;
          const uint32_t parity = (empty_phase >> stage) & 1u;
          empty_phase ^= 1u << stage;
          if (!mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, A.err, 1u << b)) break;
        }
        const uint32_t full = smem_u32(&ctl->bar[B_VFULL0 + stage]);
        const uint32_t dst = smem_u32(sm + (stage ? OFF_V1 : OFF_V0));
        mbar_arrive_expect_tx(full, 2 * kC * 64 * 2);
        tma_load_3d(dst, &tmap_v, full, 0, h, bos + c * kC);
        tma_load_3d(dst + 8192, &tmap_v, full, 64, h, bos + c * kC);
        ++issued;
      }
      // the last load of each stage must have landed before the CTA retires
      for (int c = issued - 2 > 0 ? issued - 2 : 0; c < issued; ++c) {
        const int stage = c & 1, use = c >> 1;
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&ctl->bar[B_VFULL0 + stage]), use & 1, &no_abort, A.err, 1u << 16);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t ph = 0;
      const uint32_t qg = smem_u32(sm + OFF_QG), kb = smem_u32(sm + OFF_KB), kh = smem_u32(sm + OFF_KH);
      const uint32_t zt = smem_u32(sm + OFF_ZT), st = smem_u32(sm + OFF_ST), vt = smem_u32(sm + OFF_VT);
      const uint32_t am = smem_u32(sm + OFF_AM);
      constexpr uint32_t id_m1 = idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t id_m2 = idesc_bf16_f32(128, 128, 1, 0);
      constexpr uint32_t id_m3 = idesc_bf16_f32(128, 64, 1, 0);
      constexpr uint32_t id_m4 = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t id_m5 = idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t id_m6 = idesc_bf16_f32(128, 128, 0, 1);
      for (int c = 0; c < nchunks; ++c) {
        const int stage = c & 1;
        if (!one_wait(ctl, B_PREP, ph, A.err)) break;
        const int nb = ctl->nb;
        bool ok = true;
        for (int r = 0; r < nb && ok; ++r) {
          if (r > 0) ok = one_wait(ctl, B_PREP, ph, A.err);
          if (!ok) break;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t koffb = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_bf16_ss(tbase + TM_D1, smem_desc_sw128(qg + koff, 16, 1024),
                        smem_desc_sw128(kb + koffb, 16, 1024), id_m1, (kk > 0 || r > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&ctl->bar[B_M1]));
        }
        if (!ok) break;
        if (!one_wait(ctl, B_SOLVE, ph, A.err)) break;
        if (!one_wait(ctl, B_VFULL0 + stage, ph, A.err)) break;
        const uint32_t vs = smem_u32(sm + (stage ? OFF_V1 : OFF_V0));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // M2: [0 | U^T] = V^T [0 ; T_b]^T    (A = V, MN-major; B = [0 ; T_b], K-major)
          mma_bf16_ss(tbase + TM_O, smem_desc_sw128(vs + kk * 2048, 8192, 1024),
                      smem_desc_sw128(zt + kk * 32, 16, 1024), id_m2, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // M3: W^T = (Gamma o K)^T T_b^T     (A = rows 64..127 of QG, MN-major)
          mma_bf16_ss(tbase + TM_D1, smem_desc_sw128(qg + 8192 + kk * 2048, 16384, 1024),
                      smem_desc_sw128(zt + 8192 + kk * 32, 16, 1024), id_m3, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&ctl->bar[B_M23]));
        mma_commit(smem_u32(&ctl->bar[B_VEMPTY0 + stage]));
        if (!one_wait(ctl, B_W, ph, A.err)) break;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // M4: [O^T | V~^T] += S^T [Q o Gamma ; -W]^T
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tbase + TM_O, smem_desc_sw128(st + koff, 16, 1024),
                      smem_desc_sw128(qg + koff, 16, 1024), id_m4, 1u);
        }
        mma_commit(smem_u32(&ctl->bar[B_M4]));
        if (!one_wait(ctl, B_E4, ph, A.err)) break;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // M5: O^T += V~^T A^T
          mma_bf16_ss(tbase + TM_O, smem_desc_sw128(vt + kk * 32, 16, 1024),
                      smem_desc_sw128(am + kk * 32, 16, 1024), id_m5, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // M6: D = V~^T (K o gamma_C / Gamma)   (B MN-major)
          mma_bf16_ss(tbase + TM_D6, smem_desc_sw128(vt + kk * 32, 16, 1024),
                      smem_desc_sw128(kh + kk * 2048, 8192, 1024), id_m6, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&ctl->bar[B_M56]));
      }
      // every MMA issued above has completed before TMEM is released
      mma_commit(smem_u32(&ctl->bar[B_TEARDOWN]));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&ctl->bar[B_TEARDOWN]), 0, &no_abort, A.err, 1u << 17);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- math group
    const int mtid = tid;                 // 0..255
    const int qw = warp & 3, ch = warp >> 2;
    const int p = mtid & 63, rg = mtid >> 6;
    uint32_t ph = 0;
    int seq = 0;
    const size_t sbase = ((size_t)n * H + h) * kD * kD;
    const int jrow = 32 * qw + lane;      // TMEM lane = row j (or i) of the transposed products

    // initial state -> TMEM (fp32 master) and S^T bf16 operand
    for (int blk = 0; blk < 4; ++blk) {
      const int i0 = 64 * ch + 16 * blk;
      float s[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) s[c] = a.s0 ? a.s0[sbase + (size_t)(i0 + c) * kD + jrow] : 0.f;
      tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
      st_row16_bf16(sm + OFF_ST + ch * 16384, jrow, 16 * blk, s);
    }
    tmem_wait_st();

    Prefetch pf;
    if (nchunks > 0) prefetch_chunk(pf, a, h, bos, min(kC, eos - bos), p, rg, mtid);
    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
      const int t0 = bos + c * kC;
      const int len = min(kC, eos - t0);
      // ---------------- decay prologue: cumulative log2-decay and scaled operands
      float G0[16], G1[16];
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        a0 += pf.g[r].x * kLog2e;
        a1 += pf.g[r].y * kLog2e;
        G0[r] = a0;
        G1[r] = a1;
      }
      ctl->tot[rg][2 * p] = a0;
      ctl->tot[rg][2 * p + 1] = a1;
      if (mtid < kC) ctl->bs[mtid] = pf.beta;
      math_bar();
      float ref0[4], ref1[4], run0 = 0.f, run1 = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        ref0[b] = run0;
        ref1[b] = run1;
        run0 += ctl->tot[b][2 * p];
        run1 += ctl->tot[b][2 * p + 1];
      }
      const float GC0 = run0, GC1 = run1;
      const float own0 = pick4(ref0, rg), own1 = pick4(ref1, rg);
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        G0[r] += own0;
        G1[r] += own1;
      }
      if (rg == 0) {
        ctl->gam[2 * p] = ex2(GC0);
        ctl->gam[2 * p + 1] = ex2(GC1);
      }
      if (GC0 < kSingleRefBound2 || GC1 < kSingleRefBound2) atomicOr(&ctl->slow[c & 1], 1);
      math_bar();
      const bool slow = ctl->slow[c & 1] != 0;
      if (mtid == 0) {
        ctl->slow[(c + 1) & 1] = 0;
        ctl->nb = slow ? 4 : 1;
      }
      const uint32_t half = (uint32_t)(p >> 5), col = (uint32_t)((2 * p) & 63);
      uint8_t *qg_q = sm + OFF_QG + half * 16384;
      uint8_t *kb_t = sm + OFF_KB + half * 8192;
      uint8_t *kh_t = sm + OFF_KH + half * 8192;
      if (!slow) {
        const float gc0 = ex2(GC0), gc1 = ex2(GC1);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const uint32_t row = 16 * rg + r;
          const float e0 = ex2(G0[r]), e1 = ex2(G1[r]);
          const float i0 = ex2(-G0[r]), i1 = ex2(-G1[r]);
          const float2 qv = unpack_bf16(pf.q[r]), kv = unpack_bf16(pf.k[r]);
          st_shared_u32(qg_q + sw128_offset(row, col), pack_bf16(qv.x * e0, qv.y * e1));
          st_shared_u32(qg_q + sw128_offset(64 + row, col), pack_bf16(kv.x * e0, kv.y * e1));
          const float kb0 = kv.x * i0, kb1 = kv.y * i1;
          st_shared_u32(kb_t + sw128_offset(row, col), pack_bf16(kb0, kb1));
          st_shared_u32(kh_t + sw128_offset(row, col), pack_bf16(kb0 * gc0, kb1 * gc1));
        }
        math_signal(ctl, B_PREP, mtid);
        alive = math_wait(ctl, B_M1, ph, mtid, seq, A.err);
      } else {
        for (int b = 0; b < 4 && alive; ++b) {
          const float rb0 = pick4(ref0, b), rb1 = pick4(ref1, b);
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const uint32_t row = 16 * rg + r;
            const float2 qv = unpack_bf16(pf.q[r]), kv = unpack_bf16(pf.k[r]);
            float qa = 0.f, qb = 0.f, ka = 0.f, kbv = 0.f, ba = 0.f, bb = 0.f;
            if (rg >= b) {
              const float e0 = ex2(G0[r] - rb0), e1 = ex2(G1[r] - rb1);
              qa = qv.x * e0; qb = qv.y * e1;
              ka = kv.x * e0; kbv = kv.y * e1;
            }
            if (rg == b) {
              ba = kv.x * ex2(rb0 - G0[r]);
              bb = kv.y * ex2(rb1 - G1[r]);
            }
            st_shared_u32(qg_q + sw128_offset(row, col), pack_bf16(qa, qb));
            st_shared_u32(qg_q + sw128_offset(64 + row, col), pack_bf16(ka, kbv));
            st_shared_u32(kb_t + sw128_offset(row, col), pack_bf16(ba, bb));
          }
          math_signal(ctl, B_PREP, mtid);
          alive = math_wait(ctl, B_M1, ph, mtid, seq, A.err);
        }
        if (!alive) break;
        // operands with the chunk start as reference (may underflow to 0: fine)
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const uint32_t row = 16 * rg + r;
          const float2 qv = unpack_bf16(pf.q[r]), kv = unpack_bf16(pf.k[r]);
          const float e0 = ex2(G0[r]), e1 = ex2(G1[r]);
          st_shared_u32(qg_q + sw128_offset(row, col), pack_bf16(qv.x * e0, qv.y * e1));
          st_shared_u32(qg_q + sw128_offset(64 + row, col), pack_bf16(kv.x * e0, kv.y * e1));
          st_shared_u32(kh_t + sw128_offset(row, col),
                        pack_bf16(kv.x * ex2(GC0 - G0[r]), kv.y * ex2(GC1 - G1[r])));
        }
      }
      if (!alive) break;
      // next chunk's inputs travel while this one computes
      if (c + 1 < nchunks) prefetch_chunk(pf, a, h, t0 + kC, min(kC, eos - t0 - kC), p, rg, mtid);

      // ---------------- masks, L, and T_b = (I + L)^{-1} diag(beta)
      {
        float *Lf = reinterpret_cast<float *>(sm + OFF_LF);
        float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
        float *Xf = reinterpret_cast<float *>(sm + OFF_XF);
        if (qw < 2) {
          const int r = 32 * qw + lane;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[16];
            const int s0 = 32 * ch + 16 * hh;
            tmem_ld16(tmem_addr(tbase, 32 * qw, TM_D1 + s0), v);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) v[cc] = (s0 + cc <= r) ? v[cc] : 0.f;
            st_row16_bf16(sm + OFF_AM, r, s0, v);
          }
        } else {
          const int r = 32 * (qw - 2) + lane;
          const float br = ctl->bs[r];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[16];
            const int s0 = 32 * ch + 16 * hh;
            tmem_ld16(tmem_addr(tbase, 32 * qw, TM_D1 + s0), v);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) Lf[r * LDF + s0 + cc] = (s0 + cc < r) ? br * v[cc] : 0.f;
          }
        }
        math_bar();
        // diagonal 16x16 blocks by forward substitution (one column per thread);
        // the blocks above the diagonal are zero
        if (mtid < 64) {
          const int ab = mtid >> 4, cc = mtid & 15, base = 16 * ab;
          float x[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            float acc = (rr == cc) ? 1.f : 0.f;
            if (rr > cc) {
#pragma unroll
              for (int m = 0; m < rr; ++m)
                if (m >= cc) acc -= Lf[(base + rr) * LDF + base + m] * x[m];
            }
            x[rr] = acc;
            Tf[(base + rr) * LDF + base + cc] = acc;
          }
        } else {
          for (int e = mtid - 64; e < 6 * 256; e += 192) {
            const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
            const int ab = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            Tf[(16 * ab + rr) * LDF + 16 * bb + cc] = 0.f;
          }
        }
        math_bar();
        // off-diagonal blocks by distance d: T_ab = -T_aa sum_{c=b}^{a-1} L_ac T_cb
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
          const int nblk = 4 - d;
          for (int e = mtid; e < nblk * 256; e += 256) {
            const int b = e >> 8, ab = b + d, rr = (e >> 4) & 15, cc = e & 15;
            float acc = 0.f;
            for (int cb = b; cb < ab; ++cb) {
#pragma unroll
              for (int m = 0; m < 16; ++m)
                acc += Lf[(16 * ab + rr) * LDF + 16 * cb + m] * Tf[(16 * cb + m) * LDF + 16 * b + cc];
            }
            Xf[(b * 16 + rr) * 17 + cc] = acc;
          }
          math_bar();
          for (int e = mtid; e < nblk * 256; e += 256) {
            const int b = e >> 8, ab = b + d, rr = (e >> 4) & 15, cc = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc += Tf[(16 * ab + rr) * LDF + 16 * ab + m] * Xf[(b * 16 + m) * 17 + cc];
            Tf[(16 * ab + rr) * LDF + 16 * b + cc] = -acc;
          }
          math_bar();
        }
        {
          const int r = mtid >> 2, s0 = (mtid & 3) * 16;
          float v[16];
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) v[cc] = Tf[r * LDF + s0 + cc] * ctl->bs[s0 + cc];
          st_row16_bf16(sm + OFF_ZT, 64 + r, s0, v);
        }
      }
      math_signal(ctl, B_SOLVE, mtid);

      // ---------------- W^T (TMEM) -> -W, rows 64..127 of QG
      if (!(alive = math_wait(ctl, B_M23, ph, mtid, seq, A.err))) break;
      {
        const int i = jrow;
        uint8_t *dst = sm + OFF_QG + (i >> 6) * 16384;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[16];
          const int r0 = 32 * ch + 16 * hh;
          tmem_ld16(tmem_addr(tbase, 32 * qw, TM_D1 + r0), v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc)
            *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_offset(64 + r0 + cc, i & 63)) =
                __float2bfloat16_rn(-v[cc]);
        }
      }
      math_signal(ctl, B_W, mtid);

      // ---------------- V~^T (TMEM) -> bf16 operand
      if (!(alive = math_wait(ctl, B_M4, ph, mtid, seq, A.err))) break;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v[16];
        const int r0 = 32 * ch + 16 * hh;
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_U + r0), v);
        tmem_wait_ld();
        st_row16_bf16(sm + OFF_VT, jrow, r0, v);
      }
      math_signal(ctl, B_E4, mtid);

      // ---------------- state update and output
      if (!(alive = math_wait(ctl, B_M56, ph, mtid, seq, A.err))) break;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        const int i0 = 64 * ch + 16 * blk;
        float dd[16], s[16];
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_D6 + i0), dd);
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) s[cc] = ctl->gam[i0 + cc] * s[cc] + dd[cc];
        tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        st_row16_bf16(sm + OFF_ST + ch * 16384, jrow, 16 * blk, s);
      }
      {
        __nv_bfloat16 *ostage = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_VT);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[16];
          const int r0 = 32 * ch + 16 * hh;
          tmem_ld16(tmem_addr(tbase, 32 * qw, TM_O + r0), v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) ostage[(r0 + cc) * kD + jrow] = __float2bfloat16_rn(v[cc]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      math_bar();
      {
        const uint4 *src = reinterpret_cast<const uint4 *>(sm + OFF_VT);
        uint4 *o = reinterpret_cast<uint4 *>(a.o);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int idx = it * kMathThreads + mtid, row = idx >> 4, c16 = idx & 15;
          if (row < len) o[((size_t)(t0 + row) * H + h) * (kD / 8) + c16] = src[idx];
        }
      }
    }
    // final state
    if (alive && a.sT) {
      for (int blk = 0; blk < 4; ++blk) {
        const int i0 = 64 * ch + 16 * blk;
        float s[16];
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) a.sT[sbase + (size_t)(i0 + cc) * kD + jrow] = s[cc];
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool chunk_tc_supports(const PrefillArgs &a) {
  return a.qkv == KDA_BF16 && a.out == KDA_BF16 && a.gate == KDA_F32 && a.dk == kD && a.dv == kD &&
         a.chunk == kC;
}

cudaError_t launch_chunk_tc(const PrefillArgs &a, cudaStream_t s) {
  if (a.N * a.H == 0) return cudaSuccess;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)(a.T_total > 0 ? a.T_total : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.H * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kC};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  void *wd = nullptr;
  e = cudaGetSymbolAddress(&wd, g_tc_watchdog);
  if (e != cudaSuccess) return e;
  TcArgs args{a, reinterpret_cast<unsigned int *>(wd)};
  chunk_tc_kernel<<<a.N * a.H, kThreads, SMEM_BYTES, s>>>(tmap, args);
  return cudaGetLastError();
}

cudaError_t read_tc_watchdog(unsigned int *flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_tc_watchdog, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_tc_watchdog, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace kda
