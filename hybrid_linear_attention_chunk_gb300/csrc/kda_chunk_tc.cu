// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 MMA with
// TMEM accumulators, operands in 128-byte-swizzled shared memory, inputs
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
//   T_b = (I + L)^{-1} diag(beta)   blocked substitution: CUDA cores (fp32), last level tf32 MMA
//   M2  U^T = V^T T_b^T                                          (M=128 N=64 K=64)
//   M3  W^T = (Gamma o K)^T T_b^T                                (M=128 N=64 K=64)
//   M4  V~^T = U^T - S^T W^T ;  O^T = S^T (Q o Gamma)^T          (M=128 N=64 K=128, twice)
//   M5  O^T += V~^T A^T                                          (M=128 N=64 K=64)
//   M6  S^T <- (S^T + V~^T (K / Gamma)) Diag(gamma_C)            (M=128 N=128 K=64)
// (fp32 master state in TMEM; the Diag(gamma_C) scaling is applied to the
// accumulated state in the same TMEM pass that refreshes its bf16 copy, and
// K / Gamma doubles as M1's key operand.  When the chunk took the per-tile
// range path, K / Gamma may not be formed: the state is scaled first and M6
// takes K o gamma_C / Gamma, as S^T <- S^T Diag(gamma_C) + V~^T (K o gamma_C / Gamma).)
// Every product is computed transposed so that M = 128 (dv or dk) and the
// tensor core runs at full width; TMEM lane j holds row j of the result.
// M4 reads its A operand, the bf16 copy of S^T, straight from TMEM.
//
// Two warp groups overlap consecutive chunks.  The chunk group (warps 0-7)
// runs one chunk ahead: decay prologue, M1, the UT solve, M2/M3, and the TMA
// loads of q, k, log-decay and v.  q and k land in the buffers that become
// the chunk's Q o Gamma and K o gamma_C / Gamma operands, which are then
// scaled in place.  M2/M3 complete asynchronously: their completion is what
// hands the chunk to the state group.  The state group (warps 8-11) runs the
// serial state chain: -W staging, M4, V~ staging, M5/M6, the gamma scaling,
// the bf16 state copy and the output.  Operands the state group still reads
// while the chunk group prepares the next chunk are double-buffered by chunk
// parity.  Thread 0 of each group issues that group's MMAs.
//
// Range guard ([K3-notes §2.2, Eq. 5 and Fig. 3]): with log-decay >= -5 a
// 16-token tile sums to >= -80.  If every channel's chunk total G_C is >= -80
// the chunk start serves as the single decay reference (all factors within
// e^{+-80}).  Otherwise M1 runs in four accumulating rounds, one per 16-token
// key tile b, with the cumulative decay at tile b's start as the reference:
// query-side factors are <= 1 (rows before the tile are zeroed) and key-side
// factors are <= e^{80}.
//
// Layer gates ([K3-notes §2.2]), selected at compile time: with kZ the decay
// tile is the bf16 decay logits z and the prologue forms the log-decay
// g_min Sigmoid(exp(A_h) z) (Eq. 5) in registers; with kOG the output rows are
// normalised (RMSNorm over dv, from the bf16-rounded output) and gated by
// Sigmoid(out_gate), whose tile arrives by TMA during the chunk.
//
// Every wait on an mbarrier is bounded (2 s).  On a time-out both groups
// leave their loops, drain their MMAs and copies, free TMEM and return with a
// bit set in a device word the host can read (kda_device_watchdog).
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <stddef.h>
#include <string.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

__device__ unsigned int g_tc_watchdog;  // OR of time-out codes since last cleared

namespace {
using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 384;
constexpr int kChunkThreads = 256;  // warps 0-7
constexpr int kStateThreads = 128;  // warps 8-11
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSingleRefBound2 = kSingleRefBound * kLog2e;  // the -80 bound in log2 units

// Shared-memory map (byte offsets from a 1024-aligned base).  "x2" buffers
// are indexed by chunk parity.
constexpr uint32_t OFF_QG = 0;        // 48 KB: per 64-column K-half (stride KHALF):
                                      //   [Q o Gamma, even chunks | Gamma o K | Q o Gamma, odd chunks]
constexpr uint32_t KHALF = 24576;
constexpr uint32_t OFF_KB = 49152;    // 16 KB: K / Gamma -> L, then T over it (fp32 64x64)
constexpr uint32_t OFF_TF = 65536;    // 16 KB: solve scratch: T_[01][01]^T and X^T (tf32 B operands of
                                      //   the level-2 products, 4 KB each), level-1 products (2 KB)
constexpr uint32_t OFF_KH = 81920;    // x2 16 KB: K / Gamma (B of M1, MN-major B of M6), or
                                      //   K o gamma_C / Gamma after the per-tile range path
constexpr uint32_t OFF_AM = 114688;   // x2 8 KB: A bf16, 64 rows x 64
constexpr uint32_t OFF_ZT = 131072;   // 8 KB: T_b bf16 (read by M2/M3)
constexpr uint32_t OFF_V = 139264;    // 16 KB: v tile (TMA), two 64-column boxes
constexpr uint32_t OFF_GS = 155648;   // 32 KB: log-decay tile (TMA), fp32 [64][128]
constexpr uint32_t OFF_VT = 188416;   // 16 KB: -W^T (MN-major), then V~^T, then the output tile
constexpr uint32_t OFF_PRO = 204800;  // 5 KB: decay prologue sums (written while M2/M3 may still run)
constexpr uint32_t OFF_CTL = 209920;  // 4 KB control block
constexpr uint32_t SMEM_USED = OFF_CTL + 4096;
constexpr uint32_t OFF_OG = SMEM_USED;  // 16 KB, output-gate variant only: out_gate tile (TMA), bf16 [64][128]
// + 1024 bytes of alignment slack
constexpr uint32_t smem_bytes(bool og) { return (og ? OFF_OG + 16384 : SMEM_USED) + 1024; }
static_assert(smem_bytes(true) <= 232448, "shared memory per CTA");

// TMEM columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // M1 result (chunk group)
constexpr uint32_t TM_W = 64;     // M3 result W^T (read by the state group)
constexpr uint32_t TM_U = 128;    // x2 64: U^T, V~^T after M4 (by chunk parity)
constexpr uint32_t TM_O = 256;    // O^T accumulator
constexpr uint32_t TM_STB = 320;  // bf16 S^T, two values per column (A operand of M4)
constexpr uint32_t TM_S = 384;    // fp32 master state S^T (128 columns)

enum Bar : int {
  B_M1 = 0, B_M23, B_VFULL, B_GFULL, B_QK0, B_QK1, B_TB, B_M4,
  B_M56, B_L2, B_TD_C, B_TD_S, B_OG, B_COUNT
};

struct Ctl {
  uint64_t bar[16];
  float gam[2][128];     // gamma_C per channel, by chunk parity
  float bs[64];          // beta of the chunk's rows (0 past the end)
  alignas(16) float nw[128];  // RMSNorm weight (output-gate variant), read as float4
  uint32_t tmem_slot;
  int abort;             // any thread gave up
  int go_c[2];           // chunk-group wait verdicts (double-buffered)
  int go_s[2];           // state-group wait verdicts
  int qk_iss[2], qk_lnd[2];  // q/k copies issued and waited for, by chunk parity
  int v_iss, v_lnd;          // v copies issued (chunk group) and waited for (state group)
  int og_iss, og_lnd;        // out_gate copies issued and waited for (state group)
  int slow[2];               // the chunk took the per-tile range path (by chunk parity)
};
static_assert(offsetof(Ctl, nw) % 16 == 0 && offsetof(Ctl, gam) % 16 == 0, "vector reads of the control block");
static_assert(sizeof(Ctl) <= 4096, "control block");

struct TcArgs {
  PrefillArgs a;
  unsigned int *err;
};

struct TcMaps {
  CUtensorMap q, k, v, g, og;
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

// Named barriers: 1 = chunk group (256 threads), 2 = state group (128).
__device__ __forceinline__ void bar_chunk() {
  __syncwarp();
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
// Chunk-group barrier that also returns whether any thread passed p = true.
__device__ __forceinline__ bool bar_chunk_or(bool p) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 256, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_state() {
  __syncwarp();
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Stores 16 fp32 values as bf16 at columns [c0, c0+16) of row `row` of a
// 128-byte-swizzled tile (c0 a multiple of 8 within one 64-column half).
__device__ __forceinline__ void st_row16_bf16(uint8_t *tile, uint32_t row, uint32_t c0, const float *v) {
  st_shared_v4(tile + sw128_offset(row, c0), pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
               pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  st_shared_v4(tile + sw128_offset(row, c0 + 8), pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]),
               pack_bf16(v[12], v[13]), pack_bf16(v[14], v[15]));
}

// Stores 4 fp32 values as bf16 at columns [c0, c0+4) of a 128-byte-swizzled
// tile (c0 a multiple of 4).
__device__ __forceinline__ void st_row4_bf16(uint8_t *tile, uint32_t row, uint32_t c0, const float4 &v) {
  *reinterpret_cast<uint2 *>(tile + sw128_offset(row, c0)) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
}

__device__ __forceinline__ void sts64(uint8_t *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }

__device__ __forceinline__ float4 unpack4_bf16(uint2 u) {
  const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint2 pack4_bf16(const float4 &v) {
  return make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
}

// Packs 32 fp32 values into 16 bf16 pairs (even element in the low half), the
// TMEM layout of an MMA A operand, and stores them at TMEM address taddr.
__device__ __forceinline__ void tmem_st_bf16x32(uint32_t taddr, const float (&v)[32]) {
  float w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = __uint_as_float(pack_bf16(v[2 * i], v[2 * i + 1]));
  tmem_st16(taddr, w);
}

// Shared-memory float4 load kept in program order with the other volatile
// loads, so that a batch of them issues back to back.
__device__ __forceinline__ float4 lds128(const float *p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ float f4c(const float4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ float4 mul4(const float4 &a, const float4 &b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

__device__ __forceinline__ float4 add4(const float4 &a, const float4 &b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 sub4(const float4 &a, const float4 &b) {
  return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}
__device__ __forceinline__ float4 neg4(const float4 &a) { return make_float4(-a.x, -a.y, -a.z, -a.w); }
__device__ __forceinline__ float4 ex2_4(const float4 &a) { return make_float4(ex2(a.x), ex2(a.y), ex2(a.z), ex2(a.w)); }


// acc += l[k0 + i] * t[i] for i < 8 (l: the left factor's row, four per float4)
__device__ __forceinline__ void fma8(float4 &acc, const float4 *l, int k0, const float4 (&t)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lv = f4c(l[(k0 + i) >> 2], (k0 + i) & 3);
    acc.x += lv * t[i].x; acc.y += lv * t[i].y; acc.z += lv * t[i].z; acc.w += lv * t[i].w;
  }
}


// Named barrier over the first n threads of the chunk group.
__device__ __forceinline__ void bar_sync_n(int id, int n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// fp32 64x64 matrices of the solve (L, T) are stored as two 32-column halves
// of 64 rows x 128 bytes whose 16-byte chunks are XORed with (row & 7): the
// 128-byte-swizzled K-major layout of a tf32 MMA operand.  Columns keep
// 4-float groups intact, and eight consecutive rows read at one column hit
// eight different banks.
__device__ __forceinline__ int lt_idx(int r, int c) {
  return ((c >> 5) << 11) + (r << 5) + ((((c >> 2) & 7) ^ (r & 7)) << 2) + (c & 3);
}

// Element (n, k) of a 32x32 fp32 K-major tf32 operand tile in the same layout.
__device__ __forceinline__ int tt_idx(int n, int k) { return (n << 5) + ((((k >> 2) & 7) ^ (n & 7)) << 2) + (k & 3); }

// A group-wide view of an mbarrier wait: the group's thread 0 waits, the
// group synchronises, and every thread gets the same verdict (so no thread
// can leave while others sit in a group barrier).
template <bool kChunkGroup>
__device__ __forceinline__ bool group_wait(Ctl *ctl, int b, uint32_t parity, int gtid, int &seq, unsigned int *err) {
  int *go = kChunkGroup ? ctl->go_c : ctl->go_s;
  if (gtid == 0) {
    const bool ok = mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, err, 1u << b);
    go[seq & 1] = ok && !ctl->abort;
  }
  if (kChunkGroup) bar_chunk(); else bar_state();
  const bool r = go[seq & 1] != 0;
  ++seq;
  tc_fence_after();
  return r;
}

// Single-thread wait (used by a group's thread 0 right before it issues).
__device__ __forceinline__ bool solo_wait(Ctl *ctl, int b, uint32_t parity, unsigned int *err) {
  const bool ok = mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, err, 1u << b);
  tc_fence_after();
  return ok;
}

// The group's shared-memory writes become visible to the tensor core (async
// proxy) and its TMEM accesses are ordered before what follows the barrier.
template <bool kChunkGroup>
__device__ __forceinline__ void group_publish() {
  fence_proxy_async_smem();
  tc_fence_before();
  if (kChunkGroup) bar_chunk(); else bar_state();
  tc_fence_after();
}

// ------------------------------------------------------------------- loads

struct Loader {
  const TcMaps *maps;
  Ctl *ctl;
  uint32_t sm_base;
  int h;
  int issued, landed;  // g copies
  uint32_t bytes;      // of one decay tile: fp32 log-decay or bf16 logits

  __device__ void g(int t0) {
    const uint32_t full = smem_u32(&ctl->bar[B_GFULL]);
    mbar_arrive_expect_tx(full, bytes);
    tma_load_3d(sm_base + OFF_GS, &maps->g, full, 0, h, t0);
    ++issued;
  }
  // a g copy still in flight after an abort must land before the CTA retires
  __device__ void drain(unsigned int *err) {
    volatile int no_abort = 0;
    if (issued > landed) mbar_wait(smem_u32(&ctl->bar[B_GFULL]), landed & 1, &no_abort, err, 1u << 20);
  }
};

// v of the chunk at t0 (issued by one thread of either group).
__device__ __forceinline__ void issue_v(const TcMaps *maps, Ctl *ctl, uint32_t sm_base, int h, int t0) {
  const uint32_t full = smem_u32(&ctl->bar[B_VFULL]);
  ++ctl->v_iss;
  mbar_arrive_expect_tx(full, 2 * 8192);
  tma_load_3d(sm_base + OFF_V, &maps->v, full, 0, h, t0);
  tma_load_3d(sm_base + OFF_V + 8192, &maps->v, full, 64, h, t0);
}

// out_gate tile of the chunk at t0 (state group).
__device__ __forceinline__ void issue_og(const TcMaps *maps, Ctl *ctl, uint32_t sm_base, int h, int t0) {
  const uint32_t full = smem_u32(&ctl->bar[B_OG]);
  ++ctl->og_iss;
  mbar_arrive_expect_tx(full, kC * kD * 2);
  tma_load_3d(sm_base + OFF_OG, &maps->og, full, 0, h, t0);
}


// Sigmoid of two values as 1/2 + tanh(x/2)/2, the tanh by the hardware's
// paired half-precision approximation (one special-function operation for
// two values).  Absolute error of the sigmoid < 1e-3, below the bf16 rounding
// of the gated output it scales.
__device__ __forceinline__ float2 sigmoid2_tanh(float a, float b) {
  __half2 h = __floats2half2_rn(0.5f * a, 0.5f * b);
  uint32_t t;
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<uint32_t *>(&h)));
  const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&t));
  return make_float2(fmaf(0.5f, f.x, 0.5f), fmaf(0.5f, f.y, 0.5f));
}

// Sum of squares of eight bf16 values.
__device__ __forceinline__ float sumsq8_bf16(uint4 o8) {
  const uint32_t ov[4] = {o8.x, o8.y, o8.z, o8.w};
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_bf16(ov[i]);
    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
  }
  return ss;
}

// Eight output channels (bf16 in o8) times r w Sigmoid(gate) (gate bf16 in g8).
__device__ __forceinline__ uint4 scale_gate8(uint4 o8, uint4 g8, const float *w, float r) {
  const uint32_t ov[4] = {o8.x, o8.y, o8.z, o8.w}, gv[4] = {g8.x, g8.y, g8.z, g8.w};
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = unpack_bf16(ov[i]), g = unpack_bf16(gv[i]);
    const float2 sg = sigmoid2_tanh(g.x, g.y);
    y[i] = pack_bf16(x.x * r * w[2 * i] * sg.x, x.y * r * w[2 * i + 1] * sg.y);
  }
  return make_uint4(y[0], y[1], y[2], y[3]);
}

// q and k of the chunk at t0 into the Q o Gamma and K-hat buffers of chunk
// parity par (issued by one thread of either group).
__device__ __forceinline__ void issue_qk(const TcMaps *maps, Ctl *ctl, uint32_t sm_base, int h, int t0, int par) {
  const uint32_t full = smem_u32(&ctl->bar[B_QK0 + par]);
  ++ctl->qk_iss[par];
  mbar_arrive_expect_tx(full, 4 * 8192);
  tma_load_3d(sm_base + OFF_QG + par * 16384, &maps->q, full, 0, h, t0);
  tma_load_3d(sm_base + OFF_QG + KHALF + par * 16384, &maps->q, full, 64, h, t0);
  tma_load_3d(sm_base + OFF_KH + par * 16384, &maps->k, full, 0, h, t0);
  tma_load_3d(sm_base + OFF_KH + par * 16384 + 8192, &maps->k, full, 64, h, t0);
}

// ------------------------------------------------------------- MMA batches

__device__ __forceinline__ void issue_m1(uint32_t tbase, uint32_t qg, uint32_t kb, int par, bool acc_first) {
  constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
  // A = 128 consecutive rows: [Q o Gamma ; Gamma o K] for even chunks,
  // [Gamma o K ; Q o Gamma] for odd ones (so the solve swaps lane roles)
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ka = (kk >> 2) * KHALF + par * 8192 + (kk & 3) * 32;
    const uint32_t kbo = (kk >> 2) * 8192 + (kk & 3) * 32;
    mma_bf16_ss(tbase + TM_D1, smem_desc_sw128(qg + ka, 16, 1024), smem_desc_sw128(kb + kbo, 16, 1024), id,
                (kk > 0 || acc_first) ? 1u : 0u);
  }
}

__device__ __forceinline__ void issue_m23(uint32_t tbase, uint32_t v, uint32_t qg, uint32_t zt, uint32_t tm_u) {
  constexpr uint32_t id = idesc_bf16_f32(128, 64, 1, 0);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // U^T = V^T T_b^T   (A = V, MN-major: 2 blocks of 64 columns)
    mma_bf16_ss(tbase + tm_u, smem_desc_sw128(v + kk * 2048, 8192, 1024), smem_desc_sw128(zt + kk * 32, 16, 1024),
                id, kk > 0 ? 1u : 0u);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // W^T = (Gamma o K)^T T_b^T   (A = the Gamma o K blocks, MN-major)
    mma_bf16_ss(tbase + TM_W, smem_desc_sw128(qg + 8192 + kk * 2048, KHALF, 1024),
                smem_desc_sw128(zt + kk * 32, 16, 1024), id, kk > 0 ? 1u : 0u);
}

__device__ __forceinline__ void issue_m4(uint32_t tbase, uint32_t vt, uint32_t qg, int par, uint32_t tm_u) {
  constexpr uint32_t id_w = idesc_bf16_f32(128, 64, 0, 1);
  constexpr uint32_t id_q = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)  // V~^T = U^T + S^T (-W)^T     (B = -W^T, MN-major, in the V~ buffer)
    mma_bf16_ts(tbase + tm_u, tbase + TM_STB + kk * 8, smem_desc_sw128(vt + kk * 2048, 8192, 1024), id_w, 1u);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {  // O^T = S^T (Q o Gamma)^T
    const uint32_t kb = (kk >> 2) * KHALF + par * 16384 + (kk & 3) * 32;
    mma_bf16_ts(tbase + TM_O, tbase + TM_STB + kk * 8, smem_desc_sw128(qg + kb, 16, 1024), id_q, kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void issue_m56(uint32_t tbase, uint32_t vt, uint32_t am, uint32_t kh) {
  constexpr uint32_t id5 = idesc_bf16_f32(128, 64, 0, 0);
  constexpr uint32_t id6 = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // O^T += V~^T A^T
    mma_bf16_ss(tbase + TM_O, smem_desc_sw128(vt + kk * 32, 16, 1024), smem_desc_sw128(am + kk * 32, 16, 1024),
                id5, 1u);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // S^T += V~^T (K o gamma_C / Gamma)   (B MN-major)
    mma_bf16_ss(tbase + TM_S, smem_desc_sw128(vt + kk * 32, 16, 1024),
                smem_desc_sw128(kh + kk * 2048, 8192, 1024), id6, 1u);
}

// The sequence of rank r when N packed sequences are ordered by length,
// longest first (ties by index).  Every thread of the CTA calls it; s holds
// N + 1 ints of shared scratch.
constexpr int kLongestFirstMax = 512;
__device__ int longest_first(const int32_t *cu, int N, int r, int *s, int tid) {
  for (int i = tid; i < N; i += kThreads) s[i] = cu[i + 1] - cu[i];
  __syncthreads();
  for (int j = tid; j < N; j += kThreads) {
    const int lj = s[j];
    int rank = 0;
    for (int i = 0; i < N; ++i) rank += (s[i] > lj) || (s[i] == lj && i < j);
    if (rank == r) s[N] = j;
  }
  __syncthreads();
  const int n = s[N];
  __syncthreads();  // the scratch is reused later
  return n;
}

template <bool kZ, bool kOG>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ TcMaps maps, TcArgs A) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base by pointer arithmetic on the shared array, so that the
  // compiler keeps every access through `sm` in the shared address space
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctl *ctl = reinterpret_cast<Ctl *>(sm + OFF_CTL);
  const PrefillArgs &a = A.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  // work item: (sequence n, segment, head h, kind) -- see PrefillArgs
  int item = blockIdx.x;
  const int kind = item % a.kinds;
  item /= a.kinds;
  const int h = item % H;
  item /= H;
  const int seg = item % a.nseg;
  int n = item / a.nseg;
  // Packed sequences run longest first: work items are handed to SMs in
  // index order, so a long sequence that came late would finish last.
  if (a.cu && a.N > 1 && a.N <= kLongestFirstMax)
    n = longest_first(a.cu, a.N, n, reinterpret_cast<int *>(sm + OFF_TF), tid);
  int bos, eos;
  seq_range(a, n, bos, eos);
  const int seq_bos = bos;  // checkpoints count tokens from the sequence start
  if (a.seg_tokens > 0) {
    const int sb = min(eos, bos + seg * a.seg_tokens);
    eos = min(eos, sb + a.seg_tokens);
    bos = sb;
  }
  const int nchunks = (eos - bos + kC - 1) / kC;
  const bool zero_v = kind == 1;  // transition pass: v = 0, identity entry state
  const float *s_in = (kind == 0 && a.s0) ? a.s0 + (((size_t)n * a.nseg + seg) * H + h) * kD * kD : nullptr;
  float *s_out = nullptr;
  if (a.sT) {
    if (a.kinds == 2) s_out = a.sT + ((((size_t)kind * a.N + n) * a.nseg + seg) * H + h) * kD * kD;
    else if (seg == a.nseg - 1) s_out = a.sT + ((size_t)n * H + h) * kD * kD;
  }

  if (warp == 0) {
    tmem_alloc(smem_u32(&ctl->tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(smem_u32(&ctl->bar[b]), 1);
    ctl->abort = 0;
    ctl->qk_iss[0] = ctl->qk_iss[1] = ctl->qk_lnd[0] = ctl->qk_lnd[1] = 0;
    ctl->v_iss = ctl->v_lnd = 0;
    ctl->og_iss = ctl->og_lnd = 0;
    ctl->go_c[0] = ctl->go_c[1] = ctl->go_s[0] = ctl->go_s[1] = 0;
    fence_mbar_init();
  }
  if (kOG && tid >= 64 && tid < 64 + kD) ctl->nw[tid - 64] = a.nw ? a.nw[tid - 64] : 1.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_slot;
  const uint32_t sm_base = smem_u32(sm);

  if (tid < kChunkThreads) {
    // =========================================================== chunk group
    // registers: 256 x 208 + 128 x 88 = the launch's 384 x 168
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
    const int ctid = tid;
    const int qw = warp & 3, ch = warp >> 2;
    // prologue layout: channel quad p4 (channels 4 p4 .. 4 p4 + 3) of the
    // 8-row group t8 = warp (rows [8 t8, 8 t8 + 8)); a half-warp covers one
    // 64-column K-half, and a thread's rows lie in one 16-token tile, t8 / 2
    const int p4 = ctid & 31, t8 = ctid >> 5;
    int seq = 0;
    uint32_t ph_m1 = 0, ph_m23 = 0, ph_g = 0, ph_l2 = 0;
    Loader ld{&maps, ctl, sm_base, h, 0, 0, (uint32_t)(kC * kD * (kZ ? 2 : 4))};
    // decay gate (Eq. 5) in log2 units: g log2(e) = zg_min / (1 + 2^(zs z))
    const float zs = kZ ? -expf(a.A_log[h]) * kLog2e : 0.f;
    const float zg_min = kZ ? a.g_min * kLog2e : 0.f;
    if (ctid == 0 && nchunks > 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.g);
      ld.g(bos);
      // q and k of the first two chunks; later ones are issued by the state
      // group as it frees each parity's buffers
      issue_qk(&maps, ctl, sm_base, h, bos, 0);
      if (nchunks > 1) issue_qk(&maps, ctl, sm_base, h, bos + kC, 1);
      if (!zero_v) issue_v(&maps, ctl, sm_base, h, bos);
    }
    if (zero_v)  // the v tile stays zero for the whole item
      for (int e = ctid; e < 16384 / 16; e += kChunkThreads)
        reinterpret_cast<uint4 *>(sm + OFF_V)[e] = make_uint4(0u, 0u, 0u, 0u);
    for (int e = ctid; e < 8192 / 16; e += kChunkThreads)  // T_b above the diagonal: zero for good
      reinterpret_cast<uint4 *>(sm + OFF_ZT)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (ctid < 64) {  // T_01^T in the transposed copy of T_[01][01]: zero for good
      const int n = 16 + (ctid >> 2), k0 = 4 * (ctid & 3);
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(sm + OFF_TF) + tt_idx(n, k0)) =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float beta_next = 0.f;
    if (ctid < kC && ctid < eos - bos) beta_next = __ldg(reinterpret_cast<const float *>(a.beta) + (size_t)(bos + ctid) * H + h);
    float *tot = reinterpret_cast<float *>(sm + OFF_PRO);  // [4][128] per-tile decay sums
    const float *gs = reinterpret_cast<const float *>(sm + OFF_GS);
    uint8_t *qg = sm + OFF_QG;
    bool alive = true;
    for (int m = 0; m < nchunks && alive; ++m) {
      const int par = m & 1;
      const int t0 = bos + m * kC;
      const int len = min(kC, eos - t0);
      uint8_t *kh = sm + OFF_KH + par * 16384;

      // ---------------- decay prologue: cumulative log2-decay and scaled operands
      // Each thread keeps its channel quad's cumulative decay for its 8 rows in
      // registers; the row groups' totals meet in shared memory to give every
      // row group its offset and every 16-token tile its reference (the
      // cumulative decay before its first row).
      if (!(alive = group_wait<true>(ctl, B_GFULL, ph_g, ctid, seq, A.err))) break;
      ph_g ^= 1u;
      if (ctid == 0) ld.landed = ld.issued;
      float4 Gl[8];  // cumulative log2-decay within the row group, then from the chunk start
      {
        float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int row = 8 * t8 + r;
          float4 gv;  // log2-decay
          if constexpr (kZ) {
            const float4 zv = unpack4_bf16(*reinterpret_cast<const uint2 *>(
                reinterpret_cast<const __nv_bfloat16 *>(gs) + row * kD + 4 * p4));
            gv = make_float4(__fdividef(zg_min, 1.f + ex2(zs * zv.x)), __fdividef(zg_min, 1.f + ex2(zs * zv.y)),
                             __fdividef(zg_min, 1.f + ex2(zs * zv.z)), __fdividef(zg_min, 1.f + ex2(zs * zv.w)));
          } else {
            gv = mul4(*reinterpret_cast<const float4 *>(gs + row * kD + 4 * p4),
                      make_float4(kLog2e, kLog2e, kLog2e, kLog2e));
          }
          if (row >= len) gv = make_float4(0.f, 0.f, 0.f, 0.f);  // past the end: identity step
          run = add4(run, gv);
          Gl[r] = run;
        }
        *reinterpret_cast<float4 *>(tot + t8 * 128 + 4 * p4) = run;
        if (ctid < kC) ctl->bs[ctid] = beta_next;
      }
      bar_chunk();
      if (ctid == 0 && m + 1 < nchunks) ld.g(t0 + kC);  // the log-decay tile has been consumed
      float4 ref[4], tc = make_float4(0.f, 0.f, 0.f, 0.f);  // tile references; chunk total G_C
      {
        float4 off = tc;
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const float4 tg = *reinterpret_cast<const float4 *>(tot + g8 * 128 + 4 * p4);
          if ((g8 & 1) == 0) ref[g8 >> 1] = tc;
          if (g8 == t8) off = tc;
          tc = add4(tc, tg);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) Gl[r] = add4(Gl[r], off);
      }
      const float4 gam = make_float4(ex2(tc.x), ex2(tc.y), ex2(tc.z), ex2(tc.w));
      const bool vote = fminf(fminf(tc.x, tc.y), fminf(tc.z, tc.w)) < kSingleRefBound2;
      if (ctid < kC)  // beta of the next chunk's rows, 0 past the end
        beta_next = ctid < eos - (t0 + kC)
                        ? __ldg(reinterpret_cast<const float *>(a.beta) + (size_t)(t0 + kC + ctid) * H + h)
                        : 0.f;
      // The previous chunk's M2/M3 must be done with Gamma o K and T_b before
      // this chunk overwrites them; this chunk's q and k have landed.
      if (ctid == 0) {
        bool ok = true;
        if (m >= 1) {
          ok = solo_wait(ctl, B_M23, ph_m23, A.err);
          ph_m23 ^= 1u;
        }
        if (ok) {
          ok = solo_wait(ctl, B_QK0 + par, (m >> 1) & 1, A.err);
          if (ok) ++ctl->qk_lnd[par];
        }
        ctl->go_c[seq & 1] = ok && !ctl->abort;
      }
      // the barrier also closes the range-guard vote
      const bool slow = bar_chunk_or(vote);
      alive = ctl->go_c[seq & 1] != 0;
      ++seq;
      if (!alive) break;
      // gamma_C of this parity is free only now: the q/k copy just waited for
      // was issued after the state group's last read of it (two chunks back);
      // the state group reads it after the hand-off below
      if (t8 == 0) *reinterpret_cast<float4 *>(&ctl->gam[par][4 * p4]) = gam;
      // operand tiles: channel quad p4 sits in K-half p4 / 16 at column 4 p4 mod 64
      const uint32_t half = (uint32_t)(p4 >> 4), col = (uint32_t)(4 * p4) & 63u;
      uint8_t *qb_h = qg + half * KHALF + par * 16384;  // q -> Q o Gamma (in place)
      uint8_t *gk_h = qg + half * KHALF + 8192;         // Gamma o K
      uint8_t *kb_h = sm + OFF_KB + half * 8192;        // K / Gamma
      uint8_t *kh_h = kh + half * 8192;                 // k -> K o gamma_C / Gamma (in place)
      float4 qv[8], kv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint32_t off = sw128_offset(8 * t8 + r, col);
        const bool in = 8 * t8 + r < len;  // rows past the end are zero
        qv[r] = unpack4_bf16(in ? *reinterpret_cast<const uint2 *>(qb_h + off) : make_uint2(0u, 0u));
        kv[r] = unpack4_bf16(in ? *reinterpret_cast<const uint2 *>(kh_h + off) : make_uint2(0u, 0u));
      }
      if (!slow) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // K / Gamma in place of k: M1's keys and M6's operand
          const uint32_t off = sw128_offset(8 * t8 + r, col);
          const float4 e = ex2_4(Gl[r]), i = ex2_4(neg4(Gl[r]));
          sts64(qb_h + off, pack4_bf16(mul4(qv[r], e)));
          sts64(gk_h + off, pack4_bf16(mul4(kv[r], e)));
          sts64(kh_h + off, pack4_bf16(mul4(kv[r], i)));
        }
        group_publish<true>();
        if (ctid == 0) {
          issue_m1(tbase, smem_u32(qg), sm_base + OFF_KH + par * 16384, par, false);
          mma_commit(smem_u32(&ctl->bar[B_M1]));
        }
        alive = group_wait<true>(ctl, B_M1, ph_m1, ctid, seq, A.err);
        ph_m1 ^= 1u;
      } else {
        // M1 in four accumulating rounds, one per 16-token key tile b, with
        // the cumulative decay before tile b as the reference: query rows of
        // tiles >= b, key rows of tile b only (a thread's rows are all in tile t8 / 2)
        const int tile = t8 >> 1;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          if (!alive) break;
          const float4 rb = b == 0 ? ref[0] : b == 1 ? ref[1] : b == 2 ? ref[2] : ref[3];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const uint32_t off = sw128_offset(8 * t8 + r, col);
            float4 fq = make_float4(0.f, 0.f, 0.f, 0.f), fk = fq, fb = fq;
            if (tile >= b) {
              const float4 e = ex2_4(sub4(Gl[r], rb));
              fq = mul4(qv[r], e);
              fk = mul4(kv[r], e);
            }
            if (tile == b) fb = mul4(kv[r], ex2_4(sub4(rb, Gl[r])));
            sts64(qb_h + off, pack4_bf16(fq));
            sts64(gk_h + off, pack4_bf16(fk));
            sts64(kb_h + off, pack4_bf16(fb));
          }
          group_publish<true>();
          if (ctid == 0) {
            issue_m1(tbase, smem_u32(qg), sm_base + OFF_KB, par, b > 0);
            mma_commit(smem_u32(&ctl->bar[B_M1]));
          }
          alive = group_wait<true>(ctl, B_M1, ph_m1, ctid, seq, A.err);
          ph_m1 ^= 1u;
        }
        if (!alive) break;
        // operands with the chunk start as reference (may underflow to 0: fine)
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t off = sw128_offset(8 * t8 + r, col);
          const float4 e = ex2_4(Gl[r]);
          sts64(qb_h + off, pack4_bf16(mul4(qv[r], e)));
          sts64(gk_h + off, pack4_bf16(mul4(kv[r], e)));
          sts64(kh_h + off, pack4_bf16(mul4(kv[r], ex2_4(sub4(tc, Gl[r])))));
        }
      }
      if (!alive) break;

      // ---------------- masks, L, and T_b = (I + L)^{-1} diag(beta)
      // L is stored with zeros on and above its diagonal and T is computed in
      // place over it: T is zero above the diagonal too, so the zeros L leaves
      // there are already T's.
      {
        float *Lf = reinterpret_cast<float *>(sm + OFF_KB);  // K / Gamma is dead once M1 is done
        float *TTf = reinterpret_cast<float *>(sm + OFF_TF);      // T_[01][01]^T, [32][32] K-major
        float *XTf = TTf + 1024;                                  // X^T of level 2, [32][32] K-major
        float *Xf = TTf + 2048;                                   // level-1 products
        // even chunks: TMEM lanes 0..63 hold A's rows, 64..127 L''; odd chunks the reverse
        const bool a_rows = (qw < 2) == (par == 0);
        const int r = 32 * (qw & 1) + lane;
        float v[32];  // row r, columns [32 ch, 32 ch + 32) of the Gram product
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_D1 + 32 * ch), v);
        tmem_wait_ld();
        const int s0 = 32 * ch;
        if (a_rows) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) v[cc] = (s0 + cc <= r) ? v[cc] : 0.f;
          st_row16_bf16(sm + OFF_AM + par * 8192, r, s0, v);
          st_row16_bf16(sm + OFF_AM + par * 8192, r, s0 + 16, v + 16);
        } else {
          const float br = ctl->bs[r];
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) v[cc] = (s0 + cc < r) ? br * v[cc] : 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4 *>(Lf + lt_idx(r, s0 + 4 * c4)) =
                make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
        }
        bar_chunk();
        // Diagonal 16x16 blocks: one column of T per thread, rows in groups of
        // four (left-looking).  A group first takes the contributions of the
        // rows already solved, then is solved within itself; the sum of row r
        // adds the x[r-1] term last, so consecutive rows are one multiply-add
        // apart on the dependent chain.
        if (ctid < 64) {
          const int base = 16 * (ctid >> 4), cc = ctid & 15;
          float x[16];
#pragma unroll
          for (int R = 0; R < 4; ++R) {
            float4 lr[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int q = 0; q <= R; ++q)
                lr[i][q] = *reinterpret_cast<const float4 *>(Lf + lt_idx(base + 4 * R + i, base + 4 * q));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = 4 * R + i;
              float acc = rr == cc ? 1.f : 0.f;
#pragma unroll
              for (int mm = 0; mm < rr; ++mm) acc -= f4c(lr[i][mm >> 2], mm & 3) * x[mm];
              x[rr] = acc;
            }
          }
          bar_sync_n(3, 64);  // the block's L is read in full before T overwrites it
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) Lf[lt_idx(base + rr, base + cc)] = x[rr];
          if (base < 32)  // column cc of T_00 / T_11 is row cc of the transposed copy
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<float4 *>(TTf + tt_idx(base + cc, base + 4 * j)) =
                  make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        }
        bar_chunk();
        // Off-diagonal blocks in two levels of the 2x2 block inverse
        // [[P, 0], [R, Q]]^{-1} = [[P^-1, 0], [-Q^-1 R P^-1, Q^-1]]:
        //   level 1 (16-row blocks): T_10 and T_32;
        //   level 2 (32-row blocks): T_[23][01].
        // Each output is X = R P^-1, then -Q^-1 X.  Level 1 runs on CUDA cores
        // (fp32); level 2 on the tensor core (tf32, below).  Every block of
        // T_b = T diag(beta) is written as soon as its T block is final, the
        // product outputs straight from registers or TMEM; T_b's blocks above
        // the diagonal stay zero from the start.
        const float4 *bs4 = reinterpret_cast<const float4 *>(ctl->bs);
        uint8_t *zt = sm + OFF_ZT;
        if (ctid < 128) {
          // level 1: two 16x16 outputs, 128 tasks of (row, 4 columns)
          const int blk = ctid >> 6, rr = (ctid >> 2) & 15, q4 = ctid & 3;
          const int rb = 16 * (2 * blk + 1), cb = 16 * (2 * blk);  // output block (rb, cb)
          float *X1 = Xf + blk * 256;                              // [16][16]
          float4 l[4], t[8];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) l[c4] = lds128(Lf + lt_idx(rb + rr, cb + 4 * c4));  // row of L_(rb, cb)
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k0 = 0; k0 < 16; k0 += 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = lds128(Lf + lt_idx(cb + k0 + i, cb + 4 * q4));
            fma8(acc, l, k0, t);
          }
          *reinterpret_cast<float4 *>(X1 + rr * 16 + 4 * q4) = acc;
          bar_sync_n(3, 128);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) l[c4] = lds128(Lf + lt_idx(rb + rr, rb + 4 * c4));  // row of T_(rb, rb)
          acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k0 = 0; k0 < 16; k0 += 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = lds128(X1 + (k0 + i) * 16 + 4 * q4);
            fma8(acc, l, k0, t);
          }
          acc = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
          *reinterpret_cast<float4 *>(Lf + lt_idx(rb + rr, cb + 4 * q4)) = acc;
          st_row4_bf16(zt, rb + rr, cb + 4 * q4, mul4(acc, bs4[cb / 4 + q4]));
          if (blk == 0) {  // T_10 into the transposed copy
            TTf[tt_idx(4 * q4, 16 + rr)] = acc.x;
            TTf[tt_idx(4 * q4 + 1, 16 + rr)] = acc.y;
            TTf[tt_idx(4 * q4 + 2, 16 + rr)] = acc.z;
            TTf[tt_idx(4 * q4 + 3, 16 + rr)] = acc.w;
          }
        } else if (ctid < 192) {
          // T_b of the diagonal blocks: row rr of block db, its 16 columns
          const int e = ctid - 128, db = e >> 4, rr = e & 15;
          const int row = 16 * db + rr, c0 = 16 * db;
          float v[16];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 tv = mul4(lds128(Lf + lt_idx(row, c0 + 4 * c4)), bs4[c0 / 4 + c4]);
            v[4 * c4] = tv.x; v[4 * c4 + 1] = tv.y; v[4 * c4 + 2] = tv.z; v[4 * c4 + 3] = tv.w;
          }
          st_row16_bf16(zt, row, c0, v);
        }
        // level 2 on the tensor core (tf32; the level-2 block of T is small
        // beside the diagonal, and T_b is rounded to bf16 after it):
        //   X = L_[23][01] T_[01][01], then T_[23][01] = -T_[23][23] X.
        // M = 128 rows of the row-major operand (rows 0-31 and 64-127 of the
        // product are not used), N = 32, K = 32; D in the M1 result's columns.
        group_publish<true>();
        if (ctid == 0) {
          constexpr uint32_t id = idesc_tf32_f32(128, 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_tf32_ss(tbase + TM_D1, smem_desc_sw128(sm_base + OFF_KB + kk * 32, 16, 1024),
                        smem_desc_sw128(sm_base + OFF_TF + kk * 32, 16, 1024), id, kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->bar[B_L2]));
        }
        if (!(alive = group_wait<true>(ctl, B_L2, ph_l2, ctid, seq, A.err))) break;
        ph_l2 ^= 1u;
        if ((warp & 3) == 1) {  // rows 32-63 of the product: X (TMEM lanes 32-63) -> X^T
          const int n0 = 16 * (warp >> 2);
          float x[16];
          tmem_ld16(tmem_addr(tbase, 32, TM_D1 + n0), x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) XTf[tt_idx(n0 + i, lane)] = x[i];
        }
        group_publish<true>();
        if (ctid == 0) {
          constexpr uint32_t id = idesc_tf32_f32(128, 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_tf32_ss(tbase + TM_D1 + 32, smem_desc_sw128(sm_base + OFF_KB + 8192 + kk * 32, 16, 1024),
                        smem_desc_sw128(sm_base + OFF_TF + 4096 + kk * 32, 16, 1024), id, kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->bar[B_L2]));
        }
        if (!(alive = group_wait<true>(ctl, B_L2, ph_l2, ctid, seq, A.err))) break;
        ph_l2 ^= 1u;
        if ((warp & 3) == 1) {  // rows 32-63: T_[23][23] X = -T_[23][01]  ->  T_b
          const int n0 = 16 * (warp >> 2);
          float y[16];
          tmem_ld16(tmem_addr(tbase, 32, TM_D1 + 32 + n0), y);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] *= -ctl->bs[n0 + i];
          st_row16_bf16(zt, 32 + lane, n0, y);
        }
      }
      if (ctid == 0) ctl->slow[par] = slow;
      group_publish<true>();
      // ---------------- hand the chunk to the state group, which issues M2/M3
      // (the arrive releases the chunk's shared-memory state to it)
      if (ctid == 0) mbar_arrive(smem_u32(&ctl->bar[B_TB]));
    }
    if (ctid == 0) {
      ld.drain(A.err);
      volatile int no_abort = 0;
      mma_commit(smem_u32(&ctl->bar[B_TD_C]));
      mbar_wait(smem_u32(&ctl->bar[B_TD_C]), 0, &no_abort, A.err, 1u << 23);
    }
  } else {
    // =========================================================== state group
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    const int stid = tid - kChunkThreads;  // = TMEM lane j of every state-group product
    const int qw = warp & 3;                // lane quarter, = stid >> 5
    const int j = stid;
    int seq = 0;
    uint32_t ph_m4 = 0, ph_m56 = 0;
    uint8_t *vt = sm + OFF_VT;
    if (kOG && stid == 0) tma_prefetch_desc(&maps.og);
    // entry state -> TMEM: fp32 master and the bf16 copy M4 reads (S^T row j;
    // the identity for a transition item, zero without an initial state)
#pragma unroll 1
    for (int i0 = 0; i0 < kD; i0 += 32) {
      float s[32];
#pragma unroll
      for (int c = 0; c < 32; ++c)
        s[c] = zero_v ? (i0 + c == j ? 1.f : 0.f) : (s_in ? s_in[(size_t)(i0 + c) * kD + j] : 0.f);
      tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), *reinterpret_cast<float(*)[16]>(s));
      tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0 + 16), *reinterpret_cast<float(*)[16]>(s + 16));
      tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_STB + i0 / 2), s);
    }
    tmem_wait_st();
    group_publish<false>();
    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
      const int par = c & 1;
      const int t0 = bos + c * kC;
      const int len = min(kC, eos - t0);
      const uint32_t tm_u = TM_U + par * 64;
      // ---------------- M2/M3: U^T and W^T, once the chunk group has T_b
      if (!(alive = group_wait<false>(ctl, B_TB, c & 1, stid, seq, A.err))) break;
      // (every thread is past the previous chunk's reads of the out_gate tile)
      if (kOG && stid == 0) issue_og(&maps, ctl, sm_base, h, t0);
      if (stid == 0) {
        bool ok = true;
        if (!zero_v) {
          ok = solo_wait(ctl, B_VFULL, c & 1, A.err);
          if (ok) ++ctl->v_lnd;
        }
        if (ok) {
          issue_m23(tbase, sm_base + OFF_V, sm_base + OFF_QG, sm_base + OFF_ZT, tm_u);
          mma_commit(smem_u32(&ctl->bar[B_M23]));
        }
      }
      if (!(alive = group_wait<false>(ctl, B_M23, c & 1, stid, seq, A.err))) break;
      if (stid == 0 && !zero_v && c + 1 < nchunks) issue_v(&maps, ctl, sm_base, h, t0 + kC);  // M2 is done with v

      // ---------------- -W^T (TMEM) -> MN-major operand in the V~ buffer
      {
        float v[64];
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_W), *reinterpret_cast<float(*)[32]>(v));
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_W + 32), *reinterpret_cast<float(*)[32]>(v + 32));
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) v[cc] = -v[cc];
#pragma unroll
        for (int r0 = 0; r0 < 64; r0 += 16) st_row16_bf16(vt, j, r0, v + r0);
      }
      group_publish<false>();
      if (stid == 0) {
        issue_m4(tbase, sm_base + OFF_VT, sm_base + OFF_QG, par, tm_u);
        mma_commit(smem_u32(&ctl->bar[B_M4]));
      }
      if (!(alive = group_wait<false>(ctl, B_M4, ph_m4, stid, seq, A.err))) break;
      ph_m4 ^= 1u;

      // ---------------- V~^T -> bf16 operand; after the per-tile range path,
      // S^T <- S^T Diag(gamma_C) before M6 (else the scaling follows M6)
      const bool slow = ctl->slow[par] != 0;
      {
        float v[64];
        tmem_ld32(tmem_addr(tbase, 32 * qw, tm_u), *reinterpret_cast<float(*)[32]>(v));
        tmem_ld32(tmem_addr(tbase, 32 * qw, tm_u + 32), *reinterpret_cast<float(*)[32]>(v + 32));
        tmem_wait_ld();
#pragma unroll
        for (int r0 = 0; r0 < 64; r0 += 16) st_row16_bf16(vt, j, r0, v + r0);
      }
      if (slow) {
        const float *gam = ctl->gam[par];
#pragma unroll 1
        for (int i0 = 0; i0 < kD; i0 += 32) {
          float s[32];
          tmem_ld32(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) s[cc] *= gam[i0 + cc];
          tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), *reinterpret_cast<float(*)[16]>(s));
          tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0 + 16), *reinterpret_cast<float(*)[16]>(s + 16));
        }
        tmem_wait_st();
      }
      group_publish<false>();
      if (stid == 0) {
        issue_m56(tbase, sm_base + OFF_VT, sm_base + OFF_AM + par * 8192, sm_base + OFF_KH + par * 16384);
        mma_commit(smem_u32(&ctl->bar[B_M56]));
      }
      if (!(alive = group_wait<false>(ctl, B_M56, ph_m56, stid, seq, A.err))) break;
      ph_m56 ^= 1u;

      // ---------------- S^T <- S^T Diag(gamma_C) (unless done before M6), the
      // bf16 copy of the new state (and a checkpoint of the fp32 state when
      // one ends this chunk); the output rows
      float *cp = ckpt_ptr(a, n, h, t0 + len - seq_bos);
      {
        const float *gam = ctl->gam[par];
#pragma unroll 1
        for (int i0 = 0; i0 < kD; i0 += 32) {
          float s[32];
          tmem_ld32(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
          tmem_wait_ld();
          if (!slow) {
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) s[cc] *= gam[i0 + cc];
            tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), *reinterpret_cast<float(*)[16]>(s));
            tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0 + 16), *reinterpret_cast<float(*)[16]>(s + 16));
          }
          tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_STB + i0 / 2), s);
          if (cp)
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) cp[(size_t)(i0 + cc) * kD + j] = s[cc];
        }
      }
      {
        __nv_bfloat16 *ostage = reinterpret_cast<__nv_bfloat16 *>(vt);
        float v[64];
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_O), *reinterpret_cast<float(*)[32]>(v));
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_O + 32), *reinterpret_cast<float(*)[32]>(v + 32));
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) ostage[cc * kD + j] = __float2bfloat16_rn(v[cc]);
      }
      tmem_wait_st();
      tc_fence_before();
      if constexpr (kOG) {  // the barrier also waits for this chunk's out_gate tile
        if (!(alive = group_wait<false>(ctl, B_OG, c & 1, stid, seq, A.err))) break;
        if (stid == 0) ++ctl->og_lnd;
      } else {
        bar_state();
      }
      // This parity's operand buffers are free (M4-M6 have completed and every
      // state thread has read gamma_C): q and k of the chunk two ahead land in
      // them; its A tile, gamma_C and TMEM U^T are written only after that
      // copy has been waited for.
      if (stid == 0 && c + 2 < nchunks) issue_qk(&maps, ctl, sm_base, h, t0 + 2 * kC, par);
      if (a.o) {  // segment passes of the long-sequence plan write no output
        const uint4 *src = reinterpret_cast<const uint4 *>(vt);
        uint4 *o = reinterpret_cast<uint4 *>(a.o);
        float w8[8];
        if constexpr (kOG) {
          const float4 wa = *reinterpret_cast<const float4 *>(&ctl->nw[8 * (stid & 15)]);
          const float4 wb = *reinterpret_cast<const float4 *>(&ctl->nw[8 * (stid & 15) + 4]);
          w8[0] = wa.x; w8[1] = wa.y; w8[2] = wa.z; w8[3] = wa.w;
          w8[4] = wb.x; w8[5] = wb.y; w8[6] = wb.z; w8[7] = wb.w;
        }
        if constexpr (kOG) {
          // RMSNorm and gate: a thread holds 8 channels of each of 8 rows, and
          // the 16 lanes of a half-warp share a row.  Four rows' sums of
          // squares at a time are reduced side by side so that their shuffles
          // overlap.
          const uint4 *ogt = reinterpret_cast<const uint4 *>(sm + OFF_OG);
#pragma unroll
          for (int i0 = 0; i0 < 8; i0 += 4) {
            float ss[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ss[i] = sumsq8_bf16(src[(i0 + i) * kStateThreads + stid]);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
#pragma unroll
              for (int i = 0; i < 4; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int idx = (i0 + i) * kStateThreads + stid, row = idx >> 4, c16 = idx & 15;
              const uint4 val = scale_gate8(src[idx], ogt[idx], w8, rsqrtf(ss[i] * (1.f / kD) + a.eps));
              if (row < len) o[((size_t)(t0 + row) * H + h) * (kD / 8) + c16] = val;
            }
          }
        } else {
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int idx = it * kStateThreads + stid, row = idx >> 4, c16 = idx & 15;
            if (row < len) o[((size_t)(t0 + row) * H + h) * (kD / 8) + c16] = src[idx];
          }
        }
      }
      // (the next chunk's first group wait orders these reads of the staging
      // tile before it is written again)
    }
    if (alive && s_out) {
#pragma unroll 1
      for (int i0 = 0; i0 < kD; i0 += 32) {
        float s[32];
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) s_out[(size_t)(i0 + cc) * kD + j] = s[cc];
      }
    }
    if (stid == 0) {
      volatile int no_abort = 0;
      mma_commit(smem_u32(&ctl->bar[B_TD_S]));
      mbar_wait(smem_u32(&ctl->bar[B_TD_S]), 0, &no_abort, A.err, 1u << 24);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // q/k and v copies still in flight after an abort land before the CTA retires
    volatile int no_abort = 0;
    for (int i = 0; i < 2; ++i)
      for (int n = ctl->qk_lnd[i]; n < ctl->qk_iss[i]; ++n)
        mbar_wait(smem_u32(&ctl->bar[B_QK0 + i]), n & 1, &no_abort, A.err, 1u << 25);
    for (int n = ctl->v_lnd; n < ctl->v_iss; ++n)
      mbar_wait(smem_u32(&ctl->bar[B_VFULL]), n & 1, &no_abort, A.err, 1u << 26);
    for (int n = ctl->og_lnd; n < ctl->og_iss; ++n)
      mbar_wait(smem_u32(&ctl->bar[B_OG]), n & 1, &no_abort, A.err, 1u << 27);
  }
  if (warp == 0) {
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

// [T_total, H, 128] row-major tensor; boxes of 64 tokens of one head.
// Operand layout: bf16, two 64-column boxes with the 128-byte swizzle the MMA
// operands use.  Row layout: the whole row (fp32 or bf16), unswizzled.
CUresult encode_tok_head(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *base, int T, int H,
                         bool fp32, bool operand) {
  const cuuint64_t esz = fp32 ? 4 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * esz, (cuuint64_t)H * kD * esz};
  const cuuint32_t box[3] = {operand ? 64u : (cuuint32_t)kD, 1, (cuuint32_t)kC};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             operand ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <bool kZ, bool kOG>
cudaError_t launch_variant(const TcMaps &maps, const TcArgs &args, int grid, cudaStream_t s) {
  constexpr uint32_t bytes = smem_bytes(kOG);
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<kZ, kOG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  chunk_tc_kernel<kZ, kOG><<<grid, kThreads, bytes, s>>>(maps, args);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supports(const PrefillArgs &a) {
  // (in the layer form the decay logits are bf16 like q; beta stays fp32)
  return a.qkv == KDA_BF16 && a.out == KDA_BF16 && a.gate == KDA_F32 && a.dk == kD && a.dv == kD &&
         a.chunk == kC;
}

cudaError_t launch_chunk_tc(const PrefillArgs &a, cudaStream_t s) {
  if (a.N * a.H == 0) return cudaSuccess;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  const bool z = a.A_log != nullptr, og = a.og != nullptr && a.o != nullptr;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (encode_tok_head(encode, &maps.q, a.q, a.T_total, a.H, false, true) != CUDA_SUCCESS ||
      encode_tok_head(encode, &maps.k, a.k, a.T_total, a.H, false, true) != CUDA_SUCCESS ||
      encode_tok_head(encode, &maps.v, a.v, a.T_total, a.H, false, true) != CUDA_SUCCESS ||
      encode_tok_head(encode, &maps.g, a.g, a.T_total, a.H, !z, false) != CUDA_SUCCESS ||
      (og && encode_tok_head(encode, &maps.og, a.og, a.T_total, a.H, false, false) != CUDA_SUCCESS))
    return cudaErrorInvalidValue;
  void *wd = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&wd, g_tc_watchdog);
  if (e != cudaSuccess) return e;
  TcArgs args{a, reinterpret_cast<unsigned int *>(wd)};
  const int grid = a.N * a.nseg * a.H * a.kinds;
  if (z) return og ? launch_variant<true, true>(maps, args, grid, s) : launch_variant<true, false>(maps, args, grid, s);
  return og ? launch_variant<false, true>(maps, args, grid, s) : launch_variant<false, false>(maps, args, grid, s);
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
