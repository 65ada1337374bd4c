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
// r), Gamma = exp(G), gamma_C = exp(G_C) and N = -beta o Gamma o K
// ([K3-notes §2.2, chunkwise form]):
//   M1  [A ; -L] = [Q o Gamma ; N] (K / Gamma)^T                 (M=128 N=64 K=128)
//   A  = Tril_incl(A), L strictly lower
//   T  = (I + L)^{-1} up to its 32-row diagonal blocks: recursive block inversion on CUDA cores (fp32);
//        with the output gate (kOG) also its 64-row level, as two tf32 products (M=128 N=32 K=32)
//   M4  [O^T | X] = S^T [Q o Gamma ; N]^T                        (M=128 N=128 K=128)
//   M3  X += V^T Diag(beta), so X = R^T with R = beta o (V - (Gamma o K) S)
//                                        (M=128 N=64 K=64; beta rounded to bf16)
//   M7  V~ = T R by block substitution over 32-row halves, tf32 (A read from TMEM):
//         V~_0 = T_00 R_0,  R_1 -= L_10 V~_0,  V~_1 = T_11 R_1        (M=128 N=32 K=32, three steps)
//       with kOG, whose state group carries the gate's epilogue, one product with the full T
//                                                                     (M=128 N=64 K=64)
//   M5  O^T += V~^T A^T                                           (M=128 N=64 K=64)
//   M6  S^T <- (S^T + V~^T (K / Gamma)) Diag(gamma_C)              (M=128 N=128 K=64)
// The page leaves the WY factors out; with T_b = T diag(beta) they are
// U = T_b V and W = T_b (Gamma o K), and V~ = U - W S = T R, so neither U nor W
// is formed: the state chain needs R (one product into an accumulator that
// already holds beta o V) and T, which the solve leaves in fp32.
// (fp32 master state in TMEM; the Diag(gamma_C) scaling is applied to the
// accumulated state in the same TMEM pass that refreshes its bf16 copy, and
// K / Gamma doubles as M1's key operand.  When the chunk took the per-tile
// range path, K / Gamma may not be formed: the state is scaled first and M6
// takes K o gamma_C / Gamma, as S^T <- S^T Diag(gamma_C) + V~^T (K o gamma_C / Gamma).)
// Every product is computed transposed so that M = 128 (dv or dk) and the
// tensor core runs at full width; TMEM lane j holds row j of the result.
// M4 and O read their A operand, the bf16 copy of S^T, straight from TMEM,
// M7 reads R^T (fp32) and M5/M6 read bf16 V~^T from TMEM as well.
//
// Two warp groups overlap consecutive chunks.  The chunk group (warps 0-7)
// runs one chunk ahead: decay prologue, the operands, M1 and the UT solve, and
// the TMA loads of q, k and log-decay.  q and k land in the buffers that
// become the chunk's Q o Gamma and K / Gamma operands, which are then scaled
// in place.  The state group (warps 8-11) runs the serial state chain: M4/O,
// M7, the bf16 copy of V~, M5/M6, the gamma scaling, the bf16 state copy and
// the output (one TMA store of the staging tile for a whole chunk); it also
// brings in v by TMA and writes Diag(beta) for M3.  Operands the state group
// still reads while the chunk group prepares the next chunk are
// double-buffered by chunk parity; T is single-buffered, and M1 (then the
// solve) waits for the previous chunk's M7 before L is written over T.
// Thread 0 of each group issues that group's MMAs.  With kSplit (chosen at
// launch when every chain has an SM of its own, so that the state group sets
// the pace) V~'s first half is staged in bf16, and its M5/M6 queued, while
// M7's last two steps run.  Work items that write no output (the
// long-sequence plan's pairs) form X alone and skip M5 and the staging.
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
constexpr uint32_t OFF_QG = 0;        // 64 KB: per 64-column K-half (stride KHALF), per parity (16 KB):
                                      //   [Q o Gamma | N], the 128 rows of M1's A operand
constexpr uint32_t KHALF = 32768;
constexpr uint32_t OFF_KB = 65536;    // 16 KB: L, then T over it (fp32 64x64, tf32 operand layout);
                                      //   B of M7, kept until that product is done
constexpr uint32_t OFF_TF = 81920;    // 16 KB: solve scratch: T_[01][01]^T and X^T (tf32 B operands of
                                      //   the level-64 products, 4 KB each), 16- and 32-row level products (3 KB),
                                      //   decay prologue sums (4 KB at OFF_PRO); on the per-tile range
                                      //   path, M1's key operand of one tile (all 16 KB)
constexpr uint32_t OFF_KH = 98304;    // x2 16 KB: K / Gamma (B of M1, MN-major B of M6), or
                                      //   K o gamma_C / Gamma after the per-tile range path
constexpr uint32_t OFF_AM = 131072;   // x2 8 KB: A bf16, 64 rows x 64
constexpr uint32_t OFF_V = 147456;    // 16 KB: v tile (TMA), two 64-column boxes
constexpr uint32_t OFF_GS = 163840;   // 32 KB: log-decay tile (TMA), fp32 [64][128]; with decay logits
                                      //   (bf16, 16 KB) the out_gate tile sits in the second half
constexpr uint32_t OFF_OG = OFF_GS + 16384;
constexpr uint32_t OFF_VT = 196608;   // 16 KB: output tile
constexpr uint32_t OFF_DB = 212992;   // 8 KB: Diag(beta) in bf16, K-major 64 x 64 (B operand of M3)
constexpr uint32_t OFF_CTL = 221184;  // 4 KB control block
constexpr uint32_t OFF_PRO = OFF_TF + 12288;
constexpr uint32_t SMEM_USED = OFF_CTL + 4096;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

// TMEM columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // M1 result, level-2 products (chunk group)
constexpr uint32_t TM_Y = 64;     // V~^T (fp32, M7 result)
constexpr uint32_t TM_YB = 128;   // bf16 V~^T, two values per column (A operand of M5/M6), 32 columns
constexpr uint32_t TM_O = 192;    // O^T accumulator; with TM_X the 128 columns of one M4 product
constexpr uint32_t TM_X = 256;    // S^T N^T after M4, then R^T after M3 (fp32; A operand of M7)
constexpr uint32_t TM_STB = 320;  // bf16 S^T, two values per column (A operand of M4)
constexpr uint32_t TM_S = 384;    // fp32 master state S^T (128 columns)

enum Bar : int {
  B_M1 = 0, B_M7, B_VFULL, B_GFULL, B_QK0, B_QK1, B_TB, B_M4,
  B_M56, B_M7S, B_L2, B_TD_C, B_TD_S, B_OG, B_OPS0, B_OPS1, B_COUNT
};
// B_OPS0 + (c & 1): chunk c's operands are in place (arrived once per chunk of
// that parity, so a barrier runs at most one phase ahead of its waiter: the
// next arrival on it needs the q/k copy that is issued only once chunk c's
// M5/M6 are done)

struct Ctl {
  uint64_t bar[16];
  float gam[3][128];     // gamma_C per channel, by chunk index mod 3
  alignas(16) float bsb[2][64];  // beta of a chunk's rows (0 past the end), by chunk parity: chunk group
  alignas(16) float bsx[2][64];  // the same, state group (for X)
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
static_assert(offsetof(Ctl, nw) % 16 == 0 && offsetof(Ctl, gam) % 16 == 0 && offsetof(Ctl, bsb) % 16 == 0,
              "vector reads of the control block");
static_assert(sizeof(Ctl) <= 4096, "control block");

struct TcArgs {
  PrefillArgs a;
  unsigned int *err;
};

struct TcMaps {
  CUtensorMap q, k, v, g, og, o;
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

__device__ __forceinline__ void sts64(uint8_t *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }

// beta of row `row` of the chunk at t0 into dst[row]: an asynchronous 4-byte
// copy (a plain load would hold up the next barrier until it returned), or 0
// past the end of the range.  The copy is waited for with cp_async_wait_all.
__device__ __forceinline__ void beta_async(float *dst, const float *beta, int t0, int row, int eos, int H, int h) {
  if (t0 + row < eos) {
    asm volatile(
        "{\n\t.reg .u64 g;\n\tcvta.to.global.u64 g, %1;\n\t"
        "cp.async.ca.shared.global [%0], [g], 4;\n\t}" ::"r"(smem_u32(dst + row)),
        "l"(beta + (size_t)(t0 + row) * H + h)
        : "memory");
  } else {
    dst[row] = 0.f;
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

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
// A second barrier b2 (>= 0) is waited for after the first, with parity p2.
template <bool kChunkGroup>
__device__ __forceinline__ bool group_wait(Ctl *ctl, int b, uint32_t parity, int gtid, int &seq, unsigned int *err,
                                           int b2 = -1, uint32_t p2 = 0) {
  int *go = kChunkGroup ? ctl->go_c : ctl->go_s;
  if (gtid == 0) {
    bool ok = mbar_wait(smem_u32(&ctl->bar[b]), parity, &ctl->abort, err, 1u << b);
    if (ok && b2 >= 0) ok = mbar_wait(smem_u32(&ctl->bar[b2]), p2 & 1u, &ctl->abort, err, 1u << b2);
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

// M1 of the chunk of parity par: A = the 128 rows [Q o Gamma ; N] of that
// parity (contiguous within each K-half), B = the keys kb.
__device__ __forceinline__ void issue_m1(uint32_t tbase, uint32_t qg, uint32_t kb, int par, bool acc_first) {
  constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ka = (kk >> 2) * KHALF + par * 16384 + (kk & 3) * 32;
    const uint32_t kbo = (kk >> 2) * 8192 + (kk & 3) * 32;
    mma_bf16_ss(tbase + TM_D1, smem_desc_sw128(qg + ka, 16, 1024), smem_desc_sw128(kb + kbo, 16, 1024), id,
                (kk > 0 || acc_first) ? 1u : 0u);
  }
}

// M4: [O^T | X] = S^T [Q o Gamma ; N]^T, one N = 128 product (A = bf16
// S^T in TMEM; B = the 128 rows [Q o Gamma ; N] of the chunk's parity, K-major,
// contiguous within each K-half like M1's A operand).
// With x_only (a work item that writes no output) only X = S^T N^T, from
// the N rows (the second 64 of each K-half's 128).
__device__ __forceinline__ void issue_m4(uint32_t tbase, uint32_t qg, int par, bool x_only) {
  constexpr uint32_t id = idesc_bf16_f32(128, 128, 0, 0);
  constexpr uint32_t idx = idesc_bf16_f32(128, 64, 0, 0);
  if (x_only) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t kb = (kk >> 2) * KHALF + par * 16384 + 8192 + (kk & 3) * 32;
      mma_bf16_ts(tbase + TM_X, tbase + TM_STB + kk * 8, smem_desc_sw128(qg + kb, 16, 1024), idx,
                  kk > 0 ? 1u : 0u);
    }
    return;
  }
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t kb = (kk >> 2) * KHALF + par * 16384 + (kk & 3) * 32;
    mma_bf16_ts(tbase + TM_O, tbase + TM_STB + kk * 8, smem_desc_sw128(qg + kb, 16, 1024), id, kk > 0 ? 1u : 0u);
  }
}

// M3: X += V^T Diag(beta) (A = the v tile, MN-major: two blocks of 64
// columns; B = Diag(beta), K-major).
__device__ __forceinline__ void issue_m3(uint32_t tbase, uint32_t v, uint32_t db) {
  constexpr uint32_t id = idesc_bf16_f32(128, 64, 1, 0);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_bf16_ss(tbase + TM_X, smem_desc_sw128(v + kk * 2048, 8192, 1024), smem_desc_sw128(db + kk * 32, 16, 1024),
                id, 1u);
}

// M7 in three steps over the two 32-row halves of the chunk (tf32; A from
// TMEM, one K element per column; B from the solve's buffer tt, whose
// 32-row diagonal blocks hold T_00 and T_11 and whose lower-left block holds
// -L_10):
//   step 0:  V~_0^T  = R_0^T T_00^T
//   step 1:  R_1^T  += V~_0^T (-L_10)^T
//   step 2:  V~_1^T  = R_1^T T_11^T
__device__ __forceinline__ void issue_m7_step(uint32_t tbase, uint32_t tt, int step) {
  constexpr uint32_t id = idesc_tf32_f32(128, 32);
  // (D, A column offsets; B = rows [32 (step > 0), +32) of K-half (step == 2))
  const uint32_t d = step == 0 ? TM_Y : step == 1 ? TM_X + 32 : TM_Y + 32;
  const uint32_t a = step == 0 ? TM_X : step == 1 ? TM_Y : TM_X + 32;
  const uint32_t b = tt + (step == 2 ? 8192u : 0u) + (step > 0 ? 4096u : 0u);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_tf32_ts(tbase + d, tbase + a + kk * 8, smem_desc_sw128(b + kk * 32, 16, 1024), id,
                (kk > 0 || step == 1) ? 1u : 0u);
}

// M7 as one product, V~^T = R^T T^T, with the full T in the solve's buffer
// (its two 32-column K-halves).
__device__ __forceinline__ void issue_m7_full(uint32_t tbase, uint32_t tt) {
  constexpr uint32_t id = idesc_tf32_f32(128, 64);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_tf32_ts(tbase + TM_Y, tbase + TM_X + kk * 8,
                smem_desc_sw128(tt + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id, kk > 0 ? 1u : 0u);
}

// M6 then, for a work item that writes output, M5, over the tokens of one
// 32-row half of the chunk (K-steps 2 half and 2 half + 1).
__device__ __forceinline__ void issue_m56_half(uint32_t tbase, uint32_t am, uint32_t kh, bool with_o, int half) {
  constexpr uint32_t id5 = idesc_bf16_f32(128, 64, 0, 0);
  constexpr uint32_t id6 = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const int kk = 2 * half + k2;
    mma_bf16_ts(tbase + TM_S, tbase + TM_YB + kk * 8, smem_desc_sw128(kh + kk * 2048, 8192, 1024), id6, 1u);
  }
  if (!with_o) return;
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const int kk = 2 * half + k2;
    mma_bf16_ts(tbase + TM_O, tbase + TM_YB + kk * 8, smem_desc_sw128(am + kk * 32, 16, 1024), id5, 1u);
  }
}

// M6 then, for a work item that writes output, M5 (A = bf16 V~^T in TMEM).
__device__ __forceinline__ void issue_m56(uint32_t tbase, uint32_t am, uint32_t kh, bool with_o) {
  constexpr uint32_t id5 = idesc_bf16_f32(128, 64, 0, 0);
  constexpr uint32_t id6 = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // S^T += V~^T (K / Gamma)   (B MN-major)
    mma_bf16_ts(tbase + TM_S, tbase + TM_YB + kk * 8, smem_desc_sw128(kh + kk * 2048, 8192, 1024), id6, 1u);
  if (!with_o) return;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)  // O^T += V~^T A^T
    mma_bf16_ts(tbase + TM_O, tbase + TM_YB + kk * 8, smem_desc_sw128(am + kk * 32, 16, 1024), id5, 1u);
}

// M4 (with O) and M3 of chunk c, by the state group's thread 0, once the
// chunk's operands are in place (the chunk group may still be solving for T)
// and its v tile has landed.  The bf16 state, Diag(beta) and the previous
// chunk's reads of O were ordered before this by the barrier that ended the
// previous chunk.
// A transition item (zero_v: v = 0) skips M3, whose product is zero, and an
// item without output (with_o false) forms X alone.
__device__ __forceinline__ bool issue_m43(const TcArgs &A, Ctl *ctl, uint32_t tbase, uint32_t sm_base, int c,
                                          bool zero_v, bool with_o) {
  bool ok = solo_wait(ctl, B_OPS0 + (c & 1), (c >> 1) & 1, A.err);
  if (ok && !zero_v) {
    ok = solo_wait(ctl, B_VFULL, c & 1, A.err);
    if (ok) ++ctl->v_lnd;
  }
  if (ok) {
    issue_m4(tbase, sm_base + OFF_QG, c & 1, !with_o);
    if (!zero_v) issue_m3(tbase, sm_base + OFF_V, sm_base + OFF_DB);
    mma_commit(smem_u32(&ctl->bar[B_M4]));
  }
  return ok;
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

// kSplit: M7's last two steps overlap the bf16 staging of V~'s first half
// and M5/M6 over the first 32 tokens (see the state group); chosen per launch.
template <bool kZ, bool kOG, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ TcMaps maps, TcArgs A) {
  extern __shared__ uint8_t smem_raw[];
  // Where the 64-row level of T's solve runs: in the chunk group on the
  // tensor core (the full T, one M7 product), or folded into a three-step M7
  // in the state group.  The output gate's epilogue makes the state group the
  // longer of the two per chunk, so that variant keeps the level in the chunk
  // group; without it the chunk group is the longer one.
  constexpr bool kL64 = kOG;
  // 1024-aligned base by pointer arithmetic on the shared array, so that the
  // compiler keeps every access through `sm` in the shared address space
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctl *ctl = reinterpret_cast<Ctl *>(sm + OFF_CTL);
  const PrefillArgs &a = A.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  // work item -- see PrefillArgs
  constexpr size_t DD = (size_t)kD * kD;
  int n, h, kind = 0, bos, eos, seq_bos;
  const float *s_in = nullptr;  // entry state (null: zero, or the identity for kind 1)
  float *s_out = nullptr;       // where the final state goes (nullable)
  bool out_item;                // writes outputs (and checkpoints)
  if (a.plan == 0) {
    int item = blockIdx.x;
    kind = item % a.kinds;
    item /= a.kinds;
    h = item % H;
    item /= H;
    const int seg = item % a.nseg;
    n = item / a.nseg;
    // Packed sequences run longest first: work items are handed to SMs in
    // index order, so a long sequence that came late would finish last.
    if (a.cu && a.N > 1 && a.N <= kLongestFirstMax)
      n = longest_first(a.cu, a.N, n, reinterpret_cast<int *>(sm + OFF_TF), tid);
    seq_range(a, n, bos, eos);
    seq_bos = bos;  // checkpoints count tokens from the sequence start
    if (a.seg_tokens > 0) {
      const int sb = min(eos, bos + seg * a.seg_tokens);
      eos = min(eos, sb + a.seg_tokens);
      bos = sb;
    }
    if (kind == 0 && a.s0) s_in = a.s0 + (((size_t)n * a.nseg + seg) * H + h) * DD;
    if (a.sT) {
      if (a.kinds == 2) s_out = a.sT + ((((size_t)kind * a.N + n) * a.nseg + seg) * H + h) * DD;
      else if (seg == a.nseg - 1) s_out = a.sT + ((size_t)n * H + h) * DD;
    }
    out_item = a.o != nullptr;
  } else {
    // the long-sequence plan: segment 0 items first (the longest), then the rest
    const int NH = a.N * H;
    int item = blockIdx.x, seg = 0;
    if (a.plan == 1 && item < NH) {
      n = item / H;
      h = item % H;
    } else {
      if (a.plan == 1) {
        item -= NH;
        kind = item % 2;
        item /= 2;
      }
      h = item % H;
      item /= H;
      const int nsegs = a.plan == 1 ? a.P - 2 : a.P - 1;
      seg = 1 + item % nsegs;
      n = item / nsegs;
    }
    seq_range(a, n, bos, eos);
    seq_bos = bos;
    const int sb = seg == 0 ? bos : min(eos, bos + a.seg0 + (seg - 1) * a.seg_tokens);
    eos = min(eos, seg == 0 ? bos + a.seg0 : sb + a.seg_tokens);
    bos = sb;
    const size_t nh = (size_t)n * H + h;
    if (a.plan == 1 && seg == 0) {
      s_in = a.s0 ? a.s0 + nh * DD : nullptr;
      s_out = a.E + ((size_t)n * (a.P - 1) * H + h) * DD;
      out_item = a.o != nullptr;
    } else if (a.plan == 1) {
      s_out = a.pairs + ((((size_t)kind * a.N + n) * (a.P - 2) + (seg - 1)) * H + h) * DD;
      out_item = false;
    } else {
      s_in = a.E + (((size_t)n * (a.P - 1) + (seg - 1)) * H + h) * DD;
      if (seg == a.P - 1 && a.sT) s_out = a.sT + nh * DD;
      out_item = a.o != nullptr;
    }
  }
  const int nchunks = (eos - bos + kC - 1) / kC;
  const bool zero_v = kind == 1;  // transition pass: v = 0, identity entry state

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
  const float *betap = reinterpret_cast<const float *>(a.beta);

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
    uint32_t ph_m1 = 0, ph_g = 0, ph_l2 = 0;
    Loader ld{&maps, ctl, sm_base, h, 0, 0, (uint32_t)(kC * kD * (kZ ? 2 : 4))};
    // decay gate (Eq. 5) in log2 units: g log2(e) = zg_min / (1 + 2^(zs z))
    const float zs = kZ ? -expf(a.A_log[h]) * kLog2e : 0.f;
    const float zg_min = kZ ? a.g_min * kLog2e : 0.f;
    if (ctid == 0 && nchunks > 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.g);
      ld.g(bos);
      // q and k of the first two chunks; later ones are issued by the state
      // group as it frees each parity's buffers
      issue_qk(&maps, ctl, sm_base, h, bos, 0);
      if (nchunks > 1) issue_qk(&maps, ctl, sm_base, h, bos + kC, 1);
    }
    if (ctid < kC && nchunks > 0) beta_async(ctl->bsb[0], betap, bos, ctid, eos, H, h);
    float *tot = reinterpret_cast<float *>(sm + OFF_PRO);  // [8][128] per-row-group decay sums
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
      cp_async_wait_all();  // this chunk's beta
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
      }
      bar_chunk();
      if (ctid == 0 && m + 1 < nchunks) ld.g(t0 + kC);  // the log-decay tile has been consumed
      // beta of the next chunk (its buffer was last read in the previous chunk)
      if (ctid < kC && m + 1 < nchunks) beta_async(ctl->bsb[par ^ 1], betap, t0 + kC, ctid, eos, H, h);
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
      float nb[8];  // -beta of the thread's rows (N = -beta o Gamma o K)
      {
        const float4 b0 = *reinterpret_cast<const float4 *>(&ctl->bsb[par][8 * t8]);
        const float4 b1 = *reinterpret_cast<const float4 *>(&ctl->bsb[par][8 * t8 + 4]);
        nb[0] = -b0.x; nb[1] = -b0.y; nb[2] = -b0.z; nb[3] = -b0.w;
        nb[4] = -b1.x; nb[5] = -b1.y; nb[6] = -b1.z; nb[7] = -b1.w;
      }
      // This chunk's q and k have landed (the copy was issued once the state
      // group was done with this parity's buffers, two chunks back).
      if (ctid == 0) {
        const bool ok = solo_wait(ctl, B_QK0 + par, (m >> 1) & 1, A.err);
        if (ok) ++ctl->qk_lnd[par];
        ctl->go_c[seq & 1] = ok && !ctl->abort;
      }
      // the barrier also closes the range-guard vote
      const bool slow = bar_chunk_or(vote);
      alive = ctl->go_c[seq & 1] != 0;
      ++seq;
      if (!alive) break;
      // gamma_C goes to slot m mod 3: the state group may still be reading
      // slot (m - 2) mod 3 (the q/k copy just waited for was issued once
      // chunk m - 2's M5/M6 were done, before that chunk's state refresh),
      // but it is past chunk m - 3's; it reads this slot after the hand-off below
      if (t8 == 0) *reinterpret_cast<float4 *>(&ctl->gam[m % 3][4 * p4]) = gam;
      // operand tiles: channel quad p4 sits in K-half p4 / 16 at column 4 p4 mod 64
      const uint32_t half = (uint32_t)(p4 >> 4), col = (uint32_t)(4 * p4) & 63u;
      uint8_t *qb_h = qg + half * KHALF + par * 16384;  // q -> Q o Gamma (in place)
      uint8_t *nb_h = qb_h + 8192;                      // N = -beta o Gamma o K
      uint8_t *kb_h = sm + OFF_TF + half * 8192;        // a tile's keys (per-tile range path)
      uint8_t *kh_h = kh + half * 8192;                 // k -> K / Gamma (in place)
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
          const float4 ge = mul4(kv[r], e);
          sts64(qb_h + off, pack4_bf16(mul4(qv[r], e)));
          sts64(nb_h + off, pack4_bf16(make_float4(nb[r] * ge.x, nb[r] * ge.y, nb[r] * ge.z, nb[r] * ge.w)));
          sts64(kh_h + off, pack4_bf16(mul4(kv[r], i)));
        }
        group_publish<true>();
        if (ctid == 0) {
          // the state group may start M4 and O; M1 goes in only after the
          // previous chunk's M7 (which M1 would otherwise hold up in the
          // tensor pipe, and whose T the L written below replaces)
          mbar_arrive(smem_u32(&ctl->bar[B_OPS0 + par]));
          const bool ok =
              m == 0 || mbar_wait(smem_u32(&ctl->bar[B_M7]), (m - 1) & 1, &ctl->abort, A.err, 1u << B_M7);
          tc_fence_after();
          if (ok) {
            issue_m1(tbase, smem_u32(qg), sm_base + OFF_KH + par * 16384, par, false);
            mma_commit(smem_u32(&ctl->bar[B_M1]));
          }
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
            sts64(nb_h + off, pack4_bf16(make_float4(nb[r] * fk.x, nb[r] * fk.y, nb[r] * fk.z, nb[r] * fk.w)));
            sts64(kb_h + off, pack4_bf16(fb));
          }
          group_publish<true>();
          if (ctid == 0) {
            issue_m1(tbase, smem_u32(qg), sm_base + OFF_TF, par, b > 0);
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
          const float4 ge = mul4(kv[r], e);
          sts64(qb_h + off, pack4_bf16(mul4(qv[r], e)));
          sts64(nb_h + off, pack4_bf16(make_float4(nb[r] * ge.x, nb[r] * ge.y, nb[r] * ge.z, nb[r] * ge.w)));
          sts64(kh_h + off, pack4_bf16(mul4(kv[r], ex2_4(sub4(tc, Gl[r])))));
        }
        group_publish<true>();
        if (ctid == 0) mbar_arrive(smem_u32(&ctl->bar[B_OPS0 + par]));  // the state group may start M4 and O
        // the previous chunk's M7 is done with T (L is written over it below)
        if (m > 0) alive = group_wait<true>(ctl, B_M7, (m - 1) & 1, ctid, seq, A.err);
      }
      if (!alive) break;

      // ---------------- masks, L, and T = (I + L)^{-1}
      // L is stored with zeros on and above its diagonal and T is computed in
      // place over it: T is zero above the diagonal too, so the zeros L leaves
      // there are already T's.
      {
        float *Lf = reinterpret_cast<float *>(sm + OFF_KB);
        float *TTf = reinterpret_cast<float *>(sm + OFF_TF);      // kL64: T_[01][01]^T, [32][32] K-major
        float *XTf = TTf + 1024;                                  // kL64: X^T of level 2, [32][32] K-major
        float *Xf = TTf + 2048;                                   // 16- and 32-row level products (3 KB)
        // TMEM lanes 0..63 hold A's rows, 64..127 the rows of -L (N (K / Gamma)^T)
        const bool a_rows = qw < 2;
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
          // L below the diagonal; without kL64 its lower-left 32 x 32 block is
          // kept as -L (the state group's M7 subtracts L_10 V~_0 with it)
          const float sg = (!kL64 && r >= 32 && s0 < 32) ? 1.f : -1.f;
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) v[cc] = (s0 + cc < r) ? sg * v[cc] : 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4 *>(Lf + lt_idx(r, s0 + 4 * c4)) =
                make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
        }
        bar_chunk();
        // The 32-row diagonal blocks of T = (I + L)^{-1} by recursive 2x2
        // block inversion,
        //   [[P, 0], [R, Q]]^{-1} = [[P^-1, 0], [-Q^-1 R P^-1, Q^-1]],
        // from the 8x8 diagonal blocks up: blocks of 8 by substitution, the
        // 16- and 32-row levels as X = R P^-1 then -Q^-1 X on CUDA cores (fp32,
        // every chunk-group thread).  Every T block is written in place over L
        // as soon as it is final.  Without kL64 the 64-row level is not
        // formed: the state group's M7 applies it by substitution over the two
        // 32-row halves, with -L_10 from the lower-left block.  With kL64 it is
        // formed on the tensor core (tf32, below), and the blocks of T_[01][01]
        // also go, transposed, into the B operand of its first product.
        // 8x8 diagonal blocks: one column per thread; a block's eight threads
        // share a warp, so the warp is done reading the block's L before any
        // of them writes T over it.  With kL64, threads 64..159 meanwhile
        // write the zero blocks of the transposed copy.
        if (ctid < 64) {
          const int base = 8 * (ctid >> 3), cc = ctid & 7;
          float4 lr[8][2];
#pragma unroll
          for (int r = 1; r < 8; ++r) {
            lr[r][0] = lds128(Lf + lt_idx(base + r, base));
            lr[r][1] = lds128(Lf + lt_idx(base + r, base + 4));
          }
          float x[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            float acc = r == cc ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) acc = fmaf(-f4c(lr[r][s >> 2], s & 3), x[s], acc);
            x[r] = acc;
          }
          __syncwarp();
#pragma unroll
          for (int r = 0; r < 8; ++r) Lf[lt_idx(base + r, base + cc)] = x[r];
          if (kL64 && base < 32) {  // column cc of the block is row base + cc of the transposed copy
            *reinterpret_cast<float4 *>(TTf + tt_idx(base + cc, base)) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4 *>(TTf + tt_idx(base + cc, base + 4)) = make_float4(x[4], x[5], x[6], x[7]);
          }
        } else if (kL64 && ctid < 160) {
          // zeros of T_[01][01]^T: (n 8..15, k 0..7), (n 24..31, k 16..23), (n 16..31, k 0..15)
          const int e = ctid - 64;  // 96 float4
          int n, k;
          if (e < 16) { n = 8 + (e >> 1); k = 4 * (e & 1); }
          else if (e < 32) { n = 24 + ((e - 16) >> 1); k = 16 + 4 * (e & 1); }
          else { n = 16 + ((e - 32) >> 2); k = 4 * (e & 3); }
          *reinterpret_cast<float4 *>(TTf + tt_idx(n, k)) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (ctid == 160 && m >= 1 && m + 1 < nchunks &&
                   mbar_wait(smem_u32(&ctl->bar[B_M56]), (m - 1) & 1, &ctl->abort, A.err, 1u << B_M56)) {
          // q and k of chunk m + 1 go into the buffers of chunk m - 1, whose
          // M5/M6 the state group has finished by now (this thread is idle in
          // this phase; issued a whole solve earlier than at the hand-off, the
          // copy lands before the next chunk's operand pass needs it).  B_M56
          // cannot be a phase ahead: chunk m's M5/M6 wait for this chunk's hand-off.
          issue_qk(&maps, ctl, sm_base, h, t0 + kC, par ^ 1);
        }
        bar_chunk();
        // 16-row level: four blocks, one (row i, column jj) of the output per thread
        {
          const int b = ctid >> 6, i = (ctid >> 3) & 7, jj = ctid & 7, o = 16 * b;
          float *Xb = Xf + 64 * b;  // [8][8]
          const float4 r0 = lds128(Lf + lt_idx(o + 8 + i, o)), r1 = lds128(Lf + lt_idx(o + 8 + i, o + 4));
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) acc = fmaf(f4c(k < 4 ? r0 : r1, k & 3), Lf[lt_idx(o + k, o + jj)], acc);
          Xb[8 * i + jj] = acc;
          bar_chunk();
          const float4 q0 = lds128(Lf + lt_idx(o + 8 + i, o + 8)), q1 = lds128(Lf + lt_idx(o + 8 + i, o + 12));
          float t = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) t = fmaf(f4c(k < 4 ? q0 : q1, k & 3), Xb[8 * k + jj], t);
          Lf[lt_idx(o + 8 + i, o + jj)] = -t;
          if (kL64 && o < 32) TTf[tt_idx(o + jj, o + 8 + i)] = -t;
        }
        bar_chunk();
        // 32-row level: T_10 and T_32 of the 16-row blocks, two adjacent
        // columns of one row per thread
        {
          const int blk = ctid >> 7, rr = (ctid >> 3) & 15, c2 = 2 * (ctid & 7);
          const int rb = 16 * (2 * blk + 1), cb = 32 * blk;  // output block (rb, cb)
          float *X1 = Xf + 256 + 256 * blk;                   // [16][16]
          float4 l[4];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) l[c4] = lds128(Lf + lt_idx(rb + rr, cb + 4 * c4));  // row of L_(rb, cb)
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 tv = *reinterpret_cast<const float2 *>(Lf + lt_idx(cb + k, cb + c2));
            const float lk = f4c(l[k >> 2], k & 3);
            acc.x = fmaf(lk, tv.x, acc.x);
            acc.y = fmaf(lk, tv.y, acc.y);
          }
          *reinterpret_cast<float2 *>(X1 + 16 * rr + c2) = acc;
          bar_chunk();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) l[c4] = lds128(Lf + lt_idx(rb + rr, rb + 4 * c4));  // row of T_(rb, rb)
          acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 xv = *reinterpret_cast<const float2 *>(X1 + 16 * k + c2);
            const float lk = f4c(l[k >> 2], k & 3);
            acc.x = fmaf(lk, xv.x, acc.x);
            acc.y = fmaf(lk, xv.y, acc.y);
          }
          *reinterpret_cast<float2 *>(Lf + lt_idx(rb + rr, cb + c2)) = make_float2(-acc.x, -acc.y);
          if (kL64 && blk == 0) {  // T_10 into the transposed copy
            TTf[tt_idx(c2, 16 + rr)] = -acc.x;
            TTf[tt_idx(c2 + 1, 16 + rr)] = -acc.y;
          }
        }
        if constexpr (kL64) {
          // level 2 on the tensor core (tf32):
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
          if ((warp & 3) == 1) {  // rows 32-63: T_[23][23] X = -T_[23][01]
            const int n0 = 16 * (warp >> 2);
            float y[16];
            tmem_ld16(tmem_addr(tbase, 32, TM_D1 + 32 + n0), y);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) Lf[lt_idx(32 + lane, n0 + i)] = -y[i];
          }
        }
      }
      if (ctid == 0) ctl->slow[par] = slow;
      group_publish<true>();
      // ---------------- hand the chunk to the state group (the arrive releases
      // the chunk's operands, A, T and gamma_C to it)
      if (ctid == 0) mbar_arrive(smem_u32(&ctl->bar[B_TB]));
    }
    cp_async_wait_all();
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
    uint32_t ph_m4 = 0, ph_m56 = 0, ph_m7s = 0;
    uint8_t *vt = sm + OFF_VT;
    if (stid == 0 && nchunks > 0) {
      tma_prefetch_desc(&maps.v);
      if (kOG) tma_prefetch_desc(&maps.og);
      if (!zero_v) issue_v(&maps, ctl, sm_base, h, bos);
    }
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
    // Diag(beta): zero off the diagonal for good (and the v tile of a
    // transition item, whose v is zero); the diagonal of chunk 0
    for (int e = stid; e < 8192 / 16; e += kStateThreads)
      reinterpret_cast<uint4 *>(sm + OFF_DB)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (zero_v)
      for (int e = stid; e < 16384 / 16; e += kStateThreads)
        reinterpret_cast<uint4 *>(sm + OFF_V)[e] = make_uint4(0u, 0u, 0u, 0u);
    bar_state();  // the zeros are written before the diagonal goes over them
    if (stid < kC)
      *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_DB + sw128_offset(stid, stid)) =
          __float2bfloat16_rn(stid < eos - bos ? __ldg(betap + (size_t)(bos + stid) * H + h) : 0.f);
    tmem_wait_st();
    group_publish<false>();
    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
      const int par = c & 1;
      const int t0 = bos + c * kC;
      const int len = min(kC, eos - t0);
      // beta of the next chunk's rows (for its Diag(beta))
      if (stid < kC && c + 1 < nchunks) beta_async(ctl->bsx[par ^ 1], betap, t0 + kC, stid, eos, H, h);
      // M4 and M3 (issued here rather than right after the previous chunk's
      // state refresh: there they met the chunk group's operand pass in the
      // shared-memory pipe, and the step took ~10 % longer)
      if (stid == 0) issue_m43(A, ctl, tbase, sm_base, c, zero_v, out_item);
      // ---------------- M7 once the chunk group has handed T over and M4 has
      // completed R (M7 reads it from TMEM)
      if (!(alive = group_wait<false>(ctl, B_TB, c & 1, stid, seq, A.err))) break;
      // (every thread is past the previous chunk's reads of the out_gate tile)
      if (kOG && out_item && stid == 0) issue_og(&maps, ctl, sm_base, h, t0);
      if (stid == 0 && solo_wait(ctl, B_M4, ph_m4, A.err)) {
        if constexpr (kL64) {
          issue_m7_full(tbase, sm_base + OFF_KB);
          mma_commit(smem_u32(&ctl->bar[B_M7]));
        }
        // M3 has read the v tile: the next chunk's may land
        if (!zero_v && c + 1 < nchunks) issue_v(&maps, ctl, sm_base, h, t0 + kC);
        if constexpr (!kL64) {
          // the three M7 steps, each reading from TMEM what the one before
          // wrote; with kSplit only the first here, the other two below
          bool ok = true;
          for (int step = 0; step < (kSplit ? 1 : 3) && ok; ++step) {
            issue_m7_step(tbase, sm_base + OFF_KB, step);
            if (step < 2) {
              mma_commit(smem_u32(&ctl->bar[B_M7S]));
              if constexpr (!kSplit) {
                ok = solo_wait(ctl, B_M7S, ph_m7s, A.err);
                ph_m7s ^= 1u;
              }
            }
          }
          if (ok && !kSplit) mma_commit(smem_u32(&ctl->bar[B_M7]));
        }
      }
      ph_m4 ^= 1u;
      const bool slow = ctl->slow[par] != 0;
      if constexpr (!kL64 && kSplit) {
        // Steps 1 and 2 of M7.  While they run, the group turns V~_0 (step
        // 0's result) into bf16, so that M6/M5 over the first 32 tokens follow
        // step 2 in the pipe and only the second half remains after it.  This
        // pays when the state group sets the pace (one chain per SM); when
        // the chunk group does (many chains, the long-sequence plan), the
        // later M7 costs more than it saves and the plain order is used.
        if (!(alive = group_wait<false>(ctl, B_M7S, ph_m7s, stid, seq, A.err))) break;
        ph_m7s ^= 1u;
        if (stid == 0) {
          issue_m7_step(tbase, sm_base + OFF_KB, 1);
          mma_commit(smem_u32(&ctl->bar[B_M7S]));
        }
        {
          float y[32];
          tmem_ld32(tmem_addr(tbase, 32 * qw, TM_Y), y);
          tmem_wait_ld();
          tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_YB), y);
        }
        // after the per-tile range path, S^T <- S^T Diag(gamma_C) before M6
        // (else the scaling follows M6)
        if (slow) {
          const float *gam = ctl->gam[c % 3];
#pragma unroll 1
          for (int i0 = 0; i0 < kD; i0 += 32) {
            float sv[32];
            tmem_ld32(tmem_addr(tbase, 32 * qw, TM_S + i0), sv);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) sv[cc] *= gam[i0 + cc];
            tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), *reinterpret_cast<float(*)[16]>(sv));
            tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0 + 16), *reinterpret_cast<float(*)[16]>(sv + 16));
          }
        }
        // Diag(beta) of the next chunk (M3 of this chunk is done)
        if (stid < kC && c + 1 < nchunks) {
          cp_async_wait_all();
          *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_DB + sw128_offset(stid, stid)) =
              __float2bfloat16_rn(ctl->bsx[par ^ 1][stid]);
        }
        tmem_wait_st();
        group_publish<false>();
        if (stid == 0 && solo_wait(ctl, B_M7S, ph_m7s, A.err)) {
          issue_m7_step(tbase, sm_base + OFF_KB, 2);
          mma_commit(smem_u32(&ctl->bar[B_M7]));
          issue_m56_half(tbase, sm_base + OFF_AM + par * 8192, sm_base + OFF_KH + par * 16384, out_item, 0);
        }
        ph_m7s ^= 1u;
        if (!(alive = group_wait<false>(ctl, B_M7, c & 1, stid, seq, A.err))) break;
        {
          float y[32];
          tmem_ld32(tmem_addr(tbase, 32 * qw, TM_Y + 32), y);
          tmem_wait_ld();
          tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_YB + 16), y);
        }
        tmem_wait_st();
        group_publish<false>();
        if (stid == 0) {
          issue_m56_half(tbase, sm_base + OFF_AM + par * 8192, sm_base + OFF_KH + par * 16384, out_item, 1);
          mma_commit(smem_u32(&ctl->bar[B_M56]));
          // the previous chunk's output store has read the staging tile (it is
          // written again after the barrier below)
          tma_store_wait_read();
        }
      } else {
      if (!(alive = group_wait<false>(ctl, B_M7, c & 1, stid, seq, A.err))) break;

      // ---------------- V~^T -> bf16 A operand of M5/M6; after the per-tile
      // range path, S^T <- S^T Diag(gamma_C) before M6 (else the scaling follows M6)
      {
        float y[32];
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_Y), y);
        tmem_wait_ld();
        tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_YB), y);
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_Y + 32), y);
        tmem_wait_ld();
        tmem_st_bf16x32(tmem_addr(tbase, 32 * qw, TM_YB + 16), y);
      }
      if (slow) {
        const float *gam = ctl->gam[c % 3];
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
      }
      // Diag(beta) of the next chunk (M3 of this chunk is done: M7 has completed)
      if (stid < kC && c + 1 < nchunks) {
        cp_async_wait_all();
        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_DB + sw128_offset(stid, stid)) =
            __float2bfloat16_rn(ctl->bsx[par ^ 1][stid]);
      }
      tmem_wait_st();
      group_publish<false>();
      if (stid == 0) {
        issue_m56(tbase, sm_base + OFF_AM + par * 8192, sm_base + OFF_KH + par * 16384, out_item);
        mma_commit(smem_u32(&ctl->bar[B_M56]));
        // the previous chunk's output store has read the staging tile (it is
        // written again after the barrier below)
        tma_store_wait_read();
      }
      }
      if (!(alive = group_wait<false>(ctl, B_M56, ph_m56, stid, seq, A.err))) break;
      ph_m56 ^= 1u;
      // (this parity's operand buffers are now free: the chunk group loads q
      // and k of the chunk two ahead into them)
      // ---------------- the output rows of the chunk to the staging tile (O is
      // read before the next chunk's M4 overwrites it): before the state
      // refresh, or after it with the output gate (each order measured the
      // faster one for its variant)
      auto stage_o = [&]() {
        __nv_bfloat16 *ostage = reinterpret_cast<__nv_bfloat16 *>(vt);
        float v[64];
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_O), *reinterpret_cast<float(*)[32]>(v));
        tmem_ld32(tmem_addr(tbase, 32 * qw, TM_O + 32), *reinterpret_cast<float(*)[32]>(v + 32));
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) ostage[cc * kD + j] = __float2bfloat16_rn(v[cc]);
      };
      if (!kOG && out_item) stage_o();
      // ---------------- S^T <- S^T Diag(gamma_C) (unless done before M6), the
      // bf16 copy of the new state (and a checkpoint of the fp32 state when
      // one ends this chunk)
      float *cp = out_item ? ckpt_ptr(a, n, h, t0 + len - seq_bos) : nullptr;
      {
        const float *gam = ctl->gam[c % 3];
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
      if (kOG && out_item) stage_o();
      // A whole chunk without the output gate leaves by one TMA store of the
      // staging tile; a chunk cut short by the end of its sequence (whose
      // neighbour's rows the box would cover) and the gated rows by plain stores.
      const bool tma_out = !kOG && out_item && len == kC;
      tmem_wait_st();
      tc_fence_before();
      if (tma_out) fence_proxy_async_smem();
      if (kOG && out_item) {  // the barrier also waits for this chunk's out_gate tile
        if (!(alive = group_wait<false>(ctl, B_OG, c & 1, stid, seq, A.err))) break;
        if (stid == 0) ++ctl->og_lnd;
      } else {
        bar_state();
      }
      if (tma_out && stid == 0) {
        tma_store_3d(&maps.o, sm_base + OFF_VT, 0, h, t0);
        tma_store_commit();
      }
      if (out_item && !tma_out) {  // (the pair items of the long-sequence plan write no output)
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
      // (the next chunk's group waits order these reads of the staging tile
      // before it is written again)
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
    cp_async_wait_all();
    if (stid == 0) {
      tma_store_wait_all();
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

template <bool kZ, bool kOG, bool kSplit>
cudaError_t launch_variant(const TcMaps &maps, const TcArgs &args, int grid, cudaStream_t s) {
  constexpr uint32_t bytes = SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<kZ, kOG, kSplit>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  chunk_tc_kernel<kZ, kOG, kSplit><<<grid, kThreads, bytes, s>>>(maps, args);
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
      (og && encode_tok_head(encode, &maps.og, a.og, a.T_total, a.H, false, false) != CUDA_SUCCESS) ||
      (a.o && encode_tok_head(encode, &maps.o, a.o, a.T_total, a.H, false, false) != CUDA_SUCCESS))
    return cudaErrorInvalidValue;
  void *wd = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&wd, g_tc_watchdog);
  if (e != cudaSuccess) return e;
  const int NH = a.N * a.H;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    sms = 0;
  // split M7 for an unsplit launch with at most one chain per SM (measured:
  // batch prefill 0.570 -> 0.555 ms; varlen and the long-sequence plan slower)
  const bool split = a.plan == 0 && a.kinds == 1 && a.nseg == 1 && NH <= sms;
  TcArgs args{a, reinterpret_cast<unsigned int *>(wd)};
  const int grid = a.plan == 1 ? NH + 2 * NH * (a.P - 2) : a.plan == 2 ? NH * (a.P - 1) : NH * a.nseg * a.kinds;
  if (z) {
    if (og) return launch_variant<true, true, false>(maps, args, grid, s);
    return split ? launch_variant<true, false, true>(maps, args, grid, s)
                 : launch_variant<true, false, false>(maps, args, grid, s);
  }
  // the output gate comes with the layer form, whose decay is given as logits
  // (the out_gate tile shares the decay tile's buffer, half of which bf16 logits use)
  if (og) return cudaErrorInvalidValue;
  return split ? launch_variant<false, false, true>(maps, args, grid, s)
               : launch_variant<false, false, false>(maps, args, grid, s);
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
