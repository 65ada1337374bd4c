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
//   M2  U^T = V^T T_b^T                                          (M=128 N=64 K=64)
//   M3  W^T = (Gamma o K)^T T_b^T                                (M=128 N=64 K=64)
//   M4  V~^T = U^T - S^T W^T ;  O^T = S^T (Q o Gamma)^T          (M=128 N=64 K=128, twice)
//   M5  O^T += V~^T A^T                                          (M=128 N=64 K=64)
//   S^T <- S^T Diag(gamma_C)           (fp32 master state in TMEM, scaled in place)
//   M6  S^T += V~^T (K o gamma_C / Gamma)                        (M=128 N=128 K=64)
// Every product is computed transposed so that M = 128 (dv or dk) and the
// tensor core runs at full width; TMEM lane j holds row j of the result.
//
// Two warp groups overlap consecutive chunks.  The chunk group (warps 0-7)
// runs one chunk ahead: decay prologue, M1, the UT solve, M2/M3.  The state
// group (warps 8-11) runs the serial state chain: -W staging, M4, V~ staging,
// the gamma scaling, M5/M6, the bf16 state copy and the output.  Operands the
// state group still reads while the chunk group prepares the next chunk are
// double-buffered by chunk parity.  Thread 0 of each group issues that
// group's MMAs and the chunk group's thread 0 issues the TMA loads of V.
//
// Range guard ([K3-notes §2.2, Eq. 5 and Fig. 3]): with log-decay >= -5 a
// 16-token tile sums to >= -80.  If every channel's chunk total G_C is >= -80
// the chunk start serves as the single decay reference (all factors within
// e^{+-80}).  Otherwise M1 runs in four accumulating rounds, one per 16-token
// key tile b, with the cumulative decay at tile b's start as the reference:
// query-side factors are <= 1 (rows before the tile are zeroed) and key-side
// factors are <= e^{80}.
//
// Every wait on an mbarrier is bounded (2 s).  On a time-out both groups
// leave their loops, drain their MMAs and copies, free TMEM and return with a
// bit set in a device word the host can read (kda_device_watchdog).
#include <cudaTypedefs.h>

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
constexpr uint32_t OFF_QG = 0;        // x2 32 KB: [Q o Gamma ; Gamma o K], 128 rows x 128, two K-halves;
                                      //   rows 64..127 later hold -W^T (MN-major) for the state group
constexpr uint32_t OFF_KB = 65536;    // 16 KB: K / Gamma, 64 rows x 128; then L (fp32 64x64) in the solve
constexpr uint32_t OFF_KH = 81920;    // x2 16 KB: K o gamma_C / Gamma (MN-major B of M6)
constexpr uint32_t OFF_AM = 114688;   // x2 8 KB: A bf16, 64 rows x 64
constexpr uint32_t OFF_ZT = 131072;   // 8 KB: T_b bf16, 64 rows x 64
constexpr uint32_t OFF_TF = 139264;   // 16 KB: T fp32 64x64
constexpr uint32_t OFF_XF = 155648;   // 4 KB: solve scratch fp32 [3][16][17]
constexpr uint32_t OFF_V = 159744;    // 16 KB: V tile (TMA), 64 rows x 128 as two 64-column boxes
constexpr uint32_t OFF_ST = 176128;   // 32 KB: S^T bf16, 128 rows x 128
constexpr uint32_t OFF_VT = 208896;   // 16 KB: V~^T bf16 128 rows x 64; also the output staging tile
constexpr uint32_t OFF_CTL = 225280;  // 4 KB control block
constexpr uint32_t SMEM_USED = OFF_CTL + 4096;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack

// TMEM columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // M1 result (chunk group)
constexpr uint32_t TM_W = 64;     // M3 result W^T (read by the state group)
constexpr uint32_t TM_U = 128;    // x2 64: U^T, V~^T after M4 (by chunk parity)
constexpr uint32_t TM_O = 256;    // O^T accumulator
constexpr uint32_t TM_S = 384;    // fp32 master state S^T (128 columns)

enum Bar : int {
  B_M1 = 0, B_M23, B_VFULL, B_READY0, B_READY1, B_FREE0, B_FREE1, B_WFREE, B_M4, B_M56,
  B_TD_C, B_TD_S, B_COUNT
};

struct Ctl {
  uint64_t bar[16];
  float gam[2][128];     // gamma_C per channel, by chunk parity
  float bs[64];          // beta of the chunk's rows (0 past the end)
  float tot[4][128];     // per-16-row-group log2-decay sums
  uint32_t tmem_slot;
  int abort;             // any thread gave up
  int nb;                // M1 rounds for the current chunk (1 or 4)
  int slow[2];           // range-guard vote, by chunk parity
  int go_c[2];           // chunk-group wait verdicts (double-buffered)
  int go_s[2];           // state-group wait verdicts
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

// a[i] for a runtime i without spilling the array to local memory
__device__ __forceinline__ float pick4(const float (&a)[4], int i) {
  return i == 0 ? a[0] : (i == 1 ? a[1] : (i == 2 ? a[2] : a[3]));
}

// Named barriers: 1 = chunk group (256 threads), 2 = state group (128).
__device__ __forceinline__ void bar_chunk() {
  __syncwarp();
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ void bar_state() {
  __syncwarp();
  asm volatile("bar.sync 2, 128;" ::: "memory");
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

// Inputs of one chunk held in registers by a chunk-group thread: channel pair
// (2p, 2p+1), rows [16 rg, 16 rg + 16).
// Thread layout of the prologue: channel octet o = ctid & 15 (channels
// [8o, 8o+8)), row group rg = ctid >> 4 (rows [4rg, 4rg+4)); every global
// load and shared store moves 16 bytes.
struct Prefetch {
  uint4 q[4], k[4];   // 8 bf16 each
  float4 g[4][2];     // 8 fp32 each
  float beta;
};

__device__ __forceinline__ void prefetch_chunk(Prefetch &pf, const PrefillArgs &a, int h, int t0, int len,
                                               int o, int rg, int ctid) {
  const int H = a.H;
  const uint4 *q = reinterpret_cast<const uint4 *>(a.q);
  const uint4 *k = reinterpret_cast<const uint4 *>(a.k);
  const float4 *g = reinterpret_cast<const float4 *>(a.g);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 4 * rg + r;
    if (row < len) {
      const size_t e = ((size_t)(t0 + row) * H + h) * (kD / 8) + o;  // in 8-element units
      pf.q[r] = __ldg(q + e);
      pf.k[r] = __ldg(k + e);
      pf.g[r][0] = __ldg(g + 2 * e);
      pf.g[r][1] = __ldg(g + 2 * e + 1);
    } else {
      pf.q[r] = make_uint4(0u, 0u, 0u, 0u);
      pf.k[r] = make_uint4(0u, 0u, 0u, 0u);
      pf.g[r][0] = pf.g[r][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pf.beta = 0.f;
  if (ctid < kC && ctid < len) pf.beta = __ldg(reinterpret_cast<const float *>(a.beta) + (size_t)(t0 + ctid) * H + h);
}

__device__ __forceinline__ void unpack8_bf16(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack_bf16(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void st_shared_8bf16(uint8_t *p, const float (&f)[8]) {
  st_shared_v4(p, pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

// fp32 64x64 matrices of the solve (L, T) are stored row-major with the
// column index XORed with 4*(row & 7): columns keep 4-float groups intact,
// and eight consecutive rows read at one column hit eight different banks.
__device__ __forceinline__ int swz64(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

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

// ------------------------------------------------------------- MMA batches

__device__ __forceinline__ void issue_m1(uint32_t tbase, uint32_t qg, uint32_t kb, bool acc_first) {
  constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
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
  for (int kk = 0; kk < 4; ++kk)  // W^T = (Gamma o K)^T T_b^T   (A = rows 64..127 of QG, MN-major)
    mma_bf16_ss(tbase + TM_W, smem_desc_sw128(qg + 8192 + kk * 2048, 16384, 1024),
                smem_desc_sw128(zt + kk * 32, 16, 1024), id, kk > 0 ? 1u : 0u);
}

// -W^T lives in QG rows 64..127 as an MN-major operand: i in [0,64) in the
// first K-half's rows 64..127, i in [64,128) in the second's.
__device__ __forceinline__ uint32_t wt_piece(uint32_t qg, int piece) { return qg + piece * 16384 + 8192; }

__device__ __forceinline__ void issue_m4(uint32_t tbase, uint32_t st, uint32_t qg, uint32_t tm_u) {
  constexpr uint32_t id_w = idesc_bf16_f32(128, 64, 0, 1);
  constexpr uint32_t id_q = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {  // V~^T = U^T + S^T (-W)^T
    const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
    mma_bf16_ss(tbase + tm_u, smem_desc_sw128(st + ka, 16, 1024),
                smem_desc_sw128(wt_piece(qg, kk >> 2) + (kk & 3) * 2048, 8192, 1024), id_w, 1u);
  }
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {  // O^T = S^T (Q o Gamma)^T
    const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
    mma_bf16_ss(tbase + TM_O, smem_desc_sw128(st + ka, 16, 1024), smem_desc_sw128(qg + ka, 16, 1024), id_q,
                kk > 0 ? 1u : 0u);
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
  const size_t sbase = ((size_t)n * H + h) * kD * kD;

  if (warp == 0) {
    tmem_alloc(smem_u32(&ctl->tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(smem_u32(&ctl->bar[b]), 1);
    ctl->abort = 0;
    ctl->nb = 1;
    ctl->slow[0] = ctl->slow[1] = 0;
    ctl->go_c[0] = ctl->go_c[1] = ctl->go_s[0] = ctl->go_s[1] = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_slot;
  const uint32_t sm_base = smem_u32(sm);

  if (tid < kChunkThreads) {
    // =========================================================== chunk group
    // registers: 256 x 200 + 128 x 104 = the launch's 384 x 168
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    const int ctid = tid;
    const int qw = warp & 3, ch = warp >> 2;
    const int o = ctid & 15, rg = ctid >> 4, tile = rg >> 2;  // prologue layout (see Prefetch)
    int seq = 0;
    uint32_t ph_m1 = 0, ph_m23 = 0, ph_v = 0;
    int issued_v = 0, landed_v = 0;
    if (ctid == 0 && nchunks > 0) {
      tma_prefetch_desc(&tmap_v);
      const uint32_t full = smem_u32(&ctl->bar[B_VFULL]);
      mbar_arrive_expect_tx(full, 2 * kC * 64 * 2);
      tma_load_3d(sm_base + OFF_V, &tmap_v, full, 0, h, bos);
      tma_load_3d(sm_base + OFF_V + 8192, &tmap_v, full, 64, h, bos);
      issued_v = 1;
    }
    Prefetch pf;
    if (nchunks > 0) prefetch_chunk(pf, a, h, bos, min(kC, eos - bos), o, rg, ctid);
    float *tot = reinterpret_cast<float *>(sm + OFF_TF);  // [16][128] row-group sums (T is not live yet)
    bool alive = true;
    for (int m = 0; m < nchunks && alive; ++m) {
      const int par = m & 1;
      const int t0 = bos + m * kC;
      const int len = min(kC, eos - t0);
      uint8_t *qg = sm + OFF_QG + par * 32768;
      uint8_t *kh = sm + OFF_KH + par * 16384;
      if (m >= 2 && !(alive = group_wait<true>(ctl, B_FREE0 + par, ((m >> 1) - 1) & 1, ctid, seq, A.err))) break;

      // ---------------- decay prologue: cumulative log2-decay and scaled operands
      float G[4][8];
      {
        float run[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) run[c] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float gg[8] = {pf.g[r][0].x, pf.g[r][0].y, pf.g[r][0].z, pf.g[r][0].w,
                               pf.g[r][1].x, pf.g[r][1].y, pf.g[r][1].z, pf.g[r][1].w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            run[c] += gg[c] * kLog2e;
            G[r][c] = run[c];
          }
        }
        *reinterpret_cast<float4 *>(tot + rg * 128 + 8 * o) = make_float4(run[0], run[1], run[2], run[3]);
        *reinterpret_cast<float4 *>(tot + rg * 128 + 8 * o + 4) = make_float4(run[4], run[5], run[6], run[7]);
      }
      if (ctid < kC) ctl->bs[ctid] = pf.beta;
      bar_chunk();
      // prefix over the 16 row groups: own offset and chunk total
      float own[8], GC[8];
      {
        float run[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) run[c] = own[c] = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < 16; ++g2) {
          if (g2 == rg) {
#pragma unroll
            for (int c = 0; c < 8; ++c) own[c] = run[c];
          }
          const float4 t0v = *reinterpret_cast<const float4 *>(tot + g2 * 128 + 8 * o);
          const float4 t1v = *reinterpret_cast<const float4 *>(tot + g2 * 128 + 8 * o + 4);
          run[0] += t0v.x; run[1] += t0v.y; run[2] += t0v.z; run[3] += t0v.w;
          run[4] += t1v.x; run[5] += t1v.y; run[6] += t1v.z; run[7] += t1v.w;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) GC[c] = run[c];
      }
      float gc[8];
      bool below = false;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
#pragma unroll
        for (int r = 0; r < 4; ++r) G[r][c] += own[c];
        gc[c] = ex2(GC[c]);
        below |= GC[c] < kSingleRefBound2;
      }
      if (rg == 0) {
        *reinterpret_cast<float4 *>(&ctl->gam[par][8 * o]) = make_float4(gc[0], gc[1], gc[2], gc[3]);
        *reinterpret_cast<float4 *>(&ctl->gam[par][8 * o + 4]) = make_float4(gc[4], gc[5], gc[6], gc[7]);
      }
      if (below) atomicOr(&ctl->slow[par], 1);
      bar_chunk();
      const bool slow = ctl->slow[par] != 0;
      if (ctid == 0) ctl->slow[par ^ 1] = 0;
      const uint32_t half = (uint32_t)(o >> 3), col = (uint32_t)(8 * (o & 7));
      uint8_t *qg_h = qg + half * 16384;
      uint8_t *kb_h = sm + OFF_KB + half * 8192;
      uint8_t *kh_h = kh + half * 8192;
      if (!slow) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t row = 4 * rg + r;
          float qv[8], kv[8], fq[8], fk[8], fb[8], fh[8];
          unpack8_bf16(pf.q[r], qv);
          unpack8_bf16(pf.k[r], kv);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float e = ex2(G[r][c]), i = ex2(-G[r][c]);
            fq[c] = qv[c] * e;
            fk[c] = kv[c] * e;
            fb[c] = kv[c] * i;
            fh[c] = fb[c] * gc[c];
          }
          st_shared_8bf16(qg_h + sw128_offset(row, col), fq);
          st_shared_8bf16(qg_h + sw128_offset(64 + row, col), fk);
          st_shared_8bf16(kb_h + sw128_offset(row, col), fb);
          st_shared_8bf16(kh_h + sw128_offset(row, col), fh);
        }
        group_publish<true>();
        if (ctid == 0) {
          issue_m1(tbase, smem_u32(qg), sm_base + OFF_KB, false);
          mma_commit(smem_u32(&ctl->bar[B_M1]));
        }
        alive = group_wait<true>(ctl, B_M1, ph_m1, ctid, seq, A.err);
        ph_m1 ^= 1u;
      } else {
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          if (!alive) break;
          // reference of key tile b: the cumulative decay before its first row
          float ref[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) ref[c] = 0.f;
          for (int g2 = 0; g2 < 4 * b; ++g2) {
#pragma unroll
            for (int c = 0; c < 8; ++c) ref[c] += tot[g2 * 128 + 8 * o + c];
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint32_t row = 4 * rg + r;
            float qv[8], kv[8], fq[8], fk[8], fb[8];
            unpack8_bf16(pf.q[r], qv);
            unpack8_bf16(pf.k[r], kv);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              fq[c] = fk[c] = fb[c] = 0.f;
              if (tile >= b) {
                const float e = ex2(G[r][c] - ref[c]);
                fq[c] = qv[c] * e;
                fk[c] = kv[c] * e;
              }
              if (tile == b) fb[c] = kv[c] * ex2(ref[c] - G[r][c]);
            }
            st_shared_8bf16(qg_h + sw128_offset(row, col), fq);
            st_shared_8bf16(qg_h + sw128_offset(64 + row, col), fk);
            st_shared_8bf16(kb_h + sw128_offset(row, col), fb);
          }
          group_publish<true>();
          if (ctid == 0) {
            issue_m1(tbase, smem_u32(qg), sm_base + OFF_KB, b > 0);
            mma_commit(smem_u32(&ctl->bar[B_M1]));
          }
          alive = group_wait<true>(ctl, B_M1, ph_m1, ctid, seq, A.err);
          ph_m1 ^= 1u;
        }
        if (!alive) break;
        // operands with the chunk start as reference (may underflow to 0: fine)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t row = 4 * rg + r;
          float qv[8], kv[8], fq[8], fk[8], fh[8];
          unpack8_bf16(pf.q[r], qv);
          unpack8_bf16(pf.k[r], kv);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float e = ex2(G[r][c]);
            fq[c] = qv[c] * e;
            fk[c] = kv[c] * e;
            fh[c] = kv[c] * ex2(GC[c] - G[r][c]);
          }
          st_shared_8bf16(qg_h + sw128_offset(row, col), fq);
          st_shared_8bf16(qg_h + sw128_offset(64 + row, col), fk);
          st_shared_8bf16(kh_h + sw128_offset(row, col), fh);
        }
      }
      if (!alive) break;
      // next chunk's inputs travel while this one computes
      if (m + 1 < nchunks) prefetch_chunk(pf, a, h, t0 + kC, min(kC, eos - t0 - kC), o, rg, ctid);

      // ---------------- masks, L, and T_b = (I + L)^{-1} diag(beta)
      {
        float *Lf = reinterpret_cast<float *>(sm + OFF_KB);  // K / Gamma is dead once M1 is done
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
            st_row16_bf16(sm + OFF_AM + par * 8192, r, s0, v);
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
            for (int cc = 0; cc < 16; ++cc) v[cc] = (s0 + cc < r) ? br * v[cc] : 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
              *reinterpret_cast<float4 *>(Lf + swz64(r, s0 + 4 * c4)) =
                  make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
          }
        }
        bar_chunk();
        // Diagonal 16x16 blocks by forward substitution, one column per thread:
        // x = e_c - L_blk x with x[m] = 0 for m < c, written without branches.
        if (ctid < 64) {
          const int ab = ctid >> 4, cc = ctid & 15, base = 16 * ab;
          float x[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            float acc = (rr == cc) ? 1.f : 0.f;
#pragma unroll
            for (int mm = 0; mm < rr; ++mm) acc -= Lf[swz64(base + rr, base + mm)] * x[mm];
            x[rr] = acc;
            Tf[swz64(base + rr, base + cc)] = acc;
          }
        }
        bar_chunk();
        // Off-diagonal blocks by distance d: T_ab = -T_aa sum_{c=b}^{a-1} L_ac T_cb.
        // One thread per (block, row, 4-column group); blocks above the
        // diagonal are never read (T_b below masks them).
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
          const int ntask = (4 - d) * 64;
          const int b = ctid >> 6, ab = b + d, rr = (ctid >> 2) & 15, c0 = 16 * b + 4 * (ctid & 3);
          if (ctid < ntask) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cb = b; cb < ab; ++cb) {
#pragma unroll
              for (int mm = 0; mm < 16; ++mm) {
                const float l = Lf[swz64(16 * ab + rr, 16 * cb + mm)];
                const float4 t = *reinterpret_cast<const float4 *>(Tf + swz64(16 * cb + mm, c0));
                acc.x += l * t.x; acc.y += l * t.y; acc.z += l * t.z; acc.w += l * t.w;
              }
            }
            *reinterpret_cast<float4 *>(Xf + (b * 16 + rr) * 16 + 4 * (ctid & 3)) = acc;
          }
          bar_chunk();
          if (ctid < ntask) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int mm = 0; mm < 16; ++mm) {
              const float l = Tf[swz64(16 * ab + rr, 16 * ab + mm)];
              const float4 x = *reinterpret_cast<const float4 *>(Xf + (b * 16 + mm) * 16 + 4 * (ctid & 3));
              acc.x += l * x.x; acc.y += l * x.y; acc.z += l * x.z; acc.w += l * x.w;
            }
            *reinterpret_cast<float4 *>(Tf + swz64(16 * ab + rr, c0)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
          }
          bar_chunk();
        }
        {
          const int r = ctid >> 2, s0 = (ctid & 3) * 16;
          const bool upper = (ctid & 3) > (r >> 4);  // block above the diagonal: T is zero there
          float v[16];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 t = *reinterpret_cast<const float4 *>(Tf + swz64(r, s0 + 4 * c4));
            v[4 * c4] = upper ? 0.f : t.x * ctl->bs[s0 + 4 * c4];
            v[4 * c4 + 1] = upper ? 0.f : t.y * ctl->bs[s0 + 4 * c4 + 1];
            v[4 * c4 + 2] = upper ? 0.f : t.z * ctl->bs[s0 + 4 * c4 + 2];
            v[4 * c4 + 3] = upper ? 0.f : t.w * ctl->bs[s0 + 4 * c4 + 3];
          }
          st_row16_bf16(sm + OFF_ZT, r, s0, v);
        }
      }
      group_publish<true>();

      // ---------------- U^T and W^T; then hand the chunk to the state group
      if (ctid == 0) {
        bool ok = solo_wait(ctl, B_VFULL, ph_v, A.err);
        ph_v ^= 1u;
        landed_v = ok ? issued_v : landed_v;
        if (ok && m >= 1) ok = solo_wait(ctl, B_WFREE, (m - 1) & 1, A.err);
        if (ok) {
          issue_m23(tbase, sm_base + OFF_V, smem_u32(qg), sm_base + OFF_ZT, TM_U + par * 64);
          mma_commit(smem_u32(&ctl->bar[B_M23]));
          ok = solo_wait(ctl, B_M23, ph_m23, A.err);
          ph_m23 ^= 1u;
        }
        if (ok && m + 1 < nchunks) {  // the V buffer is free again
          const uint32_t full = smem_u32(&ctl->bar[B_VFULL]);
          mbar_arrive_expect_tx(full, 2 * kC * 64 * 2);
          tma_load_3d(sm_base + OFF_V, &tmap_v, full, 0, h, t0 + kC);
          tma_load_3d(sm_base + OFF_V + 8192, &tmap_v, full, 64, h, t0 + kC);
          ++issued_v;
        }
        if (ok) mbar_arrive(smem_u32(&ctl->bar[B_READY0 + par]));
        ctl->go_c[seq & 1] = ok && !ctl->abort;
      }
      bar_chunk();
      alive = ctl->go_c[seq & 1] != 0;
      ++seq;
    }
    if (ctid == 0) {
      // outstanding V copy (only after an abort) and this group's MMAs
      volatile int no_abort = 0;
      if (issued_v > landed_v) mbar_wait(smem_u32(&ctl->bar[B_VFULL]), ph_v, &no_abort, A.err, 1u << 20);
      mma_commit(smem_u32(&ctl->bar[B_TD_C]));
      mbar_wait(smem_u32(&ctl->bar[B_TD_C]), 0, &no_abort, A.err, 1u << 21);
    }
  } else {
    // =========================================================== state group
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
    const int stid = tid - kChunkThreads;  // = TMEM lane j of every state-group product
    const int qw = warp & 3;                // lane quarter, = stid >> 5
    const int j = stid;
    int seq = 0;
    uint32_t ph_m4 = 0, ph_m56 = 0;
    // initial state -> TMEM (fp32 master) and the bf16 operand S^T
#pragma unroll 1
    for (int blk = 0; blk < 8; ++blk) {
      const int i0 = 16 * blk;
      float s[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) s[c] = a.s0 ? a.s0[sbase + (size_t)(i0 + c) * kD + j] : 0.f;
      tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
      st_row16_bf16(sm + OFF_ST + (blk >> 2) * 16384, j, 16 * (blk & 3), s);
    }
    tmem_wait_st();
    group_publish<false>();
    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
      const int par = c & 1;
      const int t0 = bos + c * kC;
      const int len = min(kC, eos - t0);
      uint8_t *qg = sm + OFF_QG + par * 32768;
      const uint32_t tm_u = TM_U + par * 64;
      if (!(alive = group_wait<false>(ctl, B_READY0 + par, (c >> 1) & 1, stid, seq, A.err))) break;

      // ---------------- -W^T (TMEM) -> MN-major operand in QG rows 64..127
      {
        uint8_t *dst = qg + (j >> 6) * 16384 + 8192;
        const uint32_t row = j & 63;
#pragma unroll
        for (int r0 = 0; r0 < 64; r0 += 16) {
          float v[16];
          tmem_ld16(tmem_addr(tbase, 32 * qw, TM_W + r0), v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) v[cc] = -v[cc];
          st_row16_bf16(dst, row, r0, v);
        }
      }
      group_publish<false>();
      if (stid == 0) {
        mbar_arrive(smem_u32(&ctl->bar[B_WFREE]));
        issue_m4(tbase, sm_base + OFF_ST, smem_u32(qg), tm_u);
        mma_commit(smem_u32(&ctl->bar[B_M4]));
      }
      if (!(alive = group_wait<false>(ctl, B_M4, ph_m4, stid, seq, A.err))) break;
      ph_m4 ^= 1u;

      // ---------------- V~^T -> bf16 operand; S^T <- S^T Diag(gamma_C)
#pragma unroll
      for (int r0 = 0; r0 < 64; r0 += 16) {
        float v[16];
        tmem_ld16(tmem_addr(tbase, 32 * qw, tm_u + r0), v);
        tmem_wait_ld();
        st_row16_bf16(sm + OFF_VT, j, r0, v);
      }
      {
        const float *gam = ctl->gam[par];
#pragma unroll 2
        for (int i0 = 0; i0 < 128; i0 += 16) {
          float s[16];
          tmem_ld16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) s[cc] *= gam[i0 + cc];
          tmem_st16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
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

      // ---------------- bf16 copy of the new state; the output rows
#pragma unroll 2
      for (int i0 = 0; i0 < 128; i0 += 16) {
        float s[16];
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        tmem_wait_ld();
        st_row16_bf16(sm + OFF_ST + (i0 >> 6) * 16384, j, i0 & 63, s);
      }
      {
        __nv_bfloat16 *ostage = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_VT);
#pragma unroll
        for (int r0 = 0; r0 < 64; r0 += 16) {
          float v[16];
          tmem_ld16(tmem_addr(tbase, 32 * qw, TM_O + r0), v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) ostage[(r0 + cc) * kD + j] = __float2bfloat16_rn(v[cc]);
        }
      }
      tc_fence_before();
      bar_state();
      {
        const uint4 *src = reinterpret_cast<const uint4 *>(sm + OFF_VT);
        uint4 *o = reinterpret_cast<uint4 *>(a.o);
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int idx = it * kStateThreads + stid, row = idx >> 4, c16 = idx & 15;
          if (row < len) o[((size_t)(t0 + row) * H + h) * (kD / 8) + c16] = src[idx];
        }
      }
      group_publish<false>();
      if (stid == 0) mbar_arrive(smem_u32(&ctl->bar[B_FREE0 + par]));
    }
    if (alive && a.sT) {
#pragma unroll 1
      for (int i0 = 0; i0 < 128; i0 += 16) {
        float s[16];
        tmem_ld16(tmem_addr(tbase, 32 * qw, TM_S + i0), s);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) a.sT[sbase + (size_t)(i0 + cc) * kD + j] = s[cc];
      }
    }
    if (stid == 0) {
      volatile int no_abort = 0;
      mma_commit(smem_u32(&ctl->bar[B_TD_S]));
      mbar_wait(smem_u32(&ctl->bar[B_TD_S]), 0, &no_abort, A.err, 1u << 22);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
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
