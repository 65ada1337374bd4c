// Long sequences: in-device context parallelism through segment affine pairs.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
//
// [K3-notes §2.5, context-parallel affine pair]: a segment maps any entry
// state to S_out = S~ + M S_in, and pairs compose.  When a batch has too few
// (sequence, head) chains to fill the GPU, every sequence is cut into P
// segments of whole chunks (segment 0 may be longer than the others) and
//   pass 1  runs segment 0 from the real initial state with outputs (its
//           final state is the entry state E_1 of segment 1) and, beside it,
//           each of segments 1 .. P-2 twice with the tensor-core kernel:
//           from S = 0 with the real v (final state S~), and from S = I with
//           v = 0 (final state M, the product of the segment's transitions),
//           without outputs;
//   pass 2  chains the entry states E_{p+1} = S~_p + M_p E_p (fp32, one CTA
//           per chain);
//   pass 3  reruns segments 1 .. P-1 from their entry states, writing o, and
//           the last segment writes the final state.
// Segment 0 needs no pair and no rerun, since its entry state is known; it
// is made longer than the others when that packs pass 1 onto the SMs better.
// Every chain's segments run in parallel in passes 1 and 3.  Kernel
// boundaries order the passes; no kernel waits on another.
#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kScanThreads = 256;

// One CTA per (sequence n, head h).  pairs: [2][N][P-1][H][D][D] (S~ then M),
// E: [N][P][H][D][D] with E[n][0][h] = first[n * first_stride + h] (first
// nullable: zero; it may be E itself).  E_p lives in shared memory between steps.
__global__ void __launch_bounds__(kScanThreads)
cp_scan_kernel(int N, int H, int P, const float *first, int first_stride, const float *__restrict__ pairs,
               float *E) {
  extern __shared__ float sE[];  // [2][D][D]
  const int nh = blockIdx.x, n = nh / H, h = nh % H;
  const int tid = threadIdx.x, j = tid & (kD - 1), half = tid >> 7;
  const size_t DD = (size_t)kD * kD;
  const size_t pair_stride = (size_t)N * (P - 1) * H * DD;  // S~ -> M
  for (int e = tid; e < kD * kD; e += kScanThreads) {
    const float v = first ? first[((size_t)n * first_stride + h) * DD + e] : 0.f;
    sE[e] = v;
    E[(((size_t)n * P + 0) * H + h) * DD + e] = v;
  }
  __syncthreads();
  for (int p = 0; p + 1 < P; ++p) {
    const float *Ecur = sE + (p & 1) * kD * kD;
    float *Enext = sE + ((p + 1) & 1) * kD * kD;
    const float *St = pairs + (((size_t)n * (P - 1) + p) * H + h) * DD;
    const float *M = St + pair_stride;
    float *Eg = E + (((size_t)n * P + p + 1) * H + h) * DD;
    // rows [64 half, 64 half + 64) of column j
    for (int i = 64 * half; i < 64 * half + 64; ++i) {
      const float *Mi = M + (size_t)i * kD;
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll 8
      for (int m = 0; m < kD; m += 4) {
        const float4 mv = __ldg(reinterpret_cast<const float4 *>(Mi + m));
        acc0 += mv.x * Ecur[(m + 0) * kD + j];
        acc1 += mv.y * Ecur[(m + 1) * kD + j];
        acc2 += mv.z * Ecur[(m + 2) * kD + j];
        acc3 += mv.w * Ecur[(m + 3) * kD + j];
      }
      const float v = St[(size_t)i * kD + j] + ((acc0 + acc1) + (acc2 + acc3));
      Enext[i * kD + j] = v;
      Eg[(size_t)i * kD + j] = v;
    }
    __syncthreads();
  }
}

// Time for items of the given lengths (in chunk steps) to run when the
// block scheduler deals them, in order, each to the SM that frees first (one
// CTA per SM).
long long makespan(std::vector<long long> lens, long long sms) {
  std::sort(lens.begin(), lens.end(), std::greater<long long>());
  std::priority_queue<long long, std::vector<long long>, std::greater<long long>> q;
  for (long long i = 0; i < sms; ++i) q.push(0);
  long long end = 0;
  for (long long l : lens) {
    const long long t = q.top() + l;
    q.pop();
    q.push(t);
    end = std::max(end, t);
  }
  return end;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

}  // namespace

// Chooses the segments of every sequence.  requested: 0 = automatic, 1 =
// never split, >1 = that many equal segments (fewer if the sequence has
// fewer chunks).  The automatic plan times pass 1 and pass 3 with the
// scheduler model above over P = 3 .. 16 and a segment 0 of 1 to 4 times the
// other segments' length, against the unsplit run.
SegPlan plan_segments(const PrefillArgs &a, int requested) {
  SegPlan pl;
  pl.P = 1;
  pl.seg_tokens = 0;
  pl.ws_bytes = 0;
  pl.seg0 = 0;
  if (requested == 1 || a.cu != nullptr || !chunk_tc_supports(a) || a.T_seq <= 0) return pl;
  const long long nc = (a.T_seq + a.chunk - 1) / a.chunk;  // chunks per sequence
  const long long chains = (long long)a.N * a.H;
  long long P = 1, len0 = 0, len = 0;  // segments; chunks of segment 0 and of the others
  if (requested > 1) {
    P = requested < nc ? requested : nc;
    len = (nc + P - 1) / P;
    len0 = len;
  } else {
    const long long sms = sm_count();
    if (chains * 2 > sms || nc < 64) return pl;
    double best = (double)((chains + sms - 1) / sms) * nc;
    for (long long cand = 3; cand <= 16 && cand <= nc; ++cand) {
      for (int r4 = 4; r4 <= 16; ++r4) {  // segment 0 = r4 / 4 segments
        const long long l = (4 * nc + r4 + 4 * (cand - 1) - 1) / (r4 + 4 * (cand - 1));
        const long long l0 = nc - (cand - 1) * l;
        const long long last = nc - l0 - (cand - 2) * l;
        if (l < 1 || l0 < l || last < 1) continue;
        std::vector<long long> p1((size_t)chains, l0), p3;
        p1.insert(p1.end(), (size_t)(2 * (cand - 2) * chains), l);
        p3.insert(p3.end(), (size_t)((cand - 2) * chains), l);
        p3.insert(p3.end(), (size_t)chains, last);
        // (a scan step, one 128 x 128 product per boundary, costs about a chunk)
        const double t = (double)(makespan(p1, sms) + makespan(p3, sms)) + (cand - 2);
        if (t < 0.97 * best) {  // (a small margin keeps ties at the simpler plan)
          best = t;
          P = cand;
          len0 = l0;
          len = l;
        }
      }
    }
  }
  if (P <= 1) return pl;
  pl.seg0 = (int)(len0 * a.chunk);
  pl.seg_tokens = (int)(len * a.chunk);
  if (pl.seg0 >= a.T_seq) return SegPlan{1, 0, 0, 0};
  pl.P = 1 + (int)((a.T_seq - pl.seg0 + pl.seg_tokens - 1) / pl.seg_tokens);
  if (pl.P <= 1) return SegPlan{1, 0, 0, 0};
  const size_t state = (size_t)kD * kD * sizeof(float);
  pl.ws_bytes = (size_t)(3 * pl.P - 5) * (size_t)a.N * a.H * state;
  return pl;
}

// The affine pair of each whole sequence of the call: kind 0 (from S = 0
// with the real v) into pairs[0][n][h], kind 1 (from S = I, v = 0) into
// pairs[1][n][h].
cudaError_t launch_affine_pair(const PrefillArgs &a, float *pairs, cudaStream_t s) {
  PrefillArgs p1 = a;
  p1.o = nullptr;
  p1.s0 = nullptr;
  p1.sT = pairs;
  p1.seg_tokens = 0;
  p1.nseg = 1;
  p1.kinds = 2;
  p1.ck = nullptr;
  p1.og = nullptr;
  return launch_chunk_tc(p1, s);
}

// Entry states E [N][P][H][D][D] of P consecutive segments from the pairs of
// the first P - 1 ([2][N][P-1][H][D][D]) and the first segment's entry s0
// (nullable: zero).
cudaError_t launch_affine_compose(int N, int H, int P, const float *s0, const float *pairs, float *E,
                                  cudaStream_t s) {
  if (N * H == 0 || P <= 0) return cudaSuccess;
  const size_t smem = 2 * (size_t)kD * kD * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(cp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cp_scan_kernel<<<N * H, kScanThreads, smem, s>>>(N, H, P, s0, H, pairs, E);
  return cudaGetLastError();
}

cudaError_t launch_chunk_tc_segmented(const PrefillArgs &a, const SegPlan &pl, void *ws, cudaStream_t s) {
  const size_t DD = (size_t)kD * kD;
  float *pairs = static_cast<float *>(ws);                                     // [2][N][P-2][H][D][D]
  float *E = pairs + (size_t)2 * a.N * (pl.P - 2) * a.H * DD;                  // [N][P-1][H][D][D]
  PrefillArgs p1 = a;  // pass 1: segment 0 with outputs, pairs of segments 1 .. P-2
  p1.plan = 1;
  p1.P = pl.P;
  p1.seg0 = pl.seg0;
  p1.seg_tokens = pl.seg_tokens;
  p1.pairs = pairs;
  p1.E = E;
  p1.sT = nullptr;
  cudaError_t e = launch_chunk_tc(p1, s);
  if (e != cudaSuccess) return e;
  if (pl.P > 2) {  // E_2 .. E_{P-1} from E_1
    const size_t smem = 2 * DD * sizeof(float);
    e = cudaFuncSetAttribute(cp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cp_scan_kernel<<<a.N * a.H, kScanThreads, smem, s>>>(a.N, a.H, pl.P - 1, E, (pl.P - 1) * a.H, pairs, E);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  PrefillArgs p3 = a;  // pass 3: segments 1 .. P-1 from their entry states
  p3.plan = 2;
  p3.P = pl.P;
  p3.seg0 = pl.seg0;
  p3.seg_tokens = pl.seg_tokens;
  p3.E = E;
  return launch_chunk_tc(p3, s);
}

}  // namespace kda
