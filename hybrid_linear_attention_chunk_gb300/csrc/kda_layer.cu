// The KDA output's per-head RMSNorm and sigmoid gate as a pass over finished
// output rows, for the CUDA-core prefill (whose CTAs each hold a dv tile, not
// whole rows).  The tensor-core prefill and the decode step apply the same
// formula in their own epilogues.
//
// Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
// (liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
//   [K3-notes §2.2, KDA output]: y = Sigmoid(W_g x) o RMSNorm(o~), per head,
//   RMSNorm(x)_j = x_j w_j / sqrt(mean_j x_j^2 + eps).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per (token, head) row

__global__ void __launch_bounds__(32 * kRowsPerBlock)
norm_gate_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= (long long)a.T_total * a.H) return;  // (uniform over the warp)
  const int dv = a.dv;
  const size_t base = (size_t)row * dv;
  float x[4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = lane + 32 * i;
    x[i] = j < dv ? ld_elem(a.o, base + j, a.out) : 0.f;
    ss += x[i] * x[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = rsqrtf(ss / (float)dv + a.eps);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = lane + 32 * i;
    if (j < dv) {
      const float w = a.nw ? a.nw[j] : 1.f;
      st_elem(a.o, base + j, x[i] * r * w * sigmoid_f(ld_elem(a.og, base + j, a.qkv)), a.out);
    }
  }
}

}  // namespace

cudaError_t launch_norm_gate(const PrefillArgs &a, cudaStream_t s) {
  const long long rows = (long long)a.T_total * a.H;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  norm_gate_kernel<<<(unsigned)blocks, 32 * kRowsPerBlock, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kda
