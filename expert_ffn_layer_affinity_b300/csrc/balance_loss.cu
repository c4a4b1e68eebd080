// Forward value of the small sequence-wise balance loss that the method keeps
// next to the bias feedback ("同时保留一个极小的序列级平衡损失", chenshi221
// DeepSeek-V3 notes, "Auxiliary-loss-free 负载均衡"; weigao.cc §3 row "A small
// sequence-wise auxiliary loss is still used").  The pages print no formula;
// this follows the plainest reading, for a sequence of T_s tokens:
//   f_i = E / (K T_s) * #{(t, k): idx[t, k] = i}
//   P_i = (1 / T_s) * sum_t s[t, i] / sum_j s[t, j]
//   L   = alpha * sum_i f_i P_i
// One CTA per sequence; warp w takes tokens w, w+8, ...; lane l owns experts
// l*VPL .. l*VPL+VPL-1.  All sums run in a fixed order (deterministic).
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

template <int VPL>
__global__ void __launch_bounds__(kWarps * 32) seq_balance_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ idx, int ldk,
    const int32_t* __restrict__ seq_offsets, int E, int K, float alpha, float* __restrict__ loss) {
  __shared__ float part_p[kWarps][32 * VPL];
  __shared__ int part_c[kWarps][32 * VPL];
  __shared__ float red[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = seq_offsets[blockIdx.x], b = seq_offsets[blockIdx.x + 1];
  const int e0 = lane * VPL;
  float P[VPL];
  int cnt[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    P[j] = 0.0f;
    cnt[j] = 0;
  }
  for (int t = a + warp; t < b; t += kWarps) {
    const float* row = scores + static_cast<size_t>(t) * E;
    float s[VPL];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      s[j] = (e0 + j < E) ? row[e0 + j] : 0.0f;
      sum = __fadd_rn(sum, s[j]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, m));
#pragma unroll
    for (int j = 0; j < VPL; ++j) P[j] = __fadd_rn(P[j], __fdiv_rn(s[j], sum));
    for (int k = 0; k < K; ++k) {
      const int e = __ldg(idx + static_cast<size_t>(t) * ldk + k);
      if (e >= e0 && e < e0 + VPL) {
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (e == e0 + j) ++cnt[j];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    part_p[warp][e0 + j] = P[j];
    part_c[warp][e0 + j] = cnt[j];
  }
  __syncthreads();
  const int Ts = b - a;
  float term = 0.0f;
  if (Ts > 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float p = 0.0f;
      int c = 0;
      for (int w = 0; w < kWarps; ++w) {
        p = __fadd_rn(p, part_p[w][e]);
        c += part_c[w][e];
      }
      const float f = static_cast<float>(static_cast<double>(E) * c / (static_cast<double>(K) * Ts));
      term = __fadd_rn(term, __fmul_rn(f, __fdiv_rn(p, static_cast<float>(Ts))));
    }
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) term = __fadd_rn(term, __shfl_xor_sync(0xFFFFFFFFu, term, m));
  if (lane == 0) red[warp] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < kWarps; ++w) tot = __fadd_rn(tot, red[w]);
    loss[blockIdx.x] = __fmul_rn(alpha, tot);
  }
}

}  // namespace

cudaError_t launch_seq_balance(const float* scores, const int32_t* idx, int ldk,
                               const int32_t* seq_offsets, int S, int E, int K, float alpha,
                               float* loss, cudaStream_t s) {
  if (S == 0) return cudaSuccess;
  const dim3 grid(S), block(kWarps * 32);
  if (E <= 32) seq_balance_kernel<1><<<grid, block, 0, s>>>(scores, idx, ldk, seq_offsets, E, K, alpha, loss);
  else if (E <= 64) seq_balance_kernel<2><<<grid, block, 0, s>>>(scores, idx, ldk, seq_offsets, E, K, alpha, loss);
  else if (E <= 128) seq_balance_kernel<4><<<grid, block, 0, s>>>(scores, idx, ldk, seq_offsets, E, K, alpha, loss);
  else if (E <= 256) seq_balance_kernel<8><<<grid, block, 0, s>>>(scores, idx, ldk, seq_offsets, E, K, alpha, loss);
  else seq_balance_kernel<16><<<grid, block, 0, s>>>(scores, idx, ldk, seq_offsets, E, K, alpha, loss);
  return cudaGetLastError();
}

}  // namespace moe
