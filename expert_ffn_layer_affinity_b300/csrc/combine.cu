// Combine and bias feedback.
//
// Combine: out[t] = y_shared[t] + sum_k gate[t,k] * y_perm[row_of[t,k]], the
// single-GPU form of the pages' all-to-all combine (weigao.cc "DeepSeek-V3
// Technical Report：中英对照解读", §2.2 table, "dispatch/combine").  Gather form:
// every output chunk is produced by exactly one thread, no atomics.
//
// Bias feedback: after the step, b_e - gamma for an overloaded expert and
// b_e + gamma for an underloaded one (chenshi221 DeepSeek-V3 notes,
// "Auxiliary-loss-free 负载均衡"; weigao.cc §3 row "The bias is updated from
// observed expert load").  "Overloaded" = above the mean load T*K/E, decided
// exactly in integers.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4& v, float g) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}

template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y_perm,
                                                      const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ gate,
                                                      const uint4* __restrict__ y_shared, int T,
                                                      int K, int chunks, uint4* __restrict__ out) {
  const size_t n = static_cast<size_t>(T) * chunks;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / chunks, c = i % chunks;
    float acc[8];
    if (y_shared != nullptr) {
      const uint4 v = __ldcs(y_shared + i);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        acc[2 * j] = f.x;
        acc[2 * j + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    }
    uint4 v[KMAX];
    float g[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        const int32_t r = __ldg(row_of + t * K + k);
        g[k] = __ldg(gate + t * K + k);
        v[k] = __ldcs(y_perm + static_cast<size_t>(r) * chunks + c);
      }
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (k < K) acc_bf16x8(acc, v[k], g[k]);
    uint4 o;
    __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) oh[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    out[i] = o;
  }
}

__global__ void __launch_bounds__(1024) bias_update_kernel(const int32_t* __restrict__ load,
                                                           float* __restrict__ bias, int T, int K,
                                                           int E, float gamma,
                                                           float* __restrict__ stats) {
  __shared__ double red_sum[32], red_sq[32];
  __shared__ int red_max[32];
  const long long target = static_cast<long long>(T) * K;
  double sum = 0.0;
  int mx = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int l = load[e];
    const long long scaled = static_cast<long long>(E) * l;
    const float b = bias[e];
    if (scaled > target) bias[e] = __fsub_rn(b, gamma);
    else if (scaled < target) bias[e] = __fadd_rn(b, gamma);
    sum += l;
    mx = l > mx ? l : mx;
  }
  if (stats == nullptr) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    const int m = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
    mx = m > mx ? m : mx;
  }
  if (lane == 0) { red_sum[warp] = sum; red_max[warp] = mx; }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  double tot = 0.0;
  int gmx = 0;
  for (int w = 0; w < nw; ++w) { tot += red_sum[w]; gmx = red_max[w] > gmx ? red_max[w] : gmx; }
  const double mean = tot / E;
  double sq = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double dlt = load[e] - mean;
    sq += dlt * dlt;
  }
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
  if (lane == 0) red_sq[warp] = sq;
  __syncthreads();
  if (threadIdx.x == 0) {
    double v = 0.0;
    for (int w = 0; w < nw; ++w) v += red_sq[w];
    const double sd = sqrt(v / E);
    stats[0] = static_cast<float>(gmx);
    stats[1] = static_cast<float>(mean);
    stats[2] = mean > 0 ? static_cast<float>(gmx / mean) : 0.0f;
    stats[3] = mean > 0 ? static_cast<float>(sd / mean) : 0.0f;
  }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* row_of, const float* gate,
                           const uint16_t* y_shared, int T, int K, int d, uint16_t* out,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int chunks = d / 8;
  const size_t n = static_cast<size_t>(T) * chunks;
  size_t blocks = (n + 255) / 256;
  const size_t cap = static_cast<size_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  const uint4* yp = reinterpret_cast<const uint4*>(y_perm);
  const uint4* ys = reinterpret_cast<const uint4*>(y_shared);
  uint4* o = reinterpret_cast<uint4*>(out);
  const int b = static_cast<int>(blocks);
  if (K <= 2) combine_kernel<2><<<b, 256, 0, s>>>(yp, row_of, gate, ys, T, K, chunks, o);
  else if (K <= 4) combine_kernel<4><<<b, 256, 0, s>>>(yp, row_of, gate, ys, T, K, chunks, o);
  else if (K <= 8) combine_kernel<8><<<b, 256, 0, s>>>(yp, row_of, gate, ys, T, K, chunks, o);
  else if (K <= 16) combine_kernel<16><<<b, 256, 0, s>>>(yp, row_of, gate, ys, T, K, chunks, o);
  else combine_kernel<32><<<b, 256, 0, s>>>(yp, row_of, gate, ys, T, K, chunks, o);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const int32_t* load, float* bias, int T, int K, int E, float gamma,
                               float* stats, cudaStream_t s) {
  int threads = ((E + 31) / 32) * 32;
  if (threads > 1024) threads = 1024;
  if (threads < 32) threads = 32;
  bias_update_kernel<<<1, threads, 0, s>>>(load, bias, T, K, E, gamma, stats);
  return cudaGetLastError();
}

}  // namespace moe
