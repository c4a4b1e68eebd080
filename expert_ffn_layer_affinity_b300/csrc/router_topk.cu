// Router selection: bias-adjusted, group-limited top-K with gates taken from
// the raw affinities, plus the per-expert load histogram.  One warp per token.
//
// Method: the selection score is affinity + bias and the bias is used only to
// choose experts ("Score = Affinity + Bias", DeepSeek V3, deepseekmodel1.org,
// section 公式解密; chenshi221 DeepSeek-V3 notes, "Auxiliary-loss-free 负载均衡");
// each token reaches at most M expert groups (same notes: "每个 token 最多发往 M
// 个节点"); loads are counted over the whole batch (qwbw.cn essay on the
// report, "统计整批样本各个专家的负载情况").
//
// Ordering: every candidate carries a 64-bit key = (orderable fp32 score << 32)
// | (0xFFFFFFFF - expert).  The largest key is the highest score, and on equal
// scores the lower expert index.  -0 is folded into +0, NaN gets the key
// class just above "excluded" (below -inf), excluded experts have key 0.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxTopPerGroup = 4;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint64_t make_key(float z, int e) {
  uint32_t ord;
  if (z != z) {
    ord = 1u;
  } else {
    uint32_t u = __float_as_uint(z);
    if (u == 0x80000000u) u = 0u;
    ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float key_value(uint64_t k) {
  const uint32_t ord = static_cast<uint32_t>(k >> 32);
  if (ord == 1u) return __uint_as_float(0x7FC00000u);
  const uint32_t u = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(u);
}

__device__ __forceinline__ int key_index(uint64_t k) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const uint64_t o = shfl_xor_u64(v, m);
    v = o > v ? o : v;
  }
  return v;
}

// Insert `k` into the descending list top[0..n) (keys are distinct unless 0).
__device__ __forceinline__ void top_insert(uint64_t (&top)[kMaxTopPerGroup], int n, uint64_t k) {
#pragma unroll
  for (int i = 0; i < kMaxTopPerGroup; ++i) {
    if (i < n && k > top[i]) {
      const uint64_t t = top[i];
      top[i] = k;
      k = t;
    }
  }
}

template <int VPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) topk_kernel(TopkArgs a) {
  extern __shared__ int32_t hist[];
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int e0 = lane * VPL;
  const int E = a.E, K = a.K, G = a.n_groups, M = a.topk_groups;
  const int gsz = E / G;
  const int lanes_per_group = gsz / VPL;  // power of two when G > 1 (host check)
  const int n_top = (K + M - 1) / M;
  const float scale = a.route_scale;

  float b[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) b[j] = (e0 + j < E) ? a.bias[e0 + j] : 0.0f;
  bool nonfinite = false;
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    if (e0 + j < E && !isfinite(b[j])) nonfinite = true;

  const int nwarps = gridDim.x * kWarpsPerBlock;
  for (int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); t < a.T; t += nwarps) {
    const float* row = a.scores + static_cast<size_t>(t) * E;
    float s[VPL];
    if (E == 32 * VPL && VPL >= 4) {
#pragma unroll
      for (int j = 0; j < VPL; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + e0 + j);
        s[j] = v.x; s[j + 1] = v.y; s[j + 2] = v.z; s[j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) s[j] = (e0 + j < E) ? row[e0 + j] : 0.0f;
    }

    uint64_t key[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (e0 + j < E) {
        if (!isfinite(s[j])) nonfinite = true;
        key[j] = make_key(__fadd_rn(s[j], b[j]), e0 + j);
      } else {
        key[j] = 0;
      }
    }

    if (G > 1) {
      // Group score: sum of the n_top largest biased scores of the group.
      uint64_t top[kMaxTopPerGroup] = {0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < VPL; ++j) top_insert(top, n_top, key[j]);
      for (int m = 1; m < lanes_per_group; m <<= 1) {
        uint64_t other[kMaxTopPerGroup];
#pragma unroll
        for (int i = 0; i < kMaxTopPerGroup; ++i) other[i] = shfl_xor_u64(top[i], m);
#pragma unroll
        for (int i = 0; i < kMaxTopPerGroup; ++i) top_insert(top, n_top, other[i]);
      }
      float gs = key_value(top[0]);
      for (int i = 1; i < n_top; ++i) gs = __fadd_rn(gs, key_value(top[i]));
      const int my_group = e0 / gsz;
      uint64_t gkey = (e0 < E) ? make_key(gs, my_group) : 0ull;
      bool kept = false;
      for (int r = 0; r < M; ++r) {
        const uint64_t m = warp_max_u64(gkey);
        if (gkey == m && m != 0ull) {
          kept = true;
          gkey = 0ull;
        }
      }
      if (!kept) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) key[j] = 0ull;
      }
    }

    int my_idx = 0;
    for (int r = 0; r < K; ++r) {
      uint64_t lm = key[0];
#pragma unroll
      for (int j = 1; j < VPL; ++j) lm = key[j] > lm ? key[j] : lm;
      const uint64_t m = warp_max_u64(lm);
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (key[j] == m) key[j] = 0ull;
      if (lane == r) my_idx = key_index(m);
    }

    const float sk = (lane < K) ? row[my_idx] : 0.0f;
    float denom = 0.0f;
    for (int r = 0; r < K; ++r) {
      const float v = __shfl_sync(kFull, sk, r);
      denom = (r == 0) ? v : __fadd_rn(denom, v);
    }
    const int ldk = K + a.n_shared_routed;
    if (lane < K) {
      const size_t o = static_cast<size_t>(t) * ldk + lane;
      a.idx[o] = my_idx;
      a.gate[o] = __fmul_rn(__fdiv_rn(sk, denom), scale);
      atomicAdd(&hist[my_idx], 1);
    } else if (lane < ldk) {
      // serving layout: shared expert j travels as routed expert E + j, gate 1
      const size_t o = static_cast<size_t>(t) * ldk + lane;
      a.idx[o] = E + (lane - K);
      a.gate[o] = 1.0f;
    }
  }
  if (__any_sync(kFull, nonfinite) && lane == 0 && a.status)
    atomicOr(reinterpret_cast<unsigned int*>(a.status), MOE_DEV_NONFINITE);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (hist[i]) atomicAdd(&a.load[i], hist[i]);
}

// w = hi + mid + lo exactly: each part is the bf16 rounding of what is left.
__global__ void router_split_kernel(const float* __restrict__ w, int E, int d,
                                    __nv_bfloat16* __restrict__ out) {
  const size_t n = static_cast<size_t>(E) * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = i / d, j = i % d;
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    __nv_bfloat16* o = out + e * 3 * d;
    o[j] = hi;
    o[d + j] = mid;
    o[2 * d + j] = lo;
  }
}

template <int VPL>
cudaError_t launch_topk_vpl(const TopkArgs& a, cudaStream_t s) {
  const int warps_needed = a.T;
  int blocks = (warps_needed + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int cap = sm_count() * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  topk_kernel<VPL><<<blocks, kWarpsPerBlock * 32, a.E * sizeof(int32_t), s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(a.load, 0, sizeof(int32_t) * a.E, s);
  if (err != cudaSuccess) return err;
  if (a.T == 0) return cudaSuccess;
  if (a.E <= 32) return launch_topk_vpl<1>(a, s);
  if (a.E <= 64) return launch_topk_vpl<2>(a, s);
  if (a.E <= 128) return launch_topk_vpl<4>(a, s);
  if (a.E <= 256) return launch_topk_vpl<8>(a, s);
  return launch_topk_vpl<16>(a, s);
}

cudaError_t launch_router_split(const float* w_r, int E, int d, uint16_t* w_split, cudaStream_t s) {
  const size_t n = static_cast<size_t>(E) * d;
  if (n == 0) return cudaSuccess;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > sm_count() * 8) blocks = sm_count() * 8;
  router_split_kernel<<<blocks, 256, 0, s>>>(w_r, E, d, reinterpret_cast<__nv_bfloat16*>(w_split));
  return cudaGetLastError();
}

}  // namespace moe
