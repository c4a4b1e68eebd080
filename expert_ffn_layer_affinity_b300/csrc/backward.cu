// Backward pass of the layer: the gather / elementwise kernels.
//
// The bias only chooses experts and never enters a gate value ("Bias
// 仅用于路由", deepseekmodel1.org, "公式解密"; chenshi221 DeepSeek-V3 notes,
// "Auxiliary-loss-free 负载均衡"), so with the chosen experts held fixed the
// gradient reaches the router through the gates, which depend on the raw
// affinities only:
//   g_k  = scale s_k / S,  S = sum over the K chosen experts of s_j
//   ds_k = scale (dg_k / S - sum_j dg_j s_j / S^2),  du_k = ds_k s_k (1 - s_k)
// The expert FFN, y = W2 (silu(a) c), a = W1 v, c = W3 v, gives
//   dh = W2^T dy, da = dh c silu'(a), dc = dh silu(a),
//   silu'(a) = sig(a) (1 + a (1 - sig(a))).
// Reductions run in a fixed order, so every result is deterministic.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}

// One warp per token: dy_perm[row_of[t,k]] = gate[t,k] dy[t] and
// dgate[t,k] = <dy[t], y_perm[row_of[t,k]]> (fp32, lane-strided partial sums
// added in a fixed butterfly).
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ y_perm,
    const int32_t* __restrict__ row_of, const float* __restrict__ gate, int T, int K, int chunks,
    uint4* __restrict__ dy_perm, float* __restrict__ dgate) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nw) {
    const uint4* dyr = dy + static_cast<size_t>(t) * chunks;
    for (int k = 0; k < K; ++k) {
      const int32_t r = __ldg(row_of + static_cast<size_t>(t) * K + k);
      const float g = __ldg(gate + static_cast<size_t>(t) * K + k);
      const uint4* yr = y_perm + static_cast<size_t>(r) * chunks;
      uint4* dr = dy_perm + static_cast<size_t>(r) * chunks;
      float acc = 0.0f;
#pragma unroll 4
      for (int c = lane; c < chunks; c += 32) {
        const uint4 a = __ldg(dyr + c);
        const uint4 b = __ldcs(yr + c);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(bf_lo(av[i]), bf_lo(bv[i]), acc);
          acc = fmaf(bf_hi(av[i]), bf_hi(bv[i]), acc);
          o[i] = pack_bf2(g * bf_lo(av[i]), g * bf_hi(av[i]));
        }
        __stcs(dr + c, make_uint4(o[0], o[1], o[2], o[3]));
      }
      acc = warp_sum(acc);
      if (lane == 0) dgate[static_cast<size_t>(t) * K + k] = acc;
    }
  }
}

// Elementwise SwiGLU backward: per row, dac = [da | dc] (2I columns) and the
// recomputed h = silu(a) c (I columns; skipped when h is null), from dh, a,
// c (I columns each).  8 columns (16 bytes of each input) per thread when
// I % 8 == 0, else 2.
template <int V>
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(
    const uint16_t* __restrict__ dh, const uint16_t* __restrict__ a,
    const uint16_t* __restrict__ c, long long R, int I, uint16_t* __restrict__ dac,
    uint16_t* __restrict__ h) {
  using Vec = typename std::conditional<V == 8, uint4, uint32_t>::type;
  constexpr int W = V / 2;  // 32-bit words per vector
  const int per_row = I / V;
  const long long n = R * per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / per_row;
    const int j = static_cast<int>(i - r * per_row) * V;  // first column
    const size_t src = static_cast<size_t>(r) * I + j;
    const Vec vh = __ldcs(reinterpret_cast<const Vec*>(dh + src));
    const Vec va = __ldcs(reinterpret_cast<const Vec*>(a + src));
    const Vec vc = __ldcs(reinterpret_cast<const Vec*>(c + src));
    const uint32_t* wh = reinterpret_cast<const uint32_t*>(&vh);
    const uint32_t* wa = reinterpret_cast<const uint32_t*>(&va);
    const uint32_t* wc = reinterpret_cast<const uint32_t*>(&vc);
    Vec oda, odc, oh;
    uint32_t* pda = reinterpret_cast<uint32_t*>(&oda);
    uint32_t* pdc = reinterpret_cast<uint32_t*>(&odc);
    uint32_t* ph = reinterpret_cast<uint32_t*>(&oh);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      float da[2], dc[2], hh[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float g = e ? bf_hi(wh[w]) : bf_lo(wh[w]);
        const float x = e ? bf_hi(wa[w]) : bf_lo(wa[w]);
        const float u = e ? bf_hi(wc[w]) : bf_lo(wc[w]);
        const float sig = 1.0f / (1.0f + expf(-x));
        const float silu = x * sig;
        da[e] = g * u * (sig * (1.0f + x * (1.0f - sig)));
        dc[e] = g * silu;
        hh[e] = silu * u;
      }
      pda[w] = pack_bf2(da[0], da[1]);
      pdc[w] = pack_bf2(dc[0], dc[1]);
      ph[w] = pack_bf2(hh[0], hh[1]);
    }
    uint16_t* drow = dac + static_cast<size_t>(r) * 2 * I;
    __stcs(reinterpret_cast<Vec*>(drow + j), oda);
    __stcs(reinterpret_cast<Vec*>(drow + I + j), odc);
    if (h) __stcs(reinterpret_cast<Vec*>(h + src), oh);
  }
}

// One warp per token: du[t,k] from the gate gradients (chosen experts only),
// and dx_router[t] = sum_k du[t,k] w_r[idx[t,k], :] in fp32.
__global__ void __launch_bounds__(256) router_bwd_token_kernel(
    const float* __restrict__ dgate, const int32_t* __restrict__ idx, int ld_idx,
    const float* __restrict__ affinity, const float* __restrict__ w_r, int T, int d, int E, int K,
    float scale, float* __restrict__ du, float* __restrict__ dx_router) {
  __shared__ int se[8][32];
  __shared__ float sdu[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nw) {
    // lanes 0..K-1 hold one chosen expert each
    int e = 0;
    float s = 0.0f, dg = 0.0f;
    if (lane < K) {
      e = __ldg(idx + static_cast<size_t>(t) * ld_idx + lane);
      s = __ldg(affinity + static_cast<size_t>(t) * E + e);
      dg = __ldg(dgate + static_cast<size_t>(t) * K + lane);
    }
    // ds_k = scale (dg_k S - sum_j dg_j s_j) / S^2 = scale sum_j s_j (dg_k - dg_j) / S^2:
    // differences first, so equal gate gradients (and K = 1) give exactly 0
    float S = 0.0f, num = 0.0f;
    for (int j = 0; j < K; ++j) {  // in rank order
      const float sj = __shfl_sync(kFull, s, j);
      const float dgj = __shfl_sync(kFull, dg, j);
      S += sj;
      num = fmaf(sj, dg - dgj, num);
    }
    const float ds = scale * (num / (S * S));
    const float duk = lane < K ? ds * s * (1.0f - s) : 0.0f;
    if (lane < K) du[static_cast<size_t>(t) * K + lane] = duk;
    if (dx_router) {
      // the K (expert, du) pairs through this warp's shared slots, so the
      // column loop needs no warp-wide exchange
      se[warp][lane] = e;
      sdu[warp][lane] = duk;
      __syncwarp();
      float* out = dx_router + static_cast<size_t>(t) * d;
      for (int c = lane; c < d; c += 32) {
        float acc = 0.0f;
        for (int k = 0; k < K; ++k)
          acc = fmaf(sdu[warp][k], __ldg(w_r + static_cast<size_t>(se[warp][k]) * d + c), acc);
        out[c] = acc;
      }
      __syncwarp();
    }
  }
}

// dw_r[e, c] = sum over the rows r of expert e (ascending) of du[row] x[tok_of[r], c].
// One block per (expert, 2048-column chunk), 8 columns (one 16-byte load of a
// token row) per thread; du_row[r] is du of the (token, slot) that row r came
// from.
__global__ void __launch_bounds__(256) router_bwd_weight_kernel(
    const float* __restrict__ du_row, const int32_t* __restrict__ tok_of,
    const int32_t* __restrict__ offsets, const uint16_t* __restrict__ x, int d, int E,
    float* __restrict__ dw_r) {
  const int e = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (e >= E || c >= d) return;
  const int r0 = offsets[e], r1 = offsets[e + 1];
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll 4
  for (int r = r0; r < r1; ++r) {
    const int t = __ldg(tok_of + r);
    const float u = __ldg(du_row + r);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + c));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = fmaf(u, bf_lo(w[j]), acc[2 * j]);
      acc[2 * j + 1] = fmaf(u, bf_hi(w[j]), acc[2 * j + 1]);
    }
  }
  float4* out = reinterpret_cast<float4*>(dw_r + static_cast<size_t>(e) * d + c);
  out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// du by row of the dispatch order: du_row[row_of[t,k]] = du[t,k].
__global__ void __launch_bounds__(256) scatter_rows_kernel(const float* __restrict__ du,
                                                           const int32_t* __restrict__ row_of,
                                                           long long n, float* __restrict__ du_row) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    du_row[row_of[i]] = du[i];
}

// dx[t] = bf16( fp32(dx_shared[t]) + dx_router[t] + sum_k fp32(dx_perm[row_of[t,k]]) ),
// the slots added in rank order.  8 columns per thread.
__global__ void __launch_bounds__(256) combine_dx_kernel(
    const uint4* __restrict__ dx_perm, const int32_t* __restrict__ row_of, int K,
    const uint4* __restrict__ dx_shared, const float4* __restrict__ dx_router, int T, int chunks,
    uint4* __restrict__ dx) {
  const long long n = static_cast<long long>(T) * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / chunks;
    const int c = static_cast<int>(i - t * chunks);
    float acc[8];
    if (dx_shared) {
      const uint4 v = __ldg(dx_shared + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = bf_lo(w[j]);
        acc[2 * j + 1] = bf_hi(w[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    }
    if (dx_router) {
      const float4 a = __ldg(dx_router + 2 * i), b = __ldg(dx_router + 2 * i + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    for (int k = 0; k < K; ++k) {
      const int32_t r = __ldg(row_of + t * K + k);
      const uint4 v = __ldcs(dx_perm + static_cast<size_t>(r) * chunks + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] += bf_lo(w[j]);
        acc[2 * j + 1] += bf_hi(w[j]);
      }
    }
    dx[i] = make_uint4(pack_bf2(acc[0], acc[1]), pack_bf2(acc[2], acc[3]), pack_bf2(acc[4], acc[5]),
                       pack_bf2(acc[6], acc[7]));
  }
}

int grid_cap(long long work, int per_block, int cap_per_sm) {
  long long b = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sm_count()) * cap_per_sm;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_combine_backward(const uint16_t* dy, const uint16_t* y_perm,
                                    const int32_t* row_of, const float* gate, int T, int K, int d,
                                    uint16_t* dy_perm, float* dgate, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  combine_bwd_kernel<<<grid_cap(T, 8, 16), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(dy), reinterpret_cast<const uint4*>(y_perm), row_of, gate, T,
      K, d / 8, reinterpret_cast<uint4*>(dy_perm), dgate);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_backward(const uint16_t* dh, const uint16_t* a, const uint16_t* c, int R,
                                   int I, uint16_t* dac, uint16_t* h, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const bool wide = I % 8 == 0 && ((reinterpret_cast<uintptr_t>(dh) | reinterpret_cast<uintptr_t>(a) |
                                     reinterpret_cast<uintptr_t>(c) | reinterpret_cast<uintptr_t>(dac) |
                                     reinterpret_cast<uintptr_t>(h)) & 15u) == 0;
  if (wide) {
    const long long n = static_cast<long long>(R) * (I / 8);
    swiglu_bwd_kernel<8><<<grid_cap(n, 256, 16), 256, 0, s>>>(dh, a, c, R, I, dac, h);
  } else {
    const long long n = static_cast<long long>(R) * (I / 2);
    swiglu_bwd_kernel<2><<<grid_cap(n, 256, 16), 256, 0, s>>>(dh, a, c, R, I, dac, h);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_backward(const float* dgate, const int32_t* idx, int ld_idx,
                                   const float* affinity, const float* w_r, const uint16_t* x,
                                   const int32_t* row_of, const int32_t* tok_of,
                                   const int32_t* offsets, int T, int d, int E, int K, float scale,
                                   float* du, float* du_row, float* dx_router, float* dw_r,
                                   cudaStream_t s) {
  if (T == 0) return cudaMemsetAsync(dw_r, 0, sizeof(float) * E * d, s);
  router_bwd_token_kernel<<<grid_cap(T, 8, 16), 256, 0, s>>>(dgate, idx, ld_idx, affinity, w_r, T,
                                                             d, E, K, scale, du, dx_router);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(T) * K;
  scatter_rows_kernel<<<grid_cap(n, 256, 8), 256, 0, s>>>(du, row_of, n, du_row);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  router_bwd_weight_kernel<<<dim3((d / 8 + 255) / 256, E), 256, 0, s>>>(du_row, tok_of, offsets, x,
                                                                         d, E, dw_r);
  return cudaGetLastError();
}

cudaError_t launch_combine_dx(const uint16_t* dx_perm, const int32_t* row_of, int K,
                              const uint16_t* dx_shared, const float* dx_router, int T, int d,
                              uint16_t* dx, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int chunks = d / 8;
  combine_dx_kernel<<<grid_cap(static_cast<long long>(T) * chunks, 256, 8), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(dx_perm), row_of, K, reinterpret_cast<const uint4*>(dx_shared),
      reinterpret_cast<const float4*>(dx_router), T, chunks, reinterpret_cast<uint4*>(dx));
  return cudaGetLastError();
}

}  // namespace moe
