// E4M3 quantization with fine-grained scaling, and the FP8 row gather.
//
// The pages quantize activations per 1 x 128 tile and weights per 128 x 128
// block, all in E4M3 (qwbw.cn essay on the report, the FP8 training passage;
// "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), section "6. FP8
// Training", row "Fine-grained quantization is used").  A block's scale is
// fp32(amax / 448) (1 for an all-zero block) and each code is the E4M3
// rounding, to nearest even and saturating at +-448, of fp32(value / scale).
//
// Activation scales are stored block-major, s[j * ld_s + row] for the 128
// columns j*128 .. j*128+127 of `row`: the GEMM epilogue then reads the
// scales of consecutive tokens from consecutive addresses.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float block_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
}

// One warp per (row, run of up to kRowBlocks consecutive 128-column blocks);
// lane l holds columns 4l .. 4l+3 of each block.  The warp loads the whole
// run before it reduces any block: a warp that moved one block per trip kept
// only 256 bytes in flight and ran the x and h quantizations at about a third
// of the HBM bandwidth.  Each block's arithmetic is unchanged.
constexpr int kRowBlocks = 8;
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ in, int rows,
                                                         int cols, uint8_t* __restrict__ q,
                                                         float* __restrict__ s, int ld_s) {
  const int lane = threadIdx.x & 31;
  const int nb = cols / 128;
  const int nrun = (nb + kRowBlocks - 1) / kRowBlocks;
  const long long total = static_cast<long long>(rows) * nrun;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
       w < total; w += nwarps) {
    const long long r = w / nrun;
    const int j0 = static_cast<int>(w - r * nrun) * kRowBlocks;
    const int n = nb - j0 < kRowBlocks ? nb - j0 : kRowBlocks;  // blocks of this run
    const size_t base = static_cast<size_t>(r) * cols + static_cast<size_t>(j0) * 128 + lane * 4;
    uint2 raw[kRowBlocks];
#pragma unroll
    for (int u = 0; u < kRowBlocks; ++u)
      raw[u] = u < n ? __ldcs(reinterpret_cast<const uint2*>(in + base + u * 128)) : make_uint2(0, 0);
#pragma unroll
    for (int u = 0; u < kRowBlocks; ++u) {
      if (u >= n) break;  // warp-uniform
      const float x0 = bf16_lo(raw[u].x), x1 = bf16_hi(raw[u].x);
      const float x2 = bf16_lo(raw[u].y), x3 = bf16_hi(raw[u].y);
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
      const float sc = block_scale(amax);
      const uint32_t lo = cvt_e4m3x2(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = cvt_e4m3x2(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      *reinterpret_cast<uint32_t*>(q + base + u * 128) = lo | (hi << 16);
      if (lane == 0) s[static_cast<size_t>(j0 + u) * ld_s + r] = sc;
    }
  }
}

// One CTA (256 threads) per 128 x 128 block.  Thread t holds row t/2,
// columns (t%2)*64 .. +63 of the block.  With a second matrix (w_pair), the
// two are written row-interleaved: output row 2i is w's row i, 2i+1 is
// w_pair's row i, and the two block scales sit side by side.  Each row of
// block scales is padded to a multiple of 4 floats, so the GEMM can fetch
// them with 16-byte TMA boxes.
__global__ void __launch_bounds__(256) quant_blocks_kernel(const uint16_t* __restrict__ w,
                                                           const uint16_t* __restrict__ w_pair,
                                                           int rows, int cols,
                                                           uint8_t* __restrict__ q,
                                                           float* __restrict__ s) {
  __shared__ float red[8];
  const int nbr = rows / 128, nbc = cols / 128, nm = w_pair ? 2 : 1;
  long long b = blockIdx.x;
  const int which = static_cast<int>(b % nm);
  b /= nm;
  const int bc = static_cast<int>(b % nbc);
  b /= nbc;
  const int br = static_cast<int>(b % nbr);
  const long long g = b / nbr;
  const int t = threadIdx.x, r = t >> 1, h = t & 1;
  const uint16_t* src = (which ? w_pair : w) +
                        (static_cast<size_t>(g) * rows + br * 128 + r) * cols + bc * 128 + h * 64;
  uint4 raw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) raw[k] = __ldg(reinterpret_cast<const uint4*>(src) + k);
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t u[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float sc = block_scale(amax);
  const size_t out_row = nm == 2 ? static_cast<size_t>(g) * 2 * rows + 2 * (br * 128 + r) + which
                                 : static_cast<size_t>(g) * rows + br * 128 + r;
  uint4* dst = reinterpret_cast<uint4*>(q + out_row * cols + bc * 128 + h * 64);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = raw[2 * k + (i >> 1)];
      const uint32_t u0 = (i & 1) ? a.z : a.x, u1 = (i & 1) ? a.w : a.y;
      const uint32_t lo = cvt_e4m3x2(__fdiv_rn(bf16_lo(u0), sc), __fdiv_rn(bf16_hi(u0), sc));
      const uint32_t hi = cvt_e4m3x2(__fdiv_rn(bf16_lo(u1), sc), __fdiv_rn(bf16_hi(u1), sc));
      o[i] = lo | (hi << 16);
    }
    dst[k] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (t == 0) {
    // rows of block scales padded to a multiple of 4 floats (16 bytes)
    const int pitch = (nm * nbc + 3) & ~3;
    s[(static_cast<size_t>(g) * nbr + br) * pitch + bc * nm + which] = sc;
  }
}

// q_perm[row_of[t, k]] = q[t] (16 bytes per thread per row); the thread that
// holds the first 16 bytes of a 128-column block also moves that block's
// scale.
__global__ void __launch_bounds__(256) gather_fp8_kernel(const uint4* __restrict__ q,
                                                         const float* __restrict__ s, int ld_in,
                                                         int T, int K, int chunks,
                                                         const int32_t* __restrict__ row_of,
                                                         uint4* __restrict__ q_perm,
                                                         float* __restrict__ s_perm, int ld_out) {
  const size_t n = static_cast<size_t>(T) * chunks;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / chunks, c = i % chunks;
    const uint4 v = __ldcs(q + i);
    const bool lead = (c & 7) == 0;
    const size_t j = c >> 3;
    const float sv = lead ? __ldg(s + j * ld_in + t) : 0.0f;
    const int32_t* rows = row_of + t * K;
    for (int k = 0; k < K; ++k) {
      const int32_t r = __ldg(rows + k);
      if (r < 0 || static_cast<size_t>(r) >= static_cast<size_t>(T) * K) continue;  // no row
      __stcs(q_perm + static_cast<size_t>(r) * chunks + c, v);
      if (lead) s_perm[j * ld_out + r] = sv;
    }
  }
}

int grid_for(long long work, int per_block, int cap_per_sm) {
  long long b = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sm_count()) * cap_per_sm;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_quantize_rows(const uint16_t* in, int rows, int cols, uint8_t* q, float* s,
                                 int ld_s, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const long long warps = static_cast<long long>(rows) * ((cols / 128 + kRowBlocks - 1) / kRowBlocks);
  quant_rows_kernel<<<grid_for(warps, 8, 16), 256, 0, st>>>(in, rows, cols, q, s, ld_s);
  return cudaGetLastError();
}

cudaError_t launch_quantize_blocks(const uint16_t* w, const uint16_t* w_pair, int groups, int rows,
                                   int cols, uint8_t* q, float* s, cudaStream_t st) {
  const long long blocks =
      static_cast<long long>(groups) * (rows / 128) * (cols / 128) * (w_pair ? 2 : 1);
  if (blocks == 0) return cudaSuccess;
  if (blocks >= (1ll << 31)) return cudaErrorInvalidValue;
  quant_blocks_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(w, w_pair, rows, cols, q, s);
  return cudaGetLastError();
}

cudaError_t launch_permute_fp8(const uint8_t* q, const float* s, int ld_in, int T, int K, int d,
                               const int32_t* row_of, uint8_t* q_perm, float* s_perm, int ld_out,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int chunks = d / 16;
  const long long n = static_cast<long long>(T) * chunks;
  gather_fp8_kernel<<<grid_for(n, 256, 8), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(q), s, ld_in, T, K, chunks, row_of,
      reinterpret_cast<uint4*>(q_perm), s_perm, ld_out);
  return cudaGetLastError();
}

}  // namespace moe
