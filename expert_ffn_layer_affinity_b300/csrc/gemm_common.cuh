// Pieces shared by the grouped-GEMM kernels (bf16 in gemm_tc.cu, FP8 in
// gemm_fp8.cu): the work-list order, tile sizing, the transposing store and
// the tensor-map encoder.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <atomic>
#include <cstdint>

#include "ptx.cuh"

namespace moe {
namespace gemm {

constexpr int kMaxGroups = 512;

// Work item w -> (group g, token tile m, weight tile n), given the per-group
// prefix of token tiles and NT weight tiles per token tile.
//
// Token tile major, weight tile fastest: the pairs that run side by side
// cover every weight tile of a token tile, and the other token tiles of the
// same group follow NT positions later (still running, sharing weights
// through L2).  Full and ragged token tiles thus spread over all pairs
// instead of repeating on the same ones (with 74 pairs and token-tile-fastest
// order, some pairs drew only full tiles and others only ragged ones: 3.53 ->
// 3.42 ms for GEMM1 at the V3 shape).  Claiming items from an atomic counter
// instead of a fixed stride measured no better.
__device__ __forceinline__ void decode_work(int w, int NT, const int* mt_prefix, int G, int& g,
                                            int& n, int& m) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mt_prefix[mid] * NT <= w) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int local = w - mt_prefix[g] * NT;
  m = local / NT;
  n = local - m * NT;
}

__device__ __forceinline__ bool wait_plain(uint32_t bar, uint32_t parity, unsigned long long ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > ns) return false;
  return true;
}

// Tokens of this tile the MMA must cover, rounded up to 32 (16 rows staged
// in each CTA of the pair).
__device__ __forceinline__ int tile_n(int rows_left, int tok_tile) {
  const int n = rows_left < tok_tile ? rows_left : tok_tile;
  return (n + 31) & ~31;
}

// Writes a 32 (weight row = output column) x 32 (token) block, held one
// output column per lane as 32 fp32 values along tokens, as 32 token rows of
// 64 bytes (bf16), or of its first cols_valid columns (a multiple of 8).
// `xp` is this warp's 32 x 80-byte staging area.
__device__ __forceinline__ void store_block_transposed(const uint32_t (&v)[32], uint8_t* xp,
                                                       int lane, __nv_bfloat16* out, long long row0,
                                                       int rows_valid, int ldo, int col,
                                                       int cols_valid = 32) {
  __nv_bfloat16* x = reinterpret_cast<__nv_bfloat16*>(xp);
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j * 40 + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
  __syncwarp();
  if (lane < rows_valid) {
    const uint4* src = reinterpret_cast<const uint4*>(xp + lane * 80);
    uint4* dst = reinterpret_cast<uint4*>(out + (row0 + lane) * ldo + col);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (8 * k < cols_valid) dst[k] = src[k];
  }
  __syncwarp();
}

// Per-group token-tile prefix and row starts, computed by one warp into
// shared memory (mt_prefix[G+1], row_start[G+1]).
template <typename OffsetFn>
__device__ __forceinline__ void build_tile_prefix(int G, int tok_tile, int lane, OffsetFn offset,
                                                  int* mt_prefix, int* row_start) {
  int carry = 0;
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int g = g0 + lane;
    int mt = 0;
    if (g < G) {
      const int a = offset(g), b = offset(g + 1);
      const int rows = b > a ? b - a : 0;
      mt = (rows + tok_tile - 1) / tok_tile;
      row_start[g] = a;
    }
    int incl = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (g < G) mt_prefix[g] = carry + incl - mt;
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) {
    mt_prefix[G] = carry;
    row_start[G] = offset(G);
  }
}

// ------------------------------------------------------------------ host side
// The driver's tensor-map encoder, looked up on first use (and again after a
// failed lookup); an atomic, so threads making their first calls together
// are safe.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// 2-D tensor [outer, inner] (inner contiguous) of `elem_bytes`-byte elements,
// box = (128 bytes of inner) x box_rows, 128-byte swizzle, zero fill outside.
inline bool make_map_sw128(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes,
                           const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, type, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace gemm
}  // namespace moe
