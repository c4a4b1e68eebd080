// Dispatch on one GPU: group the (token, slot) rows by expert in a stable
// order and gather the activations into that order.  The pages' dispatch is
// a cross-node all-to-all ("Expert parallelism requires token dispatch and
// combine", weigao.cc "DeepSeek-V3 Technical Report：中英对照解读", §2.2 table);
// on a single device it becomes a counting sort plus a row gather.
//
// Kernels:
//   1. count   per tile of kPermuteTile flat entries, count each expert
//   2. scan    per expert, exclusive scan over tiles; exclusive scan over
//              experts gives expert_offsets; tile bases = offset + tile prefix
//   3. rank    per tile: rank inside a warp with __match_any_sync, prefix over
//              the tile's warps in shared memory -> row_of / tok_of
//   4. gather  per (token, 16-byte chunk): load x once, store it to the token's
//              K rows (128-bit loads and stores)
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kTile = kPermuteTile;
constexpr int kTileWarps = kTile / 32;

__global__ void __launch_bounds__(kTile) count_kernel(const int32_t* __restrict__ idx, int R, int E,
                                                      int32_t* __restrict__ tile_counts,
                                                      int32_t* status) {
  extern __shared__ int32_t cnt[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int p = blockIdx.x * kTile + threadIdx.x;
  if (p < R) {
    const int e = idx[p];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else if (status) {
      atomicOr(reinterpret_cast<unsigned int*>(status), MOE_DEV_BAD_INDEX);
    }
  }
  __syncthreads();
  int32_t* out = tile_counts + static_cast<size_t>(blockIdx.x) * E;
  for (int i = threadIdx.x; i < E; i += blockDim.x) out[i] = cnt[i];
}

// One block.  tile_counts [n_tiles, E] is turned in place into the first row
// of each (tile, expert) in x_perm.  The tiles of each expert are split into
// `segs` runs, one thread per (run, expert), so the column sums read many
// tiles at once instead of walking all of them one after the other.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ tile_counts, int n_tiles,
                                                    int E, int32_t* __restrict__ offsets) {
  extern __shared__ int32_t sm[];  // [segs][E] run sums -> run bases, then [E] expert bases
  __shared__ int32_t warp_sums[32];
  const int segs = blockDim.x / E;  // >= 1 (E <= 512 < 1024)
  const int len = (n_tiles + segs - 1) / segs;
  int32_t* run_sum = sm;
  int32_t* base = sm + segs * E;
  const int e = threadIdx.x % E, seg = threadIdx.x / E;
  const bool active = seg < segs;
  const int t0 = seg * len, t1 = min(n_tiles, t0 + len);
  if (active) {
    int32_t sum = 0;
    for (int t = t0; t < t1; t += 8) {
      int32_t v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = (t + j < t1) ? __ldcg(tile_counts + static_cast<size_t>(t + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += v[j];
    }
    run_sum[seg * E + e] = sum;
  }
  __syncthreads();
  // per expert: exclusive scan over its runs, and its total
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int32_t run = 0;
    for (int k = 0; k < segs; ++k) {
      const int32_t v = run_sum[k * E + x];
      run_sum[k * E + x] = run;
      run += v;
    }
    base[x] = run;
  }
  __syncthreads();
  // exclusive scan of the totals over experts in chunks of blockDim.x
  int32_t carry = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int b0 = 0; b0 < E; b0 += blockDim.x) {
    const int x = b0 + threadIdx.x;
    const int32_t v = (x < E) ? base[x] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t w = (lane < nw) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) warp_sums[lane] = w;
    }
    __syncthreads();
    incl += (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (x < E) {
      offsets[x] = incl - v;
      base[x] = incl - v;
    }
    const int32_t chunk_total = warp_sums[nw - 1];
    __syncthreads();
    carry += chunk_total;
  }
  if (threadIdx.x == 0) offsets[E] = carry;
  __syncthreads();
  // each (tile, expert) entry becomes its first row: expert base + run base
  // + the counts of the earlier tiles of the run
  if (active) {
    int32_t run = base[e] + run_sum[seg * E + e];
    for (int t = t0; t < t1; t += 8) {
      int32_t v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = (t + j < t1) ? __ldcg(tile_counts + static_cast<size_t>(t + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (t + j < t1) tile_counts[static_cast<size_t>(t + j) * E + e] = run;
        run += v[j];
      }
    }
  }
}

__global__ void __launch_bounds__(kTile) rank_kernel(const int32_t* __restrict__ idx, int R, int K,
                                                     int E, const int32_t* __restrict__ tile_base,
                                                     int32_t* __restrict__ row_of,
                                                     int32_t* __restrict__ tok_of) {
  extern __shared__ int32_t wcnt[];  // [kTileWarps, E]
  for (int i = threadIdx.x; i < kTileWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p = blockIdx.x * kTile + threadIdx.x;
  int e = -1;
  if (p < R) {
    e = idx[p];
    if (e < 0 || e >= E) e = -1;
  }
  const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(same);
  __syncthreads();
  const int32_t* base = tile_base + static_cast<size_t>(blockIdx.x) * E;
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int32_t run = base[x];
    for (int w = 0; w < kTileWarps; ++w) {
      const int32_t c = wcnt[w * E + x];
      wcnt[w * E + x] = run;
      run += c;
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int32_t row = wcnt[warp * E + e] + rank;
    row_of[p] = row;
    tok_of[row] = p / K;
  }
}

// x_perm[row_of[t, k]] = x[t], 16 bytes per thread per row.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, int T, int K,
                                                     int chunks, const int32_t* __restrict__ row_of,
                                                     uint4* __restrict__ x_perm) {
  const size_t n = static_cast<size_t>(T) * chunks;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / chunks, c = i % chunks;
    const uint4 v = __ldcs(x + i);
    const int32_t* rows = row_of + t * K;
    for (int k = 0; k < K; ++k) {
      const int32_t r = __ldg(rows + k);
      // entries with an out-of-range expert id (MOE_DEV_BAD_INDEX) have no row
      if (r >= 0 && static_cast<size_t>(r) < static_cast<size_t>(T) * K)
        __stcs(x_perm + static_cast<size_t>(r) * chunks + c, v);
    }
  }
}

}  // namespace

// Scratch of moe_permute_static: the per-tile expert counts of one call live
// in this fixed device array instead of caller-provided workspace.  Every GPU
// that loads the library holds it until the process exits.  All calls share
// it, so calls whose kernels overlap on the GPU race on it.
static __device__ __align__(256) int32_t g_permute_scratch[kPermuteStaticScratchInts];

cudaError_t permute_static_scratch(int32_t** ptr) {
  // In host code the symbol is only a host-side stand-in; the device address
  // is looked up once per device, with that device current (several host
  // threads making their first call at once look it up once).
  static DeviceOnce once;
  static int32_t* cached[kMaxDevices] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  e = once_per_device(once, dev, [&]() {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (r == cudaSuccess) cached[dev] = static_cast<int32_t*>(p);
    return r;
  });
  if (e != cudaSuccess) return e;
  *ptr = cached[dev];
  return cudaSuccess;
}

size_t permute_ws_bytes(int T, int K, int E) {
  const size_t R = static_cast<size_t>(T) * K;
  const size_t n_tiles = (R + kTile - 1) / kTile;
  return n_tiles * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* idx, int T, int K, int E, const uint16_t* x, int d,
                           int32_t* offsets, int32_t* row_of, int32_t* tok_of, uint16_t* x_perm,
                           int32_t* status, int32_t* tile_counts, cudaStream_t s) {
  const int R = T * K;
  if (R == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
  const int n_tiles = (R + kTile - 1) / kTile;
  cudaError_t err;
  count_kernel<<<n_tiles, kTile, E * sizeof(int32_t), s>>>(idx, R, E, tile_counts, status);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  scan_kernel<<<1, 1024, (1024 / E + 1) * E * sizeof(int32_t), s>>>(tile_counts, n_tiles, E,
                                                                    offsets);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t rank_smem = static_cast<size_t>(kTileWarps) * E * sizeof(int32_t);
  if (rank_smem > 48 * 1024) {
    static DeviceOnce once;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    err = once_per_device(once, dev, []() {
      return cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  32 * 512 * static_cast<int>(sizeof(int32_t)));
    });
    if (err != cudaSuccess) return err;
  }
  rank_kernel<<<n_tiles, kTile, rank_smem, s>>>(idx, R, K, E, tile_counts, row_of, tok_of);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (x != nullptr && x_perm != nullptr) {
    const int chunks = d / 8;
    const size_t n = static_cast<size_t>(T) * chunks;
    size_t blocks = (n + 255) / 256;
    const size_t cap = static_cast<size_t>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    gather_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(x), T, K, chunks, row_of, reinterpret_cast<uint4*>(x_perm));
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace moe
