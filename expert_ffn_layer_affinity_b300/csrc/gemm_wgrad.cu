// Grouped weight-gradient GEMM of the expert FFN backward on the tensor cores:
//
//   out[g][m][n] = sum over the rows r of group g of A[r][m] * B[r][n]
//
// e.g. dW2[e] = dY_e^T h_e, [dW1; dW3][e] = [da | dc]_e^T x_e (the weight
// gradients of y = W2 (silu(W1 v) * (W3 v)); expert FFNs as in
// "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), §2 row
// "DeepSeekMoE").  The reduction runs over each group's tokens, so both
// operands come TRANSPOSED, K-major along the token axis: at [M, ld] and
// bt [N, ld], where group g owns columns koff[g] .. koff[g+1] (its rows,
// zero-padded to a multiple of 64; see moe_transpose_grouped).
//
// CTA pairs (tcgen05 .cta_group::2): 256 rows of M (128 per CTA) x 256 rows
// of N (128 staged in each CTA) per item, the group's k-blocks accumulated in
// one of two 256-column TMEM buffers; the epilogue of one item overlaps the
// next item's MMAs.  Each epilogue thread owns one output row and writes its
// 256 fp32 columns as contiguous 16-byte stores.  A group with no rows writes
// zeros.
//
// CTA layout (192 threads, one CTA per SM, persistent): warp 0 TMA producer,
// warp 1 TMEM allocator + MMA issuer (even CTA), warps 2..5 epilogue.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cstdint>

#include "internal.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using gemm::wait_plain;

constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;
constexpr int kStages = 6;
constexpr int kBox = 128 * BK * 2;  // 16 KB: 128 rows x 64 bf16
constexpr int kStageBytes = 2 * kBox;
constexpr int kBufCols = 256;
constexpr int kTmemCols = 2 * kBufCols;
constexpr int kNumBars = 2 * kStages + 5;
constexpr int kSmem = 1024 + kStages * kStageBytes + kNumBars * 8 + 16;
static_assert(kSmem <= 227 * 1024, "shared memory");

struct WgradParams {
  const int32_t* koff;  // [G+1] device, padded column offsets (multiples of 64)
  int G, M, N;
  float* out;  // [G, M, N]
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const WgradParams p) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* meta = smem_raw + (tiles - raw_addr) + S * kStageBytes;
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int unit_id = static_cast<int>(blockIdx.x >> 1);
  const int n_units = static_cast<int>(gridDim.x >> 1);
  const int MT = (p.M + 255) / 256, NT = (p.N + 255) / 256;
  const int total = p.G * MT * NT;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(accf_bar(b), 1);
        mbar_init(acce_bar(b), 2 * 4);  // every epilogue warp of both CTAs
      }
      mbar_init(drain_bar, 1);
      *abort_flag = 0;
      fence_mbar_init();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // item w -> group g, M tile mt, N tile nt (group-major)
  auto decode = [&](int w, int& g, int& mt, int& nt) {
    g = w / (MT * NT);
    const int r = w - g * MT * NT;
    mt = r / NT;
    nt = r - mt * NT;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, mt, nt;
        decode(w, g, mt, nt);
        const int k0 = p.koff[g], nkb = (p.koff[g + 1] - k0) / BK;
        const int arow = mt * 256 + static_cast<int>(rank) * 128;
        const int brow = nt * 256 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + s * kStageBytes;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2u * kStageBytes);
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          tma_load_2d_pair(sa, &tmA, fb, k0 + kb * BK, arow, pol);
          tma_load_2d_pair(sa + kBox, &tmB, fb, k0 + kb * BK, brow, pol);
        }
      }
      if (!ok && rank == 0) {
        const uint32_t first = it > S ? it - S : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_plain(full_bar(static_cast<int>(j % S)), (j / S) & 1u, 200000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, unit = 0;
      bool ok = true, issued = false;
      constexpr uint32_t idesc = umma_idesc_bf16(256, 256);
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, mt, nt;
        decode(w, g, mt, nt);
        const int nkb = (p.koff[g + 1] - p.koff[g]) / BK;
        if (nkb == 0) continue;  // no rows: the epilogue writes zeros
        const int b = static_cast<int>(unit & 1u);
        if (!mbar_wait(acce_bar(b), ((unit >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kBufCols);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(full_bar(s), (it / S) & 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * kStageBytes;
          const uint64_t adesc = umma_sdesc_sw128(sa);
          const uint64_t bdesc = umma_sdesc_sw128(sa + kBox);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_bf16_pair(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, idesc,
                           (kb > 0 || k > 0) ? 1u : 0u);
          issued = true;
          umma_commit_pair_mc(empty_bar(s), 0x3);
        }
        if (!ok) break;
        umma_commit_pair_mc(accf_bar(b), 0x3);
        ++unit;
      }
      if (!ok && issued) {
        umma_commit_pair_mc(drain_bar, 0x1);
        wait_plain(drain_bar, 0u, 200000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t taddr0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t unit = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      int g, mt, nt;
      decode(w, g, mt, nt);
      const int nkb = (p.koff[g + 1] - p.koff[g]) / BK;
      const int m = mt * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
      const int n0 = nt * 256;
      float* orow = p.out + (static_cast<size_t>(g) * p.M + m) * p.N + n0;
      const bool row_ok = m < p.M;
      if (nkb == 0) {
        if (row_ok)
          for (int c = 0; c < 256 && n0 + c < p.N; c += 4)
            *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int b = static_cast<int>(unit & 1u);
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(accf_bar(b), (unit >> 1) & 1u, abort_flag, p.status));
      if (!ok) break;
      ++unit;
      tc_fence_after();
      const uint32_t taddr = taddr0 + static_cast<uint32_t>(b * kBufCols);
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + c, v);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            if (n0 + c + i < p.N)
              *reinterpret_cast<float4*>(orow + c + i) =
                  make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                              __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

cudaError_t launch_grouped_wgrad(const uint16_t* at, const uint16_t* bt, long long ld,
                                 const int32_t* koff, int G, int M, int N, float* out,
                                 int32_t* status, cudaStream_t s) {
  if (G == 0 || M == 0 || N == 0) return cudaSuccess;
  CUtensorMap ta, tb;
  if (!gemm::make_map_sw128(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, at, ld, M, 128) ||
      !gemm::make_map_sw128(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, bt, ld, N, 128))
    return cudaErrorInvalidValue;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  WgradParams p{};
  p.koff = koff;
  p.G = G;
  p.M = M;
  p.N = N;
  p.out = out;
  p.status = status;
  const long long items = static_cast<long long>(G) * ((M + 255) / 256) * ((N + 255) / 256);
  int units = sm_count() / 2;
  if (items < units) units = static_cast<int>(items);
  if (units < 1) units = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wgrad_kernel, ta, tb, p);
}

}  // namespace moe
