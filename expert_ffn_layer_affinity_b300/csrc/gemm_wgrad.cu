// Grouped weight-gradient GEMM of the expert FFN backward on the tensor cores:
//
//   out[g][m][n] = sum over the rows r of group g of A[r][m] * B[r][n]
//
// e.g. dW2[e] = dY_e^T h_e and [dW1; dW3][e] = [da | dc]_e^T x_e, the weight
// gradients of y = W2 (silu(W1 v) * (W3 v)) (expert FFNs as in
// "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), §2 row
// "DeepSeekMoE").  The reduction runs over each group's tokens in dispatch
// order, so A [R, M] and B [R, N] are read as they are: both operands are
// MN-major for the MMA (64-element rows of M or N, consecutive tokens 128 B
// apart), with no transposed copies.
//
// CTA pairs (tcgen05 .cta_group::2), persistent: a work item is (group, 256
// rows of M, 256 columns of N), each CTA staging its 128 rows of M and its
// 128 columns of N for every k-block (32 of the group's tokens; 12 stages,
// finer than 6 stages of 64 tokens, measured 5-9 % faster), the even CTA
// issuing the MMAs.  A group's last k-block may run into the next group's
// tokens: its copies complete on a barrier of each CTA's own, each CTA's
// fixer warp zeroes those rows in its shared memory, and the MMA waits for
// both fixers.  Accumulators live in two 256-column TMEM buffers, so an
// item's epilogue overlaps the next item's MMAs.  The epilogue writes fp32
// 32 x 32 blocks through swizzled shared memory with TMA stores (3-D map
// [G][M][N]: a block clips at its own group's M and at N).  A group with no
// tokens gets zeros.
//
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer (even CTA), 2 tail
// fixer, 3..6 epilogue (TMEM lanes 32 (warp % 4) ..).
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

constexpr int BK = 32;                       // tokens per k-block
constexpr int TM = 256;                      // M rows per item (128 per CTA)
constexpr int TN = 256;                      // N columns per item (128 staged per CTA)
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (3 + kEpiWarps) * 32;
constexpr int kStages = 12;
constexpr int kChunk = 64 * BK * 2;              // 4 KB: 64 MN elements x 32 tokens
constexpr int kABytes = (TM / 2 / 64) * kChunk;  // 8 KB per CTA and k-block
constexpr int kBBytes = (TN / 2 / 64) * kChunk;  // 8 KB per CTA and k-block
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kOutBuf = 32 * 32 * 4;         // one 32 x 32 fp32 block
constexpr int kOutBytes = kEpiWarps * 2 * kOutBuf;  // 2 buffers per epilogue warp
constexpr int kTmemCols = 2 * TN;
constexpr int kNumBars = 4 * kStages + 5;
constexpr int kSmem = 1024 + kStages * kStageBytes + kOutBytes + kNumBars * 8 + 16;
static_assert(kSmem <= 227 * 1024, "shared memory");

// kind::f16 instruction descriptor, bf16 in, fp32 accumulate, both operands
// MN-major (the transpose bits 15 and 16); M = 256 over the pair.
constexpr uint32_t kIdesc = umma_idesc_bf16(TM, TN) | (1u << 15) | (1u << 16);

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct WgradParams {
  const int32_t* offsets;  // [G+1] device: rows of group g are offsets[g] .. offsets[g+1]
  int G, M, N;
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmO, const WgradParams p) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* tiles_ptr = smem_raw + (tiles - raw_addr);
  const uint32_t obuf = tiles + S * kStageBytes;
  uint8_t* obuf_ptr = tiles_ptr + S * kStageBytes;
  uint8_t* meta = obuf_ptr + kOutBytes;
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto fixed_bar = [&](int s) { return bars + 8u * (2 * S + s); };
  auto tfull_bar = [&](int s) { return bars + 8u * (3 * S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (4 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (4 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (4 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int unit_id = static_cast<int>(blockIdx.x >> 1);
  const int n_units = static_cast<int>(gridDim.x >> 1);
  const int MT = (p.M + TM - 1) / TM, NT = (p.N + TN - 1) / TN;
  const int total = p.G * MT * NT;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmO);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
        mbar_init(fixed_bar(s), 2);  // both CTAs' fixers
        mbar_init(tfull_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(accf_bar(b), 1);
        mbar_init(acce_bar(b), 2 * kEpiWarps);  // every epilogue warp of both CTAs
      }
      mbar_init(drain_bar, 1);
      *abort_flag = 0;
      fence_mbar_init();
      fence_async_smem();
    }
    __syncwarp();
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // item w -> group g, M tile mt, N tile nt (group-major, so a group's
  // operands stay in L2 while its items run)
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
      uint32_t it = 0, full_ph = 0, tail_ph = 0;
      // the newest fill of each stage that this CTA can wait for: the even
      // CTA counts both CTAs' whole k-blocks, each CTA its own ragged ones
      uint32_t last_bar[S], last_par[S], pending = 0;
      bool ok = true;
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, mt, nt;
        decode(w, g, mt, nt);
        const int r0 = p.offsets[g], rows = p.offsets[g + 1] - r0;
        const int nkb = (rows + BK - 1) / BK;
        const int ax = mt * TM + static_cast<int>(rank) * (TM / 2);
        const int bx = nt * TN + static_cast<int>(rank) * (TN / 2);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + s * kStageBytes, sb = sa + kABytes;
          const int y = r0 + kb * BK;
          if (rows - kb * BK < BK) {
            // ragged last k-block: this CTA's own barrier, then its fixer
            last_bar[s] = tfull_bar(s);
            last_par[s] = (tail_ph >> s) & 1u;
            tail_ph ^= 1u << s;
            pending |= 1u << s;
            mbar_arrive_expect_tx(tfull_bar(s), kStageBytes);
#pragma unroll
            for (int c = 0; c < TM / 2 / 64; ++c)
              tma_load_2d(sa + c * kChunk, &tmA, tfull_bar(s), ax + c * 64, y, pol);
#pragma unroll
            for (int c = 0; c < TN / 2 / 64; ++c)
              tma_load_2d(sb + c * kChunk, &tmB, tfull_bar(s), bx + c * 64, y, pol);
          } else {
            // whole k-block: both CTAs' copies complete on the even CTA's barrier
            if (rank == 0) {
              last_bar[s] = full_bar(s);
              last_par[s] = (full_ph >> s) & 1u;
              pending |= 1u << s;
              mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
            } else {
              pending &= ~(1u << s);
            }
            full_ph ^= 1u << s;
            const uint32_t fb = mapa_shared(full_bar(s), 0);
#pragma unroll
            for (int c = 0; c < TM / 2 / 64; ++c)
              tma_load_2d_pair(sa + c * kChunk, &tmA, fb, ax + c * 64, y, pol);
#pragma unroll
            for (int c = 0; c < TN / 2 / 64; ++c)
              tma_load_2d_pair(sb + c * kChunk, &tmB, fb, bx + c * 64, y, pol);
          }
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (int j = 0; j < S; ++j)
          if ((pending >> j) & 1u) wait_plain(last_bar[j], last_par[j], 200000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      // per-stage phase bits: fills through full_bar (whole k-blocks) and
      // through tfull_bar -> fixers -> fixed_bar (ragged last k-blocks)
      uint32_t unit = 0, full_phase = 0, fix_phase = 0, it = 0;
      bool ok = true, issued = false;
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, mt, nt;
        decode(w, g, mt, nt);
        const int rows = p.offsets[g + 1] - p.offsets[g];
        const int nkb = (rows + BK - 1) / BK;
        if (nkb == 0) continue;  // no tokens: the epilogue writes zeros
        const int b = static_cast<int>(unit & 1u);
        if (!mbar_wait(acce_bar(b), ((unit >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * TN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          const int valid = rows - kb * BK;
          bool got;
          if (valid < BK) {
            got = mbar_wait(fixed_bar(s), (fix_phase >> s) & 1u, abort_flag, p.status);
            fix_phase ^= 1u << s;
          } else {
            got = mbar_wait(full_bar(s), (full_phase >> s) & 1u, abort_flag, p.status);
            full_phase ^= 1u << s;
          }
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * kStageBytes, sb = sa + kABytes;
          const int ksteps = valid < BK ? (valid + UMMA_K - 1) / UMMA_K : BK / UMMA_K;
          for (int k = 0; k < ksteps; ++k)
            umma_bf16_pair(d_tmem, umma_sdesc_mn_sw128(sa + k * UMMA_K * 128, kChunk),
                           umma_sdesc_mn_sw128(sb + k * UMMA_K * 128, kChunk), kIdesc,
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
  } else if (warp == 2) {
    // ----------------------------------------------------------- tail fixer
    // A group's last k-block: rows valid .. BK-1 hold the next group's tokens
    // (or the fill past the tensor); zero them in every chunk of both
    // operands in this CTA.  A token row is one 128-byte line of a chunk
    // whatever the swizzle, so whole lines are cleared.
    uint32_t it = 0, tail_phase = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      int g, mt, nt;
      decode(w, g, mt, nt);
      const int rows = p.offsets[g + 1] - p.offsets[g];
      const int nkb = (rows + BK - 1) / BK;
      if (nkb == 0) continue;
      it += static_cast<uint32_t>(nkb - 1);
      const int valid = rows - (nkb - 1) * BK;
      if (valid < BK) {
        const int s = static_cast<int>(it % S);
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait(tfull_bar(s), (tail_phase >> s) & 1u, abort_flag, p.status));
        tail_phase ^= 1u << s;
        if (!ok) break;
        uint8_t* stage = tiles_ptr + s * kStageBytes;
        const int lines = BK - valid;  // per chunk
        const int n16 = (kStageBytes / kChunk) * lines * 8;
        for (int i = lane; i < n16; i += 32) {
          const int c = i / (lines * 8), rem = i - c * lines * 8;
          const int line = valid + rem / 8, part = rem & 7;
          *reinterpret_cast<uint4*>(stage + c * kChunk + line * 128 + part * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(fixed_bar(s), 0));
      }
      ++it;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t taddr0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const int e = warp - 3;
    uint8_t* my_buf = obuf_ptr + e * 2 * kOutBuf;
    const uint32_t my_buf_addr = obuf + e * 2 * kOutBuf;
    uint32_t unit = 0, slot = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      int g, mt, nt;
      decode(w, g, mt, nt);
      const int rows = p.offsets[g + 1] - p.offsets[g];
      const int m0 = mt * TM + static_cast<int>(rank) * (TM / 2) + q * 32;
      const bool zero = rows == 0;
      int b = 0;
      if (!zero) {
        b = static_cast<int>(unit & 1u);
        // a long wait: poll with short sleeps, leaving issue slots to the
        // producer and the MMA issuer on the shared sub-partitions
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait_nap(accf_bar(b), (unit >> 1) & 1u, abort_flag, p.status));
        if (!ok) break;
        ++unit;
        tc_fence_after();
      }
      const bool store = m0 < p.M;  // rows past M: release the buffer only
      const uint32_t taddr = taddr0 + static_cast<uint32_t>(b * TN);
      constexpr int kBlocks = TN / 32;
      uint32_t v[32], vn[32];
      if (!zero) {
        tmem_ld32(taddr, v);
        tmem_ld_wait();
        reg_fence32(v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
#pragma unroll 1
      for (int c = 0; c < kBlocks; ++c) {
        // next block's TMEM read in flight while this one is written out
        const bool more = !zero && c + 1 < kBlocks;
        if (more) tmem_ld32(taddr + (c + 1) * 32, vn);
        const int n = nt * TN + c * 32;
        if (store && n < p.N) {
          // the store issued from this buffer two blocks ago must have read it
          if (lane == 0) bulk_wait_read1();
          __syncwarp();
          uint8_t* buf = my_buf + (slot & 1u) * kOutBuf;
          // row `lane`, 16-byte unit j at position j ^ (lane % 8) (128-byte swizzle)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmO, my_buf_addr + (slot & 1u) * kOutBuf, n, m0, g);
            bulk_commit();
          }
          ++slot;
        }
        if (more) {
          tmem_ld_wait();
          reg_fence32(vn);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = vn[j];
        }
      }
      if (!zero) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(acce_bar(b), 0));
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA frees TMEM or exits while its peer still uses it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

bool make_out_map(CUtensorMap* m, float* out, int G, int M, int N) {
  auto fn = gemm::encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                        static_cast<cuuint64_t>(G)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(M) * N * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_wgrad(const uint16_t* a, const uint16_t* b, const int32_t* offsets,
                                 int G, int R, int M, int N, float* out, int32_t* status,
                                 cudaStream_t s) {
  if (G == 0 || M == 0 || N == 0) return cudaSuccess;
  CUtensorMap ta, tb, to;
  // A [R, M] and B [R, N] with 64 x BK boxes (64 MN elements x BK tokens);
  // R == 0 still needs valid maps, so the outer extent is at least 1
  const uint64_t rows = R > 0 ? static_cast<uint64_t>(R) : 1u;
  if (!gemm::make_map_sw128(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a, M, rows, BK) ||
      !gemm::make_map_sw128(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b, N, rows, BK) ||
      !make_out_map(&to, out, G, M, N))
    return cudaErrorInvalidValue;
  static DeviceOnce once;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = once_per_device(once, dev, []() {
    return cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (err != cudaSuccess) return err;
  WgradParams p{};
  p.offsets = offsets;
  p.G = G;
  p.M = M;
  p.N = N;
  p.status = status;
  const long long items = static_cast<long long>(G) * ((M + TM - 1) / TM) * ((N + TN - 1) / TN);
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
  return cudaLaunchKernelEx(&cfg, wgrad_kernel, ta, tb, to, p);
}

}  // namespace moe
