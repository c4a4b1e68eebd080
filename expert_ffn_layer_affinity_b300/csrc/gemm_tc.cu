// Grouped GEMMs on the fifth-generation tensor cores (tcgen05 + TMEM), fed
// by TMA.  One persistent kernel template serves the three dense
// contractions of the layer:
//
//   EPI_SWIGLU   h[r, :] = silu(a[r] . w1[g]^T) * (a[r] . w3[g]^T)  -> bf16
//                (expert up-projections; SwiGLU applied in the epilogue)
//   EPI_BF16     y[r, :] = h[r] . w2[g]^T                            -> bf16
//                (expert down-projection)
//   EPI_SIGMOID  s[t, e] = sigmoid(x[t] . w_r[e] + o[e])             -> fp32
//                (router; w_r given as an exact 3-term bf16 split laid
//                 out along K, so A's K coordinate wraps every d columns)
//
// Experts as "shared + fine-grained routed FFNs" follow weigao.cc
// "DeepSeek-V3 Technical Report：中英对照解读", §2 table rows "DeepSeekMoE" and
// "Shared experts and routed experts"; the routed groups are the rows that
// the dispatch step assigned to each expert.
//
// CTA layout (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: fills a STAGES-deep shared-memory ring
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma (M=128, N=BN, K=16)
//   warps 2..5  epilogue: tcgen05.ld from TMEM, activation, global stores
// Two TMEM accumulators (2 x BN columns) let the epilogue of one tile run
// while the next tile accumulates.  Work items are (group, n-tile, m-tile)
// triples, group-major and m-tile fastest so that the CTAs working on the
// same weight tile run side by side and share it through L2.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 512;

enum Epi : int { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_SIGMOID = 2 };

struct GemmParams {
  const int32_t* group_offsets;  // [G+1] device; nullptr = one group of rows [0, dense_rows)
  int dense_rows;
  int G;
  int N;                 // output columns of a group
  int R;                 // rows of A and of the output (stores beyond are dropped)
  int num_kb;            // reduction length / BK
  int a_k_wrap_kb;       // A's k-block = kb % a_k_wrap_kb
  int b_rows_per_group;  // rows of B's 2-D view that belong to one group
  void* out;
  int ldo;               // output row stride in elements
  const float* col_offset;  // EPI_SIGMOID: per-column logit offset or nullptr
  int32_t* status;
};

constexpr int tmem_cols_for(int n) {
  int c = 32;
  while (c < n) c <<= 1;
  return c;
}

template <int BN, int EPI, int STAGES>
struct Cfg {
  static constexpr int kBnOut = (EPI == EPI_SWIGLU) ? BN / 2 : BN;
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = tmem_cols_for(2 * BN);
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kSmem = 1024 + STAGES * kStageBytes + kNumBars * 8 + 16 +
                               2 * (kMaxGroups + 1) * 4;
  static constexpr uint32_t kIdesc = umma_idesc_bf16(BM, BN);
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=128");
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ int group_offset(const GemmParams& p, int g) {
  return p.group_offsets ? p.group_offsets[g] : (g == 0 ? 0 : p.dense_rows);
}

__device__ __forceinline__ void decode_work(int w, int NT, const int* mt_prefix, int G, int& g,
                                            int& n, int& m) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mt_prefix[mid] * NT <= w) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int mt = mt_prefix[g + 1] - mt_prefix[g];
  const int local = w - mt_prefix[g] * NT;
  n = local / mt;
  m = local - n * mt;
}

__device__ __forceinline__ bool wait_plain(uint32_t bar, uint32_t parity, unsigned long long ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > ns) return false;
  return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BN, int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const GemmParams p) {
  using C = Cfg<BN, EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* meta = smem_raw + (tiles - raw_addr) + STAGES * C::kStageBytes;
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* mt_prefix = reinterpret_cast<int*>(meta + 8 * C::kNumBars + 16);
  int* row_start = mt_prefix + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;

  if (warp == 0) {
    // per-group m-tile prefix and row starts
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      int mt = 0;
      if (g < G) {
        const int a = group_offset(p, g), b = group_offset(p, g + 1);
        const int rows = b > a ? b - a : 0;
        mt = (rows + BM - 1) / BM;
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
      row_start[G] = group_offset(p, G);
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmB2);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(accf_bar(b), 1);
        mbar_init(acce_bar(b), 128);
      }
      mbar_init(drain_bar, 1);
      *abort_flag = 0;
      fence_mbar_init();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NT = (p.N + C::kBnOut - 1) / C::kBnOut;
  const int total = mt_prefix[G] * NT;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        int g, n, m;
        decode_work(w, NT, mt_prefix, G, g, n, m);
        const int a_row = row_start[g] + m * BM;
        const int b_row = g * p.b_rows_per_group + n * C::kBnOut;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = static_cast<int>(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + s * C::kStageBytes;
          const uint32_t sb = sa + C::kABytes;
          mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
          tma_load_2d(sa, &tmA, full_bar(s), (kb % p.a_k_wrap_kb) * BK, a_row, pol_a);
          if (EPI == EPI_SWIGLU) {
            tma_load_2d(sb, &tmB, full_bar(s), kb * BK, b_row, pol_b);
            tma_load_2d(sb + C::kBBytes / 2, &tmB2, full_bar(s), kb * BK, b_row, pol_b);
          } else {
            tma_load_2d(sb, &tmB, full_bar(s), kb * BK, b_row, pol_b);
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        const uint32_t first = it > STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_plain(full_bar(static_cast<int>(j % STAGES)), (j / STAGES) & 1u, 200000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tile = 0;
      bool ok = true;
      bool issued = false;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++tile) {
        const int ab = static_cast<int>(tile & 1u);
        const uint32_t aph = (tile >> 1) & 1u;
        if (!mbar_wait(acce_bar(ab), aph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * BN);
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = static_cast<int>(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(full_bar(s), ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * C::kStageBytes;
          const uint64_t adesc = umma_sdesc_sw128(sa);
          const uint64_t bdesc = umma_sdesc_sw128(sa + C::kABytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_bf16(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, C::kIdesc,
                      (kb > 0 || k > 0) ? 1u : 0u);
          issued = true;
          umma_commit(empty_bar(s));
        }
        if (!ok) break;
        umma_commit(accf_bar(ab));
      }
      if (!ok && issued) {
        umma_commit(drain_bar);
        wait_plain(drain_bar, 0u, 200000000ull);
      }
    }
    __syncwarp();
  } else {
    // epilogue warps 2..5; warp w may read TMEM lanes 32*(w%4) .. +31
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    uint32_t tile = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++tile) {
      int g, n, m;
      decode_work(w, NT, mt_prefix, G, g, n, m);
      const int ab = static_cast<int>(tile & 1u);
      const uint32_t aph = (tile >> 1) & 1u;
      bool ok = mbar_wait(accf_bar(ab), aph, abort_flag, p.status);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      const int rows_g = row_start[g + 1] - row_start[g];
      const int local_row = m * BM + r_in_tile;
      const long long orow = static_cast<long long>(row_start[g]) + local_row;
      const bool row_ok = local_row < rows_g && orow < p.R;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(ab * BN);
      if (EPI == EPI_SWIGLU) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
        for (int c = 0; c < C::kBnOut; c += 32) {
          uint32_t ra[32], rc[32];
          tmem_ld32(taddr + c, ra);
          tmem_ld32(taddr + C::kBnOut + c, rc);
          tmem_ld_wait();
          const int col = n * C::kBnOut + c;
          if (row_ok && col < p.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a0 = __uint_as_float(ra[2 * i]), a1 = __uint_as_float(ra[2 * i + 1]);
              const float c0 = __uint_as_float(rc[2 * i]), c1 = __uint_as_float(rc[2 * i + 1]);
              const float h0 = a0 * __frcp_rn(1.0f + __expf(-a0)) * c0;
              const float h1 = a1 * __frcp_rn(1.0f + __expf(-a1)) * c1;
              pk[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(out + orow * p.ldo + col);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else if (EPI == EPI_BF16) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t ra[32];
          tmem_ld32(taddr + c, ra);
          tmem_ld_wait();
          const int col = n * BN + c;
          if (row_ok && col < p.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(out + orow * p.ldo + col);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        float* out = reinterpret_cast<float*>(p.out);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t ra[32];
          tmem_ld32(taddr + c, ra);
          tmem_ld_wait();
          const int col = n * BN + c;
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int cc = col + i;
              if (cc < p.N) {
                float u = __uint_as_float(ra[i]);
                if (p.col_offset) u = u + p.col_offset[cc];
                out[orow * p.ldo + cc] = 1.0f / (1.0f + expf(-u));
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acce_bar(ab));
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor [outer, inner] (inner contiguous), box = 64 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int EPI, int STAGES>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                        const GemmParams& p, int max_works, cudaStream_t s) {
  using C = Cfg<BN, EPI, STAGES>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, EPI, STAGES>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  int grid = sm_count();
  if (max_works < grid) grid = max_works;
  if (grid < 1) grid = 1;
  gemm_kernel<BN, EPI, STAGES><<<grid, kThreads, C::kSmem, s>>>(a, b, b2, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_swiglu(const uint16_t* a, const int32_t* offsets, int G, int R, int d,
                                  int I, const uint16_t* w1, const uint16_t* w3,
                                  const uint16_t* w2, uint16_t* h, uint16_t* y, int32_t* status,
                                  cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  CUtensorMap ta, tb1, tb3, th, tb2;
  if (!make_map(&ta, a, d, R, BM) || !make_map(&tb1, w1, d, static_cast<uint64_t>(G) * I, 128) ||
      !make_map(&tb3, w3, d, static_cast<uint64_t>(G) * I, 128) || !make_map(&th, h, I, R, BM) ||
      !make_map(&tb2, w2, I, static_cast<uint64_t>(G) * d, 256))
    return cudaErrorInvalidValue;
  const int m_tiles_max = (R + BM - 1) / BM + G;
  GemmParams p1{};
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = d / BK;
  p1.a_k_wrap_kb = d / BK;
  p1.b_rows_per_group = I;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  cudaError_t e = launch_gemm<256, EPI_SWIGLU, 4>(ta, tb1, tb3, p1, m_tiles_max * ((I + 127) / 128), s);
  if (e != cudaSuccess) return e;
  GemmParams p2 = p1;
  p2.N = d;
  p2.num_kb = I / BK;
  p2.a_k_wrap_kb = I / BK;
  p2.b_rows_per_group = d;
  p2.out = y;
  p2.ldo = d;
  return launch_gemm<256, EPI_BF16, 4>(th, tb2, tb2, p2, m_tiles_max * ((d + 255) / 256), s);
}

cudaError_t launch_router_gemm(const uint16_t* x, const uint16_t* w_split, const float* offset,
                               int T, int d, int E, float* scores, int32_t* status,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int BNr = E <= 32 ? 32 : (E <= 64 ? 64 : 128);
  CUtensorMap ta, tb;
  if (!make_map(&ta, x, d, T, BM) || !make_map(&tb, w_split, 3ull * d, E, BNr))
    return cudaErrorInvalidValue;
  GemmParams p{};
  p.group_offsets = nullptr;
  p.dense_rows = T;
  p.G = 1;
  p.N = E;
  p.R = T;
  p.num_kb = 3 * d / BK;
  p.a_k_wrap_kb = d / BK;
  p.b_rows_per_group = 0;
  p.out = scores;
  p.ldo = E;
  p.col_offset = offset;
  p.status = status;
  const int works = ((T + BM - 1) / BM) * ((E + BNr - 1) / BNr);
  if (BNr == 32) return launch_gemm<32, EPI_SIGMOID, 8>(ta, tb, tb, p, works, s);
  if (BNr == 64) return launch_gemm<64, EPI_SIGMOID, 8>(ta, tb, tb, p, works, s);
  return launch_gemm<128, EPI_SIGMOID, 6>(ta, tb, tb, p, works, s);
}

}  // namespace moe
