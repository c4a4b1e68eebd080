// FP8 (E4M3) grouped expert GEMMs with fine-grained scaling on the
// fifth-generation tensor cores.
//
// Method (qwbw.cn essay on the report, the FP8 training passage;
// "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), section "6. FP8
// Training", rows "Fine-grained quantization is used" and "Accumulation
// precision still matters"): both GEMM operands are E4M3 with one fp32 scale
// per 1 x 128 activation tile and per 128 x 128 weight block, and the tensor
// core's partial sums are promoted to fp32 on the CUDA cores every Nc = 128
// reduction elements.  Here a 128-deep k-block is exactly one promotion
// interval and one scale block:
//
//   P_j      = sum over the 128 k of k-block j of qw[row, k] * qa[tok, k]
//              (tensor core, into its own TMEM buffer)
//   acc     += P_j * (sw[row block, j] * sa[j, tok])   (fp32 FFMA, registers)
//
//   F8_SWIGLU  h[tok, i] = bf16(silu(acc_w1) * acc_w3)
//   F8_DOWN    y[tok, c] = bf16(acc)
//
// Layout: CTA pairs (cta_group::2) with 256 weight rows on M (128 per CTA)
// and up to 256 tokens on N, as in the bf16 kernel.  For SwiGLU the weights
// are stored row-interleaved (row 2i = w1 row i, row 2i+1 = w3 row i), so
// the gate and up values of one output column sit in neighbouring TMEM lanes
// and meet with one shuffle.  TMEM holds two 256-column partial buffers: the
// MMA fills one while the epilogue promotes the other.
//
// CTA layout (384 threads, one CTA per SM, persistent):
//   warp 0       TMA producer (one 128-deep k-block of both operands per stage)
//   warp 1       TMEM allocator; lane 0 of the even CTA issues the MMAs
//   warps 2, 3   idle
//   warps 4..11  epilogue: two warps per TMEM lane quarter, each owning 128 of
//                the 256 token columns (128 fp32 accumulators per thread); all
//                eight stage the per-column scale products of the next k-block
// Registers: the first warpgroup gives its registers up (setmaxnreg.dec to
// kCtrlRegs) and the two epilogue warpgroups take them (setmaxnreg.inc to
// kEpiRegs).  The host checks, before every launch, that the split fits the
// registers the CTA is launched with.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using gemm::decode_work;
using gemm::kMaxGroups;
using gemm::store_block_transposed;
using gemm::tile_n;
using gemm::wait_plain;

constexpr int BK = 128;      // E4M3 values (bytes) per k-block = promotion interval
constexpr int UMMA_K = 32;   // reduction depth of one kind::f8f6f4 instruction
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;  // first epilogue warp (warpgroups 1 and 2)
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kCtrlRegs = 56, kEpiRegs = 224;
// registers the split needs at launch, per CTA
constexpr int kSplitRegs = 128 * kCtrlRegs + 32 * kEpiWarps * kEpiRegs;
constexpr int kStages = 6;
constexpr int kTokTile = 256;
constexpr int kA = 128 * BK, kB = 128 * BK;  // per CTA: 128 weight rows, up to 128 token rows
constexpr int kStageBytes = kA + kB;
constexpr int kBufCols = 256;
constexpr int kTmemCols = 2 * kBufCols;
constexpr int kXposeBytes = kEpiWarps * 32 * 80;
constexpr int kScaleFloats = 2 * 2 * 256;  // [buffer][w1 / w3 variant][token column]
// full[S], empty[S], accf[2], acce[2], drain, sfull[2]
constexpr int kNumBars = 2 * kStages + 7;
constexpr int kSmem = 1024 + kStages * kStageBytes + kXposeBytes + kScaleFloats * 4 +
                      kNumBars * 8 + 16 + 2 * (kMaxGroups + 1) * 4;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");

enum Fp8Mode : int { F8_SWIGLU = 0, F8_DOWN = 1 };

struct Fp8Params {
  const int32_t* group_offsets;  // [G+1] device
  int G;
  int N;                 // output columns of a group (I for SwiGLU, d for the down projection)
  int R;                 // token rows
  int num_kb;            // reduction length / 128
  int w_rows_per_group;  // weight operand rows per group (2I interleaved, or d)
  const float* a_scale;  // [num_kb][ld_as]
  int ld_as;
  const float* w_scale;  // SwiGLU [G][I/128][num_kb][2]; down [G][d/128][num_kb]
  void* out;             // bf16 [R, ldo]
  int ldo;
  int32_t* status;
};

struct Item {
  int g, n, m;
  long long row0;  // first token row of the tile
  int rows_tile;   // token rows of the tile that belong to the group
  int n_eff;       // MMA N (rows_tile rounded up to 32)
};

__device__ __forceinline__ Item item_of(int w, int NT, const int* mt_prefix, const int* row_start,
                                        int G) {
  Item it;
  decode_work(w, NT, mt_prefix, G, it.g, it.n, it.m);
  const int rows_g = row_start[it.g + 1] - row_start[it.g];
  const int tok0 = it.m * kTokTile;
  it.row0 = static_cast<long long>(row_start[it.g]) + tok0;
  it.rows_tile = (rows_g - tok0) < kTokTile ? rows_g - tok0 : kTokTile;
  it.n_eff = tile_n(rows_g - tok0, kTokTile);
  return it;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const Fp8Params p) {
  constexpr int kColTile = (MODE == F8_SWIGLU) ? 128 : 256;  // output columns per pair
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* xpose = smem_raw + (tiles - raw_addr) + S * kStageBytes;
  float* sc = reinterpret_cast<float*>(xpose + kXposeBytes);
  uint8_t* meta = reinterpret_cast<uint8_t*>(sc + kScaleFloats);
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  auto sfull_bar = [&](int b) { return bars + 8u * (2 * S + 5 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* mt_prefix = reinterpret_cast<int*>(meta + 8 * kNumBars + 16);
  int* row_start = mt_prefix + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const uint32_t rank = cluster_ctarank();
  const int unit_id = static_cast<int>(blockIdx.x >> 1);
  const int n_units = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    gemm::build_tile_prefix(G, kTokTile, lane, [&](int g) { return p.group_offsets[g]; },
                            mt_prefix, row_start);
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(accf_bar(b), 1);
        mbar_init(acce_bar(b), 2 * kEpiWarps);  // every epilogue warp of both CTAs
        mbar_init(sfull_bar(b), kEpiWarps);     // every epilogue warp of this CTA
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
  cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NT = (p.N + kColTile - 1) / kColTile;
  const int total = mt_prefix[G] * NT;
  const int nkb = p.num_kb;

  if (warp < kEpiWarp0) {
    setmaxnreg_dec<kCtrlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_tok = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      for (int w = unit_id; w < total && ok; w += n_units) {
        const Item t = item_of(w, NT, mt_prefix, row_start, G);
        const int tok_row = static_cast<int>(t.row0) + static_cast<int>(rank) * (t.n_eff / 2);
        const int w_row = t.g * p.w_rows_per_group + t.n * 256 + static_cast<int>(rank) * 128;
        for (int j = 0; j < nkb; ++j, ++it) {
          const int s = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = tiles + s * kStageBytes;
          // both CTAs' copies complete on the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2u * kStageBytes);
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          tma_load_2d_pair(sa, &tmW, fb, j * BK, w_row, pol_w);
          tma_load_2d_pair(sa + kA, &tmX, fb, j * BK, tok_row, pol_tok);
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
      for (int w = unit_id; w < total && ok; w += n_units) {
        const Item t = item_of(w, NT, mt_prefix, row_start, G);
        const uint32_t idesc = umma_idesc_e4m3(256, t.n_eff);
        for (int j = 0; j < nkb; ++j, ++it, ++unit) {
          const int b = static_cast<int>(unit & 1u);
          if (!mbar_wait(acce_bar(b), ((unit >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(full_bar(s), (it / S) & 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * kStageBytes;
          const uint64_t adesc = umma_sdesc_sw128(sa);
          const uint64_t bdesc = umma_sdesc_sw128(sa + kA);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kBufCols);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_f8_pair(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, idesc, k > 0 ? 1u : 0u);
          issued = true;
          umma_commit_pair_mc(empty_bar(s), 0x3);
          umma_commit_pair_mc(accf_bar(b), 0x3);
        }
      }
      if (!ok && issued) {
        umma_commit_pair_mc(drain_bar, 0x1);
        wait_plain(drain_bar, 0u, 200000000ull);
      }
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<kEpiRegs>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;  // 0..7
    const int q = warp & 3;         // this warp may read TMEM lanes 32q .. 32q+31
    const int half = ew >> 2;       // token columns half*128 .. half*128+127
    const int col_thr = ew * 32 + lane;  // the token column whose scales this thread stages
    uint8_t* xp = xpose + ew * 32 * 80;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);

    // scale of (item, k-block j) for column col_thr: activation scale and the
    // weight scale(s) of this CTA's rows
    auto fetch = [&](const Item& t, int j, float& sa, float& s0, float& s1) {
      sa = 0.0f;
      if (col_thr < t.rows_tile && t.row0 + col_thr < p.R)
        sa = __ldg(p.a_scale + static_cast<long long>(j) * p.ld_as + t.row0 + col_thr);
      if (MODE == F8_SWIGLU) {
        const float2 wv = __ldg(reinterpret_cast<const float2*>(p.w_scale) +
                                static_cast<long long>(t.g * (p.N / 128) + t.n) * p.num_kb + j);
        s0 = wv.x;
        s1 = wv.y;
      } else {
        const int blk = t.n * 2 + static_cast<int>(rank);
        s0 = (blk * 128 < p.N)
                 ? __ldg(p.w_scale + static_cast<long long>(t.g * (p.N / 128) + blk) * p.num_kb + j)
                 : 0.0f;
        s1 = 0.0f;
      }
    };

    uint32_t unit = 0;
    bool ok = true;
    float nsa = 0.0f, ns0 = 0.0f, ns1 = 0.0f;
    if (unit_id < total) fetch(item_of(unit_id, NT, mt_prefix, row_start, G), 0, nsa, ns0, ns1);
    for (int w = unit_id; w < total && ok; w += n_units) {
      const Item t = item_of(w, NT, mt_prefix, row_start, G);
      const bool has_next = w + n_units < total;
      const Item nx = has_next ? item_of(w + n_units, NT, mt_prefix, row_start, G) : t;
      int nc = t.n_eff - half * 128;
      nc = nc < 0 ? 0 : (nc > 128 ? 128 : nc);
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;

      for (int j = 0; j < nkb; ++j, ++unit) {
        const int bsel = static_cast<int>(unit & 1u);
        const uint32_t par = (unit >> 1) & 1u;
        float* scb = sc + bsel * 512;
        scb[col_thr] = nsa * ns0;
        if (MODE == F8_SWIGLU) scb[256 + col_thr] = nsa * ns1;
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull_bar(bsel));
        if (j + 1 < nkb) fetch(t, j + 1, nsa, ns0, ns1);
        else if (has_next) fetch(nx, 0, nsa, ns0, ns1);
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(sfull_bar(bsel), par, abort_flag, p.status));
        if (!ok) break;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(accf_bar(bsel), par, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const float* srow = scb + ((MODE == F8_SWIGLU && (lane & 1)) ? 256 : 0) + half * 128;
        const uint32_t taddr =
            tmem_base + lane_base + static_cast<uint32_t>(bsel * kBufCols + half * 128);
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          if (c < nc) {
            uint32_t v[32];
            tmem_ld32(taddr + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 s4 = *reinterpret_cast<const float4*>(srow + c + i);
              acc[c + i] = fmaf(__uint_as_float(v[i]), s4.x, acc[c + i]);
              acc[c + i + 1] = fmaf(__uint_as_float(v[i + 1]), s4.y, acc[c + i + 1]);
              acc[c + i + 2] = fmaf(__uint_as_float(v[i + 2]), s4.z, acc[c + i + 2]);
              acc[c + i + 3] = fmaf(__uint_as_float(v[i + 3]), s4.w, acc[c + i + 3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(bsel), 0));
      }
      if (!ok) break;

      // ---- store this thread's 128 token columns
      if (MODE == F8_SWIGLU) {
        const int ibase = t.n * 128 + static_cast<int>(rank) * 64 + q * 16;  // first h column
        const bool odd = (lane & 1) != 0;
        const int pcol = lane >> 1;
        __nv_bfloat16* x = reinterpret_cast<__nv_bfloat16*>(xp);
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          if (c < nc) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float o = __shfl_xor_sync(0xFFFFFFFFu, acc[c + i], 1);
              const float a = odd ? o : acc[c + i];
              const float u = odd ? acc[c + i] : o;
              h[i] = a * __frcp_rn(1.0f + __expf(-a)) * u;
            }
            // stage [32 tokens][16 h columns]: even lanes tokens 0..15, odd
            // lanes tokens 16..31 (rows an odd distance apart: no bank clash)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int row = odd ? 16 + (i ^ 1) : i;
              x[row * 16 + pcol] = __float2bfloat16_rn(odd ? h[16 + (i ^ 1)] : h[i]);
            }
            __syncwarp();
            const int t0 = half * 128 + c;
            int valid = t.rows_tile - t0;
            valid = valid > 32 ? 32 : valid;
            const long long last = t.row0 + t0 + valid;
            if (last > p.R) valid -= static_cast<int>(last - p.R);
            if (lane < valid && ibase < p.N) {
              const uint4* src = reinterpret_cast<const uint4*>(xp + lane * 32);
              uint4* dst = reinterpret_cast<uint4*>(out + (t.row0 + t0 + lane) * p.ldo + ibase);
              dst[0] = src[0];
              dst[1] = src[1];
            }
            __syncwarp();
          }
        }
      } else {
        const int colbase = t.n * 256 + static_cast<int>(rank) * 128 + q * 32;
        if (colbase < p.N) {
#pragma unroll
          for (int c = 0; c < 128; c += 32) {
            if (c < nc) {
              uint32_t v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(acc[c + i]);
              const int t0 = half * 128 + c;
              int valid = t.rows_tile - t0;
              valid = valid > 32 ? 32 : valid;
              const long long last = t.row0 + t0 + valid;
              if (last > p.R) valid -= static_cast<int>(last - p.R);
              store_block_transposed(v, xp, lane, out, t.row0 + t0, valid, p.ldo, colbase);
            }
          }
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA frees TMEM or exits while its peer still uses it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  return gemm::make_map_sw128(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ptr, inner, outer, 128);
}

template <int MODE>
cudaError_t launch_fp8(const CUtensorMap& w, const CUtensorMap& x, const Fp8Params& p,
                       int max_units, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    // The register split (setmaxnreg) must fit what the CTA is launched with,
    // or the increasing warps would wait for registers that never come.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fp8_gemm_kernel<MODE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < kSplitRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(fp8_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  int units = sm_count() / 2;
  if (max_units < units) units = max_units;
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
  return cudaLaunchKernelEx(&cfg, fp8_gemm_kernel<MODE>, w, x, p);
}

}  // namespace

cudaError_t launch_grouped_swiglu_fp8(const uint8_t* a_q, const float* a_s, int ld_as,
                                      const int32_t* offsets, int G, int R, int d, int I,
                                      const uint8_t* w13_q, const float* w13_s,
                                      const uint8_t* w2_q, const float* w2_s, uint16_t* h,
                                      uint8_t* h_q, float* h_s, uint16_t* y, int32_t* status,
                                      cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  CUtensorMap tw13, tx, tw2, th;
  if (!make_map_u8(&tw13, w13_q, d, static_cast<uint64_t>(G) * 2 * I) ||
      !make_map_u8(&tx, a_q, d, R) ||
      !make_map_u8(&tw2, w2_q, I, static_cast<uint64_t>(G) * d) ||
      !make_map_u8(&th, h_q, I, R))
    return cudaErrorInvalidValue;
  Fp8Params p1{};
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = d / BK;
  p1.w_rows_per_group = 2 * I;
  p1.a_scale = a_s;
  p1.ld_as = ld_as;
  p1.w_scale = w13_s;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  const int mt = (R + kTokTile - 1) / kTokTile + G;
  cudaError_t e = launch_fp8<F8_SWIGLU>(tw13, tx, p1, mt * (I / 128), s);
  if (e != cudaSuccess) return e;
  e = launch_quantize_rows(h, R, I, h_q, h_s, R, s);
  if (e != cudaSuccess) return e;
  Fp8Params p2 = p1;
  p2.N = d;
  p2.num_kb = I / BK;
  p2.w_rows_per_group = d;
  p2.a_scale = h_s;
  p2.ld_as = R;
  p2.w_scale = w2_s;
  p2.out = y;
  p2.ldo = d;
  return launch_fp8<F8_DOWN>(tw2, th, p2, mt * ((d + 255) / 256), s);
}

}  // namespace moe
