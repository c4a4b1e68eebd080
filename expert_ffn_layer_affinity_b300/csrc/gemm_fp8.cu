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
//   P_j      = sum over the 128 k of k-block j of qa[tok, k] * qw[row, k]
//              (tensor core, into its own TMEM buffer)
//   acc     += P_j * (sa[j, tok] * sw[row block, j])   (fp32 FFMA, registers)
//
//   F8_SWIGLU  h[tok, i] = bf16(silu(acc_w1) * acc_w3)
//   F8_DOWN    y[tok, c] = bf16(acc)
//
// Layout: CTA pairs (cta_group::2).  TOKENS are on the MMA's M side (256 per
// pair tile, 128 in each CTA's TMEM lanes) and 256 WEIGHT rows on N (128
// staged in each CTA).  Each epilogue thread thus owns one token and 128
// weight columns: its activation scale is one number per k-block and the
// weight scales are at most two, so the promotion is a plain fused
// multiply-add per accumulator with no per-column scale traffic, and TMEM
// is read in the fast 32x32b shape.  (The other orientation, weights on M as
// in the bf16 kernel, needs a per-token-column scale for every accumulator;
// measured on B300, its shared-memory scale reads and the slower 16x256b
// TMEM shape cost about twice as much per k-block.)  Reading each k-block's
// fp32 partial out of TMEM is what bounds this kernel; ragged token tiles
// only waste tensor-core work, which is not the limit.
//
// For SwiGLU the weights are stored row-interleaved (row 2i = w1 row i, row
// 2i+1 = w3 row i), so the gate and up values of one output column are
// neighbouring accumulators of the same thread.  TMEM holds two 256-column
// partial buffers: the MMA fills one while the epilogue promotes the other,
// and each buffer goes back as soon as its last chunk is in registers.
// Scales arrive by TMA with the operands, into a ring of scale slots.
//
// CTA layout (384 threads, one CTA per SM, persistent):
//   warp 0       TMA producer (operands and scales of one k-block per stage)
//   warp 1       TMEM allocator; lane 0 of the even CTA issues the MMAs
//   warps 2, 3   idle
//   warps 4..11  epilogue: two warps per TMEM lane quarter (32 tokens), one
//                for weight columns 0..127, one for 128..255
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
constexpr int kA = 128 * BK, kB = 128 * BK;  // per CTA: 128 token rows, 128 weight rows
constexpr int kStageBytes = kA + kB;
constexpr int kBufCols = 256;
constexpr int kTmemCols = 2 * kBufCols;
// scale slot: activation scales of tokens x0 .. x0+263 (x0 = first token
// rounded down to a multiple of 4, two boxes of 128 and 136), then a box of
// 2 x 4 weight scales; each box starts on a 128-byte boundary
constexpr int kSaBox1 = 128, kSaBox2 = 136, kSwBox = 4, kSwRows = 2;
constexpr int kSlotW = 1152;       // byte offset of the weight-scale box
constexpr int kSlotBytes = 1280;
constexpr int kScaleTx = 4 * (kSaBox1 + kSaBox2 + kSwBox * kSwRows);
constexpr int kSlots = 8;          // producer runs at most 8 k-blocks ahead of the epilogue
// full[S], empty[S], accf[2], acce[2], drain, safull[8], saempty[8]
constexpr int kNumBars = 2 * kStages + 5 + 2 * kSlots;
constexpr int kSmem = 1024 + kStages * kStageBytes + kSlots * kSlotBytes + kNumBars * 8 + 16 +
                      2 * (kMaxGroups + 1) * 4;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kSlotBytes % 128 == 0 && kSlotW % 128 == 0 && 4 * (kSaBox1 + kSaBox2) <= kSlotW &&
                  kSlotW + 4 * kSwBox * kSwRows <= kSlotBytes,
              "scale boxes start on 128-byte boundaries and fit the slot");
static_assert(kSmem <= 227 * 1024, "shared memory");

enum Fp8Mode : int { F8_SWIGLU = 0, F8_DOWN = 1 };

struct Fp8Params {
  const int32_t* group_offsets;  // [G+1] device
  int G;
  int N;                 // output columns of a group (I for SwiGLU, d for the down projection)
  int R;                 // token rows
  int num_kb;            // reduction length / 128
  int w_rows_per_group;  // weight operand rows per group (2I interleaved, or d)
  void* out;             // bf16 [R, ldo]
  int ldo;
  int32_t* status;
};

struct Item {
  int g, n, m;
  long long row0;  // first token row of the tile
  int rows_tile;   // token rows of the tile that belong to the group
};

__device__ __forceinline__ Item item_of(int w, int NT, const int* mt_prefix, const int* row_start,
                                        int G) {
  Item it;
  decode_work(w, NT, mt_prefix, G, it.g, it.n, it.m);
  const int rows_g = row_start[it.g + 1] - row_start[it.g];
  const int tok0 = it.m * kTokTile;
  it.row0 = static_cast<long long>(row_start[it.g]) + tok0;
  it.rows_tile = (rows_g - tok0) < kTokTile ? rows_g - tok0 : kTokTile;
  return it;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmSa1,
                    const __grid_constant__ CUtensorMap tmSa2,
                    const __grid_constant__ CUtensorMap tmSw, const Fp8Params p) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* ring = smem_raw + (tiles - raw_addr) + S * kStageBytes;
  const uint32_t ring_addr = tiles + S * kStageBytes;
  uint8_t* meta = ring + kSlots * kSlotBytes;
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  auto safull_bar = [&](int k) { return bars + 8u * (2 * S + 5 + k); };
  auto saempty_bar = [&](int k) { return bars + 8u * (2 * S + 5 + kSlots + k); };
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
      tma_prefetch_desc(&tmSa1);
      tma_prefetch_desc(&tmSa2);
      tma_prefetch_desc(&tmSw);
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
      }
      for (int k = 0; k < kSlots; ++k) {
        mbar_init(safull_bar(k), 1);
        mbar_init(saempty_bar(k), kEpiWarps);   // every epilogue warp of this CTA
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

  // 256 weight rows per pair tile: 128 h columns (SwiGLU, w1/w3 interleaved)
  // or 256 output columns (down projection)
  const int NT = (MODE == F8_SWIGLU) ? p.N / 128 : (p.N + 255) / 256;
  const int total = mt_prefix[G] * NT;
  const int nkb = p.num_kb;

  if (warp < kEpiWarp0) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        const uint64_t pol_tok = l2_policy_evict_last();
        const uint64_t pol_w = l2_policy_evict_normal();
        uint32_t it = 0;
        bool ok = true;
        for (int w = unit_id; w < total && ok; w += n_units) {
          const Item t = item_of(w, NT, mt_prefix, row_start, G);
          const int tok_row = static_cast<int>(t.row0) + static_cast<int>(rank) * 128;
          const int w_row = t.g * p.w_rows_per_group + t.n * 256 + static_cast<int>(rank) * 128;
          const int sa_x = static_cast<int>(t.row0) & ~3;
          // weight-scale rows of the tile: SwiGLU one (w1 and w3 side by
          // side), down projection the tile's two 128-row blocks
          const int sw_row = (MODE == F8_SWIGLU) ? t.g * (p.N / 128) + t.n
                                                 : t.g * (p.N / 128) + t.n * 2;
          for (int j = 0; j < nkb; ++j, ++it) {
            const int s = static_cast<int>(it % S);
            const int k = static_cast<int>(it % kSlots);
            if (!mbar_wait(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag, p.status) ||
                !mbar_wait(saempty_bar(k), ((it / kSlots) & 1u) ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            // this CTA's scales of the k-block, into its own slot
            const uint32_t slot = ring_addr + static_cast<uint32_t>(k * kSlotBytes);
            mbar_arrive_expect_tx(safull_bar(k), kScaleTx);
            tma_load_2d(slot, &tmSa1, safull_bar(k), sa_x, j, pol_tok);
            tma_load_2d(slot + 4 * kSaBox1, &tmSa2, safull_bar(k), sa_x + kSaBox1, j, pol_tok);
            tma_load_2d(slot + kSlotW, &tmSw, safull_bar(k), (j * (MODE == F8_SWIGLU ? 2 : 1)) & ~3,
                        sw_row, pol_w);
            // operands: both CTAs' copies complete on the even CTA's barrier
            const uint32_t sa = tiles + s * kStageBytes;
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2u * kStageBytes);
            const uint32_t fb = mapa_shared(full_bar(s), 0);
            tma_load_2d_pair(sa, &tmX, fb, j * BK, tok_row, pol_tok);
            tma_load_2d_pair(sa + kA, &tmW, fb, j * BK, w_row, pol_w);
          }
        }
        if (!ok) {
          // let this CTA's own copies land before the CTA can exit
          const uint32_t first = it > kSlots ? it - kSlots : 0u;
          for (uint32_t j = first; j < it; ++j)
            wait_plain(safull_bar(static_cast<int>(j % kSlots)), (j / kSlots) & 1u, 200000000ull);
          if (rank == 0) {
            const uint32_t f2 = it > S ? it - S : 0u;
            for (uint32_t j = f2; j < it; ++j)
              wait_plain(full_bar(static_cast<int>(j % S)), (j / S) & 1u, 200000000ull);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      if (lane == 0 && rank == 0) {
        uint32_t it = 0;
        bool ok = true, issued = false;
        constexpr uint32_t idesc = umma_idesc_e4m3(256, 256);
        for (int w = unit_id; w < total && ok; w += n_units) {
          for (int j = 0; j < nkb; ++j, ++it) {
            const int b = static_cast<int>(it & 1u);
            if (!mbar_wait(acce_bar(b), ((it >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
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
            const uint64_t adesc = umma_sdesc_sw128(sa);        // tokens
            const uint64_t bdesc = umma_sdesc_sw128(sa + kA);   // weights
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
    const int q = warp & 3;           // this warp may read TMEM lanes 32q .. 32q+31
    const int half = ew >> 2;         // weight columns half*128 .. half*128+127
    const int tl = static_cast<int>(rank) * 128 + q * 32 + lane;  // token within the tile
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           static_cast<uint32_t>(half * 128);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);

    uint32_t u = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      const Item t = item_of(w, NT, mt_prefix, row_start, G);
      // tokens of this warp's lane quarter that belong to the tile
      const bool active = static_cast<int>(rank) * 128 + q * 32 < t.rows_tile;
      const bool mine = tl < t.rows_tile && t.row0 + tl < p.R;
      const int xoff = (static_cast<int>(t.row0) & 3) + tl;
      // acc[c][i]: weight columns half*128 + 32c + 2i and + 2i + 1
      float2 acc[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[c][i] = make_float2(0.0f, 0.0f);

      for (int j = 0; j < nkb; ++j, ++u) {
        const int k = static_cast<int>(u % kSlots);
        const int bsel = static_cast<int>(u & 1u);
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait(safull_bar(k), (u / kSlots) & 1u, abort_flag, p.status) &&
                            mbar_wait(accf_bar(bsel), (u >> 1) & 1u, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        // this token's scale products for the k-block: (gate, up) columns for
        // SwiGLU, the column half's block for the down projection
        const float* sl = reinterpret_cast<const float*>(ring + k * kSlotBytes);
        const float sa = mine ? sl[xoff] : 0.0f;
        float2 sc;
        if (MODE == F8_SWIGLU) {
          const float* sw = sl + kSlotW / 4 + ((2 * j) & 3);
          sc = make_float2(sa * sw[0], sa * sw[1]);
        } else {
          const float wv = sl[kSlotW / 4 + half * kSwBox + (j & 3)];
          sc = make_float2(sa * wv, sa * wv);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(saempty_bar(k));
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(acce_bar(bsel), 0));
        };
        auto promote = [&](float2 (&a)[16], const uint32_t (&r)[32]) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            a[i] = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                              sc, a[i]);
        };
        const uint32_t col0 = static_cast<uint32_t>(bsel * kBufCols);
        if (!active) {
          release();
        } else {
          // two register buffers: chunk c+1 loads while chunk c is promoted
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr + col0, r0);
          tmem_ld_wait();
          reg_fence32(r0);
          tmem_ld32(taddr + col0 + 32, r1);
          promote(acc[0], r0);
          tmem_ld_wait();
          reg_fence32(r1);
          tmem_ld32(taddr + col0 + 64, r0);
          promote(acc[1], r1);
          tmem_ld_wait();
          reg_fence32(r0);
          tmem_ld32(taddr + col0 + 96, r1);
          promote(acc[2], r0);
          tmem_ld_wait();
          reg_fence32(r1);
          release();
          promote(acc[3], r1);
        }
      }
      if (!ok) break;

      // ---- store this token's row segment
      if (mine) {
        __nv_bfloat16* orow = out + (t.row0 + tl) * p.ldo;
        if (MODE == F8_SWIGLU) {
          // columns 2i / 2i+1 of the tile are gate / up of h column
          // n*128 + half*64 + (32c + 2i) / 2
          uint4* dst = reinterpret_cast<uint4*>(orow + t.n * 128 + half * 64);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t hw[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float g0 = acc[c][i].x, u0 = acc[c][i].y;
              const float g1 = acc[c][i + 1].x, u1 = acc[c][i + 1].y;
              const float h0 = g0 * __frcp_rn(1.0f + __expf(-g0)) * u0;
              const float h1 = g1 * __frcp_rn(1.0f + __expf(-g1)) * u1;
              const __nv_bfloat162 pr = __floats2bfloat162_rn(h0, h1);
              hw[i / 2] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            dst[2 * c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dst[2 * c + 1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          }
        } else {
          const int col = t.n * 256 + half * 128;
          if (col < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(acc[c][i].x, acc[c][i].y);
                v[i] = *reinterpret_cast<const uint32_t*>(&pr);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[4 * c + e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
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

// fp32 rows [outer, inner] (inner % 4 == 0), box = box_inner x box_rows, no swizzle.
bool make_map_f32_rows(CUtensorMap* m, const float* ptr, uint64_t inner, uint64_t outer,
                       uint32_t box_inner, uint32_t box_rows = 1) {
  auto fn = gemm::encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_fp8(const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap& sa1,
                       const CUtensorMap& sa2, const CUtensorMap& sw, const Fp8Params& p,
                       int max_units, cudaStream_t s) {
  static DeviceOnce once;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = once_per_device(once, dev, []() {
    // The register split (setmaxnreg) must fit what the CTA is launched with,
    // or the increasing warps would wait for registers that never come.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fp8_gemm_kernel<MODE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < kSplitRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(fp8_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (err != cudaSuccess) return err;
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
  return cudaLaunchKernelEx(&cfg, fp8_gemm_kernel<MODE>, w, x, sa1, sa2, sw, p);
}

}  // namespace

int fp8_scale_pitch(int pairs, int cols) { return (pairs * (cols / 128) + 3) & ~3; }

cudaError_t launch_grouped_swiglu_fp8(const uint8_t* a_q, const float* a_s, int ld_as,
                                      const int32_t* offsets, int G, int R, int d, int I,
                                      const uint8_t* w13_q, const float* w13_s,
                                      const uint8_t* w2_q, const float* w2_s, uint16_t* h,
                                      uint8_t* h_q, float* h_s, uint16_t* y, int32_t* status,
                                      cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups || ld_as % 4) return cudaErrorInvalidValue;
  const int ld_h = (R + 3) & ~3;
  const int kb1 = d / BK, kb2 = I / BK;
  CUtensorMap tw13, tx, tw2, th, ta1, ta2, tsw13, th1, th2, tsw2;
  if (!make_map_u8(&tw13, w13_q, d, static_cast<uint64_t>(G) * 2 * I) ||
      !make_map_u8(&tx, a_q, d, R) ||
      !make_map_u8(&tw2, w2_q, I, static_cast<uint64_t>(G) * d) ||
      !make_map_u8(&th, h_q, I, R) ||
      !make_map_f32_rows(&ta1, a_s, ld_as, kb1, kSaBox1) ||
      !make_map_f32_rows(&ta2, a_s, ld_as, kb1, kSaBox2) ||
      !make_map_f32_rows(&tsw13, w13_s, fp8_scale_pitch(2, d), static_cast<uint64_t>(G) * (I / 128),
                         kSwBox, kSwRows) ||
      !make_map_f32_rows(&th1, h_s, ld_h, kb2, kSaBox1) ||
      !make_map_f32_rows(&th2, h_s, ld_h, kb2, kSaBox2) ||
      !make_map_f32_rows(&tsw2, w2_s, fp8_scale_pitch(1, I), static_cast<uint64_t>(G) * (d / 128),
                         kSwBox, kSwRows))
    return cudaErrorInvalidValue;
  // decode-sized groups (fewer than 64 rows on average): weights on M and the
  // few tokens on N waste less than 256-token tiles
  if (static_cast<long long>(R) < 64ll * G)
    return launch_grouped_swiglu_fp8_small(a_q, ld_as, offsets, G, R, d, I, w13_q, w2_q, h, h_q, h_s,
                                           y, status, ta1, ta2, tsw13, th1, th2, tsw2, s);
  Fp8Params p1{};
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = kb1;
  p1.w_rows_per_group = 2 * I;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  const int mt = (R + kTokTile - 1) / kTokTile + G;
  cudaError_t e = launch_fp8<F8_SWIGLU>(tw13, tx, ta1, ta2, tsw13, p1, mt * (I / 128), s);
  if (e != cudaSuccess) return e;
  e = launch_quantize_rows(h, R, I, h_q, h_s, ld_h, s);
  if (e != cudaSuccess) return e;
  Fp8Params p2 = p1;
  p2.N = d;
  p2.num_kb = kb2;
  p2.w_rows_per_group = d;
  p2.out = y;
  p2.ldo = d;
  return launch_fp8<F8_DOWN>(tw2, th, th1, th2, tsw2, p2, mt * ((d + 255) / 256), s);
}

}  // namespace moe
