// FP8 (E4M3) grouped expert GEMMs for SMALL token groups (decode-sized
// batches): the same method and scale layouts as gemm_fp8.cu (promotion of
// each 128-deep k-block's fp32 partial with activation x weight scales), in
// the other orientation -- 256 WEIGHT rows on the MMA's M side and the
// group's tokens on N, rounded up to 32 -- so a group of a few tokens costs
// an N=32 MMA and a 32-column promotion instead of a 256-token tile.
//
// Per k-block the producer fetches the tile's activation scales and this
// CTA's weight scale(s) by TMA into a ring of scale slots; a stager warp turns
// them into per-token-column products (activation x weight scale) four
// k-blocks ahead.  The epilogue reads TMEM in the 16x256b shape (4 rows x 32
// token columns per thread), so one 8-byte product load serves 8
// accumulators.  For SwiGLU the weight rows are interleaved (2i = w1 row i,
// 2i+1 = w3 row i); gate and up meet by a shuffle between lanes 4 apart.
//
// CTA layout (384 threads, one CTA per SM, persistent):
//   warp 0       TMA producer (operands and scales of one k-block per stage)
//   warp 1       TMEM allocator; lane 0 of the even CTA issues the MMAs
//   warp 2       scale stager
//   warp 3       idle
//   warps 4..11  epilogue: two warps per TMEM lane quarter, each owning 128 of
//                the 256 token columns
// Registers: setmaxnreg moves registers from the first warpgroup to the two
// epilogue warpgroups; the host checks the split against the launch.
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
// scale slot: activation scales of tokens x0 .. x0+263 (x0 = first token
// rounded down to a multiple of 4, two boxes of 128 and 136), then a box of
// 4 weight scales; each box starts on a 128-byte boundary
constexpr int kSaBox1 = 128, kSaBox2 = 136, kSwBox = 4;
constexpr int kSlotW = 1152;       // byte offset of the weight-scale box
constexpr int kSlotBytes = 1280;
// the weight-scale box carries two rows (the layout gemm_fp8.cu fetches);
// this orientation uses the first
constexpr int kScaleTx = 4 * (kSaBox1 + kSaBox2 + 2 * kSwBox);
constexpr int kSlots = 8;          // producer runs at most 8 k-blocks ahead of the epilogue
constexpr int kProdBufs = 4;       // scale-product buffers (see the epilogue)
// [w1 variant: 256 token columns][8 floats pad][w3 variant: 256 columns]: the
// pad puts the two variants' same columns in different banks
constexpr int kVar1 = 264;
constexpr int kProdFloats = kVar1 + 256;
// full[S], empty[S], accf[2], acce[2], drain, sfull[4], safull[8], saempty[8], pempty[4]
constexpr int kNumBars = 2 * kStages + 5 + 2 * kProdBufs + 2 * kSlots;
constexpr int kSmem = 1024 + kStages * kStageBytes + kSlots * kSlotBytes +
                      kProdBufs * kProdFloats * 4 + kNumBars * 8 + 16 + 2 * (kMaxGroups + 1) * 4;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(kSlotBytes % 128 == 0 && kSlotW % 128 == 0 && 4 * (kSaBox1 + kSaBox2) <= kSlotW,
              "scale boxes start on 128-byte boundaries");
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
    fp8_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmSa1,
                    const __grid_constant__ CUtensorMap tmSa2,
                    const __grid_constant__ CUtensorMap tmSw, const Fp8Params p) {
  constexpr int kColTile = (MODE == F8_SWIGLU) ? 128 : 256;  // output columns per pair
  constexpr int kNm = (MODE == F8_SWIGLU) ? 2 : 1;             // weight scales per k-block
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* ring = smem_raw + (tiles - raw_addr) + S * kStageBytes;
  const uint32_t ring_addr = tiles + S * kStageBytes;
  float* prod = reinterpret_cast<float*>(ring + kSlots * kSlotBytes);
  uint8_t* meta = reinterpret_cast<uint8_t*>(prod + kProdBufs * kProdFloats);
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  auto sfull_bar = [&](int b) { return bars + 8u * (2 * S + 5 + b); };
  auto safull_bar = [&](int k) { return bars + 8u * (2 * S + 5 + kProdBufs + k); };
  auto saempty_bar = [&](int k) { return bars + 8u * (2 * S + 5 + kProdBufs + kSlots + k); };
  auto pempty_bar = [&](int b) { return bars + 8u * (2 * S + 5 + kProdBufs + 2 * kSlots + b); };
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
      for (int b = 0; b < kProdBufs; ++b) {
        mbar_init(sfull_bar(b), 1);            // the scale stager
        mbar_init(pempty_bar(b), kEpiWarps);   // every epilogue warp of this CTA
      }
      for (int k = 0; k < kSlots; ++k) {
        mbar_init(safull_bar(k), 1);
        mbar_init(saempty_bar(k), 1);          // the scale stager
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
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        const uint64_t pol_tok = l2_policy_evict_last();
        const uint64_t pol_w = l2_policy_evict_normal();
        uint32_t it = 0;
        bool ok = true;
        for (int w = unit_id; w < total && ok; w += n_units) {
          const Item t = item_of(w, NT, mt_prefix, row_start, G);
          const int tok_row = static_cast<int>(t.row0) + static_cast<int>(rank) * (t.n_eff / 2);
          const int w_row = t.g * p.w_rows_per_group + t.n * 256 + static_cast<int>(rank) * 128;
          const int sa_x = static_cast<int>(t.row0) & ~3;
          const int sw_row = (MODE == F8_SWIGLU) ? t.g * (p.N / 128) + t.n
                                                 : t.g * (p.N / 128) + t.n * 2 + static_cast<int>(rank);
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
            tma_load_2d(slot + kSlotW, &tmSw, safull_bar(k), (j * kNm) & ~3, sw_row, pol_w);
            // operands: both CTAs' copies complete on the even CTA's barrier
            const uint32_t sa = tiles + s * kStageBytes;
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2u * kStageBytes);
            const uint32_t fb = mapa_shared(full_bar(s), 0);
            tma_load_2d_pair(sa, &tmW, fb, j * BK, w_row, pol_w);
            tma_load_2d_pair(sa + kA, &tmX, fb, j * BK, tok_row, pol_tok);
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
        for (int w = unit_id; w < total && ok; w += n_units) {
          const Item t = item_of(w, NT, mt_prefix, row_start, G);
          const uint32_t idesc = umma_idesc_e4m3(256, t.n_eff);
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
    } else if (warp == 2) {
      // ------------------------------------------------------ scale stager
      // Per k-block: the activation scale of each token column times this
      // CTA's weight scale(s), into product buffer v % 4 (8 columns per lane).
      uint32_t v = 0;
      bool ok = true;
      for (int w = unit_id; w < total && ok; w += n_units) {
        const Item t = item_of(w, NT, mt_prefix, row_start, G);
        const int x0 = static_cast<int>(t.row0) & 3;
        for (int j = 0; j < nkb; ++j, ++v) {
          const int k = static_cast<int>(v % kSlots);
          const int b = static_cast<int>(v % kProdBufs);
          ok = __all_sync(0xFFFFFFFFu,
                          mbar_wait(safull_bar(k), (v / kSlots) & 1u, abort_flag, p.status) &&
                              mbar_wait(pempty_bar(b), ((v / kProdBufs) & 1u) ^ 1u, abort_flag,
                                        p.status));
          if (!ok) break;
          const float* sl = reinterpret_cast<const float*>(ring + k * kSlotBytes);
          const float* sw = sl + kSlotW / 4 + ((j * kNm) & 3);
          const float w0 = sw[0], w1 = (MODE == F8_SWIGLU) ? sw[1] : 0.0f;
          float* pb = prod + b * kProdFloats;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int col = lane + 32 * i;
            const float a = col < t.rows_tile ? sl[x0 + col] : 0.0f;
            pb[col] = a * w0;
            if (MODE == F8_SWIGLU) pb[kVar1 + col] = a * w1;
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(sfull_bar(b));
            mbar_arrive(saempty_bar(k));
          }
        }
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kEpiRegs>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;      // 0..7
    const int q = warp & 3;               // this warp may read TMEM lanes 32q .. 32q+31
    const int half = ew >> 2;             // token columns half*128 .. half*128+127
    const int tq = lane & 3, tr = lane >> 2;
    const uint32_t taddr_lo = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t taddr_hi = tmem_base + (static_cast<uint32_t>(q * 32 + 16) << 16);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);

    // TMEM reads of chunk c (32 token columns) of the buffer at column col0
    auto tld = [&](uint32_t col0, int c, uint32_t (&lo)[16], uint32_t (&hi)[16]) {
      tmem_ld16x256b_x4(taddr_lo + col0 + 32 * c, lo);
      tmem_ld16x256b_x4(taddr_hi + col0 + 32 * c, hi);
    };

    uint32_t u = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      const Item t = item_of(w, NT, mt_prefix, row_start, G);
      int nc = t.n_eff - half * 128;
      nc = nc < 0 ? 0 : (nc > 128 ? 128 : nc);
      const int nch = nc / 32;
      // acc[c][m][k]: chunk c (32 columns), repeat m (8 columns), row slot k
      // (rows tr, tr+8, tr+16, tr+24 of this warp's lane quarter); .x/.y =
      // columns half*128 + 32c + 8m + 2tq + {0, 1}
      float2 acc[4][4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[c][m][k] = make_float2(0.0f, 0.0f);

      for (int j = 0; j < nkb; ++j, ++u) {
        const int pbi = static_cast<int>(u % kProdBufs);
        const int bsel = static_cast<int>(u & 1u);
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait(sfull_bar(pbi), (u / kProdBufs) & 1u, abort_flag, p.status) &&
                            mbar_wait(accf_bar(bsel), (u >> 1) & 1u, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const float* srow = prod + pbi * kProdFloats + ((MODE == F8_SWIGLU && (tr & 1)) ? kVar1 : 0) +
                            half * 128 + 2 * tq;
        const uint32_t col0 = static_cast<uint32_t>(bsel * kBufCols + half * 128);
        // hand the TMEM buffer back as soon as its last chunk is in registers
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(acce_bar(bsel), 0));
        };
        // acc += P * (activation scale x weight scale), one chunk
        auto promote = [&](float2 (&a)[4][4], const uint32_t (&lo)[16], const uint32_t (&hi)[16],
                           int c) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float2 sc2 = *reinterpret_cast<const float2*>(srow + 32 * c + 8 * m);
            a[m][0] = __ffma2_rn(make_float2(__uint_as_float(lo[4 * m]), __uint_as_float(lo[4 * m + 1])),
                                 sc2, a[m][0]);
            a[m][1] = __ffma2_rn(make_float2(__uint_as_float(lo[4 * m + 2]),
                                             __uint_as_float(lo[4 * m + 3])), sc2, a[m][1]);
            a[m][2] = __ffma2_rn(make_float2(__uint_as_float(hi[4 * m]), __uint_as_float(hi[4 * m + 1])),
                                 sc2, a[m][2]);
            a[m][3] = __ffma2_rn(make_float2(__uint_as_float(hi[4 * m + 2]),
                                             __uint_as_float(hi[4 * m + 3])), sc2, a[m][3]);
          }
        };
        // two register buffers: chunk c+1 loads while chunk c is promoted
        uint32_t lo0[16], hi0[16], lo1[16], hi1[16];
        if (nch > 0) tld(col0, 0, lo0, hi0);
        tmem_ld_wait();
        reg_fence16(lo0);
        reg_fence16(hi0);
        if (nch > 1) tld(col0, 1, lo1, hi1);
        else release();
        if (nch > 0) promote(acc[0], lo0, hi0, 0);
        if (nch > 1) {
          tmem_ld_wait();
          reg_fence16(lo1);
          reg_fence16(hi1);
          if (nch > 2) tld(col0, 2, lo0, hi0);
          else release();
          promote(acc[1], lo1, hi1, 1);
        }
        if (nch > 2) {
          tmem_ld_wait();
          reg_fence16(lo0);
          reg_fence16(hi0);
          if (nch > 3) tld(col0, 3, lo1, hi1);
          else release();
          promote(acc[2], lo0, hi0, 2);
        }
        if (nch > 3) {
          tmem_ld_wait();
          reg_fence16(lo1);
          reg_fence16(hi1);
          release();
          promote(acc[3], lo1, hi1, 3);
        }
        // the products of this k-block are no longer read
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty_bar(pbi));
      }
      if (!ok) break;

      // ---- store (tokens half*128 + 32c + 8m + 2tq + e, e = 0, 1)
      const int t0 = half * 128;
      int nvalid = t.rows_tile - t0;
      if (nvalid > nc) nvalid = nc;
      const long long over = t.row0 + t0 + nvalid - p.R;
      if (over > 0) nvalid -= static_cast<int>(over);
      __nv_bfloat16* obase = out + (t.row0 + t0) * p.ldo;
      if (MODE == F8_SWIGLU) {
        // rows tr + 8k are gate (tr even) or up (tr odd) of h column
        // tr/2 + 4k; the partner row sits in lane ^ 4.  The gate lane makes
        // and stores h for the even token of each pair, the up lane for the
        // odd one.
        const bool up = (tr & 1) != 0;
        const int colb = t.n * 128 + static_cast<int>(rank) * 64 + q * 16 + (tr >> 1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (32 * c < nc) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int tok = 32 * c + 8 * m + 2 * tq + (up ? 1 : 0);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 mine = acc[c][m][k];
                const float ox = __shfl_xor_sync(0xFFFFFFFFu, mine.x, 4);
                const float oy = __shfl_xor_sync(0xFFFFFFFFu, mine.y, 4);
                const float g = up ? oy : mine.x;
                const float v = up ? mine.y : ox;
                const float h = g * __frcp_rn(1.0f + __expf(-g)) * v;
                if (tok < nvalid)
                  obase[static_cast<long long>(tok) * p.ldo + colb + 4 * k] = __float2bfloat16_rn(h);
              }
            }
          }
        }
      } else {
        const int colb = t.n * 256 + static_cast<int>(rank) * 128 + q * 32 + tr;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (32 * c < nc) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int tok = 32 * c + 8 * m + 2 * tq;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int col = colb + 8 * k;
                if (col < p.N) {
                  if (tok < nvalid)
                    obase[static_cast<long long>(tok) * p.ldo + col] =
                        __float2bfloat16_rn(acc[c][m][k].x);
                  if (tok + 1 < nvalid)
                    obase[static_cast<long long>(tok + 1) * p.ldo + col] =
                        __float2bfloat16_rn(acc[c][m][k].y);
                }
              }
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

bool make_map_u8_swap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  return gemm::make_map_sw128(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ptr, inner, outer, 128);
}

template <int MODE>
cudaError_t launch_fp8_swap(const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap& sa1,
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
    cudaError_t e = cudaFuncGetAttributes(&fa, fp8_swap_kernel<MODE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < kSplitRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(fp8_swap_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
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
  return cudaLaunchKernelEx(&cfg, fp8_swap_kernel<MODE>, w, x, sa1, sa2, sw, p);
}

}  // namespace

// Both GEMMs of moe_grouped_swiglu_fp8 in the small-group orientation; maps
// and scale layouts as in launch_grouped_swiglu_fp8.
cudaError_t launch_grouped_swiglu_fp8_small(const uint8_t* a_q, int ld_as, const int32_t* offsets,
                                            int G, int R, int d, int I, const uint8_t* w13_q,
                                            const uint8_t* w2_q, uint16_t* h, uint8_t* h_q,
                                            float* h_s, uint16_t* y, int32_t* status,
                                            const CUtensorMap& ta1, const CUtensorMap& ta2,
                                            const CUtensorMap& tsw13, const CUtensorMap& th1,
                                            const CUtensorMap& th2, const CUtensorMap& tsw2,
                                            cudaStream_t s) {
  CUtensorMap tw13, tx, tw2, th;
  if (!make_map_u8_swap(&tw13, w13_q, d, static_cast<uint64_t>(G) * 2 * I) ||
      !make_map_u8_swap(&tx, a_q, d, R) ||
      !make_map_u8_swap(&tw2, w2_q, I, static_cast<uint64_t>(G) * d) ||
      !make_map_u8_swap(&th, h_q, I, R))
    return cudaErrorInvalidValue;
  Fp8Params p1{};
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = d / BK;
  p1.w_rows_per_group = 2 * I;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  const int mt = (R + kTokTile - 1) / kTokTile + G;
  cudaError_t e = launch_fp8_swap<F8_SWIGLU>(tw13, tx, ta1, ta2, tsw13, p1, mt * (I / 128), s);
  if (e != cudaSuccess) return e;
  e = launch_quantize_rows(h, R, I, h_q, h_s, (R + 3) & ~3, s);
  if (e != cudaSuccess) return e;
  Fp8Params p2 = p1;
  p2.N = d;
  p2.num_kb = I / BK;
  p2.w_rows_per_group = d;
  p2.out = y;
  p2.ldo = d;
  return launch_fp8_swap<F8_DOWN>(tw2, th, th1, th2, tsw2, p2, mt * ((d + 255) / 256), s);
}

}  // namespace moe
