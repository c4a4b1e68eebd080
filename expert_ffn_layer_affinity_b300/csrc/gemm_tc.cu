// Grouped GEMMs on the fifth-generation tensor cores (tcgen05 + TMEM), fed
// by TMA.  One persistent, warp-specialised kernel template serves the three
// dense contractions of the layer:
//
//   MODE_SWIGLU  h[r, :] = silu(a[r] . w1[g]^T) * (a[r] . w3[g]^T)  -> bf16
//   MODE_DOWN    y[r, :] = h[r] . w2[g]^T                            -> bf16
//   MODE_ROUTER  s[t, e] = sigmoid(x[t] . w_r[e] + o[e])             -> fp32
//   MODE_DGRAD   o[r, :] = a[r] . [w[g] ; w'[g]]                     -> bf16
//
// MODE_DGRAD is the data-gradient product of the backward pass, e.g.
// dh = dy . W2 and dv = [da | dc] . [W1 ; W3]: the weights stay in their
// forward layout [K, N] (N contiguous) and are read MN-major by the MMA
// (the transpose bit of A), up to two stacked parts along K from two maps.
//
// Experts as shared + fine-grained routed FFNs follow weigao.cc "DeepSeek-V3
// Technical Report：中英对照解读", §2 table rows "DeepSeekMoE" and "Shared
// experts and routed experts"; a group is the run of rows the dispatch step
// gave to one expert.
//
// Expert modes run on CTA PAIRS (clusters of two, tcgen05 .cta_group::2).
// The pair puts 256 WEIGHT rows on the MMA's M side (128 in each CTA) and up
// to 256 of the group's TOKENS on the N side (half staged in each CTA), with
// N chosen per tile as the tokens left rounded up to 16.  Each CTA thus
// stages 16 KB of weights and 16 KB of tokens per 64-deep k-block for a
// 256 x 256 x 64 MMA step: a third less shared-memory fill traffic per FLOP
// than one CTA can reach.  Padding with N rounded to 16 costs about 3% of the
// MMA work at the V3 loads (6% at 32, 23% with 128-row token tiles).  The epilogue reads the [weight row x token] accumulator of its
// own CTA, transposes it through shared memory and writes token-major rows.
//
// Router mode keeps tokens on M (128) and experts on N (128).  Its K loop is
// cut into chunks of 4 k-blocks; each chunk is accumulated by the tensor core
// into its own TMEM buffer and the epilogue adds the chunk partials in fp32
// registers.  Long tensor-core accumulation chains lose precision; the short
// chains keep the logits' error well inside the 1e-5 near-tie margin used to
// judge routing.
//
// CTA layout (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: fills a STAGES-deep shared-memory ring
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma and commits (in a
//               pair, only the even CTA issues; its commits reach both CTAs)
//   warps 2..5  epilogue: tcgen05.ld from TMEM, activation, global stores
//
// The MMA issuer is the critical path: a tcgen05.mma of the pair costs the
// issuing thread about the same whatever N is, so a k-block of a ragged tile
// takes as long as a full one.  The issuer's loop keeps only the barrier
// wait, four MMAs and the commit per k-block (ring slot and parity stepped,
// descriptors offset from slot 0), and the epilogue warps, which share the
// SM sub-partitions with the issuer and the producer, poll their
// accumulator barrier with short sleeps instead of spinning (measured on the
// V3 routed call: about 20% fewer cycles, outputs bit-identical).
// Work items are (group, token tile, column tile), group-major and column
// tile fastest (see decode_work), handed out with a fixed stride.
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

constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;
using gemm::kMaxGroups;
using gemm::decode_work;
using gemm::wait_plain;
using gemm::store_block_transposed;
constexpr int kRouterChunkKb = 4;

// Tokens of a pair tile the MMA covers: the rows left, at most tok_tile,
// rounded up to 16 (8 staged in each CTA of the pair, one swizzle atom; the
// MMA's N is a multiple of 16).  Rows past the group's end are computed and
// never stored.
__device__ __forceinline__ int tile_n(int rows_left, int tok_tile) {
  const int n = rows_left < tok_tile ? rows_left : tok_tile;
  return (n + 15) & ~15;
}

enum Mode : int { MODE_SWIGLU = 0, MODE_DOWN = 1, MODE_ROUTER = 2, MODE_DGRAD = 3 };

template <int MODE>
struct Tr;
// SwiGLU pair tile: 128 output columns x up to 256 tokens.  Each CTA's 128
// M rows are the 64 w1 rows (TMEM lanes 0..63, the gate) and the 64 matching
// w3 rows (lanes 64..127, the up projection) of its 64 output columns.  The
// epilogue warps reading lanes 64..127 hand their values to the warps
// reading lanes 0..63 through a double-buffered shared-memory exchange.
template <>
struct Tr<MODE_SWIGLU> {
  static constexpr bool kPair = true;
  static constexpr int kTokTile = 256, kColTile = 128, kStages = 3, kBoxes = 2, kBufs = 2,
                       kBufCols = 256;
  static constexpr int kA = 128 * BK * 2, kB = 128 * BK * 2;  // per CTA and 64-wide k-block
};
// Down-projection pair tile: 256 output columns x up to 256 tokens.
template <>
struct Tr<MODE_DOWN> {
  static constexpr bool kPair = true;
  static constexpr int kTokTile = 256, kColTile = 256, kStages = 3, kBoxes = 2, kBufs = 2,
                       kBufCols = 256;
  static constexpr int kA = 128 * BK * 2, kB = 128 * BK * 2;
};
// Data-gradient pair tile: as MODE_DOWN, the weight tile staged MN-major
// (two 64-column chunks of 64 k-rows per CTA).
template <>
struct Tr<MODE_DGRAD> : Tr<MODE_DOWN> {};
template <>
struct Tr<MODE_ROUTER> {
  static constexpr bool kPair = false;
  static constexpr int kTokTile = 128, kColTile = 128, kStages = 3, kBoxes = 2, kBufs = 4,
                       kBufCols = 128;
  static constexpr int kA = 128 * BK * 2, kB = 128 * BK * 2;      // token tile, w_split tile
};

template <int MODE>
struct Cfg : Tr<MODE> {
  using T = Tr<MODE>;
  // A stage holds kBoxes consecutive 64-wide k-blocks of both operands, laid
  // out [A_0 .. A_{n-1}][B_0 .. B_{n-1}].  Every mode takes two boxes per
  // stage in three stages: the MMA issuer then waits and commits once per 128
  // of K (eight MMAs) instead of once per 64 (measured on the V3 shape: the
  // routed call 3% fewer SM cycles and 1.7% shorter steps from a cold start,
  // the route call 5% faster; outputs bit-identical).
  static constexpr int kStageBytes = T::kBoxes * (T::kA + T::kB);
  static constexpr int kTmemCols = T::kBufs * T::kBufCols;
  static constexpr int kNumBars = 2 * T::kStages + 2 * T::kBufs + 1;
  // epilogue staging: four per-warp 32 x 80-byte blocks (SwiGLU), or a
  // CTA-wide [2][32 tokens][128 columns] tile that the four epilogue warps
  // fill together (down and data-gradient modes)
  static constexpr int kXposeBytes = (MODE == MODE_ROUTER) ? 0
                                     : (MODE == MODE_DOWN || MODE == MODE_DGRAD) ? 2 * 32 * 128 * 2
                                                                                 : 4 * 32 * 80;
  // SwiGLU: 2 warp pairs x 2 buffers x 32 lanes x 33 fp32 (one padded row per lane)
  static constexpr int kXchgBytes = (MODE == MODE_SWIGLU) ? 2 * 2 * 32 * 33 * 4 : 0;
  static constexpr int kSmem = 1024 + T::kStages * kStageBytes + kXposeBytes + kXchgBytes +
                               (kNumBars + 8) * 8 + 16 + 2 * (kMaxGroups + 1) * 4;
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kTmemCols <= 512, "tensor memory");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct GemmParams {
  const int32_t* group_offsets;  // [G+1] device; nullptr = one group of rows [0, dense_rows)
  int dense_rows;
  int G;
  int N;                 // output columns of a group
  int R;                 // rows of the token operand and of the output
  int num_kb;            // reduction length / BK
  int a_k_wrap_kb;       // router: x's k-block = kb % a_k_wrap_kb
  int w_rows_per_group;  // rows of the weight operand's 2-D view per group
  int w_part_kb;         // DGRAD: k-blocks from tmA, the rest from tmA2
  void* out_a;           // SWIGLU: also store the pre-activations a and c (or nullptr)
  void* out_c;
  int splits;            // ROUTER: the k-blocks of a tile split over this many CTAs (>= 1)
  float* partial;        // ROUTER, splits > 1: raw logit sums [splits][R][ldo]
  void* out;
  int ldo;               // output row stride in elements
  const float* col_offset;  // router: per-expert logit offset or nullptr
  int w13_3d;               // SwiGLU: tmA is a 3-D map fetching w1 and w3 rows in one box
  int32_t* status;
  int w_tiled;  // expert modes: weights in the box-contiguous layout (see tile_expert_weights)
};

__device__ __forceinline__ int group_offset(const GemmParams& p, int g) {
  return p.group_offsets ? p.group_offsets[g] : (g == 0 ? 0 : p.dense_rows);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using C = Cfg<MODE>;
  constexpr bool PAIR = C::kPair;
  constexpr int S = C::kStages, NB = C::kBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles = (raw_addr + 1023u) & ~1023u;
  uint8_t* xpose = smem_raw + (tiles - raw_addr) + S * C::kStageBytes;
  float* xchg = reinterpret_cast<float*>(xpose + C::kXposeBytes);
  uint8_t* meta = xpose + C::kXposeBytes + C::kXchgBytes;
  const uint32_t bars = smem_u32(meta);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * S + NB + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 2 * NB);
  // SwiGLU exchange: xfull / xempty for (warp pair, buffer)
  auto xfull_bar = [&](int pr, int b) { return bars + 8u * (C::kNumBars + 2 * pr + b); };
  auto xempty_bar = [&](int pr, int b) { return bars + 8u * (C::kNumBars + 4 + 2 * pr + b); };
  // epilogue row gather (down and data-gradient modes): the four epilogue
  // warps meet once per 32-token chunk
  static_assert(kThreads == 6 * 32, "the row-gather barrier counts four epilogue warps");
  const uint32_t gather_bar = bars + 8u * C::kNumBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * (C::kNumBars + 8));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* mt_prefix = reinterpret_cast<int*>(meta + 8 * (C::kNumBars + 8) + 16);
  int* row_start = mt_prefix + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  // CTA pairs: rank 0 issues the MMAs; both iterate the same work list.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit_id = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (warp == 0) {
    gemm::build_tile_prefix(G, C::kTokTile, lane, [&](int g) { return group_offset(p, g); },
                            mt_prefix, row_start);
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      if (MODE == MODE_SWIGLU && !p.w13_3d) tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < NB; ++b) {
        mbar_init(accf_bar(b), 1);
        mbar_init(acce_bar(b), PAIR ? 256 : 128);
      }
      mbar_init(drain_bar, 1);
      // outside SwiGLU the first of these is the epilogue warps' row-gather
      // barrier (one arrival per warp)
      for (int i = 0; i < 8; ++i)
        mbar_init(bars + 8u * (C::kNumBars + i), (i == 0 && MODE != MODE_SWIGLU) ? 4 : 1);
      *abort_flag = 0;
      fence_mbar_init();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NT = (p.N + C::kColTile - 1) / C::kColTile;
  // the router may split a tile's k-blocks over `splits` work items (whole
  // chunks of kRouterChunkKb each); item w is (tile w / splits, split w % splits)
  const int splits = (MODE == MODE_ROUTER && p.splits > 1) ? p.splits : 1;
  const int total = mt_prefix[G] * NT * splits;
  const int split_kb = (MODE == MODE_ROUTER)
                           ? ((p.num_kb + kRouterChunkKb - 1) / kRouterChunkKb + splits - 1) / splits *
                                 kRouterChunkKb
                           : p.num_kb;
  auto kb_range = [&](int w, int& kb_lo, int& kb_hi) {
    const int sp = w % splits;
    kb_lo = sp * split_kb;
    kb_hi = kb_lo + split_kb < p.num_kb ? kb_lo + split_kb : p.num_kb;
  };
  const int chunk_kb = (MODE == MODE_ROUTER) ? kRouterChunkKb : p.num_kb;
  // Rows per token tile of a group of rows_g rows (expert modes): the group's
  // ceil(rows_g / 256) tiles share its rows evenly, rounded up to 16, so no
  // tile is a sliver.  A tile's MMAs cost the issuer about the same whatever
  // their N, so 300 rows as 160 + 144 cost less than as 256 + 48.  (The
  // fallback to 256 guards the last tile against being empty; no group of
  // up to 200000 rows needs it.)  Each token's arithmetic is unchanged.
  auto tile_rows = [&](int rows_g) {
    if (MODE == MODE_ROUTER || rows_g <= C::kTokTile) return C::kTokTile;
    const int nt = (rows_g + C::kTokTile - 1) / C::kTokTile;
    const int per = ((rows_g + nt - 1) / nt + 15) & ~15;
    return (nt - 1) * per < rows_g ? per : C::kTokTile;
  };
  const int num_st = (p.num_kb + C::kBoxes - 1) / C::kBoxes;           // stages per tile
  // stages per TMEM unit (a router chunk holds whole stages)
  const int chunk_st = (MODE == MODE_ROUTER) ? kRouterChunkKb / C::kBoxes : num_st;
  static_assert(kRouterChunkKb % C::kBoxes == 0, "router chunks hold whole stages");
  // the stages of item w: its k-blocks kBoxes at a time (the last stage may
  // hold fewer boxes)
  auto st_range = [&](int w, int& st_lo, int& st_hi) {
    int kb_lo, kb_hi;
    kb_range(w, kb_lo, kb_hi);
    st_lo = kb_lo / C::kBoxes;
    st_hi = (kb_hi + C::kBoxes - 1) / C::kBoxes;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_tok = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, n, m, st_lo, st_hi;
        decode_work(w / splits, NT, mt_prefix, G, g, n, m);
        st_range(w, st_lo, st_hi);
        const int rows_g = row_start[g + 1] - row_start[g];
        const int per = tile_rows(rows_g);
        int tok_row = row_start[g] + m * per;
        int w_row = g * p.w_rows_per_group + n * C::kColTile;
        if (PAIR) {
          tok_row += static_cast<int>(rank) * (tile_n(rows_g - m * per, per) / 2);
          w_row += static_cast<int>(rank) * (MODE == MODE_SWIGLU ? 64 : 128);
        }
        for (int st = st_lo; st < st_hi; ++st, ++it) {
          const int s = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int kb0 = st * C::kBoxes;
          const int nbox = (p.num_kb - kb0) < C::kBoxes ? p.num_kb - kb0 : C::kBoxes;
          const uint32_t sa = tiles + s * C::kStageBytes;
          const uint32_t sb = sa + C::kBoxes * C::kA;
          const uint32_t bytes = static_cast<uint32_t>(nbox * (C::kA + C::kB));
          if (MODE == MODE_ROUTER) {
            mbar_arrive_expect_tx(full_bar(s), bytes);
            for (int j = 0; j < nbox; ++j) {
              tma_load_2d(sa + static_cast<uint32_t>(j * C::kA), &tmA, full_bar(s),
                          ((kb0 + j) % p.a_k_wrap_kb) * BK, tok_row, pol_tok);
              tma_load_2d(sb + static_cast<uint32_t>(j * C::kB), &tmB, full_bar(s), (kb0 + j) * BK,
                          w_row, pol_w);
            }
          } else {
            // both CTAs' copies complete on the even CTA's barrier
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * bytes);
            const uint32_t fb = mapa_shared(full_bar(s), 0);
            for (int j = 0; j < nbox; ++j) {
              const uint32_t aj = sa + static_cast<uint32_t>(j * C::kA);
              const int kx = (kb0 + j) * BK;
              if ((MODE == MODE_SWIGLU || MODE == MODE_DOWN) && p.w_tiled) {
                // box-contiguous weights: box (group, row tile of this CTA,
                // k-block) is 128 rows of 128 B at row (index * 128) of a
                // [boxes * 128, 64] view; SwiGLU boxes alternate w1 and w3 rows
                const int row_tiles = MODE == MODE_SWIGLU ? p.N / 64 : p.N / 128;
                const long long box =
                    (static_cast<long long>(g) * row_tiles + n * 2 + static_cast<int>(rank)) *
                        p.num_kb + (kb0 + j);
                tma_load_2d_pair(aj, &tmA, fb, 0, static_cast<int>(box * 128), pol_w);
              } else if (MODE == MODE_SWIGLU && p.w13_3d) {
                tma_load_3d_pair(aj, &tmA, fb, kx, w_row, 0, pol_w);  // w1 rows, then w3 rows
              } else if (MODE == MODE_SWIGLU) {
                tma_load_2d_pair(aj, &tmA, fb, kx, w_row, pol_w);
                tma_load_2d_pair(aj + 64 * 128, &tmA2, fb, kx, w_row, pol_w);
              } else if (MODE == MODE_DGRAD) {
                // weights [K, N]: rows are k, columns the output columns of
                // this CTA's 128 (two 64-wide chunks)
                const int kb = kb0 + j;
                const bool second = kb >= p.w_part_kb;
                const int krow = g * p.w_rows_per_group + (second ? kb - p.w_part_kb : kb) * BK;
                const int ncol = n * C::kColTile + static_cast<int>(rank) * 128;
                tma_load_2d_pair(aj, second ? &tmA2 : &tmA, fb, ncol, krow, pol_w);
                tma_load_2d_pair(aj + 64 * BK * 2, second ? &tmA2 : &tmA, fb, ncol + 64, krow, pol_w);
              } else {
                tma_load_2d_pair(aj, &tmA, fb, kx, w_row, pol_w);
              }
            }
            for (int j = 0; j < nbox; ++j)
              tma_load_2d_pair(sb + static_cast<uint32_t>(j * C::kB), &tmB, fb, (kb0 + j) * BK,
                               tok_row, pol_tok);
          }
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
      uint32_t unit = 0;
      int slot = 0;        // ring slot of the next stage
      uint32_t fph = 0;    // parity of that slot's full barrier
      bool ok = true, issued = false;
      // shared-memory descriptors of slot 0; slot s starts s * kStageBytes
      // further on (the start-address field counts 16-byte units)
      const uint64_t a_desc0 =
          MODE == MODE_DGRAD ? umma_sdesc_mn_sw128(tiles) : umma_sdesc_sw128(tiles);
      const uint64_t b_desc0 = umma_sdesc_sw128(tiles + C::kBoxes * C::kA);
      constexpr uint64_t kSlotStep = C::kStageBytes >> 4;
      // the next 16 of K: 32 bytes along a K-major row, or 16 128-byte rows
      // of an MN-major chunk
      constexpr uint64_t a_step = MODE == MODE_DGRAD ? (16 * 128) >> 4 : 2;
      for (int w = unit_id; w < total && ok; w += n_units) {
        int g, n, m, st_lo, st_hi;
        decode_work(w / splits, NT, mt_prefix, G, g, n, m);
        st_range(w, st_lo, st_hi);
        uint32_t idesc;
        if (MODE == MODE_ROUTER) {
          idesc = umma_idesc_bf16(128, C::kColTile);
        } else {
          const int rows_g = row_start[g + 1] - row_start[g];
          const int per = tile_rows(rows_g);
          idesc = umma_idesc_bf16(256, tile_n(rows_g - m * per, per)) |
                  (MODE == MODE_DGRAD ? (1u << 15) : 0u);  // A (weights) MN-major
        }
        for (int st0 = st_lo; st0 < st_hi && ok; st0 += chunk_st, ++unit) {
          const int b = static_cast<int>(unit % NB);
          const uint32_t bph = (unit / NB) & 1u;
          if (!mbar_wait(acce_bar(b), bph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * C::kBufCols);
          const int st1 = (st0 + chunk_st < st_hi) ? st0 + chunk_st : st_hi;
          uint32_t acc = 0u;  // the unit's first MMA overwrites its accumulator
          for (int st = st0; st < st1; ++st) {
            if (!mbar_wait(full_bar(slot), fph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t soff = static_cast<uint64_t>(slot) * kSlotStep;
            const int nbox = C::kBoxes == 1 ? 1
                             : (p.num_kb - st * C::kBoxes < C::kBoxes ? p.num_kb - st * C::kBoxes
                                                                        : C::kBoxes);
#pragma unroll
            for (int j = 0; j < C::kBoxes; ++j) {
              if (j >= nbox) break;
              const uint64_t adesc = a_desc0 + soff + static_cast<uint64_t>((j * C::kA) >> 4);
              const uint64_t bdesc = b_desc0 + soff + static_cast<uint64_t>((j * C::kB) >> 4);
#pragma unroll
              for (int k = 0; k < BK / UMMA_K; ++k) {
                if (PAIR) umma_bf16_pair(d_tmem, adesc + a_step * k, bdesc + 2ull * k, idesc, acc);
                else umma_bf16(d_tmem, adesc + a_step * k, bdesc + 2ull * k, idesc, acc);
                acc = 1u;
              }
            }
            issued = true;
            if (PAIR) umma_commit_pair_mc(empty_bar(slot), 0x3);
            else umma_commit(empty_bar(slot));
            if (++slot == S) {
              slot = 0;
              fph ^= 1u;
            }
          }
          if (!ok) break;
          if (PAIR) umma_commit_pair_mc(accf_bar(b), 0x3);
          else umma_commit(accf_bar(b));
        }
      }
      if (!ok && issued) {
        if (PAIR) umma_commit_pair_mc(drain_bar, 0x1);
        else umma_commit(drain_bar);
        wait_plain(drain_bar, 0u, 200000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp may read TMEM lanes 32q .. 32q+31
    uint8_t* xp = xpose + q * 32 * 80;
    uint32_t unit = 0, xchunk = 0;
    bool ok = true;
    for (int w = unit_id; w < total && ok; w += n_units) {
      int g, n, m, kb_lo, kb_hi;
      decode_work(w / splits, NT, mt_prefix, G, g, n, m);
      kb_range(w, kb_lo, kb_hi);
      const int rows_g = row_start[g + 1] - row_start[g];
      const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
      if (MODE == MODE_ROUTER) {
        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
        for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += chunk_kb, ++unit) {
          const int b = static_cast<int>(unit % NB);
          const uint32_t bph = (unit / NB) & 1u;
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_nap(accf_bar(b), bph, abort_flag, p.status));
          if (!ok) break;
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(b * C::kBufCols);
#pragma unroll
          for (int c = 0; c < 128; c += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c + i] = __fadd_rn(acc[c + i], __uint_as_float(r[i]));
          }
          tc_fence_before();
          mbar_arrive(acce_bar(b));
        }
        if (!ok) break;
        const int row_local = m * 128 + q * 32 + lane;
        if (row_local < rows_g && row_local < p.R) {
          const int col0 = n * 128;
          if (splits > 1) {
            // this split's sum of its chunk partials; router_finish adds the
            // splits in order, then the offset and the sigmoid
            float* out = p.partial + (static_cast<long long>(w % splits) * p.R + row_local) * p.ldo;
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (col0 + i < p.N) out[col0 + i] = acc[i];
          } else {
            float* out = reinterpret_cast<float*>(p.out) + static_cast<long long>(row_local) * p.ldo;
#pragma unroll
            for (int i = 0; i < 128; ++i) {
              const int cc = col0 + i;
              if (cc < p.N) {
                float u = acc[i];
                if (p.col_offset) u = __fadd_rn(u, p.col_offset[cc]);
                out[cc] = 1.0f / (1.0f + expf(-u));
              }
            }
          }
        }
      } else {
        const int b = static_cast<int>(unit % NB);
        const uint32_t bph = (unit / NB) & 1u;
        ++unit;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait_nap(accf_bar(b), bph, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const int per = tile_rows(rows_g);
        const int tok0 = m * per;
        const int n_eff = tile_n(rows_g - tok0, per);
        const int rows_tile = (rows_g - tok0) < per ? rows_g - tok0 : per;
        const int col = n * C::kColTile +
                        (MODE == MODE_SWIGLU ? 64 * static_cast<int>(rank) + 32 * (q & 1)
                                             : 128 * static_cast<int>(rank) + 32 * q);
        const long long row0 = static_cast<long long>(row_start[g]) + tok0;
        const bool col_ok = col < p.N;
        const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(b * C::kBufCols);
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        for (int c = 0; c < n_eff && ok; c += 32, ++xchunk) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          int valid = rows_tile - c;
          if (valid > 32) valid = 32;
          const long long last = row0 + c + valid;
          if (last > p.R) valid -= static_cast<int>(last - p.R);
          if (MODE == MODE_SWIGLU && p.w_tiled) {
            // box-contiguous weights interleave the rows: TMEM lane 2i holds
            // the gate (w1 row i) and lane 2i + 1 the up value (w3 row i) of
            // output column i, so a lane pair of this warp owns 16 columns;
            // the even lane finishes tokens 0..15 of the chunk, the odd lane
            // tokens 16..31, after swapping halves with one shuffle each
            const bool odd = (lane & 1) != 0;
            const int tcol = n * C::kColTile + 64 * static_cast<int>(rank) + 16 * q;
            __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(xp);  // [32 tokens][16 columns]
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float mine = __uint_as_float(odd ? v[k] : v[16 + k]);
              const float other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
              const float gate = odd ? other : __uint_as_float(v[k]);
              const float up = odd ? __uint_as_float(v[16 + k]) : other;
              // silu(gate) * up; the fast division (about 2 ulp in fp32, far
              // below the bf16 rounding of h) instead of a correctly rounded
              // reciprocal: the SwiGLU epilogue is on the critical path of
              // short items (mid layer: 0.686 -> 0.624 ms per step)
              const float hv = __fdividef(gate, 1.0f + __expf(-gate)) * up;
              st[((odd ? 16 : 0) + k) * 16 + (lane >> 1)] = __float2bfloat16_rn(hv);
            }
            __syncwarp();
            if (tcol < p.N && lane < valid) {
              const uint4* src = reinterpret_cast<const uint4*>(xp + lane * 32);
              uint4* dst = reinterpret_cast<uint4*>(out + (row0 + c + lane) * p.ldo + tcol);
              dst[0] = src[0];
              dst[1] = src[1];
            }
            __syncwarp();
          } else if (MODE == MODE_SWIGLU) {
            // pair (q, q + 2): lanes 64..127 (up) hand over to lanes 0..63 (gate)
            const int pr = q & 1, xb = static_cast<int>(xchunk & 1u);
            const uint32_t xph = (xchunk >> 1) & 1u;
            float* xrow = xchg + ((pr * 2 + xb) * 32 + lane) * 33;
            if (q >= 2) {
              ok = __all_sync(0xFFFFFFFFu,
                              mbar_wait(xempty_bar(pr, xb), xph ^ 1u, abort_flag, p.status));
              if (!ok) break;
#pragma unroll
              for (int j = 0; j < 32; ++j) xrow[j] = __uint_as_float(v[j]);
              __syncwarp();
              if (lane == 0) mbar_arrive(xfull_bar(pr, xb));
            } else {
              ok = __all_sync(0xFFFFFFFFu, mbar_wait(xfull_bar(pr, xb), xph, abort_flag, p.status));
              if (!ok) break;
              if (p.out_a != nullptr && col_ok) {
                // training: keep a = v.w1 and c = v.w3 for the backward pass
                uint32_t cv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) cv[j] = __float_as_uint(xrow[j]);
                store_block_transposed(v, xp, lane, static_cast<__nv_bfloat16*>(p.out_a), row0 + c,
                                       valid, p.ldo, col);
                store_block_transposed(cv, xp, lane, static_cast<__nv_bfloat16*>(p.out_c), row0 + c,
                                       valid, p.ldo, col);
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float a = __uint_as_float(v[j]);
                v[j] = __float_as_uint(__fdividef(a, 1.0f + __expf(-a)) * xrow[j]);  // as above
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(xempty_bar(pr, xb));
              if (col_ok) store_block_transposed(v, xp, lane, out, row0 + c, valid, p.ldo, col);
            }
          } else {
            // the CTA's 128 columns of the chunk's 32 tokens, gathered from the
            // four epilogue warps into one tile, then written as whole 256-byte
            // token rows instead of each lane storing 64 bytes of a different
            // row (the store transactions share the SM's L1 data path with the
            // MMA's operand reads; bit-identical).  The SwiGLU epilogue keeps
            // per-warp stores: there the extra meeting per chunk cost the
            // mid layer 1.9% (its 32-k-block items leave the epilogue little
            // slack) and gained nothing measurable at the V3 shape.
            __nv_bfloat16* tile =
                reinterpret_cast<__nv_bfloat16*>(xpose) + (xchunk & 1u) * (32 * 128);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              tile[j * 128 + 32 * q + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
            __syncwarp();
            if (lane == 0) mbar_arrive(gather_bar);
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(gather_bar, xchunk & 1u, abort_flag, p.status));
            if (!ok) break;
            const int cbase = n * C::kColTile + 128 * static_cast<int>(rank);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 8 * q + 2 * i + (lane >> 4);
              const int cc = (lane & 15) * 8;
              if (r < valid && cbase + cc < p.N)
                *reinterpret_cast<uint4*>(out + (row0 + c + r) * p.ldo + cbase + cc) =
                    *reinterpret_cast<const uint4*>(tile + r * 128 + cc);
            }
          }
        }
        if (!ok) break;
        tc_fence_before();
        mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // no CTA frees TMEM or exits while its peer still uses it
  tc_fence_after();
  if (warp == 1) {
    if (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using gemm::encode_fn;

// 2-D bf16 tensor [outer, inner] (inner contiguous), box = 64 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  return gemm::make_map_sw128(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, inner, outer, box_rows);
}

// w1 and w3 of one allocation, w3 a fixed positive byte distance after w1:
// a 3-D map [2][rows][inner] whose box {64, 64, 2} brings 64 rows of w1 and
// the same 64 rows of w3 in one copy.
bool make_map_w13(CUtensorMap* m, const void* w1, const void* w3, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(w1), b = reinterpret_cast<uintptr_t>(w3);
  if (b <= a) return false;
  const uint64_t dist = b - a;
  if (dist % 16 || dist >= (1ull << 40) || dist < rows * inner * 2) return false;
  cuuint64_t dims[3] = {inner, rows, 2};
  cuuint64_t strides[2] = {inner * 2, dist};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w1), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                        const GemmParams& p, int max_units, cudaStream_t s) {
  using C = Cfg<MODE>;
  static DeviceOnce once;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = once_per_device(once, dev, []() {
    return cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmem);
  });
  if (err != cudaSuccess) return err;
  const int per_unit = C::kPair ? 2 : 1;
  int units = sm_count() / per_unit;
  if (max_units < units) units = max_units;
  if (units < 1) units = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * per_unit), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(per_unit);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<MODE>, a, a2, b, p);
}

}  // namespace

cudaError_t launch_grouped_swiglu(const uint16_t* a, const int32_t* offsets, int G, int R, int d,
                                  int I, const uint16_t* w1, const uint16_t* w3,
                                  const uint16_t* w2, uint16_t* h, uint16_t* y, int32_t* status,
                                  cudaStream_t s, uint16_t* a_out, uint16_t* c_out) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  using C1 = Cfg<MODE_SWIGLU>;
  using C2 = Cfg<MODE_DOWN>;
  CUtensorMap tw1, tw3, tx, tw2, th;
  if (!make_map(&tw1, w1, d, static_cast<uint64_t>(G) * I, 64) ||
      !make_map(&tw3, w3, d, static_cast<uint64_t>(G) * I, 64) ||
      !make_map(&tx, a, d, R, 128) ||
      !make_map(&tw2, w2, I, static_cast<uint64_t>(G) * d, 128) ||
      !make_map(&th, h, I, R, 128))
    return cudaErrorInvalidValue;
  CUtensorMap tw13;
  const bool w13 = make_map_w13(&tw13, w1, w3, d, static_cast<uint64_t>(G) * I);
  GemmParams p1{};
  p1.w13_3d = w13 ? 1 : 0;
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = d / BK;
  p1.a_k_wrap_kb = d / BK;
  p1.w_rows_per_group = I;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  p1.out_a = a_out;
  p1.out_c = c_out;
  const int mt1 = (R + C1::kTokTile - 1) / C1::kTokTile + G;
  cudaError_t e = launch_gemm<MODE_SWIGLU>(w13 ? tw13 : tw1, tw3, tx, p1, mt1 * ((I + 127) / 128), s);
  if (e != cudaSuccess) return e;
  GemmParams p2 = p1;
  p2.out_a = p2.out_c = nullptr;
  p2.w13_3d = 0;
  p2.N = d;
  p2.num_kb = I / BK;
  p2.a_k_wrap_kb = I / BK;
  p2.w_rows_per_group = d;
  p2.out = y;
  p2.ldo = d;
  const int mt2 = (R + C2::kTokTile - 1) / C2::kTokTile + G;
  return launch_gemm<MODE_DOWN>(tw2, tw2, th, p2, mt2 * ((d + 255) / 256), s);
}

namespace {
// out = the box-contiguous copy of a weight tensor (see launch_tile_expert_weights):
// 16-byte chunk q of the output holds source row `src_row`, columns
// kb*64 + c8*8 .. +7.
__global__ void __launch_bounds__(256) tile_weights_kernel(const uint4* __restrict__ w1,
                                                           const uint4* __restrict__ w3,
                                                           long long G, int rows, int cols,
                                                           int tile_rows, uint4* __restrict__ out) {
  const int kbs = cols / 64;
  const int tiles = rows / tile_rows;  // row tiles per group (SwiGLU: 64 rows of w1 and of w3)
  const int box_rows = w3 ? 2 * tile_rows : tile_rows;
  const long long n = G * tiles * kbs * box_rows * 8;
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < n;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(q & 7);
    long long t = q >> 3;
    const int r = static_cast<int>(t % box_rows);
    t /= box_rows;
    const int kb = static_cast<int>(t % kbs);
    t /= kbs;
    const int tile = static_cast<int>(t % tiles);
    const long long g = t / tiles;
    // SwiGLU boxes alternate the rows: row 2i is w1 row i, row 2i + 1 is w3 row i
    const bool second = w3 != nullptr && (r & 1);
    const long long src_row = g * rows + static_cast<long long>(tile) * tile_rows +
                              (w3 != nullptr ? (r >> 1) : r);
    const uint4* src = second ? w3 : w1;
    out[q] = src[src_row * (cols / 8) + kb * 8 + c8];
  }
}
}  // namespace

// Box-contiguous copies of the expert weights, so that every 128-row x
// 64-column box the grouped GEMM stages is 16 KB of consecutive memory (one
// DRAM stream per box instead of 128 strided rows):
//   w13_tiled [G][I/64][d/64][128][64]: row 2i of a box is w1 row t*64 + i of
//     group g and row 2i + 1 the same row of w3 (so the gate and up values of
//     an output column land in neighbouring TMEM lanes of one epilogue warp),
//     columns kb*64 .. kb*64+63;
//   w2_tiled  [G][d/128][I/64][128][64]: rows t*128 .. t*128+127 of w2[g].
cudaError_t launch_tile_expert_weights(const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                                       int G, int I, int d, uint16_t* w13_tiled,
                                       uint16_t* w2_tiled, cudaStream_t s) {
  const int blocks = sm_count() * 8;
  if (w1 && w3 && w13_tiled)
    tile_weights_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(w1),
                                               reinterpret_cast<const uint4*>(w3), G, I, d, 64,
                                               reinterpret_cast<uint4*>(w13_tiled));
  if (w2 && w2_tiled)
    tile_weights_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(w2), nullptr, G, d,
                                               I, 128, reinterpret_cast<uint4*>(w2_tiled));
  return cudaGetLastError();
}

// The grouped SwiGLU experts on box-contiguous weights (same arithmetic and
// order as launch_grouped_swiglu, so bit-identical outputs).
cudaError_t launch_grouped_swiglu_tiled(const uint16_t* a, const int32_t* offsets, int G, int R,
                                        int d, int I, const uint16_t* w13_tiled,
                                        const uint16_t* w2_tiled, uint16_t* h, uint16_t* y,
                                        int32_t* status, cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  using C1 = Cfg<MODE_SWIGLU>;
  using C2 = Cfg<MODE_DOWN>;
  CUtensorMap tw13, tx, tw2, th;
  if (!make_map(&tw13, w13_tiled, 64, static_cast<uint64_t>(G) * (I / 64) * (d / 64) * 128, 128) ||
      !make_map(&tw2, w2_tiled, 64, static_cast<uint64_t>(G) * (d / 128) * (I / 64) * 128, 128) ||
      !make_map(&tx, a, d, R, 128) || !make_map(&th, h, I, R, 128))
    return cudaErrorInvalidValue;
  GemmParams p1{};
  p1.w_tiled = 1;
  p1.group_offsets = offsets;
  p1.G = G;
  p1.N = I;
  p1.R = R;
  p1.num_kb = d / BK;
  p1.a_k_wrap_kb = d / BK;
  p1.w_rows_per_group = I;
  p1.out = h;
  p1.ldo = I;
  p1.status = status;
  const int mt1 = (R + C1::kTokTile - 1) / C1::kTokTile + G;
  cudaError_t e = launch_gemm<MODE_SWIGLU>(tw13, tw13, tx, p1, mt1 * ((I + 127) / 128), s);
  if (e != cudaSuccess) return e;
  GemmParams p2 = p1;
  p2.N = d;
  p2.num_kb = I / BK;
  p2.a_k_wrap_kb = I / BK;
  p2.w_rows_per_group = d;
  p2.out = y;
  p2.ldo = d;
  const int mt2 = (R + C2::kTokTile - 1) / C2::kTokTile + G;
  return launch_gemm<MODE_DOWN>(tw2, tw2, th, p2, mt2 * ((d + 255) / 256), s);
}

cudaError_t launch_grouped_gemm_nt(const uint16_t* a, const int32_t* offsets, int G, int R, int K,
                                   int N, const uint16_t* w, uint16_t* out, int32_t* status,
                                   cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  using C2 = Cfg<MODE_DOWN>;
  CUtensorMap tw, ta;
  if (!make_map(&tw, w, K, static_cast<uint64_t>(G) * N, 128) || !make_map(&ta, a, K, R, 128))
    return cudaErrorInvalidValue;
  GemmParams p{};
  p.group_offsets = offsets;
  p.G = G;
  p.N = N;
  p.R = R;
  p.num_kb = K / BK;
  p.a_k_wrap_kb = K / BK;
  p.w_rows_per_group = N;
  p.out = out;
  p.ldo = N;
  p.status = status;
  const int mt = (R + C2::kTokTile - 1) / C2::kTokTile + G;
  return launch_gemm<MODE_DOWN>(tw, tw, ta, p, mt * ((N + 255) / 256), s);
}

cudaError_t launch_grouped_gemm_kn(const uint16_t* a, const int32_t* offsets, int G, int R, int K,
                                   int N, const uint16_t* w0, int K0, const uint16_t* w1,
                                   uint16_t* out, int32_t* status, cudaStream_t s) {
  if (R == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups) return cudaErrorInvalidValue;
  using C = Cfg<MODE_DGRAD>;
  CUtensorMap tw0, tw1, ta;
  const int K1 = K - K0;
  if (!make_map(&tw0, w0, N, static_cast<uint64_t>(G) * K0, BK) ||
      !make_map(&tw1, K1 > 0 ? w1 : w0, N, static_cast<uint64_t>(G) * (K1 > 0 ? K1 : K0), BK) ||
      !make_map(&ta, a, K, R, 128))
    return cudaErrorInvalidValue;
  GemmParams p{};
  p.group_offsets = offsets;
  p.G = G;
  p.N = N;
  p.R = R;
  p.num_kb = K / BK;
  p.a_k_wrap_kb = K / BK;
  p.w_rows_per_group = K0;  // rows of each part per group: K0 and K1
  p.w_part_kb = K0 / BK;
  p.out = out;
  p.ldo = N;
  p.status = status;
  // (the second part's rows per group equal the first's whenever it exists)
  const int mt = (R + C::kTokTile - 1) / C::kTokTile + G;
  return launch_gemm<MODE_DGRAD>(tw0, tw1, ta, p, mt * ((N + 255) / 256), s);
}

namespace {
// scores[t, e] = sigmoid(sum over the splits, in order, of partial[s, t, e] + o[e])
__global__ void __launch_bounds__(256) router_finish_kernel(const float* __restrict__ partial,
                                                            int splits, long long n, int E,
                                                            const float* __restrict__ offset,
                                                            float* __restrict__ scores) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float u = partial[i];
    for (int sp = 1; sp < splits; ++sp) u = __fadd_rn(u, partial[sp * n + i]);
    if (offset) u = __fadd_rn(u, offset[i % E]);
    scores[i] = 1.0f / (1.0f + expf(-u));
  }
}
}  // namespace

int router_splits(int T, int d, int E, int sms) {
  const int units = ((T + 127) / 128) * ((E + 127) / 128);
  const int chunks = (3 * d / BK + kRouterChunkKb - 1) / kRouterChunkKb;
  int sp = units >= sms ? 1 : sms / units;
  if (sp > chunks) sp = chunks;
  if (sp < 1) sp = 1;
  const int per = (chunks + sp - 1) / sp;  // no empty split
  return (chunks + per - 1) / per;
}

cudaError_t launch_router_gemm(const uint16_t* x, const uint16_t* w_split, const float* offset,
                               int T, int d, int E, float* scores, int32_t* status,
                               cudaStream_t s, float* partial, size_t partial_bytes) {
  if (T == 0) return cudaSuccess;
  CUtensorMap ta, tb;
  if (!make_map(&ta, x, d, T, 128) || !make_map(&tb, w_split, 3ull * d, E, 128))
    return cudaErrorInvalidValue;
  GemmParams p{};
  p.group_offsets = nullptr;
  p.dense_rows = T;
  p.G = 1;
  p.N = E;
  p.R = T;
  p.num_kb = 3 * d / BK;
  p.a_k_wrap_kb = d / BK;
  p.w_rows_per_group = 0;
  p.out = scores;
  p.ldo = E;
  p.col_offset = offset;
  p.status = status;
  // small batches fill the GPU by splitting each tile's reduction
  int splits = router_splits(T, d, E, sm_count());
  const size_t need = static_cast<size_t>(splits) * T * E * sizeof(float);
  if (splits > 1 && (partial == nullptr || partial_bytes < need)) splits = 1;
  p.splits = splits;
  p.partial = splits > 1 ? partial : nullptr;
  const int works = ((T + 127) / 128) * ((E + 127) / 128) * splits;
  cudaError_t e = launch_gemm<MODE_ROUTER>(ta, ta, tb, p, works, s);
  if (e != cudaSuccess || splits == 1) return e;
  const long long n = static_cast<long long>(T) * E;
  long long blocks = (n + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  router_finish_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(partial, splits, n, E, offset,
                                                                 scores);
  return cudaGetLastError();
}

}  // namespace moe
