/*
 * moe.h -- C ABI of libmoe_b300.so: the forward pass of a DeepSeekMoE layer
 * with auxiliary-loss-free load balancing, on one NVIDIA B300 (sm_103a).
 *
 * The layer (one step over a batch of T tokens):
 *   1. affinity   s[t,e] = sigmoid(x[t,:] . w_r[e,:] (+ o[e]))
 *   2. selection  top-K experts of the biased score z = s + b (the bias only
 *                 chooses experts), optionally limited to M of G expert groups
 *   3. gates      g[t,k] = scale * s[t,idx_k] / sum_j s[t,idx_j]  (raw s only)
 *   4. dispatch   rows grouped by expert, SwiGLU experts + shared experts,
 *                 weighted combine
 *   5. feedback   per-expert load over the batch; b_e -= gamma if overloaded,
 *                 b_e += gamma if underloaded
 * Sources: "Score = Affinity + Bias" and "Bias 仅用于路由" (DeepSeek V3,
 * deepseekmodel1.org, section 公式解密); the bias update and node-limited
 * routing (DeepSeek-V3 Technical Report reading notes, chenshi221.pages.dev,
 * section "Auxiliary-loss-free 负载均衡"); §3 of "DeepSeek-V3 Technical Report：
 * 中英对照解读" (weigao.cc); dispatch/combine (same page, §2.2 table row
 * "Expert parallelism requires token dispatch and combine").
 *
 * Conventions shared by every call:
 *  - All pointers are DEVICE pointers owned by the caller unless a comment says
 *    otherwise; the library never allocates, frees or synchronises (except the
 *    one-time per-device set-up noted below) and keeps no state between calls.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream).
 *  - Arguments are validated synchronously; a negative moe_status is returned
 *    and nothing is launched.  Conditions only the device can see (a bounded
 *    wait that ran out, non-finite scores, out-of-range expert indices) are
 *    OR-ed as MOE_DEV_* bits into the caller's int32 `status_dev` word, which
 *    the caller zeroes and reads back when it chooses.
 *  - Dtypes: bf16 = IEEE bfloat16 bit patterns (uint16), fp32 = float,
 *    indices int32.  Matrices are row-major with the reduction dimension
 *    contiguous; base pointers must be 16-byte aligned.
 *  - Shape limits: d % 64 == 0, I % 64 == 0, 1 <= K <= E <= 512, E % n_groups
 *    == 0, 1 <= topk_groups <= n_groups, T*K < 2^31.  Anything else returns
 *    MOE_ERR_UNSUPPORTED_SHAPE; there is no fallback path.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int moe_status;
typedef void* moe_stream_t; /* a cudaStream_t */

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad enum */
#define MOE_ERR_UNSUPPORTED_SHAPE (-2) /* outside the limits above */
#define MOE_ERR_CUDA (-3)              /* a CUDA runtime/driver call failed */
#define MOE_ERR_WORKSPACE (-4)         /* workspace smaller than required */
#define MOE_ERR_SCRATCH_LIMIT (-5)     /* shape needs more than a fixed scratch array holds */

/* Bits OR-ed into *status_dev by the kernels. */
#define MOE_DEV_TIMEOUT 1u    /* a bounded mbarrier wait ran out (the kernel returned early) */
#define MOE_DEV_NONFINITE 2u  /* a NaN/Inf affinity or bias was seen (selection still completes, NaN ranks lowest) */
#define MOE_DEV_BAD_INDEX 4u  /* an expert index outside [0, E) was given to moe_permute (entry skipped) */

/* ABI version of this header: 1. */
int moe_abi_version(void);

/* Bytes of device workspace the calls below need for a layer of this shape
 * (the caller allocates it once; 256-byte aligned).  Covers the router's
 * affinity buffer (T*E fp32), then, in one shared region, the router GEMM's
 * split-reduction scratch (small T: each output tile's reduction spread over
 * several CTAs) and the permute's per-tile expert counts. */
size_t moe_workspace_bytes(int T, int d, int E, int K, int I);

/* How many CTAs share each output tile's reduction in the router GEMM of
 * moe_router_topk on the current device (1: no split; above 1 one more small
 * kernel adds the splits).  Host-only query.  The count depends on T and on
 * the device's SM count, and the affinities' last bits depend on the count
 * (see moe_router_topk). */
int moe_router_splits(int T, int d, int E);

/* One-time router weight preparation: splits fp32 w_r [E, d] exactly into
 * three bf16 parts hi + mid + lo (each the bf16 rounding of the remainder),
 * stored side by side as w_split [E, 3*d] bf16, so the tensor-core router
 * GEMM forms every product x*w exactly and only accumulates in fp32.  The
 * report keeps MoE gating in high precision (qwbw.cn essay on the report,
 * "MoE门控...依然保留BF16或者FP32高精度"). */
moe_status moe_router_prepare(const float* w_r, int E, int d, void* w_split_bf16,
                              moe_stream_t stream);

/* Steps 1-3 and the load count of step 5.
 *  x_bf16        [T, d] activations, or NULL to select from `scores_in`.
 *  w_split_bf16  [E, 3d] from moe_router_prepare (ignored when x is NULL).
 *  scores_in     [T, E] fp32 affinities s, used when x is NULL (this is how
 *                the selection is checked bit-for-bit against a reference).
 *  logit_offset  [E] fp32 added to the logits before the sigmoid, or NULL.
 *  bias          [E] fp32 per-expert selection bias b.
 *  n_groups, topk_groups  G and M of the group limit (1, 1 = no limit).  A
 *                group's score is the sum of its ceil(K/M) largest z.
 *  route_scale   multiplies the normalised gates.
 *  n_shared_routed  serving layout of the report's decode deployment, where
 *                the shared expert travels as one more routed expert ("每个
 *                token ... 9个专家", qwbw.cn essay on the report): 0 = off;
 *                n > 0 appends ids E .. E+n-1 with gate 1.0 after the K routed
 *                ones, so rows of topk_idx / topk_gate have K+n entries and
 *                the shared experts run inside the routed grouped GEMM (their
 *                weights stored as groups E .. E+n-1).  Loads count the K
 *                routed experts only.  K + n <= 32.
 * Outputs: topk_idx [T, K(+n)] int32 in rank order (z descending, lower expert
 *  index first on equal z, -0 == +0, NaN below every number); topk_gate
 *  [T, K(+n)] fp32; expert_load [E] int32 (overwritten: zeroed then counted);
 *  affinity_out [T, E] fp32 or NULL (the s used, when x is given).
 * Fp32 rule (bit-exact against a reference fed the same s): z = s + b; group
 *  score = top1 + top2 (+ ...); denom = s_1 + s_2 + ... in rank order;
 *  g = (s_k / denom) * scale, each one IEEE fp32 operation.
 * Workspace: `ws` of `ws_bytes` >= moe_workspace_bytes(...); with x given and
 *  a smaller workspace (or none next to affinity_out) the router GEMM runs
 *  without splitting its reduction.
 * Batch dependence: the router GEMM adds the same exact products in an
 *  order that depends on its split count (moe_router_splits, chosen from T
 *  and the device's SM count), so a token's affinities may differ in their
 *  last bits between batch sizes or devices, and on a near tie its chosen
 *  experts with them.  Every split count stays within 4e-6 of the exact
 *  affinity at d = 7168. */
moe_status moe_router_topk(const void* x_bf16, const void* w_split_bf16,
                           const float* scores_in, const float* logit_offset,
                           const float* bias, int T, int d, int E, int K,
                           int n_groups, int topk_groups, float route_scale,
                           int n_shared_routed, int32_t* topk_idx, float* topk_gate,
                           int32_t* expert_load,
                           float* affinity_out, int32_t* status_dev, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* Step 4a, dispatch.  Rows of expert e are the (t, k) pairs with
 * topk_idx[t,k] == e, in ascending (t, k) order; experts follow one another
 * in ascending order.
 *  expert_offsets [E+1] int32: row range of each expert (exclusive scan of loads).
 *  row_of [T, K] int32: row of x_perm holding (t, k).
 *  tok_of [T*K] int32: token of each row.
 *  x_perm [T*K, d] bf16: x_perm[row_of[t,k]] = x[t]  (skipped when x_bf16 is NULL). */
moe_status moe_permute(const int32_t* topk_idx, int T, int K, int E, const void* x_bf16,
                       int d, int32_t* expert_offsets, int32_t* row_of, int32_t* tok_of,
                       void* x_perm_bf16, int32_t* status_dev, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Allocation-free variant of moe_permute.  (The method has no counterpart of
 * this: it only changes where the call keeps its temporary data.)
 *
 * For callers that cannot allocate device memory at call time: for example a
 * plugin running inside a host application that owns every device allocation
 * through its own pool and hands out no workspace, or a latency-critical
 * serving loop that must never call cudaMalloc once it has started (an
 * allocation can synchronise the device and stall every stream).  Arguments,
 * outputs and results are exactly those of moe_permute; only the workspace
 * is gone.
 *
 * The per-tile expert counts go to a fixed array of 65536 int32 (256 KiB)
 * compiled into this library, which every GPU that loads the library keeps
 * until the process exits.  Limit: ceil(T*K / 1024) * E <= 65536 (for
 * instance T*K <= 262144 with E = 256); larger shapes return
 * MOE_ERR_SCRATCH_LIMIT before anything is launched.  Each call overwrites
 * the counts it uses, so nothing has to be cleared between calls.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture.  All calls share the one array: calls whose kernels can overlap on
 * the GPU (other streams, other host threads) race on it, so the caller must
 * serialise them.  No device memory is allocated or freed by this call. */
moe_status moe_permute_static(const int32_t* topk_idx, int T, int K, int E, const void* x_bf16,
                              int d, int32_t* expert_offsets, int32_t* row_of, int32_t* tok_of,
                              void* x_perm_bf16, int32_t* status_dev, moe_stream_t stream);

/* Step 4b, grouped SwiGLU experts: for each group g and each row r in
 * [group_offsets[g], group_offsets[g+1]):
 *   h[r]  = silu(a[r] . w1[g]^T) * (a[r] . w3[g]^T)      (bf16 [R, I], fp32 accumulate)
 *   y[r]  = h[r] . w2[g]^T                                (bf16 [R, d])
 * with silu(v) = v / (1 + exp(-v)).  a [R, d], w1/w3 [G, I, d], w2 [G, d, I],
 * all bf16.  group_offsets is a DEVICE array of G+1 non-decreasing row
 * offsets with group_offsets[G] <= R.  The routed experts use G = E with the
 * offsets of moe_permute; shared experts use G = 1, offsets {0, T}, a = x and
 * their weights side by side (width n_shared*I), which equals summing them.
 * Runs on the tensor cores (tcgen05, TMEM accumulators, TMA-fed). */
moe_status moe_grouped_swiglu(const void* a_bf16, const int32_t* group_offsets, int n_groups,
                              int R, int d, int I, const void* w1_bf16, const void* w3_bf16,
                              const void* w2_bf16, void* h_bf16, void* y_bf16,
                              int32_t* status_dev, moe_stream_t stream);

/* Box-contiguous copies of expert weights for moe_grouped_swiglu_tiled.  The
 * grouped GEMM stages its weights as boxes of 128 rows x 64 columns; in the
 * [rows, cols] layout above every box is 128 strided 128-byte pieces, in
 * these copies it is 16 KB of consecutive memory, which the GPU's memory
 * streams more efficiently.  Same values, rearranged (a one-time copy, like
 * moe_router_prepare; the method is unchanged):
 *  w13_tiled [G][I/64][d/64][128][64] bf16: box (g, t, kb) holds rows
 *    t*64 .. t*64+63 of w1[g] and of w3[g], alternating (box row 2i is w1
 *    row t*64+i, box row 2i+1 is w3 row t*64+i), columns kb*64 .. kb*64+63;
 *  w2_tiled  [G][d/128][I/64][128][64] bf16: box (g, t, kb) holds rows
 *    t*128 .. t*128+127 of w2[g], columns kb*64 .. kb*64+63.
 * w1, w3 [G, I, d] and w2 [G, d, I] as for moe_grouped_swiglu; either the
 * w1/w3/w13_tiled triple or the w2/w2_tiled pair may be all NULL to skip it.
 * d % 128 == 0 and I % 64 == 0, else MOE_ERR_UNSUPPORTED_SHAPE. */
moe_status moe_tile_expert_weights(const void* w1_bf16, const void* w3_bf16, const void* w2_bf16,
                                   int n_groups, int I, int d, void* w13_tiled_bf16,
                                   void* w2_tiled_bf16, moe_stream_t stream);

/* moe_grouped_swiglu on the box-contiguous weights of moe_tile_expert_weights:
 * the same kernels and the same arithmetic in the same order, so h and y are
 * bit-identical to moe_grouped_swiglu's on the same weights.  The alternating
 * w1/w3 rows put each output column's gate and up values in neighbouring
 * lanes of one epilogue warp, which finishes the SwiGLU with a register
 * shuffle instead of a shared-memory exchange between warps (faster where
 * the reduction is short: the mid layer's d = 2048).  Requires
 * d % 128 == 0 and I % 64 == 0.  Same expert FFN (weigao.cc notes, §2 table
 * row "DeepSeekMoE"). */
moe_status moe_grouped_swiglu_tiled(const void* a_bf16, const int32_t* group_offsets,
                                    int n_groups, int R, int d, int I, const void* w13_tiled_bf16,
                                    const void* w2_tiled_bf16, void* h_bf16, void* y_bf16,
                                    int32_t* status_dev, moe_stream_t stream);

/* The same call for a training step: also writes the pre-activations
 * pre_a[r] = a[r] . w1[g]^T and pre_c[r] = a[r] . w3[g]^T (bf16 [R, I] each),
 * which the backward pass needs (da = dh c silu'(a), dc = dh silu(a)), from
 * the GEMM's own fp32 accumulators. */
moe_status moe_grouped_swiglu_save(const void* a_bf16, const int32_t* group_offsets,
                                   int n_groups, int R, int d, int I, const void* w1_bf16,
                                   const void* w3_bf16, const void* w2_bf16, void* h_bf16,
                                   void* y_bf16, void* pre_a_bf16, void* pre_c_bf16,
                                   int32_t* status_dev, moe_stream_t stream);

/* Step 4c, combine:
 *   out[t] = bf16( y_shared[t] + sum_k topk_gate[t,k] * y_perm[row_of[t,k]] )
 * accumulated in fp32 in rank order (y_shared may be NULL).  Gather form:
 * no atomics, deterministic. */
moe_status moe_combine(const void* y_perm_bf16, const int32_t* row_of, const float* topk_gate,
                       const void* y_shared_bf16, int T, int K, int d, void* out_bf16,
                       moe_stream_t stream);

/* Serving-side redundant experts (host call, no device work).  The report's
 * prefill deployment keeps 32 redundant experts, re-placed from observed
 * load ("32个冗余专家", qwbw.cn essay on the report).  Plans n_redundant extra
 * copies from per-expert loads: slot e is expert e; slots E..E+n_redundant-1
 * are copies, each given in turn to the expert with the largest load per copy
 * (lower index on ties; this minimises the largest load per copy).
 *  load_host [E] int32 (host): observed loads.
 *  slot_start_host [E+1], slots_host [E+n_redundant] (host, out): CSR list of
 *    each expert's slots (its own slot first).
 *  expert_of_slot_host [E+n_redundant] (host, out): logical expert of each
 *    slot (copy weights accordingly). */
moe_status moe_replica_plan(const int32_t* load_host, int E, int n_redundant,
                            int32_t* slot_start_host, int32_t* slots_host,
                            int32_t* expert_of_slot_host);

/* Device remap to physical slots: entry (t, k) of logical expert e in [0, E)
 * becomes slots[slot_start[e] + t mod c_e] (c_e = copies of e); ids >= E
 * (shared experts in the serving layout) become id + n_redundant, so the
 * physical layout is [E experts][n_redundant copies][shared].  slot_start
 * and slots are DEVICE copies of the plan.  phys_idx [T, K] int32. */
moe_status moe_replica_remap(const int32_t* topk_idx, int T, int K, int E, int n_redundant,
                             const int32_t* slot_start, const int32_t* slots, int32_t* phys_idx,
                             moe_stream_t stream);

/* Forward value of the small sequence-wise balance loss kept next to the bias
 * feedback ("同时保留一个极小的序列级平衡损失", chenshi221 DeepSeek-V3 notes,
 * "Auxiliary-loss-free 负载均衡"; weigao.cc §3).  The pages print no formula;
 * the reading taken, per sequence of T_s tokens:
 *   f_i = E / (K T_s) * #{(t, k < K): topk_idx[t, k] = i}
 *   P_i = (1 / T_s) * sum_t scores[t, i] / sum_j scores[t, j]
 *   loss = alpha * sum_i f_i P_i
 *  scores [T, E] fp32 affinities (e.g. affinity_out of moe_router_topk);
 *  topk_idx [T, ldk] int32, first K columns used (ldk = K, or K + shared
 *  experts in the serving layout); seq_offsets [S+1] DEVICE int32 token
 *  ranges of the S sequences; loss_out [S] fp32.  Sums in a fixed order. */
moe_status moe_seq_balance_loss(const float* scores, const int32_t* topk_idx, int ldk,
                                const int32_t* seq_offsets, int S, int E, int K, float alpha,
                                float* loss_out, moe_stream_t stream);

/* ---------------------------------------------------------------- FP8 path
 * E4M3 expert GEMMs with fine-grained scaling: activations scaled per 1 x 128
 * tile, weights per 128 x 128 block, tensor-core partial sums promoted to
 * fp32 every 128 reduction elements (qwbw.cn essay on the report, the FP8
 * training passage; "DeepSeek-V3 Technical Report：中英对照解读", weigao.cc,
 * section "6. FP8 Training").  Gating, dispatch maps and the combine stay
 * those of the bf16 calls above.
 *
 * Quantization rule of every block: scale = fp32(amax / 448) with amax the
 * largest |value| of the block (NaN ignored), scale = 1 for an all-zero
 * block; code = E4M3 rounding (nearest, ties to even, saturating at +-448)
 * of fp32(value / scale).  Codes are E4M3 bytes (uint8).
 *
 * Activation scales are stored BLOCK-MAJOR: s[j * ld_s + row] is the scale
 * of columns j*128 .. j*128+127 of `row` (ld_s >= rows).
 * Shape limits: cols, d and I multiples of 128. */

/* Quantize bf16 rows [rows, cols] per 1 x 128 tile: q_out uint8 [rows, cols],
 * s_out fp32 [cols/128][ld_s]. */
moe_status moe_quantize_fp8(const void* x_bf16, int rows, int cols, void* q_out, float* s_out,
                            int ld_s, moe_stream_t stream);

/* Quantize weights bf16 [groups, rows, cols] per 128 x 128 block (rows and
 * cols multiples of 128).
 *  w_pair_bf16 == NULL: q_out uint8 [groups, rows, cols], s_out fp32
 *    [groups, rows/128, pitch] with pitch = round_up(cols/128, 4): scale of
 *    block (r, c) at [g, r, c] (the down projection w2, rows = d).
 *  w_pair_bf16 != NULL (a second matrix of the same shape): the two are
 *    written ROW-INTERLEAVED for the SwiGLU GEMM, q_out uint8
 *    [groups, 2*rows, cols] with row 2i = w_bf16 row i and row 2i+1 =
 *    w_pair_bf16 row i; s_out fp32 [groups, rows/128, pitch] with pitch =
 *    round_up(2*cols/128, 4): the two matrices' block scales side by side,
 *    block (r, c) of w_bf16 at [g, r, 2c], of w_pair_bf16 at [g, r, 2c+1].
 *    Pass w1 and w3.
 * Padding floats at the end of each scale row are not written.  The
 * quantized layout is what moe_grouped_swiglu_fp8 reads. */
moe_status moe_quantize_weights_fp8(const void* w_bf16, const void* w_pair_bf16, int groups,
                                    int rows, int cols, void* q_out, float* s_out,
                                    moe_stream_t stream);

/* Dispatch of quantized activations: q_perm[row_of[t,k]] = q_in[t] (d bytes
 * per row) and s_perm[j * ld_out + row_of[t,k]] = s_in[j * ld_in + t] for
 * every block j.  row_of [T, K] from moe_permute (x may be NULL there).
 * ld_in >= T, ld_out >= T*K. */
moe_status moe_permute_fp8(const void* q_in, const float* s_in, int ld_in, int T, int K, int d,
                           const int32_t* row_of, void* q_perm, float* s_perm, int ld_out,
                           moe_stream_t stream);

/* FP8 grouped SwiGLU experts: for group g (rows group_offsets[g] ..
 * group_offsets[g+1] of a):
 *   h = bf16(silu(a . w1[g]^T) * (a . w3[g]^T)),  h quantized per 1 x 128,
 *   y = bf16(h . w2[g]^T)
 * with every product an E4M3 GEMM promoted to fp32 per 128-deep block.
 *  a_q uint8 [R, d], a_s fp32 [d/128][ld_as] (ld_as >= R, ld_as % 4 == 0,
 *  so that rows of scales can be fetched by TMA);
 *  group_offsets [n_groups+1] DEVICE int32, 1 <= n_groups <= 512;
 *  w13_q / w13_s and w2_q / w2_s as written by moe_quantize_weights_fp8
 *  (w1 paired with w3; w2 alone, rows = d);
 *  h_bf16 [R, I] and h_q uint8 [R, I], h_s fp32 [I/128][round_up(R, 4)]:
 *  scratch that holds h (bf16 and quantized) on return; y_bf16 [R, d].
 * Shared experts: n_groups = 1, offsets {0, T}, I = n_shared * expert width. */
moe_status moe_grouped_swiglu_fp8(const void* a_q, const float* a_s, int ld_as,
                                  const int32_t* group_offsets, int n_groups, int R, int d, int I,
                                  const void* w13_q, const float* w13_s, const void* w2_q,
                                  const float* w2_s, void* h_bf16, void* h_q, float* h_s,
                                  void* y_bf16, int32_t* status_dev, moe_stream_t stream);

/* Failure detection self-test: one small kernel waits, with the bounded wait
 * every pipelined kernel here uses, on a barrier nothing arrives on.  After
 * limit_ns (1 us .. 1 s) it records MOE_DEV_TIMEOUT in status_dev (DEVICE,
 * OR-ed in) and returns; the context stays usable.  Lets a caller check that
 * a stalled pipeline surfaces as a status instead of a hang. */
moe_status moe_wait_selftest(long long limit_ns, int32_t* status_dev, moe_stream_t stream);

/* ---------------------------------------------------------- backward pass
 * Gradients of the layer output for a fixed choice of experts.  The bias only
 * chooses experts and never enters a gate value ("Bias 仅用于路由",
 * deepseekmodel1.org, "公式解密"; chenshi221 notes, "Auxiliary-loss-free
 * 负载均衡"), so the router receives gradient through the gates, which depend
 * on the raw affinities only, and the bias receives none:
 *   g_k = scale s_k / S (S = sum of the K chosen s_j),
 *   ds_k = scale (dg_k / S - sum_j dg_j s_j / S^2), du_k = ds_k s_k (1 - s_k).
 * Expert FFN y = W2 (silu(a) c), a = W1 v, c = W3 v:
 *   dh = W2^T dy, da = dh c silu'(a), dc = dh silu(a), dv = W1^T da + W3^T dc,
 *   dW2 = dy h^T, dW1 = da v^T, dW3 = dc v^T.
 * Reductions run in a fixed order (results are deterministic).  The weight
 * gradients are fp32; the activation gradients bf16. */

/* Combine backward: dy_perm[row_of[t,k]] = gate[t,k] dy[t] and
 * dgate[t,k] = <dy[t], y_perm[row_of[t,k]]> (fp32).
 *  dy, y_perm bf16 [T, d] / [T*K, d] (y_perm = the experts' outputs the forward
 *  combined); row_of [T, K]; gate fp32 [T, K]; dy_perm bf16 [T*K, d] out;
 *  dgate fp32 [T, K] out.  d % 8 == 0. */
moe_status moe_combine_backward(const void* dy_bf16, const void* y_perm_bf16,
                                const int32_t* row_of, const float* gate, int T, int K, int d,
                                void* dy_perm_bf16, float* dgate, moe_stream_t stream);

/* Elementwise SwiGLU backward per row: from dh, a = v.W1^T, c = v.W3^T
 * (bf16 [R, I] each) write dac = [da | dc] (bf16 [R, 2I]) and the recomputed
 * h = silu(a) c (bf16 [R, I]; NULL skips it).  I % 2 == 0. */
moe_status moe_swiglu_backward(const void* dh_bf16, const void* a_bf16, const void* c_bf16, int R,
                               int I, void* dac_bf16, void* h_bf16, moe_stream_t stream);

/* Grouped bf16 GEMM on the tensor cores: out[r] = a[r] . w[g]^T for the rows r
 * of group g (group_offsets [G+1] DEVICE).  a [R, K], w [G, N, K], out [R, N]
 * bf16; K % 64 == 0, N % 8 == 0, 1 <= G <= 512.  Recomputes a = v W1^T and
 * c = v W3^T in the backward pass. */
moe_status moe_grouped_gemm(const void* a_bf16, const int32_t* group_offsets, int n_groups, int R,
                            int K, int N, const void* w_bf16, void* out_bf16, int32_t* status_dev,
                            moe_stream_t stream);

/* Grouped data-gradient GEMM: out[r] = a[r] . w[g] for the rows r of group g,
 * the weights in their forward layout w [G, K, N] (N contiguous), or stacked
 * along K from two halves w0, w1 [G, K/2, N] each (w1 NULL: one part):
 * dh = (g dy) . W2 with W2 [E, d, I], and dv = [da | dc] . [W1 ; W3] with
 * W1, W3 [E, I, d].  a [R, K], out [R, N] bf16; each part's K % 64 == 0,
 * N % 8 == 0, 1 <= G <= 512. */
moe_status moe_grouped_gemm_kn(const void* a_bf16, const int32_t* group_offsets, int n_groups,
                               int R, int K, int N, const void* w0_bf16, const void* w1_bf16,
                               void* out_bf16, int32_t* status_dev, moe_stream_t stream);

/* Grouped weight-gradient GEMM: out[g][m][n] = sum over the rows r of group
 * g of A[r][m] B[r][n], fp32 [G, M, N], reading the dispatch-order buffers as
 * they are: A bf16 [R, M] (e.g. g dy or [da | dc]) and B bf16 [R, N] (h or
 * the dispatched tokens), groups by group_offsets [G+1] (DEVICE, as written
 * by moe_permute).  M % 8 == 0, N % 8 == 0.  A group with no rows gets zeros. */
moe_status moe_grouped_gemm_wgrad(const void* a_bf16, const void* b_bf16,
                                  const int32_t* group_offsets, int n_groups, int R, int M, int N,
                                  float* out, int32_t* status_dev, moe_stream_t stream);

/* Router backward (chosen experts only): du fp32 [T, K] from dgate [T, K],
 * the chosen experts topk_idx [T, ldk] (first K columns) and the forward's
 * affinities fp32 [T, E]; dx_router fp32 [T, d] = du . w_r (or NULL);
 * dw_r fp32 [E, d] = du^T x, summed per expert over its rows of the dispatch
 * order (row_of [T, K], tok_of [T*K], expert_offsets [E+1] from moe_permute).
 * du_row fp32 [T*K]: scratch.  x bf16 [T, d], w_r fp32 [E, d]; d % 8 == 0,
 * x and dw_r 16-byte aligned. */
moe_status moe_router_backward(const float* dgate, const int32_t* topk_idx, int ldk,
                               const float* affinity, const float* w_r, const void* x_bf16,
                               const int32_t* row_of, const int32_t* tok_of,
                               const int32_t* expert_offsets, int T, int d, int E, int K,
                               float route_scale, float* du, float* du_row, float* dx_router,
                               float* dw_r, moe_stream_t stream);

/* Input gradient: dx[t] = bf16( dx_shared[t] + dx_router[t] + sum_k
 * dx_perm[row_of[t,k]] ) with fp32 sums in rank order.  dx_perm bf16 [T*K, d];
 * dx_shared bf16 [T, d] or NULL; dx_router fp32 [T, d] or NULL; dx bf16 [T, d]. */
moe_status moe_combine_dx(const void* dx_perm_bf16, const int32_t* row_of, int K,
                          const void* dx_shared_bf16, const float* dx_router, int T, int d,
                          void* dx_bf16, moe_stream_t stream);

/* Step 5, bias feedback after the step:
 *   bias[e] = bias[e] - gamma  if E*load[e] > T*K   (overloaded)
 *   bias[e] = bias[e] + gamma  if E*load[e] < T*K   (underloaded)
 *   unchanged                  if equal
 * each one fp32 operation.  stats_out [4] fp32 (max load, mean load,
 * max/mean, coefficient of variation = population standard deviation over
 * the mean; all taken over the E experts, untouched ones as load 0; all 0
 * when no load was counted) or NULL. */
moe_status moe_bias_update(const int32_t* expert_load, float* bias, int T, int K, int E,
                           float gamma, float* stats_out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
