// C ABI of libmoe_b300.so (declared in include/moe.h): argument checks, the
// workspace layout, and the kernel launches of each step.
#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>

#include <nvtx3/nvToolsExt.h>
#include "internal.h"

namespace {
// An NVTX range around every entry point, named after it: a profiler shows
// which call each kernel belongs to; without one attached it costs a check.
struct Trace {
  explicit Trace(const char* name) { nvtxRangePushA(name); }
  ~Trace() { nvtxRangePop(); }
};
}  // namespace
#define MOE_TRACE() Trace moe_trace_(__func__)
#include "../../include/moe.h"

namespace moe {

int sm_count() {
  static DeviceOnce once;
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int n = 0;
  const cudaError_t e = once_per_device(once, dev, [&]() {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    if (dev >= 0 && dev < kMaxDevices) cached[dev] = n;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return 148;
  return (dev >= 0 && dev < kMaxDevices) ? cached[dev] : n;
}

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorInvalidValue) return MOE_ERR_INVALID_ARG;
  return MOE_ERR_CUDA;
}

// Workspace layout: [router scores T*E fp32][permute tile counts].
size_t ws_router_bytes(int T, int E) { return align_up(static_cast<size_t>(T) * E * sizeof(float)); }

// Scratch of the router GEMM's split reduction (small batches): at most
// splits * T * E floats with splits * ceil(T/128) * ceil(E/128) <= the SM
// count (bounded by 160 here) and splits <= the 4-k-block chunks of 3d.  It
// shares the workspace region after the scores with the permute's counts:
// the router's reduction is finished before the permute runs.
size_t ws_router_partial_bound(int T, int d, int E) {
  if (d < 64) return 0;
  const long long chunks = (3ll * d / 64 + 3) / 4;
  long long n = 160ll * 128 * 128;
  if (chunks * T * E < n) n = chunks * T * E;
  return align_up(static_cast<size_t>(n) * sizeof(float));
}

bool routing_shape_ok(int T, int E, int K, int G, int M) {
  if (T < 0 || E < 1 || E > 512 || K < 1 || K > E || K > 32) return false;
  if (G < 1 || M < 1 || M > G || E % G) return false;
  if (static_cast<long long>(T) * K >= (1ll << 31)) return false;
  if (G > 1) {
    const int vpl = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : 16;
    const int gsz = E / G;
    if (gsz % vpl) return false;
    const int lanes = gsz / vpl;
    if (lanes & (lanes - 1)) return false;
    const int n_top = (K + M - 1) / M;
    if (n_top > 4 || n_top > gsz || K > M * gsz) return false;
  }
  return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 1; }

size_t moe_workspace_bytes(int T, int d, int E, int K, int I) {
  (void)I;
  if (T < 0 || E < 1 || K < 1) return 0;
  const size_t perm = align_up(permute_ws_bytes(T, K, E));
  const size_t part = ws_router_partial_bound(T, d, E);
  return ws_router_bytes(T, E) + (perm > part ? perm : part);
}

int moe_router_splits(int T, int d, int E) {
  if (T < 1 || d < 64 || E < 1) return 1;
  return router_splits(T, d, E, sm_count());
}

moe_status moe_router_prepare(const float* w_r, int E, int d, void* w_split_bf16,
                              moe_stream_t stream) {
  MOE_TRACE();
  if (!w_r || !w_split_bf16 || E < 1 || d < 1) return MOE_ERR_INVALID_ARG;
  if (d % 64 || E > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_router_split(w_r, E, d, static_cast<uint16_t*>(w_split_bf16),
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_topk(const void* x_bf16, const void* w_split_bf16, const float* scores_in,
                           const float* logit_offset, const float* bias, int T, int d, int E,
                           int K, int n_groups, int topk_groups, float route_scale,
                           int n_shared_routed, int32_t* topk_idx, float* topk_gate,
                           int32_t* expert_load,
                           float* affinity_out, int32_t* status_dev, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
  MOE_TRACE();
  if (!bias || !expert_load || T < 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !topk_gate)) return MOE_ERR_INVALID_ARG;
  if (!routing_shape_ok(T, E, K, n_groups, topk_groups)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n_shared_routed < 0) return MOE_ERR_INVALID_ARG;
  if (K + n_shared_routed > 32 || E + n_shared_routed > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* scores = scores_in;
  if (x_bf16 != nullptr) {
    if (!w_split_bf16) return MOE_ERR_INVALID_ARG;
    if (d < 64 || d % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(w_split_bf16)) return MOE_ERR_UNSUPPORTED_SHAPE;
    float* buf = affinity_out;
    if (buf == nullptr) {
      if (!ws || ws_bytes < ws_router_bytes(T, E)) return MOE_ERR_WORKSPACE;
      buf = static_cast<float*>(ws);
    }
    // the split reduction's scratch follows the scores region (when the
    // workspace has room; otherwise the GEMM runs unsplit)
    float* partial = nullptr;
    size_t partial_bytes = 0;
    if (ws && ws_bytes > ws_router_bytes(T, E)) {
      partial = reinterpret_cast<float*>(static_cast<char*>(ws) + ws_router_bytes(T, E));
      partial_bytes = ws_bytes - ws_router_bytes(T, E);
    }
    const cudaError_t e = launch_router_gemm(static_cast<const uint16_t*>(x_bf16),
                                             static_cast<const uint16_t*>(w_split_bf16),
                                             logit_offset, T, d, E, buf, status_dev, s, partial,
                                             partial_bytes);
    if (e != cudaSuccess) return cuda_status(e);
    scores = buf;
  } else if (scores_in == nullptr && T > 0) {
    return MOE_ERR_INVALID_ARG;
  }
  TopkArgs a{};
  a.scores = scores;
  a.bias = bias;
  a.T = T;
  a.E = E;
  a.K = K;
  a.n_groups = n_groups;
  a.topk_groups = topk_groups;
  a.route_scale = route_scale;
  a.n_shared_routed = n_shared_routed;
  a.idx = topk_idx;
  a.gate = topk_gate;
  a.load = expert_load;
  a.status = status_dev;
  return cuda_status(launch_topk(a, s));
}

moe_status moe_permute(const int32_t* topk_idx, int T, int K, int E, const void* x_bf16, int d,
                       int32_t* expert_offsets, int32_t* row_of, int32_t* tok_of,
                       void* x_perm_bf16, int32_t* status_dev, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || E < 1 || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_of || !tok_of)) return MOE_ERR_INVALID_ARG;
  if (E > 512 || K > 32 || static_cast<long long>(T) * K >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (x_bf16 != nullptr) {
    if (!x_perm_bf16) return MOE_ERR_INVALID_ARG;
    if (d < 8 || d % 8 || !aligned16(x_bf16) || !aligned16(x_perm_bf16))
      return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  const size_t need = permute_ws_bytes(T, K, E);
  const size_t off = ws_router_bytes(T, E);
  if (T > 0 && (!ws || ws_bytes < off + need)) return MOE_ERR_WORKSPACE;
  int32_t* tile_counts =
      T > 0 ? reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off) : nullptr;
  return cuda_status(launch_permute(topk_idx, T, K, E, static_cast<const uint16_t*>(x_bf16), d,
                                    expert_offsets, row_of, tok_of,
                                    static_cast<uint16_t*>(x_perm_bf16), status_dev, tile_counts,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute_static(const int32_t* topk_idx, int T, int K, int E, const void* x_bf16,
                              int d, int32_t* expert_offsets, int32_t* row_of, int32_t* tok_of,
                              void* x_perm_bf16, int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || E < 1 || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_of || !tok_of)) return MOE_ERR_INVALID_ARG;
  if (E > 512 || K > 32 || static_cast<long long>(T) * K >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (x_bf16 != nullptr) {
    if (!x_perm_bf16) return MOE_ERR_INVALID_ARG;
    if (d < 8 || d % 8 || !aligned16(x_bf16) || !aligned16(x_perm_bf16))
      return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  if (permute_ws_bytes(T, K, E) > kPermuteStaticScratchInts * sizeof(int32_t))
    return MOE_ERR_SCRATCH_LIMIT;
  int32_t* scratch = nullptr;
  if (T > 0) {
    const cudaError_t e = permute_static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return cuda_status(launch_permute(topk_idx, T, K, E, static_cast<const uint16_t*>(x_bf16), d,
                                    expert_offsets, row_of, tok_of,
                                    static_cast<uint16_t*>(x_perm_bf16), status_dev, scratch,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_tile_expert_weights(const void* w1_bf16, const void* w3_bf16, const void* w2_bf16,
                                   int n_groups, int I, int d, void* w13_tiled_bf16,
                                   void* w2_tiled_bf16, moe_stream_t stream) {
  MOE_TRACE();
  if (n_groups < 1 || I < 1 || d < 1) return MOE_ERR_INVALID_ARG;
  const bool has13 = w1_bf16 || w3_bf16 || w13_tiled_bf16;
  const bool has2 = w2_bf16 || w2_tiled_bf16;
  if (!has13 && !has2) return MOE_ERR_INVALID_ARG;
  if (has13 && (!w1_bf16 || !w3_bf16 || !w13_tiled_bf16)) return MOE_ERR_INVALID_ARG;
  if (has2 && (!w2_bf16 || !w2_tiled_bf16)) return MOE_ERR_INVALID_ARG;
  if (d % 128 || I % 64 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  for (const void* q : {w1_bf16, w3_bf16, w2_bf16, static_cast<const void*>(w13_tiled_bf16),
                        static_cast<const void*>(w2_tiled_bf16)})
    if (q && !aligned16(q)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_tile_expert_weights(
      static_cast<const uint16_t*>(w1_bf16), static_cast<const uint16_t*>(w3_bf16),
      static_cast<const uint16_t*>(w2_bf16), n_groups, I, d, static_cast<uint16_t*>(w13_tiled_bf16),
      static_cast<uint16_t*>(w2_tiled_bf16), static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_swiglu_tiled(const void* a_bf16, const int32_t* group_offsets,
                                    int n_groups, int R, int d, int I, const void* w13_tiled_bf16,
                                    const void* w2_tiled_bf16, void* h_bf16, void* y_bf16,
                                    int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || d < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_bf16 || !group_offsets || !w13_tiled_bf16 || !w2_tiled_bf16 || !h_bf16 ||
                !y_bf16))
    return MOE_ERR_INVALID_ARG;
  if (d % 128 || I % 64 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_bf16) || !aligned16(w13_tiled_bf16) || !aligned16(w2_tiled_bf16) ||
                !aligned16(h_bf16) || !aligned16(y_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_swiglu_tiled(
      static_cast<const uint16_t*>(a_bf16), group_offsets, n_groups, R, d, I,
      static_cast<const uint16_t*>(w13_tiled_bf16), static_cast<const uint16_t*>(w2_tiled_bf16),
      static_cast<uint16_t*>(h_bf16), static_cast<uint16_t*>(y_bf16), status_dev,
      static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_swiglu(const void* a_bf16, const int32_t* group_offsets, int n_groups,
                              int R, int d, int I, const void* w1_bf16, const void* w3_bf16,
                              const void* w2_bf16, void* h_bf16, void* y_bf16,
                              int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || d < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_bf16 || !group_offsets || !w1_bf16 || !w3_bf16 || !w2_bf16 || !h_bf16 ||
                !y_bf16))
    return MOE_ERR_INVALID_ARG;
  if (d % 64 || I % 64 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_bf16) || !aligned16(w1_bf16) || !aligned16(w3_bf16) ||
                !aligned16(w2_bf16) || !aligned16(h_bf16) || !aligned16(y_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_swiglu(
      static_cast<const uint16_t*>(a_bf16), group_offsets, n_groups, R, d, I,
      static_cast<const uint16_t*>(w1_bf16), static_cast<const uint16_t*>(w3_bf16),
      static_cast<const uint16_t*>(w2_bf16), static_cast<uint16_t*>(h_bf16),
      static_cast<uint16_t*>(y_bf16), status_dev, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_swiglu_save(const void* a_bf16, const int32_t* group_offsets,
                                   int n_groups, int R, int d, int I, const void* w1_bf16,
                                   const void* w3_bf16, const void* w2_bf16, void* h_bf16,
                                   void* y_bf16, void* pre_a_bf16, void* pre_c_bf16,
                                   int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R > 0 && (!pre_a_bf16 || !pre_c_bf16)) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!aligned16(pre_a_bf16) || !aligned16(pre_c_bf16))) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R < 0 || n_groups < 1 || d < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_bf16 || !group_offsets || !w1_bf16 || !w3_bf16 || !w2_bf16 || !h_bf16 ||
                !y_bf16))
    return MOE_ERR_INVALID_ARG;
  if (d % 64 || I % 64 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_bf16) || !aligned16(w1_bf16) || !aligned16(w3_bf16) ||
                !aligned16(w2_bf16) || !aligned16(h_bf16) || !aligned16(y_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_swiglu(
      static_cast<const uint16_t*>(a_bf16), group_offsets, n_groups, R, d, I,
      static_cast<const uint16_t*>(w1_bf16), static_cast<const uint16_t*>(w3_bf16),
      static_cast<const uint16_t*>(w2_bf16), static_cast<uint16_t*>(h_bf16),
      static_cast<uint16_t*>(y_bf16), status_dev, static_cast<cudaStream_t>(stream),
      static_cast<uint16_t*>(pre_a_bf16), static_cast<uint16_t*>(pre_c_bf16)));
}

// ------------------------------------------------------------------ FP8 path
moe_status moe_quantize_fp8(const void* x_bf16, int rows, int cols, void* q_out, float* s_out,
                            int ld_s, moe_stream_t stream) {
  MOE_TRACE();
  if (rows < 0 || cols < 1 || ld_s < rows) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!x_bf16 || !q_out || !s_out)) return MOE_ERR_INVALID_ARG;
  if (cols % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0 && (!aligned16(x_bf16) || !aligned16(q_out) ||
                   (reinterpret_cast<uintptr_t>(s_out) & 3u)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_quantize_rows(static_cast<const uint16_t*>(x_bf16), rows, cols,
                                          static_cast<uint8_t*>(q_out), s_out, ld_s,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_weights_fp8(const void* w_bf16, const void* w_pair_bf16, int groups,
                                    int rows, int cols, void* q_out, float* s_out,
                                    moe_stream_t stream) {
  MOE_TRACE();
  if (groups < 0 || rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (groups > 0 && (!w_bf16 || !q_out || !s_out)) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (groups > 0 && (!aligned16(w_bf16) || !aligned16(q_out) ||
                     (w_pair_bf16 && !aligned16(w_pair_bf16)) ||
                     (reinterpret_cast<uintptr_t>(s_out) & 3u)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_quantize_blocks(
      static_cast<const uint16_t*>(w_bf16), static_cast<const uint16_t*>(w_pair_bf16), groups,
      rows, cols, static_cast<uint8_t*>(q_out), s_out, static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute_fp8(const void* q_in, const float* s_in, int ld_in, int T, int K, int d,
                           const int32_t* row_of, void* q_perm, float* s_perm, int ld_out,
                           moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || d < 1 || ld_in < T) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * K >= (1ll << 31) || static_cast<long long>(ld_out) < 1ll * T * K)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!q_in || !s_in || !row_of || !q_perm || !s_perm)) return MOE_ERR_INVALID_ARG;
  if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!aligned16(q_in) || !aligned16(q_perm))) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_permute_fp8(static_cast<const uint8_t*>(q_in), s_in, ld_in, T, K, d,
                                        row_of, static_cast<uint8_t*>(q_perm), s_perm, ld_out,
                                        static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_swiglu_fp8(const void* a_q, const float* a_s, int ld_as,
                                  const int32_t* group_offsets, int n_groups, int R, int d, int I,
                                  const void* w13_q, const float* w13_s, const void* w2_q,
                                  const float* w2_s, void* h_bf16, void* h_q, float* h_s,
                                  void* y_bf16, int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || d < 1 || I < 1 || ld_as < R) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_q || !a_s || !group_offsets || !w13_q || !w13_s || !w2_q || !w2_s ||
                !h_bf16 || !h_q || !h_s || !y_bf16))
    return MOE_ERR_INVALID_ARG;
  if (d % 128 || I % 128 || n_groups > 512 || ld_as % 4)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_q) || !aligned16(w13_q) || !aligned16(w2_q) || !aligned16(h_bf16) ||
                !aligned16(h_q) || !aligned16(y_bf16) || !aligned16(w13_s) ||
                !aligned16(w2_s) || !aligned16(a_s) || !aligned16(h_s)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_swiglu_fp8(
      static_cast<const uint8_t*>(a_q), a_s, ld_as, group_offsets, n_groups, R, d, I,
      static_cast<const uint8_t*>(w13_q), w13_s, static_cast<const uint8_t*>(w2_q), w2_s,
      static_cast<uint16_t*>(h_bf16), static_cast<uint8_t*>(h_q), h_s,
      static_cast<uint16_t*>(y_bf16), status_dev, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------ self-test
moe_status moe_wait_selftest(long long limit_ns, int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (!status_dev || limit_ns < 1000 || limit_ns > 1000000000ll) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_selftest(static_cast<unsigned long long>(limit_ns), status_dev,
                                          static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ backward
moe_status moe_combine_backward(const void* dy_bf16, const void* y_perm_bf16,
                                const int32_t* row_of, const float* gate, int T, int K, int d,
                                void* dy_perm_bf16, float* dgate, moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || K > 32 || d < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!dy_bf16 || !y_perm_bf16 || !row_of || !gate || !dy_perm_bf16 || !dgate))
    return MOE_ERR_INVALID_ARG;
  if (d % 8) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!aligned16(dy_bf16) || !aligned16(y_perm_bf16) || !aligned16(dy_perm_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_combine_backward(
      static_cast<const uint16_t*>(dy_bf16), static_cast<const uint16_t*>(y_perm_bf16), row_of,
      gate, T, K, d, static_cast<uint16_t*>(dy_perm_bf16), dgate, static_cast<cudaStream_t>(stream)));
}

moe_status moe_swiglu_backward(const void* dh_bf16, const void* a_bf16, const void* c_bf16, int R,
                               int I, void* dac_bf16, void* h_bf16, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || I < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!dh_bf16 || !a_bf16 || !c_bf16 || !dac_bf16)) return MOE_ERR_INVALID_ARG;
  if (I % 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && ((reinterpret_cast<uintptr_t>(dh_bf16) | reinterpret_cast<uintptr_t>(a_bf16) |
                 reinterpret_cast<uintptr_t>(c_bf16) | reinterpret_cast<uintptr_t>(dac_bf16) |
                 reinterpret_cast<uintptr_t>(h_bf16)) & 3u))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_swiglu_backward(
      static_cast<const uint16_t*>(dh_bf16), static_cast<const uint16_t*>(a_bf16),
      static_cast<const uint16_t*>(c_bf16), R, I, static_cast<uint16_t*>(dac_bf16),
      static_cast<uint16_t*>(h_bf16), static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm(const void* a_bf16, const int32_t* group_offsets, int n_groups, int R,
                            int K, int N, const void* w_bf16, void* out_bf16, int32_t* status_dev,
                            moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_bf16 || !group_offsets || !w_bf16 || !out_bf16)) return MOE_ERR_INVALID_ARG;
  if (K % 64 || N % 8 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_bf16) || !aligned16(w_bf16) || !aligned16(out_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_gemm_nt(
      static_cast<const uint16_t*>(a_bf16), group_offsets, n_groups, R, K, N,
      static_cast<const uint16_t*>(w_bf16), static_cast<uint16_t*>(out_bf16), status_dev,
      static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm_kn(const void* a_bf16, const int32_t* group_offsets, int n_groups,
                               int R, int K, int N, const void* w0_bf16, const void* w1_bf16,
                               void* out_bf16, int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!a_bf16 || !group_offsets || !w0_bf16 || !out_bf16)) return MOE_ERR_INVALID_ARG;
  const int K0 = w1_bf16 ? K / 2 : K;
  if (K0 % 64 || (w1_bf16 && K % 128) || N % 8 || n_groups > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R > 0 && (!aligned16(a_bf16) || !aligned16(w0_bf16) || !aligned16(out_bf16) ||
                (w1_bf16 && !aligned16(w1_bf16))))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_grouped_gemm_kn(
      static_cast<const uint16_t*>(a_bf16), group_offsets, n_groups, R, K, N,
      static_cast<const uint16_t*>(w0_bf16), K0, static_cast<const uint16_t*>(w1_bf16),
      static_cast<uint16_t*>(out_bf16), status_dev, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm_wgrad(const void* a_bf16, const void* b_bf16,
                                  const int32_t* group_offsets, int n_groups, int R, int M, int N,
                                  float* out, int32_t* status_dev, moe_stream_t stream) {
  MOE_TRACE();
  if (R < 0 || n_groups < 1 || M < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  if (!group_offsets || !out || (R > 0 && (!a_bf16 || !b_bf16))) return MOE_ERR_INVALID_ARG;
  if (M % 8 || N % 8 || n_groups > 65535) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(out) || (R > 0 && (!aligned16(a_bf16) || !aligned16(b_bf16))))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  // with no rows the maps still need a valid address: the output stands in
  const void* a = R > 0 ? a_bf16 : out;
  const void* b = R > 0 ? b_bf16 : out;
  return cuda_status(launch_grouped_wgrad(static_cast<const uint16_t*>(a),
                                          static_cast<const uint16_t*>(b), group_offsets, n_groups,
                                          R, M, N, out, status_dev,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_backward(const float* dgate, const int32_t* topk_idx, int ldk,
                               const float* affinity, const float* w_r, const void* x_bf16,
                               const int32_t* row_of, const int32_t* tok_of,
                               const int32_t* expert_offsets, int T, int d, int E, int K,
                               float route_scale, float* du, float* du_row, float* dx_router,
                               float* dw_r, moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || d < 1 || E < 1 || K < 1 || K > 32 || K > E || ldk < K) return MOE_ERR_INVALID_ARG;
  if (!dw_r || (T > 0 && (!dgate || !topk_idx || !affinity || !w_r || !x_bf16 || !row_of ||
                          !tok_of || !expert_offsets || !du || !du_row)))
    return MOE_ERR_INVALID_ARG;
  if (E > 65535 || d % 8 || !aligned16(dw_r) || (T > 0 && !aligned16(x_bf16)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_router_backward(
      dgate, topk_idx, ldk, affinity, w_r, static_cast<const uint16_t*>(x_bf16), row_of, tok_of,
      expert_offsets, T, d, E, K, route_scale, du, du_row, dx_router, dw_r,
      static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_dx(const void* dx_perm_bf16, const int32_t* row_of, int K,
                          const void* dx_shared_bf16, const float* dx_router, int T, int d,
                          void* dx_bf16, moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || d < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!dx_perm_bf16 || !row_of || !dx_bf16)) return MOE_ERR_INVALID_ARG;
  if (d % 8) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!aligned16(dx_perm_bf16) || !aligned16(dx_bf16) ||
                (dx_shared_bf16 && !aligned16(dx_shared_bf16)) || (dx_router && !aligned16(dx_router))))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_combine_dx(static_cast<const uint16_t*>(dx_perm_bf16), row_of, K,
                                       static_cast<const uint16_t*>(dx_shared_bf16), dx_router, T, d,
                                       static_cast<uint16_t*>(dx_bf16),
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_replica_plan(const int32_t* load_host, int E, int n_redundant,
                            int32_t* slot_start_host, int32_t* slots_host,
                            int32_t* expert_of_slot_host) {
  MOE_TRACE();
  if (!load_host || !slot_start_host || !slots_host || !expert_of_slot_host || E < 1 ||
      n_redundant < 0)
    return MOE_ERR_INVALID_ARG;
  if (E + n_redundant > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  return replica_plan(load_host, E, n_redundant, slot_start_host, slots_host, expert_of_slot_host)
             ? MOE_OK
             : MOE_ERR_INVALID_ARG;
}

moe_status moe_replica_remap(const int32_t* topk_idx, int T, int K, int E, int n_redundant,
                             const int32_t* slot_start, const int32_t* slots, int32_t* phys_idx,
                             moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || E < 1 || n_redundant < 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !slot_start || !slots || !phys_idx)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_replica_remap(topk_idx, T, K, E, n_redundant, slot_start, slots,
                                          phys_idx, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const void* y_perm_bf16, const int32_t* row_of, const float* topk_gate,
                       const void* y_shared_bf16, int T, int K, int d, void* out_bf16,
                       moe_stream_t stream) {
  MOE_TRACE();
  if (T < 0 || K < 1 || d < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!y_perm_bf16 || !row_of || !topk_gate || !out_bf16)) return MOE_ERR_INVALID_ARG;
  if (d % 8 || K > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!aligned16(y_perm_bf16) || !aligned16(out_bf16) ||
                (y_shared_bf16 && !aligned16(y_shared_bf16))))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_combine(static_cast<const uint16_t*>(y_perm_bf16), row_of, topk_gate,
                                    static_cast<const uint16_t*>(y_shared_bf16), T, K, d,
                                    static_cast<uint16_t*>(out_bf16),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_seq_balance_loss(const float* scores, const int32_t* topk_idx, int ldk,
                                const int32_t* seq_offsets, int S, int E, int K, float alpha,
                                float* loss_out, moe_stream_t stream) {
  MOE_TRACE();
  if (S < 0 || E < 1 || K < 1 || ldk < K) return MOE_ERR_INVALID_ARG;
  if (S > 0 && (!scores || !topk_idx || !seq_offsets || !loss_out)) return MOE_ERR_INVALID_ARG;
  if (E > 512 || K > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_seq_balance(scores, topk_idx, ldk, seq_offsets, S, E, K, alpha,
                                        loss_out, static_cast<cudaStream_t>(stream)));
}

moe_status moe_bias_update(const int32_t* expert_load, float* bias, int T, int K, int E,
                           float gamma, float* stats_out, moe_stream_t stream) {
  MOE_TRACE();
  if (!expert_load || !bias || T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_bias_update(expert_load, bias, T, K, E, gamma, stats_out,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
