// Internal launch interface between the C ABI (moe_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace moe {

int sm_count();  // SMs of the current device (cached per device)

// One-time set-up per device (a kernel attribute, a looked-up address, a
// device property), safe when several host threads make their first calls
// at the same time: the first caller on a device runs `init` under a lock
// and marks the device done only when `init` succeeded; later callers see
// the mark (acquire) without locking.  Devices beyond kMaxDevices run
// `init` on every call.
constexpr int kMaxDevices = 64;
struct DeviceOnce {
  std::atomic<bool> done[kMaxDevices] = {};
  std::mutex lock;
};
template <typename F>
cudaError_t once_per_device(DeviceOnce& once, int dev, F&& init) {
  if (dev < 0 || dev >= kMaxDevices) return init();
  if (once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> guard(once.lock);
  if (once.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = init();
  if (e == cudaSuccess) once.done[dev].store(true, std::memory_order_release);
  return e;
}

// ---- router selection (router_topk.cu)
struct TopkArgs {
  const float* scores;     // [T, E] affinities
  const float* bias;       // [E]
  int T, E, K, n_groups, topk_groups;
  float route_scale;
  int n_shared_routed;     // shared experts appended as ids E.. with gate 1 (0 = none)
  int32_t* idx;            // [T, K + n_shared_routed]
  float* gate;             // [T, K + n_shared_routed]
  int32_t* load;           // [E], zeroed before the launch
  int32_t* status;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);

// ---- router weight split (router_topk.cu)
cudaError_t launch_router_split(const float* w_r, int E, int d, uint16_t* w_split, cudaStream_t s);

// ---- permute (permute.cu)
constexpr int kPermuteTile = 1024;   // (token, slot) entries per counting tile
size_t permute_ws_bytes(int T, int K, int E);
// Fixed device scratch for the allocation-free permute: (T*K/1024 rounded up)
// x E counts of int32, at most this many.
constexpr size_t kPermuteStaticScratchInts = 65536;  // 256 KiB
cudaError_t permute_static_scratch(int32_t** ptr);
cudaError_t launch_permute(const int32_t* idx, int T, int K, int E, const uint16_t* x, int d,
                           int32_t* offsets, int32_t* row_of, int32_t* tok_of, uint16_t* x_perm,
                           int32_t* status, int32_t* tile_counts, cudaStream_t s);

// ---- combine + bias update (combine.cu)
cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* row_of, const float* gate,
                           const uint16_t* y_shared, int T, int K, int d, uint16_t* out,
                           cudaStream_t s);
cudaError_t launch_bias_update(const int32_t* load, float* bias, int T, int K, int E, float gamma,
                               float* stats, cudaStream_t s);

// ---- redundant expert copies (replicas.cu)
bool replica_plan(const int32_t* load, int E, int n_redundant, int32_t* slot_start, int32_t* slots,
                  int32_t* expert_of_slot);
cudaError_t launch_replica_remap(const int32_t* idx, int T, int K, int E, int n_redundant,
                                 const int32_t* slot_start, const int32_t* slots, int32_t* phys,
                                 cudaStream_t s);

// ---- sequence-wise balance loss (balance_loss.cu)
cudaError_t launch_seq_balance(const float* scores, const int32_t* idx, int ldk,
                               const int32_t* seq_offsets, int S, int E, int K, float alpha,
                               float* loss, cudaStream_t s);

// ---- tensor-core GEMMs (gemm_tc.cu)
// Router logits + sigmoid: s[t, e] = sigmoid(sum_j x[t,j] w[e,j] + o[e]) with
// w given as the exact bf16 split [E, 3d].
// Router GEMM; with `partial` (a caller scratch of partial_bytes) small batches
// split each tile's reduction over several CTAs (router_splits of them).
int router_splits(int T, int d, int E, int sms);
cudaError_t launch_router_gemm(const uint16_t* x, const uint16_t* w_split, const float* offset,
                               int T, int d, int E, float* scores, int32_t* status,
                               cudaStream_t s, float* partial = nullptr, size_t partial_bytes = 0);
// Grouped SwiGLU experts (GEMM1 + fused SwiGLU, then GEMM2).
cudaError_t launch_grouped_swiglu(const uint16_t* a, const int32_t* offsets, int G, int R, int d,
                                  int I, const uint16_t* w1, const uint16_t* w3,
                                  const uint16_t* w2, uint16_t* h, uint16_t* y, int32_t* status,
                                  cudaStream_t s, uint16_t* a_out = nullptr,
                                  uint16_t* c_out = nullptr);

// Box-contiguous expert weights and the grouped SwiGLU reading them.
cudaError_t launch_tile_expert_weights(const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                                       int G, int I, int d, uint16_t* w13_tiled,
                                       uint16_t* w2_tiled, cudaStream_t s);
cudaError_t launch_grouped_swiglu_tiled(const uint16_t* a, const int32_t* offsets, int G, int R,
                                        int d, int I, const uint16_t* w13_tiled,
                                        const uint16_t* w2_tiled, uint16_t* h, uint16_t* y,
                                        int32_t* status, cudaStream_t s);

// ---- FP8 path (quant_fp8.cu, gemm_fp8.cu)
cudaError_t launch_quantize_rows(const uint16_t* in, int rows, int cols, uint8_t* q, float* s,
                                 int ld_s, cudaStream_t st);
cudaError_t launch_quantize_blocks(const uint16_t* w, const uint16_t* w_pair, int groups, int rows,
                                   int cols, uint8_t* q, float* s, cudaStream_t st);
cudaError_t launch_permute_fp8(const uint8_t* q, const float* s, int ld_in, int T, int K, int d,
                               const int32_t* row_of, uint8_t* q_perm, float* s_perm, int ld_out,
                               cudaStream_t st);
cudaError_t launch_grouped_swiglu_fp8(const uint8_t* a_q, const float* a_s, int ld_as,
                                      const int32_t* offsets, int G, int R, int d, int I,
                                      const uint8_t* w13_q, const float* w13_s,
                                      const uint8_t* w2_q, const float* w2_s, uint16_t* h,
                                      uint8_t* h_q, float* h_s, uint16_t* y, int32_t* status,
                                      cudaStream_t s);

// Small-group orientation of the FP8 grouped experts (gemm_fp8_small.cu),
// chosen by launch_grouped_swiglu_fp8; the scale maps are the caller's.
cudaError_t launch_grouped_swiglu_fp8_small(const uint8_t* a_q, int ld_as, const int32_t* offsets,
                                            int G, int R, int d, int I, const uint8_t* w13_q,
                                            const uint8_t* w2_q, uint16_t* h, uint8_t* h_q,
                                            float* h_s, uint16_t* y, int32_t* status,
                                            const CUtensorMap& ta1, const CUtensorMap& ta2,
                                            const CUtensorMap& tsw13, const CUtensorMap& th1,
                                            const CUtensorMap& th2, const CUtensorMap& tsw2,
                                            cudaStream_t s);

// ---- self-test of the bounded device wait (selftest.cu)
cudaError_t launch_wait_selftest(unsigned long long limit_ns, int32_t* status, cudaStream_t s);

// ---- backward (backward.cu, gemm_wgrad.cu, gemm_tc.cu)
cudaError_t launch_grouped_gemm_kn(const uint16_t* a, const int32_t* offsets, int G, int R, int K,
                                   int N, const uint16_t* w0, int K0, const uint16_t* w1,
                                   uint16_t* out, int32_t* status, cudaStream_t s);
cudaError_t launch_grouped_gemm_nt(const uint16_t* a, const int32_t* offsets, int G, int R, int K,
                                   int N, const uint16_t* w, uint16_t* out, int32_t* status,
                                   cudaStream_t s);
cudaError_t launch_grouped_wgrad(const uint16_t* a, const uint16_t* b, const int32_t* offsets,
                                 int G, int R, int M, int N, float* out, int32_t* status,
                                 cudaStream_t s);
cudaError_t launch_combine_backward(const uint16_t* dy, const uint16_t* y_perm,
                                    const int32_t* row_of, const float* gate, int T, int K, int d,
                                    uint16_t* dy_perm, float* dgate, cudaStream_t s);
cudaError_t launch_swiglu_backward(const uint16_t* dh, const uint16_t* a, const uint16_t* c, int R,
                                   int I, uint16_t* dac, uint16_t* h, cudaStream_t s);
cudaError_t launch_router_backward(const float* dgate, const int32_t* idx, int ld_idx,
                                   const float* affinity, const float* w_r, const uint16_t* x,
                                   const int32_t* row_of, const int32_t* tok_of,
                                   const int32_t* offsets, int T, int d, int E, int K, float scale,
                                   float* du, float* du_row, float* dx_router, float* dw_r,
                                   cudaStream_t s);
cudaError_t launch_combine_dx(const uint16_t* dx_perm, const int32_t* row_of, int K,
                              const uint16_t* dx_shared, const float* dx_router, int T, int d,
                              uint16_t* dx, cudaStream_t s);


}  // namespace moe
