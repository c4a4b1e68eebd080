// Serving-side redundant experts.  The report's prefill deployment keeps 32
// redundant experts and re-places them periodically from observed load
// statistics ("32个冗余专家", qwbw.cn essay on the report; weigao.cc
// "DeepSeek-V3 Technical Report：中英对照解读", §7 deployment notes).
//
// A plan gives every logical expert one or more physical slots: slot e is
// expert e itself, slots E .. E+n_redundant-1 are extra copies.  Extra copies
// go, one at a time, to the expert whose load per copy is currently the
// largest (lower expert index on ties), which minimises the largest load per
// copy.  The remap sends (token t, slot k) of logical expert e to copy
// t mod c_e of e, so every copy of a hot expert takes an equal share of its
// tokens and the layer's result is unchanged (copies hold identical weights).
#include <cuda_runtime.h>
#include <cstdint>
#include <vector>

#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) remap_kernel(const int32_t* __restrict__ idx, int T, int K,
                                                    int E, int n_redundant,
                                                    const int32_t* __restrict__ slot_start,
                                                    const int32_t* __restrict__ slots,
                                                    int32_t* __restrict__ phys) {
  const long long n = static_cast<long long>(T) * K;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = idx[i];
    int out;
    if (e >= 0 && e < E) {
      const int s0 = slot_start[e], c = slot_start[e + 1] - s0;
      const int t = static_cast<int>(i / K);
      out = c > 0 ? slots[s0 + t % c] : e;
    } else {
      out = e >= E ? e + n_redundant : e;  // ids past the routed experts keep their place after the copies
    }
    phys[i] = out;
  }
}

}  // namespace

bool replica_plan(const int32_t* load, int E, int n_redundant, int32_t* slot_start, int32_t* slots,
                  int32_t* expert_of_slot) {
  if (E < 1 || n_redundant < 0) return false;
  std::vector<long long> copies(E, 1);
  std::vector<int32_t> extra_of(n_redundant);
  for (int r = 0; r < n_redundant; ++r) {
    int best = 0;
    for (int e = 1; e < E; ++e) {
      // load[e] / copies[e] > load[best] / copies[best], exactly in integers
      const long long lhs = static_cast<long long>(load[e] < 0 ? 0 : load[e]) * copies[best];
      const long long rhs = static_cast<long long>(load[best] < 0 ? 0 : load[best]) * copies[e];
      if (lhs > rhs) best = e;
    }
    copies[best] += 1;
    extra_of[r] = best;
  }
  int pos = 0;
  for (int e = 0; e < E; ++e) {
    slot_start[e] = pos;
    slots[pos++] = e;
    for (int r = 0; r < n_redundant; ++r)
      if (extra_of[r] == e) slots[pos++] = E + r;
  }
  slot_start[E] = pos;
  for (int s = 0; s < E; ++s) expert_of_slot[s] = s;
  for (int r = 0; r < n_redundant; ++r) expert_of_slot[E + r] = extra_of[r];
  return true;
}

cudaError_t launch_replica_remap(const int32_t* idx, int T, int K, int E, int n_redundant,
                                 const int32_t* slot_start, const int32_t* slots, int32_t* phys,
                                 cudaStream_t s) {
  const long long n = static_cast<long long>(T) * K;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  remap_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(idx, T, K, E, n_redundant, slot_start,
                                                          slots, phys);
  return cudaGetLastError();
}

}  // namespace moe
