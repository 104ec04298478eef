// topk.cuh -- one token's top-k selection by one warp (router logits ->
// expert indices and renormalised softmax weights), shared by the routing
// kernels and the fused decode layer.
//
// The router of "Perplexity libera Lily, un motor de IA que supera a MLX-LM
// en Apple Silicon" (diariobitcoin.com), section "Qwen3.6 combina tres
// cargas de trabajo", scores every expert and keeps k of them per token.
// Ties go to the lower expert index, a NaN logit ranks as -infinity, -0
// ranks equal to +0; the weights are the softmax over the selected logits
// (equal to the softmax over all experts renormalised over the k).
#pragma once

#include "moe_common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t order_key(float f) {   // monotone float -> uint32
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One token's selection by one warp, from its logits row (read through L2:
// the row may have been written by other CTAs of the same launch). Lane j < k
// gets the j-th selected expert and its renormalised softmax weight.
// The warp's top-k of one row of E values, given as lane + 32 i -> lv[i]
// (entries past E ignored).
template <int VPL>   // values per lane, E <= 32 * VPL
__device__ __forceinline__ void topk_select(const float (&lv)[VPL], int E, int k, int& idx,
                                            float& w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const float l = lv[i];
    key[i] = order_key(isnan(l) ? -INFINITY : l + 0.0f);   // + 0 turns -0 into +0
  }
  uint32_t live = 0;   // bit i: lane's value i not selected yet and e < E
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) live |= 1u << i;
  float sel_v0 = 0.f, zsum = 0.f, my_val = 0.f;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best live value (lowest i, i.e. lowest expert, on ties)
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (((live >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
      }
    // every real key is above 0, so a lane with nothing live never wins
    const uint32_t m = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == m) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
    const int be = (int)__reduce_min_sync(0xffffffffu, cand);
    if ((be & 31) == lane) live &= ~(1u << (be >> 5));
    const float bv = key_value(m);
    if (j == 0) sel_v0 = bv;
    const float pj = expf(bv - sel_v0);
    zsum += pj;
    if (lane == j) {
      my_idx = be;
      my_val = pj;
    }
  }
  idx = my_idx;
  w = my_val / zsum;
}

template <int VPL>   // values per lane, E <= 32 * VPL
__device__ __forceinline__ void topk_warp(const float* __restrict__ row, int E, int k,
                                          int& idx, float& w) {
  const int lane = threadIdx.x & 31;
  float lv[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    lv[i] = e < E ? __ldcg(row + e) : -INFINITY;
  }
  topk_select<VPL>(lv, E, k, idx, w);
}

}  // namespace moe
