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
// The warp's top-k of one row of E <= 256 values, 8 per lane (lane + 32 i ->
// lv[i]; entries past E ignored): the same choices, weights and bits as the
// scan below, faster. Each lane sorts its 8 (key, expert) pairs once (a
// 19-comparator network, keys descending, lower expert first on equal
// keys), so a round is two warp reductions over the lanes' heads and a pop
// of the winner's head; the exponentials are taken after the rounds and
// summed in selection order, as the scan does.
__device__ __forceinline__ void topk_select8(const float (&lv)[8], int E, int k, int& idx,
                                             float& w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[8];
  int ix[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float l = lv[i];
    ix[i] = lane + 32 * i;
    // every real key is above 0: entries past E sort last and never win
    key[i] = ix[i] < E ? order_key(isnan(l) ? -INFINITY : l + 0.0f) : 0u;   // + 0: -0 -> +0
  }
  auto cswap = [&](int a, int b) {
    const bool sw = key[b] > key[a] || (key[b] == key[a] && ix[b] < ix[a]);
    const uint32_t ka = key[a], kb = key[b];
    const int ia = ix[a], ib = ix[b];
    key[a] = sw ? kb : ka;
    key[b] = sw ? ka : kb;
    ix[a] = sw ? ib : ia;
    ix[b] = sw ? ia : ib;
  };
  cswap(0, 2); cswap(1, 3); cswap(4, 6); cswap(5, 7);
  cswap(0, 4); cswap(1, 5); cswap(2, 6); cswap(3, 7);
  cswap(0, 1); cswap(2, 3); cswap(4, 5); cswap(6, 7);
  cswap(2, 4); cswap(3, 5);
  cswap(1, 4); cswap(3, 6);
  cswap(1, 2); cswap(3, 4); cswap(5, 6);
  uint32_t my_key = 0u;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t cand = (key[0] == m && key[0] != 0u) ? (uint32_t)ix[0] : 0xffffffffu;
    const int be = (int)__reduce_min_sync(0xffffffffu, cand);
    if (ix[0] == be) {   // this lane's head was taken: the next one moves up
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        key[i] = key[i + 1];
        ix[i] = ix[i + 1];
      }
      key[7] = 0u;
    }
    if (lane == j) {
      my_idx = be;
      my_key = m;
    }
  }
  const float v0 = key_value(__shfl_sync(0xffffffffu, my_key, 0));
  const float pj = lane < k ? expf(key_value(my_key) - v0) : 0.f;
  float zsum = 0.f;
  for (int j = 0; j < k; ++j) zsum += __shfl_sync(0xffffffffu, pj, j);
  idx = my_idx;
  w = pj / zsum;
}

// The warp's top-k of one row of E values, given as lane + 32 i -> lv[i]
// (entries past E ignored).
template <int VPL>   // values per lane, E <= 32 * VPL
__device__ __forceinline__ void topk_select(const float (&lv)[VPL], int E, int k, int& idx,
                                            float& w) {
  if constexpr (VPL == 8) {
    topk_select8(lv, E, k, idx, w);
    return;
  }
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
