// Top-k softmax routing of one token by one warp: shared by the routing
// kernel and the single-launch decode layer, so that both give the same
// bits.
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Order used by the top-k: larger logit first, equal logits -> lower expert id
// first, NaN after every number (NaNs among themselves by id).  Each logit
// becomes one 64-bit key whose unsigned order is exactly that order: the high
// word is the value mapped to an order-preserving integer (-0 taken as +0,
// NaN -> 1, below -inf), the low word is ~id; 0 marks "taken / absent".
MOE_D uint64_t route_key(float v, int e) {
  uint32_t ord;
  if (v != v) {
    ord = 1u;
  } else {
    const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0
    ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return (static_cast<uint64_t>(ord) << 32) | (0xffffffffu - static_cast<uint32_t>(e));
}

MOE_D float route_key_value(uint64_t key) {
  const uint32_t ord = static_cast<uint32_t>(key >> 32);
  if (ord == 1u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

// The top-k of one token's E logits (row) by the calling warp.  Lane l holds
// the keys of experts l, l+32, ... in registers (NPL per lane, NPL*32 >= E)
// and its own best; every round takes the warp-wide maximum key (5 shuffle
// levels), and the owning lane retires that key and recomputes its best.
// Lane j < k returns slot j: its expert id and its weight
// w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0); the return value tells
// whether the row holds a NaN (every lane).
template <int NPL>
MOE_D bool route_token(const float* row, int E, int k, int lane, int& id, float& wt) {
  uint64_t key[NPL];
  bool any_nan = false;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    key[i] = 0;
    if (e < E) {
      const float v = __ldg(row + e);
      any_nan |= (v != v);
      key[i] = route_key(v, e);
    }
  }
  const bool nan = __any_sync(0xffffffffu, any_nan);
  uint64_t best = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) best = key[i] > best ? key[i] : best;
  uint64_t mine = 0;  // lane j keeps the key of slot j
  for (int j = 0; j < k; ++j) {
    uint64_t m = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, m, o);
      m = other > m ? other : m;
    }
    if (lane == j) mine = m;
    const int wid = static_cast<int>(0xffffffffu - static_cast<uint32_t>(m));
    if ((wid & 31) == lane) {  // retire the winner, recompute this lane's best
      const int slot = wid >> 5;
      best = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (i == slot) key[i] = 0;
        best = key[i] > best ? key[i] : best;
      }
    }
  }
  // softmax over the selected logits, relative to the largest (slot 0)
  float l = route_key_value(mine);
  l = (l != l) ? -INFINITY : l;
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  const float z = (lane < k) ? expf(l - l0) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);
  id = static_cast<int>(0xffffffffu - static_cast<uint32_t>(mine));
  wt = z / sum;
  return nan;
}

}  // namespace moe
