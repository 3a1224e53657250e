// One row of a 128-key score tile, prepared for the online-softmax step of
// "MiniPaged-Qwen: Qwen3 Prefill FlashAttention" section 4 in the exp2 form
// of "NVIDIA闪存注意力实操" section "在线Softmax算法" (scores in log2 units,
// log2(e) folded into the scale). Both attention kernels use it.
//
// The scale may be any nonzero finite number here (a zero scale reaches the
// kernels as scale 1 with Q read as zeros, which gives the same scores). The
// row maximum of the scaled scores is what the recurrence needs; for a
// negative scale it is the scale times the smallest raw score.
#pragma once

#include "ptx_sm103.cuh"

namespace fa {

// s: the row's 128 raw scores q.k (fp32, straight from Q K^T).
// sl2: softmax scale * log2(e), nonzero.
// masked: some key of this tile is hidden from this row (warp-uniform);
// lim: keys c < lim are visible (used only when masked).
//
// Hidden keys get the raw score that ranks below every other one under the
// scale's sign (-inf for sl2 > 0, +inf for sl2 < 0), so that their exponent
// s * sl2 - m is -inf and their weight 0. Returns the raw score x whose
// scaled value x * sl2 is the row's largest in this tile: max(s) for
// sl2 > 0, min(s) for sl2 < 0 (x * sl2 = -inf when no key is visible).
__device__ __forceinline__ float prepare_row(float (&s)[128], bool masked, int lim, float sl2) {
  const bool pos = sl2 > 0.0f;
  if (masked) {
    const float hide = pos ? -__int_as_float(0x7f800000) : __int_as_float(0x7f800000);
#pragma unroll
    for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : hide;
  }
  // eight independent chains of three-input max (or min)
  float mq[8];
  if (pos) {
#pragma unroll
    for (int q = 0; q < 8; ++q) mq[q] = fmaxf(s[2 * q], s[2 * q + 1]);   // columns 0 .. 15
#pragma unroll
    for (int c = 16; c < 128; c += 16) {
#pragma unroll
      for (int q = 0; q < 8; ++q) mq[q] = ptx::max3(mq[q], s[c + 2 * q], s[c + 2 * q + 1]);
    }
    return ptx::max3(ptx::max3(mq[0], mq[1], mq[2]), ptx::max3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) mq[q] = fminf(s[2 * q], s[2 * q + 1]);
#pragma unroll
  for (int c = 16; c < 128; c += 16) {
#pragma unroll
    for (int q = 0; q < 8; ++q) mq[q] = ptx::min3(mq[q], s[c + 2 * q], s[c + 2 * q + 1]);
  }
  return ptx::min3(ptx::min3(mq[0], mq[1], mq[2]), ptx::min3(mq[3], mq[4], mq[5]), fminf(mq[6], mq[7]));
}

}  // namespace fa
