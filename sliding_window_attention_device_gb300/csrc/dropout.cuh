// Attention dropout: the keep decisions of every (query head, query position,
// key position) pair, drawn on the device.
//
// blockdiag_cp.kernels `_cp_blockdiag_varlen` (and the FlashAttention varlen
// helpers of gemma4_moe.cp_attention) take `dropout_p`, the chance that an
// attention weight is dropped. It acts on the softmax probabilities P: a
// weight is kept with probability 1 - p and then scaled by the inverse of that
// probability (inverted dropout), so the forward output is sum_s P_ps Z_ps v_s
// with Z in {0, scale}; the softmax normaliser and the LSE stay the undropped
// ones.
//
// The random bits come from Philox-4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), a counter-based
// generator, so any kernel can draw any pair's decision without state:
//   counter = (s / 8, p, h, b), key = (seed_lo, seed_hi), with global
//   positions p (query) and s (key), query head h and batch row b;
//   the 128-bit output holds eight 16-bit draws u, key s taking piece s mod 8
//   (word (s mod 8) / 2, low half for even s, high half for odd s);
//   kept iff u >= T, T = round(p * 2^16); scale = 2^16 / (2^16 - T).
// One call therefore covers eight consecutive keys of one query row. Threads
// that own a query row (forward, fixed-order dq pass) draw their own rows;
// threads that own a key row (backward main kernels) share each call among
// the eight lanes whose keys it covers, through warp shuffles.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace bd {

// Philox-4x32 with ten rounds: each round multiplies words 0 and 2 by the
// round multipliers (full 64-bit products), mixes the high halves with words
// 1 and 3 and the key; the key advances by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(x0, x1, x2, x3);
}

// Keep bits of the eight keys 8k .. 8k+7 of one query row: bit e set iff the
// 16-bit draw of key 8k+e is >= t (a draw's high half >= t iff the word is
// >= t << 16).
__device__ __forceinline__ uint32_t keep_byte(const uint4 r, uint32_t t) {
  const uint32_t th = t << 16;
  return ((r.x & 0xFFFFu) >= t ? 1u : 0u) | (r.x >= th ? 2u : 0u) | ((r.y & 0xFFFFu) >= t ? 4u : 0u) |
         (r.y >= th ? 8u : 0u) | ((r.z & 0xFFFFu) >= t ? 16u : 0u) | (r.z >= th ? 32u : 0u) |
         ((r.w & 0xFFFFu) >= t ? 64u : 0u) | (r.w >= th ? 128u : 0u);
}

// Keep mask of one query row (global position p, head h, batch row b) over
// the 128 keys s0 .. s0+127: bit c of m[c / 32] is the decision of key s0 + c.
// The keys span 16 Philox calls, 17 when s0 is not a multiple of 8.
__device__ __forceinline__ void row_keep_mask(const Geom& g, int b, int h, int p, int s0, uint32_t (&m)[4]) {
  const uint32_t g0 = static_cast<uint32_t>(s0) >> 3, sh = static_cast<uint32_t>(s0) & 7u;
  uint32_t w[5] = {0u, 0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 17; ++i) {
    if (i < 16 || sh != 0) {
      const uint4 r = philox4x32_10(g0 + i, static_cast<uint32_t>(p), static_cast<uint32_t>(h),
                                    static_cast<uint32_t>(b), g.seed_lo, g.seed_hi);
      w[i >> 2] |= keep_byte(r, g.drop_t) << (8 * (i & 3));
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) m[k] = __funnelshift_r(w[k], w[k + 1], sh);
}

// Keep mask of this lane's key over the query rows p0 .. p0 + 8*NB - 1: bit c
// is the decision of (p0 + c, key). Every lane of the warp calls it together
// with the same p0, h, b; lane l's key is s_w + l (consecutive keys). The
// warp's 32 keys lie in 4 or 5 groups of eight; per batch of eight rows, lane
// L draws group G0 + (L mod 4) of row L / 4 and, when a fifth group exists,
// lanes L = 0 mod 4 also draw it; each lane then takes its bit from the lane
// that drew its (row, group).
template <int NB>
__device__ __forceinline__ uint64_t key_keep_mask(const Geom& g, int b, int h, int p0, int s_w, int lane) {
  const uint32_t G0 = static_cast<uint32_t>(s_w) >> 3;
  const bool five = (((static_cast<uint32_t>(s_w) + 31u) >> 3) - G0) == 4u;
  const uint32_t s = static_cast<uint32_t>(s_w + lane);
  const uint32_t gi = (s >> 3) - G0;                      // 0..4
  const int src = gi < 4u ? static_cast<int>(gi) : 0;     // lane offset of the drawer within a row's four
  const uint32_t bit = (gi < 4u ? 0u : 8u) + (s & 7u);    // bit of the drawn pair of bytes
  uint64_t mask = 0;
#pragma unroll
  for (int j0 = 0; j0 < 8 * NB; j0 += 8) {
    const uint32_t pp = static_cast<uint32_t>(p0 + j0 + (lane >> 2));
    uint32_t ab = keep_byte(philox4x32_10(G0 + (lane & 3), pp, static_cast<uint32_t>(h), static_cast<uint32_t>(b),
                                          g.seed_lo, g.seed_hi),
                            g.drop_t);
    if (five && (lane & 3) == 0)
      ab |= keep_byte(philox4x32_10(G0 + 4u, pp, static_cast<uint32_t>(h), static_cast<uint32_t>(b), g.seed_lo,
                                    g.seed_hi),
                      g.drop_t)
            << 8;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const uint32_t v = __shfl_sync(0xffffffffu, ab, 4 * jj + src);
      mask |= static_cast<uint64_t>((v >> bit) & 1u) << (j0 + jj);
    }
  }
  return mask;
}

}  // namespace bd
