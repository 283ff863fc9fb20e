// Per-row pieces shared by the fixed-order dq passes that stream K/V (and, at
// D = 512, Q / dO) through a chunk ring: forming dS from S and dP in tensor
// memory, and writing dQ columns from tensor memory to the dq rows.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pipeline.cuh"

namespace bd {

// dS of this thread's q row over one 128-key tile, pre-scaled:
//   P  = 2^(scale log2(e) s - lse log2(e)) on the allowed keys [a_lo, e_hi]
//        (all of them when `full`, none when `dead`),
//   dS = P (scale dP - scale delta),
// as bf16 pairs (keys 2e, 2e + 1 of half hf in pk[hf][e]). t_s / t_dp: the
// row's S and dP columns in tensor memory (128 each); nl2 = -lse log2(e),
// ndl = -scale delta. With attention dropout (kDrop), key c's dP counts only
// when bit c of km is set and is scaled by drop_scale: dS = P (Z dP - delta).
template <bool kDrop = false>
__device__ __forceinline__ void dq_form_ds(uint32_t t_s, uint32_t t_dp, float scale, float nl2, float ndl,
                                           bool dead, bool full, int a_lo, int e_hi, uint32_t (&pk)[2][32],
                                           const uint32_t (&km)[4] = {0u, 0u, 0u, 0u}, float drop_scale = 1.0f) {
  const float2 sl2 = make_float2(scale * 1.4426950408889634f, scale * 1.4426950408889634f);
  const float scd = kDrop ? scale * drop_scale : scale;
  const float2 sc = make_float2(scd, scd), nl2v = make_float2(nl2, nl2), ndlv = make_float2(ndl, ndl);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t sr[64], dr[64];
    tmem_ld32(t_s + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_ld32(t_s + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_ld32(t_dp + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
    tmem_ld32(t_dp + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
    tmem_wait_ld();
    tmem_regs_ready<64>(sr);
    tmem_regs_ready<64>(dr);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = 64 * hf + 2 * e;
      const float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), sl2, nl2v);
      float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
      if (dead) {
        p0 = 0.f;
        p1 = 0.f;
      } else if (!full) {
        p0 = (c >= a_lo && c <= e_hi) ? p0 : 0.f;
        p1 = (c + 1 >= a_lo && c + 1 <= e_hi) ? p1 : 0.f;
      }
      float dp0 = __uint_as_float(dr[2 * e]), dp1 = __uint_as_float(dr[2 * e + 1]);
      if constexpr (kDrop) {
        const uint32_t kb = km[c >> 5] >> (c & 31);
        dp0 = (kb & 1u) ? dp0 : 0.f;
        dp1 = (kb & 2u) ? dp1 : 0.f;
      }
      const float2 d = __ffma2_rn(make_float2(dp0, dp1), sc, ndlv);
      const float2 ds = __fmul2_rn(make_float2(p0, p1), d);
      pk[hf][e] = pack_bf16x2(ds.x, ds.y);
    }
  }
}

// Columns [0, ncols) of this thread's dQ row in tensor memory (from t_dq) into
// dq at element `elem_off` (fp32 or bf16); `store` false: read only (the
// tensor-memory loads are warp-collective).
__device__ __forceinline__ void dq_store_cols(uint32_t t_dq, int ncols, void* dq, size_t elem_off, int dq_bf16,
                                              bool store) {
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t o[32];
    tmem_ld32(t_dq + c, o);
    tmem_wait_ld();
    if (!store) continue;
    if (dq_bf16) {
      uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dq) + elem_off + c);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        d4[e] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * e]), __uint_as_float(o[8 * e + 1])),
                           pack_bf16x2(__uint_as_float(o[8 * e + 2]), __uint_as_float(o[8 * e + 3])),
                           pack_bf16x2(__uint_as_float(o[8 * e + 4]), __uint_as_float(o[8 * e + 5])),
                           pack_bf16x2(__uint_as_float(o[8 * e + 6]), __uint_as_float(o[8 * e + 7])));
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(dq) + elem_off + c);
#pragma unroll
      for (int e = 0; e < 8; ++e) d4[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
    }
  }
}

}  // namespace bd
