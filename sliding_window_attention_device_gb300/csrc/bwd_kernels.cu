// K4a / K4 / K4b: backward of per-document causal attention for one CP shard.
//
// Reference (NeMo AutoModel API): gemma4_moe.cp_local_ring
// `sliding_ring_compute_fa_bwd` -- backward from the saved out / LSE with no
// forward recompute; blockdiag_cp.exchange `_AllGatherSeqDiff` -- a K/V
// position's gradient is the sum of every query's contribution. With
// P = exp(scale q.k - lse) on allowed pairs, delta = rowsum(dout * out):
//   dV += P^T dO,  dP = dO V^T,  dS = P (dP - delta),
//   dK += scale dS^T Q,  dQ += scale dS K,
// dK / dV summed over the Hq/Hkv query heads of a group.
//
// K4 design (GB300): one CTA per (128-row K/V tile, kv head), longest first.
// The CTA keeps K and V in shared memory and loops over the query heads of
// the group and over the 64-row q tiles that attend its keys. All products
// are tcgen05 MMAs with fp32 accumulators in tensor memory, computed in the
// transposed orientation so that the key tile is the M = 128 side:
//   S^T = K Q^T, dP^T = V dO^T                       (cols [0,64), [64,128))
//   dV += P^T dO  (P^T bf16 written back over S^T)    (cols [256, 256+Dp))
//   dK += dS^T Q  (dS^T bf16 in shared memory)        (cols [384, 384+Dp))
//   dQ^T = K^T dS^T, read out and added to an fp32    (cols [128,192))
//   accumulator in global memory with red.global.add.
// dK / dV never leave tensor memory until the last q tile, so the GQA sum is
// exact and deterministic. For D = 256 the dK / dV columns are produced in
// two passes of 128 (the S / dP products are recomputed in the second pass)
// because 2 x 256 fp32 columns would fill the whole tensor memory.
//   warp 0  loads (TMA for K, V, Q, dO; the q rows' lse / delta / mask bounds)
//   warp 1  issues the MMAs          warp 2  owns the tensor memory
//   warps 4-7 and 12-15  P, dS (thread = key row; q columns 0-31 / 32-63)
//   warps 8-11  dQ read-out (thread = d row)
// With attention dropout (kDrop) each P / dS warp draws its 32 keys' keep
// masks over the half's q columns (dropout.cuh); dropped weights are zeroed in
// P^T, dS = P (Z dP - delta), and dV is scaled by the keep scale when written.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// ----------------------------------------------------------------- K4a
// delta[row] = sum_d dout[row, d] * out[row, d] (fp32) and, given an
// accumulator, dq_acc[row, :] = 0.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ dout,
                                                      const __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ delta, float* __restrict__ dq_acc,
                                                      long long n_rows, const int32_t* status) {
  pdl_begin();
  if (*reinterpret_cast<const volatile int*>(status) != 0) return;
  constexpr int kLanes = D / 8 < 32 ? D / 8 : 32;  // threads per row
  constexpr int kVec = D / 8 / kLanes;              // 8-element (16 B) pieces per thread
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n_rows * kLanes;
       t += nthreads) {
    const long long row = t / kLanes;
    const int part = static_cast<int>(t % kLanes);
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const uint4 a = reinterpret_cast<const uint4*>(dout + row * D)[part + u * kLanes];
      const uint4 o = reinterpret_cast<const uint4*>(out + row * D)[part + u * kLanes];
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(o2[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int o = kLanes / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, kLanes);
    if (part == 0) delta[row] = acc;
    if (dq_acc) {  // none: delta only (the fixed-order dq pass writes dq itself)
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        float4* z = reinterpret_cast<float4*>(dq_acc + row * D + (part + u * kLanes) * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ----------------------------------------------------------------- K4b
// dq = scale * dq_acc in the requested dtype (8 elements per thread).
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ dq_acc, void* __restrict__ dq,
                                                         long long n_elems, float scale, int to_bf16,
                                                         const int32_t* status) {
  pdl_begin();
  if (*reinterpret_cast<const volatile int*>(status) != 0) return;
  const long long n8 = n_elems / 8;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += nthreads) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 c = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    if (to_bf16) {
      uint4 w;
      w.x = pack_bf16x2(a.x * scale, a.y * scale);
      w.y = pack_bf16x2(a.z * scale, a.w * scale);
      w.z = pack_bf16x2(c.x * scale, c.y * scale);
      w.w = pack_bf16x2(c.z * scale, c.w * scale);
      reinterpret_cast<uint4*>(dq)[t] = w;
    } else {
      reinterpret_cast<float4*>(dq)[2 * t] = make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale);
      reinterpret_cast<float4*>(dq)[2 * t + 1] = make_float4(c.x * scale, c.y * scale, c.z * scale, c.w * scale);
    }
  }
}

// ------------------------------------------------------------------ K4
template <int D>
struct BwdCfg {
  static constexpr int kDp = D < 128 ? D : 128;  // dK / dV columns per pass
  static constexpr int kPasses = D / kDp;
  static constexpr int kNsq = D == 256 ? 1 : (D == 128 ? 3 : 4);  // Q / dO stages
  // dQ^T is double-buffered in tensor memory: columns [128,192) and [192,256).
  static constexpr uint32_t kColS = 0, kColDp = 64, kColDq = 128, kColDv = 256, kColDk = 384;
  // For D <= 128 the dq partial tile is staged in shared memory (64 q x 64 d
  // fp32 per slot) and added to the accumulator with TMA bulk reduce-add;
  // D = 256 has no shared memory left and uses red.add.
  static constexpr bool kTmaDq = D <= 128;
  static constexpr int kDqChunks = kDp / 64;
  static constexpr int kStageSlots = kTmaDq ? kDqChunks : 0;
};

template <int SLOTS>
struct DqStage {
  alignas(1024) float buf[SLOTS][kBwdQ * 64];
};
template <>
struct DqStage<0> {};

template <int D, int NSQ>
struct BwdSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kKChunk = kTile * 128;  // 128 rows x 128 B
  static constexpr int kQChunk = kBwdQ * 128;  // 64 rows x 128 B
  // v must directly follow k: for D = 64 the dQ^T product reads A rows
  // 64..127 (d >= 64, discarded) from the 16 KB after k.
  alignas(1024) uint8_t k[kChunks][kKChunk];
  alignas(1024) uint8_t v[kChunks][kKChunk];
  alignas(1024) uint8_t q[NSQ][kChunks][kQChunk];
  alignas(1024) uint8_t dout[NSQ][kChunks][kQChunk];
  alignas(1024) uint8_t ds[kKChunk];  // dS^T, 128 keys x 64 q, bf16, 128B-swizzled
  DqStage<BwdCfg<D>::kStageSlots> stage;
  alignas(16) float lse2[2][kBwdQ];  // per q row: lse * log2(e), by tile parity
  alignas(16) float delta[2][kBwdQ];
  // the Q / dO stage in two groups (chunks [g kDp/64, (g+1) kDp/64) of both):
  // a tile frees the group its dK / dV products do not read as soon as its S
  // and dP products are done, so the next tile's copy of it starts early
  uint64_t kv_full, grp_full[2], grp_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full[2], dq_empty[2], acc_full, acc_empty, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, kt, q64_lo, nq64, n_real, skip, mode, n_att;
};

constexpr int kBwdThreads = 512;
constexpr int kZeroCtasBwd = 152;  // CTAs that carry the zero-fill (the first wave on 152 SMs)
// What a backward CTA does, from its position in the work list.
constexpr int kBwdModeIdle = 0;  // past the attended tiles (their dK / dV zeroed by the working CTAs)
constexpr int kBwdModeWork = 1;  // an attended K/V tile

// kDq: with the dq products (else dK / dV only, for the fixed-order dq pass).
template <int D, bool kDq, bool kDrop>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_dq, const int32_t* __restrict__ seg, const Geom g,
               const float* __restrict__ lse, const float* __restrict__ delta, float* __restrict__ dq_acc,
               void* __restrict__ dk, void* __restrict__ dv, int grads_bf16, int32_t* status) {
  pdl_begin();
  using Cfg = BwdCfg<D>;
  constexpr int NSQ = Cfg::kNsq, kDp = Cfg::kDp, kPasses = Cfg::kPasses;
  static_assert(NSQ == 1 && kPasses == 2, "one Q / dO stage in two groups, two passes over D (D = 256)");
  constexpr int kGrp = kDp / 64;  // 64-column chunks per group
  using Smem = BwdSmem<D, NSQ>;
  constexpr int kChunks = Smem::kChunks;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw so the compiler keeps the shared address space
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = blockIdx.x % g.Hkv;
  volatile int* vstatus = status;

  const int item = blockIdx.x / g.Hkv;
  if (tid == 0) {
    // the attended K/V tiles lead the work list; the grid must cover them
    const int n_att = seg[g.off[BD_SEG_OFF_COUNTS] + 3];
    int mode = kBwdModeIdle;
    s.n_att = -1;
    if (n_att < 0 || n_att > g.B * g.nkt || n_att > static_cast<int>(gridDim.x) / g.Hkv) {
      atomicOr(status, BD_STATUS_BOUNDS);
    } else {
      mode = item < n_att ? kBwdModeWork : kBwdModeIdle;
      s.n_att = n_att;
    }
    s.mode = mode;
  }
  __syncthreads();
  // dK / dV of the tiles no local row attends are zero. With at least a wave
  // of working CTAs, warps 2-3 of the first kZeroCtasBwd of them write these
  // rows during their main loop (their tiles lead the longest-first list, so
  // these CTAs run longest); with fewer, every CTA of the grid takes a share,
  // the idle ones with all their threads.
  const int n_att_s = s.n_att;
  const int n_zw = n_att_s * g.Hkv >= kZeroCtasBwd ? kZeroCtasBwd : static_cast<int>(gridDim.x);
  if (s.mode != kBwdModeWork) {
    if (n_att_s >= 0 && static_cast<int>(blockIdx.x) < n_zw)
      zero_unattended_kv(seg, g, n_att_s, static_cast<int>(blockIdx.x), n_zw, tid, kBwdThreads, dk, dv, grads_bf16,
                         status);
    return;
  }

  if (tid == 0) {
    const int wi = seg[g.off[BD_SEG_OFF_BWD_WORK] + item];
    int ok = wi >= 0 && wi < g.B * g.nkt;
    const int b = ok ? wi / g.nkt : 0, kt = ok ? wi % g.nkt : 0;
    const int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
    ok = ok && hdr[kHdrMagic] == kSegMagic && hdr[kHdrRowOffset] == g.row_offset && hdr[kHdrL] == g.L &&
         hdr[kHdrKvOffset] == g.kv_offset && hdr[kHdrSkv] == g.S_kv && hdr[kHdrWindow] == g.window &&
         hdr[kHdrSfull] == g.S_full;
    const int n_real = hdr[BD_SEG_N_REAL];
    const int32_t* qr = seg + g.off[BD_SEG_OFF_KT_QRANGE] + (b * g.nkt + kt) * 2;
    const int qlo = qr[0], qhi = qr[1];
    // an attended tile has a non-empty q range
    ok = ok && n_real >= 0 && n_real <= g.L && qlo >= 0 && qhi <= n_real && qlo < qhi;
    const int nq64 = qhi > qlo ? (qhi - 1) / kBwdQ - qlo / kBwdQ + 1 : 0;
    if (!ok) atomicOr(status, BD_STATUS_BOUNDS);
    s.b = b;
    s.kt = kt;
    s.q64_lo = qlo / kBwdQ;
    s.nq64 = nq64;
    s.n_real = n_real;
    s.skip = (!ok || *vstatus != 0) ? 1 : 0;
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.grp_full[i], 1);
      mbar_init(&s.grp_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.p_full, 256);
    mbar_init(&s.ds_full, 256);
    mbar_init(&s.ds_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.dq_full[i], 1);
      mbar_init(&s.dq_empty[i], 128);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 256);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, kt = s.kt, q64_lo = s.q64_lo, nq64 = s.nq64, n_real = s.n_real;
  const int G = g.G;
  const int n_it_pass = G * nq64;
  const int n_it = kPasses * n_it_pass;
  // dK / dV row j of this (batch row, kv head): kv_row(g, b, hk, j)
  // P / dS warpgroups: warps 4-7 (half 0, q columns 0-31) and 12-15 (half 1, 32-63)
  const bool is_pds = (warp >= 4 && warp < 8) || warp >= 12;
  const int half = warp >= 12 ? 1 : 0;

  auto store_row = [&](void* base, size_t elem_off, const float* vals32) {
    if (grads_bf16) {
      uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + elem_off);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint4 w;
        w.x = pack_bf16x2(vals32[8 * e + 0], vals32[8 * e + 1]);
        w.y = pack_bf16x2(vals32[8 * e + 2], vals32[8 * e + 3]);
        w.z = pack_bf16x2(vals32[8 * e + 4], vals32[8 * e + 5]);
        w.w = pack_bf16x2(vals32[8 * e + 6], vals32[8 * e + 7]);
        p[e] = w;
      }
    } else {
      float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem_off);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        p[e] = make_float4(vals32[4 * e + 0], vals32[4 * e + 1], vals32[4 * e + 2], vals32[4 * e + 3]);
    }
  };

  if (warp == 2) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;

  auto decode = [&](int it, int& pass, int& h, int& q0) {
    pass = it / n_it_pass;
    const int rem = it - pass * n_it_pass;
    const int gq = rem / nq64;
    h = hk * G + gq;
    q0 = (q64_lo + rem - gq * nq64) * kBwdQ;
  };

  if (warp == 0) {
    // -------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_dout);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.kv_full, 2 * kChunks * Smem::kKChunk);
      for (int c = 0; c < kChunks; ++c) {
        tma_load_3d(s.k[c], &tm_k, &s.kv_full, c * 64, g.kv_tm ? b * g.Hkv + hk : kt * kTile, g.kv_tm ? kt * kTile : b * g.Hkv + hk);
        tma_load_3d(s.v[c], &tm_v, &s.kv_full, c * 64, g.kv_tm ? b * g.Hkv + hk : kt * kTile, g.kv_tm ? kt * kTile : b * g.Hkv + hk);
      }
    }
    int issued[2] = {0, 0};
    bool stopped = false;
    for (int it = 0; it < n_it && !stopped; ++it) {
      int pass, h, q0;
      decode(it, pass, h, q0);
      // the per-row values are fetched before waiting for the free stage so
      // that their global-load latency overlaps the wait
      float l2[2], dl[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = q0 + lane + 32 * e;
        l2[e] = 0.f;
        dl[e] = 0.f;
        if (i < n_real) {
          const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
          l2[e] = lse[row] * 1.4426950408889634f;
          dl[e] = delta[row] * g.scale;  // dS is formed pre-scaled: scale * P (dP - delta)
        }
      }
      // the group the previous tile freed early first, then the other
      const int ge = it > 0 ? 1 - (it - 1) / n_it_pass : 0;
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int gr = k == 0 ? ge : 1 - ge;
        if (it > 0 && !warp_wait(&s.grp_empty[gr], (it - 1) & 1, &s.abort_flag, vstatus)) {
          stopped = true;
          break;
        }
        if (k == 0) {  // this tile's row values (slot it & 1: tile it - 2's, read long before)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = lane + 32 * e;
            s.lse2[it & 1][c] = l2[e];
            s.delta[it & 1][c] = dl[e];
          }
          __syncwarp();
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.grp_full[gr], 2 * kGrp * Smem::kQChunk);
          for (int c = gr * kGrp; c < (gr + 1) * kGrp; ++c) {
            tma_load_3d(s.q[0][c], &tm_q, &s.grp_full[gr], c * 64, q0, b * g.Hq + h);
            tma_load_3d(s.dout[0][c], &tm_dout, &s.grp_full[gr], c * 64, q0, b * g.Hq + h);
          }
        }
        ++issued[gr];
      }
    }
    if (lane == 0) {
      if (stopped) {
        s.abort_flag = 1;
        atomicOr(status, BD_STATUS_TIMEOUT);
      }
      // no copy into this CTA's shared memory may still be in flight at exit
      mbar_wait_drain(&s.kv_full, 0);
      for (int gr = 0; gr < 2; ++gr)
        if (issued[gr] > 0) mbar_wait_drain(&s.grp_full[gr], (issued[gr] - 1) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idST = idesc_bf16(128, kBwdQ, false, false);
      constexpr uint32_t idDKV = idesc_bf16(128, kDp, false, true);
      constexpr uint32_t idDQ = idesc_bf16(128, kBwdQ, true, true);
      const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);              // K-major operands
      const uint64_t dMN_q = umma_desc_sw128(0, Smem::kQChunk, 1024);      // MN-major, 64-row chunks
      const uint64_t dMN_k = umma_desc_sw128(0, Smem::kKChunk, 1024);      // MN-major, 128-row chunks
      const uint32_t a_k = smem_u32(s.k[0]), a_v = smem_u32(s.v[0]), a_ds = smem_u32(s.ds);
      const uint32_t a_q = smem_u32(s.q[0][0]), a_do = smem_u32(s.dout[0][0]);
      // X^T = A B^T over the head-dim chunks of group gr (A = K or V, B = Q or dO)
      auto issue_grp = [&](uint32_t col, uint32_t a_base, uint32_t b_base, int gr, bool first) {
#pragma unroll
        for (int kk = 0; kk < 4 * kGrp; ++kk) {
          const int ks = gr * 4 * kGrp + kk;
          const uint32_t off_a = (ks >> 2) * Smem::kKChunk + (ks & 3) * 32;
          const uint32_t off_b = (ks >> 2) * Smem::kQChunk + (ks & 3) * 32;
          umma_ss(tbase + col, desc_at(dK_major, a_base + off_a), desc_at(dK_major, b_base + off_b), idST,
                  (first && kk == 0) ? 0u : 1u);
        }
      };
      auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
      // S^T and dP^T of tile t: the group the previous tile freed early (and
      // whose copy started first) first; then the group tile t's dK / dV do not
      // read is free again once these are done
      auto issue_sdp = [&](int t) -> bool {
        const int ge = t > 0 ? 1 - (t - 1) / n_it_pass : 0, gl = 1 - ge;
        if (!wait(&s.grp_full[ge], t & 1)) return false;
        tc_fence_after();
        issue_grp(Cfg::kColS, a_k, a_q, ge, true);
        issue_grp(Cfg::kColDp, a_v, a_do, ge, true);
        if (!wait(&s.grp_full[gl], t & 1)) return false;
        tc_fence_after();
        issue_grp(Cfg::kColS, a_k, a_q, gl, false);
        umma_commit(&s.s_full);
        issue_grp(Cfg::kColDp, a_v, a_do, gl, false);
        umma_commit(&s.dp_full);
        umma_commit(&s.grp_empty[1 - t / n_it_pass]);
        return true;
      };
      bool ok = wait(&s.kv_full, 0) && issue_sdp(0);
      for (int it = 0; ok && it < n_it; ++it) {
        int pass, h, q0;
        decode(it, pass, h, q0);
        const bool first_of_pass = (it % n_it_pass) == 0;
        const bool last_of_pass = (it % n_it_pass) == n_it_pass - 1;
        const uint32_t pass_off_q = pass * kGrp * Smem::kQChunk;  // this pass's group of Q / dO chunks
        if (first_of_pass && pass > 0 && !wait(&s.acc_empty, (pass - 1) & 1)) { ok = false; break; }
        // dV += P^T dO[:, pass]; P^T is bf16 in tensor memory, q columns 0-31 at
        // column offset 0 and 32-63 at offset 48 (each half writes over its own S^T)
        if (!wait(&s.p_full, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBwdQ / 16; ++ks) {
          const uint32_t a_col = Cfg::kColS + (ks < 2 ? ks * 8 : 48 + (ks - 2) * 8);
          umma_ts(tbase + Cfg::kColDv, tbase + a_col, desc_at(dMN_q, a_do + pass_off_q + ks * 2048), idDKV,
                  (!first_of_pass || ks > 0) ? 1u : 0u);
        }
        // dK += dS^T Q[:, pass] ; dQ^T = K[:, pass]^T dS^T
        if (!wait(&s.ds_full, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBwdQ / 16; ++ks)
          umma_ss(tbase + Cfg::kColDk, desc_at(dK_major, a_ds + ks * 32), desc_at(dMN_q, a_q + pass_off_q + ks * 2048),
                  idDKV, (!first_of_pass || ks > 0) ? 1u : 0u);
        if constexpr (kDq) {
          const int bq = it & 1;  // dQ^T tensor-memory buffer
          if (it >= 2 && !wait(&s.dq_empty[bq], ((it >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_kpass = a_k + pass * (kDp / 64) * Smem::kKChunk;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_ss(tbase + Cfg::kColDq + 64 * bq, desc_at(dMN_k, a_kpass + ks * 2048),
                    desc_at(dMN_k, a_ds + ks * 2048), idDQ, ks > 0 ? 1u : 0u);
          umma_commit(&s.dq_full[bq]);
        }
        umma_commit(&s.ds_empty);
        umma_commit(&s.grp_empty[pass]);  // this pass's group: read by dV, dK above
        if (last_of_pass) umma_commit(&s.acc_full);
        if (it + 1 < n_it && !issue_sdp(it + 1)) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        s.abort_flag = 1;
        atomicOr(status, BD_STATUS_TIMEOUT);
      }
      umma_commit(&s.mma_drain);
      mbar_wait_drain(&s.mma_drain, 0);
    }
  } else if (is_pds) {
    // ---------------------------- P and dS (key rows; one half of the q columns)
    const int r = (warp & 3) * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int j = kt * kTile + r;  // K/V buffer row of this thread
    const int c0 = half * 32;      // first q column of this half
    const float sl2 = g.scale * 1.4426950408889634f;
    uint8_t* ds_row = s.ds + r * 128;
    // A real row p >= key s attends s iff p lies in the document that contains
    // s (documents are contiguous runs) and, with a window, p - s < W. So the
    // rows attending s are [s, min(doc_end(s), s + W)) intersected with the
    // real rows. doc_end(s) is fixed for the CTA: find it once from cu_q.
    const int key = g.kv_offset + j;  // global position of this thread's key
    int doc_end = -0x40000000;        // keys no local row attends
    {
      const int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
      const int32_t* cu_q = seg + g.off[BD_SEG_OFF_CU_Q] + b * (g.L + 1);
      const int n_seg = hdr[BD_SEG_N_SEG];
      if (n_seg > 0 && key >= hdr[BD_SEG_S_FIRST] && key < hdr[BD_SEG_REAL_END]) {
        int k = 0;  // segment containing key: the last k with row_offset + cu_q[k] <= key
        if (key >= g.row_offset) {
          int a = 0, e = n_seg - 1;
          while (a < e) {
            const int mid = (a + e + 1) >> 1;
            if (g.row_offset + cu_q[mid] <= key) a = mid; else e = mid - 1;
          }
          k = a;
        }
        doc_end = g.row_offset + cu_q[k + 1];
      }
    }
    const int win_end = g.window > 0 ? key + g.window : 0x3fffffff;
    const int row_end = min(doc_end, win_end);  // rows [key, row_end) attend this key
    // dropout: scale * keep scale multiplies a kept dP (a dropped one is zero)
    const float sc_dp = kDrop ? g.scale * g.drop_scale : g.scale;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;  // slot of this tile's row values
      int pass, h, q0;
      decode(it, pass, h, q0);
      uint64_t km = 0;  // dropout: keep bits of this key over the half's 32 q columns
      if constexpr (kDrop)
        km = key_keep_mask<4>(g, b, h, g.row_offset + q0 + c0, g.kv_offset + kt * kTile + (warp & 3) * 32, lane);
      // the early group's copy also publishes this tile's row values
      const int ge = it > 0 ? 1 - (it - 1) / n_it_pass : 0;
      if (!warp_wait(&s.grp_full[ge], it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      if (!warp_wait(&s.s_full, it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(tbase + lane_off + Cfg::kColS + c0, sr);
      tmem_wait_ld();
      // q columns [c_lo, c_hi) of this tile attend the key (relative to c0)
      const int row0 = g.row_offset + q0;
      const int c_lo = max(0, key - row0) - c0;
      const int c_hi = min(min(kBwdQ, n_real - q0), row_end - row0) - c0;
      float p[32];
      const float4* l4 = reinterpret_cast<const float4*>(s.lse2[st] + c0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l = l4[c4];
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * c4 + e;
          const float pe = fast_exp2(__uint_as_float(sr[c]) * sl2 - lv[e]);
          p[c] = (c >= c_lo && c < c_hi) ? pe : 0.f;
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if constexpr (kDrop)
          pk[c] = pack_bf16x2(((km >> (2 * c)) & 1u) ? p[2 * c] : 0.f, ((km >> (2 * c + 1)) & 1u) ? p[2 * c + 1] : 0.f);
        else
          pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
      }
      tmem_st16(tbase + lane_off + Cfg::kColS + 48 * half, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);

      if (!warp_wait(&s.dp_full, it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(tbase + lane_off + Cfg::kColDp + c0, sr);
      tmem_wait_ld();
      const float4* d4 = reinterpret_cast<const float4*>(s.delta[st] + c0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 dl = d4[c4];
        const int c = 4 * c4;
        float dp[4] = {__uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), __uint_as_float(sr[c + 2]),
                       __uint_as_float(sr[c + 3])};
        if constexpr (kDrop) {
#pragma unroll
          for (int e = 0; e < 4; ++e) dp[e] = ((km >> (c + e)) & 1u) ? dp[e] : 0.f;
        }
        pk[2 * c4] = pack_bf16x2(p[c] * fmaf(dp[0], sc_dp, -dl.x), p[c + 1] * fmaf(dp[1], sc_dp, -dl.y));
        pk[2 * c4 + 1] = pack_bf16x2(p[c + 2] * fmaf(dp[2], sc_dp, -dl.z), p[c + 3] * fmaf(dp[3], sc_dp, -dl.w));
      }
      if (it > 0 && !warp_wait(&s.ds_empty, (it - 1) & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      // this half's 64 B of the key row of dS^T, 128B-swizzled K-major layout
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int c16 = 4 * half + k4;
        const uint4 w = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
        *reinterpret_cast<uint4*>(ds_row + ((c16 ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&s.ds_full);

      if ((it % n_it_pass) == n_it_pass - 1) {
        // end of a pass: write this thread's dK / dV row (its half of the pass's columns)
        if (!warp_wait(&s.acc_full, pass & 1, &s.abort_flag, vstatus)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = half * (kDp / 2); c < (half + 1) * (kDp / 2); c += 32) {
          uint32_t vv[32];
          float f[32];
          tmem_ld32(tbase + lane_off + Cfg::kColDv + c, vv);
          tmem_wait_ld();
          if (j < g.S_kv) {
            const float dvs = kDrop ? g.drop_scale : 1.0f;  // dropout: the keep scale of P^T
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(vv[e]) * dvs;
            store_row(dv, kv_row(g, b, hk, j) * D + pass * kDp + c, f);
          }
          tmem_ld32(tbase + lane_off + Cfg::kColDk + c, vv);
          tmem_wait_ld();
          if (j < g.S_kv) {
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(vv[e]);  // dS was pre-scaled
            store_row(dk, kv_row(g, b, hk, j) * D + pass * kDp + c, f);
          }
        }
        tc_fence_before();
        mbar_arrive(&s.acc_empty);
      }
    }
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    }
  } else if (warp == 2 || warp == 3) {
    if (static_cast<int>(blockIdx.x) < n_zw)
      zero_unattended_kv(seg, g, n_att_s, static_cast<int>(blockIdx.x), n_zw, tid - 64, 64, dk, dv, grads_bf16, status);
  } else if (kDq && warp >= 8 && warp < 12) {
    // ----------------------------------------------- dQ read-out (d rows)
    const int r = tid - 256;  // d index within the pass == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool active = (warp & 3) * 32 < kDp;  // D = 64: lanes 64..127 hold nothing useful
    const bool issuer = tid == 256;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      int pass, h, q0;
      decode(it, pass, h, q0);
      const int bq = it & 1;
      bool got = warp_wait(&s.dq_full[bq], (it >> 1) & 1, &s.abort_flag, vstatus);
      uint32_t qv[64];
      if (got) {
        tc_fence_after();
        if (active) {
          const uint32_t col = Cfg::kColDq + 64 * bq;
          tmem_ld32(tbase + lane_off + col, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
          tmem_ld32(tbase + lane_off + col + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(&s.dq_empty[bq]);
      }
      if constexpr (Cfg::kTmaDq) {
        // Stage this iteration's 64 x kDp tile in shared memory and add it to
        // the accumulator with TMA bulk reduce-add. The previous iteration's
        // reduce must have finished reading the slots first; the barrier also
        // makes the abort decision uniform over the warpgroup.
        if (issuer) bulk_wait_group_read<0>();
        if (!named_bar_and(1, 128, got)) {
          ok = false;
          break;
        }
        if (active) {
          float* slot = s.stage.buf[r >> 6];
#pragma unroll
          for (int c = 0; c < kBwdQ; ++c) slot[c * 64 + (r & 63)] = __uint_as_float(qv[c]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (issuer) {
#pragma unroll
          for (int ch = 0; ch < Cfg::kDqChunks; ++ch)
            tma_reduce_add_3d(&tm_dq, s.stage.buf[ch], pass * kDp + ch * 64, q0, b * g.Hq + h);
          bulk_commit_group();
        }
      } else {
        if (!got) {
          ok = false;
          break;
        }
        if (active) {
          float* base = dq_acc + ((static_cast<size_t>(b) * g.Hq + h) * g.L) * D + pass * kDp + r;
          const int cmax = min(kBwdQ, n_real - q0);
          if (cmax >= kBwdQ) {  // full tile: no per-value row check on the red stream
#pragma unroll
            for (int c = 0; c < kBwdQ; ++c) red_add_f32(base + static_cast<size_t>(q0 + c) * D, __uint_as_float(qv[c]));
          } else {
#pragma unroll
            for (int c = 0; c < kBwdQ; ++c)
              if (c < cmax) red_add_f32(base + static_cast<size_t>(q0 + c) * D, __uint_as_float(qv[c]));
          }
        }
      }
    }
    if (Cfg::kTmaDq && issuer) bulk_wait_group<0>();
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

unsigned grid_for(long long work_items) {
  const long long blocks = (work_items + 255) / 256;
  return static_cast<unsigned>(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
}

template <int D, bool kDq>
cudaError_t launch_main_d(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mdq, const int32_t* seg, const Geom& g, const float* lse,
                          const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                          cudaStream_t st) {
  const size_t smem = sizeof(BwdSmem<D, BwdCfg<D>::kNsq>) + 1024;  // + 1 KB to align the swizzled tiles
  auto kern = g.drop_t ? bwd_kernel<D, kDq, true> : bwd_kernel<D, kDq, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // only tiles some local row can reach by position get a working CTA; with
  // none reachable, B CTAs per kv head still zero dK / dV
  const int reach = kv_tiles_reachable(g);
  const long long grid = static_cast<long long>(g.B) * (reach > 0 ? reach : 1) * g.Hkv;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kBwdThreads), smem, st, mq,
      mdo, mk, mv, mdq, seg, g, lse, delta, dq_acc, dk, dv, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}
}  // namespace

// Workspace: fp32 dq accumulator [B,Hq,L,D], then fp32 delta [B,Hq,L].
size_t bwd_workspace_bytes(const Geom& g) {
  const size_t rows = static_cast<size_t>(g.B) * g.Hq * g.L;
  return align256(rows * g.D * 4) + align256(rows * 4);
}

static float* ws_delta(const Geom& g, void* workspace) {
  const size_t rows = static_cast<size_t>(g.B) * g.Hq * g.L;
  return reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * g.D * 4));
}

// K4a: delta (in the workspace) and a zeroed dq accumulator: `dq_f32` when
// given (the fp32 dq output itself), else the workspace's.
namespace {
cudaError_t launch_pre(const Geom& g, const void* dout, const void* out, void* workspace, float* dq_acc,
                       int32_t* status, cudaStream_t st);
}  // namespace

cudaError_t launch_bwd_prep(const Geom& g, const void* dout, const void* out, void* workspace, float* dq_f32,
                            int32_t* status, cudaStream_t st) {
  return launch_pre(g, dout, out, workspace, dq_f32 ? dq_f32 : static_cast<float*>(workspace), status, st);
}

// delta only, for the fixed-order dq pass
cudaError_t launch_bwd_delta(const Geom& g, const void* dout, const void* out, void* workspace, int32_t* status,
                             cudaStream_t st) {
  return launch_pre(g, dout, out, workspace, nullptr, status, st);
}

const float* bwd_delta_ptr(const Geom& g, void* workspace) { return ws_delta(g, workspace); }

namespace {
cudaError_t launch_pre(const Geom& g, const void* dout, const void* out, void* workspace, float* dq_acc,
                       int32_t* status, cudaStream_t st) {
  const long long rows = static_cast<long long>(g.B) * g.Hq * g.L;
  const __nv_bfloat16* dob = static_cast<const __nv_bfloat16*>(dout);
  const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(out);
  float* delta = ws_delta(g, workspace);
  const unsigned grid = grid_for(rows * (g.D / 8 < 32 ? g.D / 8 : 32));
  switch (g.D) {
    case 64: if (const cudaError_t le = launch_pdl(bwd_pre_kernel<64>, dim3(grid), dim3(256), 0, st, dob, ob, delta,
        dq_acc, rows, status); le != cudaSuccess) return le; break;
    case 128: if (const cudaError_t le = launch_pdl(bwd_pre_kernel<128>, dim3(grid), dim3(256), 0, st, dob, ob,
        delta, dq_acc, rows, status); le != cudaSuccess) return le; break;
    case 256: if (const cudaError_t le = launch_pdl(bwd_pre_kernel<256>, dim3(grid), dim3(256), 0, st, dob, ob,
        delta, dq_acc, rows, status); le != cudaSuccess) return le; break;
    case 512: if (const cudaError_t le = launch_pdl(bwd_pre_kernel<512>, dim3(grid), dim3(256), 0, st, dob, ob,
        delta, dq_acc, rows, status); le != cudaSuccess) return le; break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd128_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                               const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                               const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                               cudaStream_t st);
cudaError_t launch_bwd512_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                               const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                               const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                               cudaStream_t st);

// Rows of the q / dout TMA boxes the backward main kernel for this head dim expects.
int bwd_q_box_rows(int D) { return D <= 128 ? 128 : kBwdQ; }

// K4: dK, dV and the dq accumulation (scale * dS K: the kernels form dS
// pre-scaled) into the workspace's fp32 accumulator (`mdq` maps it as
// [B*Hq][L][D] with 64 x 64 boxes) or, when `dq_f32` is given, straight into
// that fp32 dq output.
cudaError_t launch_bwd_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdq, const int32_t* seg, const Geom& g, const float* lse, void* dk,
                            void* dv, int bf16, void* workspace, float* dq_f32, int32_t* status, cudaStream_t st) {
  float* dq_acc = dq_f32 ? dq_f32 : static_cast<float*>(workspace);
  const float* delta = ws_delta(g, workspace);
  switch (g.D) {
    case 64:
    case 128:  // 128-row q tiles (bwd128_kernel.cu); q / dout maps use 128-row boxes
      return launch_bwd128_main(mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status, st);
    case 256:
      return launch_main_d<256, true>(mq, mdo, mk, mv, mdq, seg, g, lse, delta, dq_acc, dk, dv, bf16, status, st);
    case 512:  // the head dim of the outputs split over four CTAs (bwd512_kernel.cu)
      return launch_bwd512_main(mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status, st);
    default: return cudaErrorInvalidValue;
  }
}

// K4 without the dq products (D = 64 / 128 / 256 / 512; for D >= 256 the
// q / dout maps have kBwdQ-row boxes): dK, dV and the zero-fill only, for the
// fixed-order dq pass.
cudaError_t launch_bwd_main_nodq(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                                 void* dk, void* dv, int bf16, void* workspace, int32_t* status, cudaStream_t st) {
  if (g.D != 64 && g.D != 128 && g.D != 256 && g.D != 512) return cudaErrorInvalidValue;
  if (g.D == 512)
    return launch_bwd512_main(mq, mdo, mk, mv, seg, g, lse, ws_delta(g, workspace), nullptr, dk, dv, bf16, status,
                              st);
  if (g.D == 256)  // the dq map is not read without the dq products
    return launch_main_d<256, false>(mq, mdo, mk, mv, mq, seg, g, lse, ws_delta(g, workspace), nullptr, dk, dv, bf16,
                                     status, st);
  return launch_bwd128_main(mq, mdo, mk, mv, seg, g, lse, ws_delta(g, workspace), nullptr, dk, dv, bf16, status,
                            st);
}

// K4b: dq = the accumulator (already scaled) in the gradient dtype.
cudaError_t launch_bwd_finalize(const Geom& g, void* dq, int bf16, void* workspace, int32_t* status,
                                cudaStream_t st) {
  const long long n = static_cast<long long>(g.B) * g.Hq * g.L * g.D;
  if (const cudaError_t le = launch_pdl(dq_convert_kernel, dim3(grid_for(n / 8)), dim3(256), 0, st,
      static_cast<const float*>(workspace), dq, n, 1.0f, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
