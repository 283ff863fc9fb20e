// K4, head dims 64 and 128: the backward main kernel with 128-row q tiles.
//
// Same mathematics as the 64-row kernel in bwd_kernels.cu (gemma4_moe.
// cp_local_ring `sliding_ring_compute_fa_bwd`: backward from the saved out /
// LSE; blockdiag_cp.exchange `_AllGatherSeqDiff`: a K/V position's gradient
// is the sum of all its queries' contributions), tiled for tcgen05 issue
// efficiency: every product is an M = 128, N = 128 MMA (an N = 64 MMA runs at
// ~65% of the tensor rate on this part), so each 128 x 128 (key, query) tile
// costs 5 x (D/16 or 8) instructions.
//
// One CTA per (128-row K/V tile, kv head), longest first; it loops over the
// group's query heads and the 128-row q tiles that attend its keys.
//   tensor memory  [0,128)   S^T = K Q^T, then P^T (bf16, packed in place)
//                  [128,256) dP^T = V dO^T, then dQ^T = K^T dS^T
//                  [256,384) dV += P^T dO        [384,512) dK += dS^T Q
//   shared memory  K, V (resident), Q / dO (two stages), dS^T (bf16)
//   warp 0 TMA + per-row lse / delta; warp 1 MMA issue; warp 2 tensor memory;
//   warps 4-7 and 12-15 P and dS (thread = key row, q columns 0-63 / 64-127);
//   warps 8-11 read dQ^T (thread = d row) and add it to the fp32 accumulator
//   with red.global.add (128-byte coalesced per warp instruction).
// With attention dropout (kDrop) each P / dS warp draws its 32 keys' keep
// masks over the tile's q columns before S arrives; the dropped weights are
// zeroed in P^T (the dV operand), dS = P (Z dP - delta) takes the same
// decisions, and dV is scaled by the keep scale when it is written.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

namespace {

constexpr int kQ = 128;          // q rows per tile
constexpr int kThreads = 512;
constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;
constexpr int kZeroCtas = 152;  // CTAs that carry the zero-fill (the first wave on 152 SMs)

template <int D>
struct Tiles {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunk = 128 * 128;  // 128 rows x 128 B (64 bf16)
  // v directly follows k: for D = 64 the dQ^T product reads A rows 64..127
  // (d >= 64, discarded) from the 16 KB after k.
  alignas(1024) uint8_t k[kChunks][kChunk];
  alignas(1024) uint8_t v[kChunks][kChunk];
  alignas(1024) uint8_t q[2][kChunks][kChunk];
  alignas(1024) uint8_t dout[2][kChunks][kChunk];
  alignas(1024) uint8_t ds[2][kChunk];  // dS^T: 128 keys x 128 q, two 64-column chunks, 128B-swizzled
};

struct Ctl {
  float lse2[2][kQ];  // per q row: lse * log2(e)
  float delta[2][kQ];
  uint64_t kv_full, q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full, dq_empty, acc_full, acc_empty, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, kt, q_lo, nq, n_real, skip, mode, n_att;
};

// What a CTA does, from its position in the backward work list.
constexpr int kModeIdle = 0;  // past the attended tiles (their dK / dV zeroed by the working CTAs)
constexpr int kModeWork = 1;  // an attended K/V tile

__device__ __forceinline__ void red_add(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ uint32_t dyn_smem_bytes() {
  uint32_t n;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
  return n;
}

}  // namespace

template <int D>
__host__ __device__ constexpr size_t bwd128_smem_bytes() {
  return sizeof(Tiles<D>) + sizeof(Ctl);
}

// kDq: also the dq products and their reductions (else dK / dV only, for a
// separate deterministic dq pass)
template <int D, bool kDq, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    bwd128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                  const float* __restrict__ delta, float* __restrict__ dq_acc,
                  void* __restrict__ dk, void* __restrict__ dv, int grads_bf16, int32_t* status) {
  pdl_begin();
  using T = Tiles<D>;
  constexpr int kChunks = T::kChunks;
  constexpr int kChunk = T::kChunk;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t align_off = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (align_off + bwd128_smem_bytes<D>() > dyn_smem_bytes()) {  // the layout must fit the allocation
    if (threadIdx.x == 0) atomicOr(status, BD_STATUS_BOUNDS);
    return;
  }
  T& t = *reinterpret_cast<T*>(smem_raw + align_off);
  Ctl& s = *reinterpret_cast<Ctl*>(smem_raw + align_off + sizeof(T));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = blockIdx.x % g.Hkv;
  volatile int* vstatus = status;

  const int item = blockIdx.x / g.Hkv;
  if (tid == 0) {
    // the attended K/V tiles lead the work list; the grid must cover them
    const int n_att = seg[g.off[BD_SEG_OFF_COUNTS] + 3];
    int mode = kModeIdle;
    s.n_att = -1;
    if (n_att < 0 || n_att > g.B * g.nkt || n_att > static_cast<int>(gridDim.x) / g.Hkv) {
      atomicOr(status, BD_STATUS_BOUNDS);
    } else {
      mode = item < n_att ? kModeWork : kModeIdle;
      s.n_att = n_att;
    }
    s.mode = mode;
  }
  __syncthreads();
  // dK / dV of the tiles no local row attends are zero. With at least a wave
  // of working CTAs, warps 2-3 of the first kZeroCtas of them write these rows
  // during their main loop (their tiles lead the longest-first list, so these
  // CTAs run longest); with fewer, every CTA of the grid takes a share, the
  // idle ones with all their threads.
  const int n_att_s = s.n_att;
  const int n_zw = n_att_s * g.Hkv >= kZeroCtas ? kZeroCtas : static_cast<int>(gridDim.x);
  if (s.mode != kModeWork) {
    if (n_att_s >= 0 && static_cast<int>(blockIdx.x) < n_zw)
      zero_unattended_kv(seg, g, n_att_s, static_cast<int>(blockIdx.x), n_zw, tid, kThreads, dk, dv, grads_bf16,
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
    if (!ok) atomicOr(status, BD_STATUS_BOUNDS);
    s.b = b;
    s.kt = kt;
    s.q_lo = qlo / kQ;
    s.nq = qhi > qlo ? (qhi - 1) / kQ - qlo / kQ + 1 : 0;
    s.n_real = n_real;
    s.skip = (!ok || *vstatus != 0) ? 1 : 0;
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.p_full, 256);
    mbar_init(&s.ds_full, 256);
    mbar_init(&s.ds_empty, 1);
    mbar_init(&s.dq_full, 1);
    mbar_init(&s.dq_empty, 128);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 256);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, kt = s.kt, q_lo = s.q_lo, nq = s.nq, n_real = s.n_real;
  const int G = g.G;
  const int n_it = G * nq;  // iteration it: query head hk*G + it / nq, q tile q_lo + it % nq
  // dK / dV row j of this (batch row, kv head): kv_row(g, b, hk, j)
  const bool is_pds = (warp >= 4 && warp < 8) || warp >= 12;
  const int half = warp >= 12 ? 1 : 0;

  auto store_row = [&](void* base, size_t elem_off, const float* vals32) {
    if (grads_bf16) {
      uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + elem_off);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        p[e] = make_uint4(pack_bf16x2(vals32[8 * e + 0], vals32[8 * e + 1]),
                          pack_bf16x2(vals32[8 * e + 2], vals32[8 * e + 3]),
                          pack_bf16x2(vals32[8 * e + 4], vals32[8 * e + 5]),
                          pack_bf16x2(vals32[8 * e + 6], vals32[8 * e + 7]));
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

  if (warp == 0) {
    // -------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_dout);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.kv_full, 2 * kChunks * kChunk);
      for (int c = 0; c < kChunks; ++c) {
        tma_load_3d(t.k[c], &tm_k, &s.kv_full, c * 64, g.kv_tm ? b * g.Hkv + hk : kt * kTile, g.kv_tm ? kt * kTile : b * g.Hkv + hk);
        tma_load_3d(t.v[c], &tm_v, &s.kv_full, c * 64, g.kv_tm ? b * g.Hkv + hk : kt * kTile, g.kv_tm ? kt * kTile : b * g.Hkv + hk);
      }
    }
    int issued = 0, gq = 0, qt = 0;  // (head, q tile) of iteration `it`
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;
      const int h = hk * G + gq, q0 = (q_lo + qt) * kQ;
      // fetch this tile's per-row values before waiting for the free stage
      float l2[4], dl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = q0 + lane + 32 * e;
        l2[e] = 0.f;
        dl[e] = 0.f;
        if (i < n_real) {
          const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
          l2[e] = lse[row] * 1.4426950408889634f;
          dl[e] = delta[row] * g.scale;  // dS is formed pre-scaled: scale * P (dP - delta)
        }
      }
      if (it >= 2 && !warp_wait(&s.q_empty[st], ((it >> 1) - 1) & 1, &s.abort_flag, vstatus)) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s.lse2[st][lane + 32 * e] = l2[e];
        s.delta[st][lane + 32 * e] = dl[e];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.q_full[st], 2 * kChunks * kChunk);
        for (int c = 0; c < kChunks; ++c) {
          tma_load_3d(t.q[st][c], &tm_q, &s.q_full[st], c * 64, q0, b * g.Hq + h);
          tma_load_3d(t.dout[st][c], &tm_dout, &s.q_full[st], c * 64, q0, b * g.Hq + h);
        }
      }
      ++issued;
      if (++qt == nq) {
        qt = 0;
        ++gq;
      }
    }
    if (lane == 0) {
      if (issued < n_it) {
        s.abort_flag = 1;
        atomicOr(status, BD_STATUS_TIMEOUT);
      }
      mbar_wait_drain(&s.kv_full, 0);
      for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it) mbar_wait_drain(&s.q_full[it & 1], (it >> 1) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idST = idesc_bf16(128, kQ, false, false);  // S^T, dP^T
      constexpr uint32_t idDKV = idesc_bf16(128, D, false, true);   // dV, dK
      constexpr uint32_t idDQ = idesc_bf16(128, kQ, true, true);    // dQ^T
      const uint64_t dKm = umma_desc_sw128(0, 16, 1024);       // K-major operands
      const uint64_t dMN = umma_desc_sw128(0, kChunk, 1024);   // MN-major, 16 KB between 64-column chunks
      const uint32_t a_k = smem_u32(t.k[0]), a_v = smem_u32(t.v[0]), a_ds = smem_u32(t.ds[0]);
      const uint32_t a_q = smem_u32(t.q[0][0]), a_do = smem_u32(t.dout[0][0]);
      constexpr uint32_t kStage = kChunks * kChunk;
      // X^T = A B^T over the head dim, A = K or V (128 keys), B = Q or dO (128 q rows)
      auto issue_t = [&](uint32_t col, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kChunk + (ks & 3) * 32;
          umma_ss(tbase + col, desc_at(dKm, a_base + off), desc_at(dKm, b_base + off), idST, ks > 0 ? 1u : 0u);
        }
      };
      auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
      bool ok = wait(&s.kv_full, 0) && wait(&s.q_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_t(kColS, a_k, a_q);
        umma_commit(&s.s_full);
        issue_t(kColDp, a_v, a_do);
        umma_commit(&s.dp_full);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it & 1;
        // dV += P^T dO : P^T (bf16) sits in tensor memory over S^T, q columns
        // 0-63 at column 0 and 64-127 at column 64 (each half over its own S^T)
        if (!wait(&s.p_full, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kQ / 16; ++ks) {
          const uint32_t a_col = kColS + (ks < 4 ? ks * 8 : 64 + (ks - 4) * 8);
          umma_ts(tbase + kColDv, tbase + a_col, desc_at(dMN, a_do + st * kStage + ks * 2048), idDKV,
                  (it > 0 || ks > 0) ? 1u : 0u);
        }
        // S^T of the next tile can go in now (the dV product above was issued
        // first, so it reads P^T before S^T is overwritten)
        if (it + 1 < n_it) {
          if (!wait(&s.q_full[st ^ 1], ((it + 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_t(kColS, a_k, a_q + (st ^ 1) * kStage);
          umma_commit(&s.s_full);
        }
        // dQ^T = K^T dS^T into the dP^T columns (dS is written, so dP^T was read)
        if (!wait(&s.ds_full, it & 1)) { ok = false; break; }
        tc_fence_after();
        if constexpr (kDq) {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_ss(tbase + kColDp, desc_at(dMN, a_k + ks * 2048), desc_at(dMN, a_ds + ks * 2048), idDQ,
                    ks > 0 ? 1u : 0u);
          umma_commit(&s.dq_full);
        }
        // dK += dS^T Q
#pragma unroll
        for (int ks = 0; ks < kQ / 16; ++ks)
          umma_ss(tbase + kColDk, desc_at(dKm, a_ds + (ks >> 2) * kChunk + (ks & 3) * 32),
                  desc_at(dMN, a_q + st * kStage + ks * 2048), idDKV, (it > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.ds_empty);
        umma_commit(&s.q_empty[st]);
        if (it + 1 == n_it) umma_commit(&s.acc_full);
        // dP^T of the next tile once dQ^T has been read out of those columns
        if (it + 1 < n_it) {
          if (kDq && !wait(&s.dq_empty, it & 1)) { ok = false; break; }
          tc_fence_after();
          issue_t(kColDp, a_v, a_do + (st ^ 1) * kStage);
          umma_commit(&s.dp_full);
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
    const int j = kt * kTile + r;
    const int c0 = half * 64;  // first q column of this half
    const float sl2 = g.scale * 1.4426950408889634f;
    uint8_t* ds_row = t.ds[half] + r * 128;
    // A real row p >= key s attends s iff p lies in the document that contains
    // s (documents are contiguous runs) and, with a window, p - s < W: rows
    // [s, min(doc_end(s), s + W)) of the real rows. doc_end(s) is fixed for
    // the CTA; find it once from cu_q.
    const int key = g.kv_offset + j;
    int doc_end = -0x40000000;  // keys no local row attends
    {
      const int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
      const int32_t* cu_q = seg + g.off[BD_SEG_OFF_CU_Q] + b * (g.L + 1);
      const int n_seg = hdr[BD_SEG_N_SEG];
      if (n_seg > 0 && key >= hdr[BD_SEG_S_FIRST] && key < hdr[BD_SEG_REAL_END]) {
        int k = 0;  // the last segment with row_offset + cu_q[k] <= key
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
    const int row_end = min(doc_end, g.window > 0 ? key + g.window : 0x3fffffff);
    // dropout: scale * keep scale multiplies a kept dP (a dropped one is zero)
    const float sc_dp = kDrop ? g.scale * g.drop_scale : g.scale;
    bool ok = true;
    int qt = 0, gq = 0;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;
      const int q0 = (q_lo + qt) * kQ;
      uint64_t km = 0;  // dropout: keep bits of this key over the half's 64 q columns
      if constexpr (kDrop)
        km = key_keep_mask<8>(g, b, hk * G + gq, g.row_offset + q0 + c0, g.kv_offset + kt * kTile + (warp & 3) * 32,
                              lane);
      if (++qt == nq) {
        qt = 0;
        ++gq;
      }
      if (!warp_wait(&s.q_full[st], (it >> 1) & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      if (!warp_wait(&s.s_full, it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      tc_fence_after();
      // q columns [c_lo, c_hi) of this tile attend the key (relative to c0)
      const int row0 = g.row_offset + q0;
      const int c_lo = max(0, key - row0) - c0;
      const int c_hi = min(min(kQ, n_real - q0), row_end - row0) - c0;
      float p[64];  // P in fp32, kept for dS
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t sr[32];
        tmem_ld32(tbase + lane_off + kColS + c0 + 32 * h2, sr);
        tmem_wait_ld();
        const float4* l4 = reinterpret_cast<const float4*>(s.lse2[st] + c0 + 32 * h2);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l = l4[c4];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 32 * h2 + 4 * c4 + e;
            const float pe = fast_exp2(__uint_as_float(sr[4 * c4 + e]) * sl2 - lv[e]);
            p[c] = (c >= c_lo && c < c_hi) ? pe : 0.f;
          }
        }
        // packed bf16 P of these 32 q columns over S^T columns this half has read
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = 32 * h2 + 2 * e;
          if constexpr (kDrop)
            pk[e] = pack_bf16x2(((km >> c) & 1u) ? p[c] : 0.f, ((km >> (c + 1)) & 1u) ? p[c + 1] : 0.f);
          else
            pk[e] = pack_bf16x2(p[c], p[c + 1]);
        }
        tmem_st16(tbase + lane_off + kColS + c0 + 16 * h2, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);

      if (!warp_wait(&s.dp_full, it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      tc_fence_after();
      // the previous tile's dK / dQ products must be done reading dS^T
      if (it > 0 && !warp_wait(&s.ds_empty, (it - 1) & 1, &s.abort_flag, vstatus)) { ok = false; break; }
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {  // 16 q columns at a time
        uint32_t sr[16];
        tmem_ld16(tbase + lane_off + kColDp + c0 + 16 * h4, sr);
        tmem_wait_ld();
        const float4* d4 = reinterpret_cast<const float4*>(s.delta[st] + c0 + 16 * h4);
        uint32_t dsk[8];  // dS of 16 q columns, bf16 pairs
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const float4 dl = d4[c4];
          const int c = 16 * h4 + 4 * c4;
          float dp[4] = {__uint_as_float(sr[4 * c4]), __uint_as_float(sr[4 * c4 + 1]), __uint_as_float(sr[4 * c4 + 2]),
                         __uint_as_float(sr[4 * c4 + 3])};
          if constexpr (kDrop) {
#pragma unroll
            for (int e = 0; e < 4; ++e) dp[e] = ((km >> (c + e)) & 1u) ? dp[e] : 0.f;
          }
          dsk[2 * c4] = pack_bf16x2(p[c] * fmaf(dp[0], sc_dp, -dl.x), p[c + 1] * fmaf(dp[1], sc_dp, -dl.y));
          dsk[2 * c4 + 1] = pack_bf16x2(p[c + 2] * fmaf(dp[2], sc_dp, -dl.z), p[c + 3] * fmaf(dp[3], sc_dp, -dl.w));
        }
        // 32 B of this key row of dS^T (128B-swizzled K-major layout)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int c16 = 2 * h4 + k2;
          *reinterpret_cast<uint4*>(ds_row + ((c16 ^ (r & 7)) << 4)) =
              make_uint4(dsk[4 * k2], dsk[4 * k2 + 1], dsk[4 * k2 + 2], dsk[4 * k2 + 3]);
        }
      }
      tc_fence_before();  // the dP^T reads above complete before dQ^T may overwrite those columns
      fence_proxy_async_smem();
      mbar_arrive(&s.ds_full);
    }
    if (ok) {
      // write this thread's dK / dV row (its half of the columns)
      if (!warp_wait(&s.acc_full, 0, &s.abort_flag, vstatus)) {
        ok = false;
      } else {
        tc_fence_after();
#pragma unroll 1
        for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
          uint32_t vv[32];
          float f[32];
          tmem_ld32(tbase + lane_off + kColDv + c, vv);
          tmem_wait_ld();
          if (j < g.S_kv) {
            const float dvs = kDrop ? g.drop_scale : 1.0f;  // dropout: the keep scale of P^T
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(vv[e]) * dvs;
            store_row(dv, kv_row(g, b, hk, j) * D + c, f);
          }
          tmem_ld32(tbase + lane_off + kColDk + c, vv);
          tmem_wait_ld();
          if (j < g.S_kv) {
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(vv[e]);  // dS was pre-scaled
            store_row(dk, kv_row(g, b, hk, j) * D + c, f);
          }
        }
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
    const int r = tid - 256;  // d index == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool active = (warp & 3) * 32 < D;  // D = 64: lanes 64..127 hold nothing useful
    bool ok = true;
    int gq = 0, qt = 0;
    for (int it = 0; it < n_it; ++it) {
      const int h = hk * G + gq, q0 = (q_lo + qt) * kQ;
      if (++qt == nq) {
        qt = 0;
        ++gq;
      }
      if (!warp_wait(&s.dq_full, it & 1, &s.abort_flag, vstatus)) { ok = false; break; }
      tc_fence_after();
      // two halves of 64 q columns; the columns are released after the second read
      float* base = dq_acc + ((static_cast<size_t>(b) * g.Hq + h) * g.L + q0) * D + r;
      const int cmax = min(kQ, n_real - q0);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t qv[64];
        if (active) {
          tmem_ld32(tbase + lane_off + kColDp + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
          tmem_ld32(tbase + lane_off + kColDp + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
          tmem_wait_ld();
        }
        if (hh == 1) {
          tc_fence_before();
          mbar_arrive(&s.dq_empty);
        }
        if (active) {
          // these warps issue one red per value and nothing else: a full
          // tile takes the loop without a per-value row check
          if (cmax >= kQ) {
#pragma unroll
            for (int c = 0; c < 64; ++c) red_add(base + static_cast<size_t>(64 * hh + c) * D, __uint_as_float(qv[c]));
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (64 * hh + c < cmax) red_add(base + static_cast<size_t>(64 * hh + c) * D, __uint_as_float(qv[c]));
          }
        }
      }
    }
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
template <int D>
cudaError_t launch128(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk, const CUtensorMap& mv,
                      const int32_t* seg, const Geom& g, const float* lse, const float* delta, float* dq_acc,
                      void* dk, void* dv, int bf16, int32_t* status, cudaStream_t st) {
  constexpr size_t need = bwd128_smem_bytes<D>();
  // request the layout plus alignment slack, up to the per-block maximum; the
  // kernel verifies at run time that its 1024-byte-aligned layout fits
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const size_t smem = need + 1024 <= static_cast<size_t>(max_optin) ? need + 1024 : static_cast<size_t>(max_optin);
  if (smem < need) return cudaErrorInvalidValue;
  // no accumulator: dK / dV only
  auto kern = g.drop_t ? (dq_acc ? bwd128_kernel<D, true, true> : bwd128_kernel<D, false, true>)
                       : (dq_acc ? bwd128_kernel<D, true, false> : bwd128_kernel<D, false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // only tiles some local row can reach by position get a working CTA; with
  // none reachable, B CTAs per kv head still zero dK / dV
  const int reach = kv_tiles_reachable(g);
  const long long grid = static_cast<long long>(g.B) * (reach > 0 ? reach : 1) * g.Hkv;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, st, mq, mdo,
      mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}
}  // namespace

// Backward main kernel for D = 64 / 128 (q and dout maps must use 128-row boxes).
cudaError_t launch_bwd128_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                               const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                               const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                               cudaStream_t st) {
  switch (g.D) {
    case 64: return launch128<64>(mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status, st);
    case 128: return launch128<128>(mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bd
