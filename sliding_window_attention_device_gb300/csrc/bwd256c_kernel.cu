// K4h: the backward main kernel for head dim 256 (the Gemma4 sliding-window
// layers), on a pair of CTAs per K/V tile.
//
// Same mathematics as K4 (gemma4_moe.cp_local_ring `sliding_ring_compute_fa_bwd`:
// backward from the saved out / LSE; blockdiag_cp.exchange `_AllGatherSeqDiff`:
// a K/V position's gradient is the sum of all its queries' contributions).
// With P = exp(scale q.k - lse) on allowed pairs and delta = rowsum(dO * O):
//   dV += P^T dO,  dP = dO V^T,  dS = P (dP - delta),  dK += scale dS^T Q,
//   dQ += scale dS K, dK / dV summed over the Hq/Hkv query heads of a group.
//
// Design (GB300). At D = 256 a whole K/V tile (128 KB) and two Q / dO stages
// (128 KB) do not fit in one CTA's shared memory, and dK / dV of 128 keys over
// all 256 columns (2 x 256 fp32 columns) would fill the whole tensor memory.
// So each 128-row K/V tile (and kv head) is worked by a cluster of two CTAs,
// CTA c owning the head-dim half [128 c, 128 c + 128) of K, V, Q and dO:
//   S^T = K Q^T and dP^T = V dO^T split over the head dim: each CTA forms
//   the partial products of its half (M = 128 keys, N = 64 q rows) and the
//   two exchange them through distributed shared memory, so both hold the
//   full S^T and dP^T and form the same P and dS;
//   dV[:, c] += P^T dO[:, c], dK[:, c] += dS^T Q[:, c] and dQ^T[c] =
//   K[:, c]^T dS^T need only the CTA's own half.
// Every product is computed once (no second pass over D), and the freed
// shared memory holds two Q / dO stages.
//   tensor memory  [0,64) partial S^T, then P^T (bf16)   [64,128) partial dP^T
//                  [128,256) dQ^T (two buffers)   [256,384) dV half   [384,512) dK half
//   shared memory  K, V halves (resident), Q / dO halves (two stages), dS^T,
//                  the peer's partial S^T and dP^T (fp32, swizzled rows)
//   warp 0 TMA + per-row lse / delta; warp 1 MMA issue; warp 2 tensor memory;
//   warps 4-7 and 12-15 exchange, P and dS (thread = key row, q columns
//   0-31 / 32-63); warps 8-11 read dQ^T (thread = d row of the half) and add
//   it to the fp32 accumulator with red.global.add.
// With attention dropout (kDrop) each P / dS warp draws its 32 keys' keep
// masks (dropout.cuh); dropped weights are zeroed in P^T, dS = P (Z dP -
// delta), and dV is scaled by the keep scale when written.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

namespace {

constexpr int kDc = 256;         // head dim
constexpr int kHalf = 128;       // head-dim columns per CTA
constexpr int kQc = 64;          // q rows per tile
constexpr int kThreadsC = 512;
constexpr uint32_t kColSc = 0, kColDpc = 64, kColDqc = 128, kColDvc = 256, kColDkc = 384;
constexpr int kKChunkC = kTile * 128;  // 128 rows x 128 B (64 bf16)
constexpr int kQChunkC = kQc * 128;    // 64 rows x 128 B

struct Bwd256cSmem {
  alignas(1024) uint8_t k[2][kKChunkC];       // K[:, half]: two 64-column chunks
  alignas(1024) uint8_t v[2][kKChunkC];
  alignas(1024) uint8_t q[2][2][kQChunkC];    // [stage][chunk]
  alignas(1024) uint8_t dout[2][2][kQChunkC];
  alignas(1024) uint8_t ds[kKChunkC];         // dS^T: 128 keys x 64 q, bf16, 128B-swizzled
  alignas(1024) float xs[kTile * kQc];        // the peer's partial S^T, [key][q], 16-byte pieces swizzled
  alignas(1024) float xdp[kTile * kQc];       // the peer's partial dP^T
  alignas(16) float lse2[2][kQc];             // per q row of a stage: lse * log2(e)
  alignas(16) float delta[2][kQc];            // per q row: scale * delta
  uint64_t kv_full, q_full[2], q_empty[2];
  uint64_t sdp_full, x_full, x_empty, p_full, ds_full, ds_empty, dq_full[2], dq_empty[2], acc_full, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, kt, q64_lo, nq64, n_real, skip, mode;
};
static_assert(sizeof(Bwd256cSmem) + 1024 <= 232448, "shared memory per CTA");

// ---------------------------------------------------------- cluster helpers
// Address in the peer CTA's shared memory of this CTA's `local` object.
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t peer_rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(peer_rank));
  return r;
}

__device__ __forceinline__ void st_peer_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// One arrival on a barrier in the peer CTA, ordered after this thread's
// earlier shared-memory accesses (release at cluster scope).
__device__ __forceinline__ void arrive_peer(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}

__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Warp-wide bounded wait on a barrier the peer CTA arrives on (acquire at
// cluster scope, so the peer's stores before its arrivals are visible); the
// same limits and abort rules as the other pipeline waits.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, int* abort_flag,
                                                  volatile int* gstatus) {
  bool ok = try_wait_cluster(bar, parity);
  uint64_t t0 = 0;
  uint32_t n = 0;
  while (!ok) {
    if (try_wait_cluster(bar, parity)) {
      ok = true;
      break;
    }
    if ((++n & 255u) == 0u) {
      if (*abort_flag) break;
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      const uint64_t waited = now - t0;
      if (waited > kWaitLimitNs) break;
      if (waited > 100000ull && (*gstatus & kAbortBits)) break;
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void red_add_c(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Byte offset of the 16-byte piece `piece` (0..15) of key row r in an
// exchange buffer ([128 keys][64 q] fp32, 256 B per row): pieces are
// XOR-swizzled by the row within 128-byte halves, so the 32 rows a warp
// touches at once spread over all banks.
__device__ __forceinline__ uint32_t xoff(int r, int piece) {
  return static_cast<uint32_t>(r) * 256u + static_cast<uint32_t>(((piece & 8) | ((piece ^ r) & 7)) << 4);
}

constexpr int kModeIdleC = 0, kModeWorkC = 1;

template <bool kDq, bool kDrop>
__global__ void __launch_bounds__(kThreadsC, 1)
    bwd256c_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                   const float* __restrict__ delta, float* __restrict__ dq_acc, void* __restrict__ dk,
                   void* __restrict__ dv, int grads_bf16, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  Bwd256cSmem& s = *reinterpret_cast<Bwd256cSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = blockIdx.x & 1u, peer = rank ^ 1u;  // cluster of two consecutive CTAs
  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int hk = unit % g.Hkv, item = unit / g.Hkv;
  volatile int* vstatus = status;

  if (tid == 0) {
    // the attended K/V tiles lead the work list; both CTAs read the same count
    const int n_att = seg[g.off[BD_SEG_OFF_COUNTS] + 3];
    int mode = kModeIdleC;
    if (n_att < 0 || n_att > g.B * g.nkt || n_att > static_cast<int>(gridDim.x / 2) / g.Hkv)
      atomicOr(status, BD_STATUS_BOUNDS);
    else
      mode = item < n_att ? kModeWorkC : kModeIdleC;
    s.mode = mode;
  }
  __syncthreads();
  if (s.mode != kModeWorkC) return;  // both CTAs of an idle cluster leave here

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
    ok = ok && n_real >= 0 && n_real <= g.L && qlo >= 0 && qhi <= n_real && qlo < qhi;
    if (!ok) atomicOr(status, BD_STATUS_BOUNDS);
    s.b = b;
    s.kt = kt;
    s.q64_lo = ok ? qlo / kQc : 0;
    s.nq64 = ok ? (qhi - 1) / kQc - qlo / kQc + 1 : 0;
    s.n_real = n_real;
    s.skip = (!ok || *vstatus != 0) ? 1 : 0;
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.dq_full[i], 1);
      mbar_init(&s.dq_empty[i], 128);
    }
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.x_full, 256);   // the peer's 256 P / dS threads, one arrival each per tile
    mbar_init(&s.x_empty, 256);
    mbar_init(&s.p_full, 256);
    mbar_init(&s.ds_full, 256);
    mbar_init(&s.ds_empty, 1);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  // no CTA touches its peer's shared memory before the peer's barriers exist;
  // from here on every thread of both CTAs reaches the final cluster barrier
  cluster_sync_all();
  // a skipping CTA (bad table or an earlier error) still joins the final
  // barrier; its peer's waits on it give up within their limits
  const bool run = !s.skip;
  const int b = s.b, kt = s.kt, q64_lo = s.q64_lo, nq64 = s.nq64, n_real = s.n_real;
  const int G = g.G;
  const int n_it = G * nq64;  // iteration it: query head hk*G + it / nq64, q tile q64_lo + it % nq64
  const bool is_pds = (warp >= 4 && warp < 8) || warp >= 12;
  const int half = warp >= 12 ? 1 : 0;
  const int d0 = static_cast<int>(rank) * kHalf;  // this CTA's head-dim columns
  auto decode = [&](int it, int& h, int& q0) {
    const int gq = it / nq64;
    h = hk * G + gq;
    q0 = (q64_lo + it - gq * nq64) * kQc;
  };

  if (run && warp == 2) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;

  if (!run) {
    // nothing to do
  } else if (warp == 0) {
    // -------------------------------------------------------------- loads
    const int pl = b * g.Hkv + hk;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_dout);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.kv_full, 4 * kKChunkC);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(s.k[c], &tm_k, &s.kv_full, d0 + c * 64, g.kv_tm ? pl : kt * kTile, g.kv_tm ? kt * kTile : pl);
        tma_load_3d(s.v[c], &tm_v, &s.kv_full, d0 + c * 64, g.kv_tm ? pl : kt * kTile, g.kv_tm ? kt * kTile : pl);
      }
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;
      int h, q0;
      decode(it, h, q0);
      // the per-row values are fetched before waiting for the free stage
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
      if (it >= 2 && !warp_wait(&s.q_empty[st], ((it >> 1) - 1) & 1, &s.abort_flag, vstatus)) break;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s.lse2[st][lane + 32 * e] = l2[e];
        s.delta[st][lane + 32 * e] = dl[e];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.q_full[st], 4 * kQChunkC);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(s.q[st][c], &tm_q, &s.q_full[st], d0 + c * 64, q0, b * g.Hq + h);
          tma_load_3d(s.dout[st][c], &tm_dout, &s.q_full[st], d0 + c * 64, q0, b * g.Hq + h);
        }
      }
      ++issued;
    }
    if (lane == 0) {
      if (issued < n_it) {
        s.abort_flag = 1;
        atomicOr(status, BD_STATUS_TIMEOUT);
      }
      // no copy into this CTA's shared memory may still be in flight at exit
      mbar_wait_drain(&s.kv_full, 0);
      for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it) mbar_wait_drain(&s.q_full[it & 1], (it >> 1) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idST = idesc_bf16(128, kQc, false, false);   // partial S^T, dP^T
      constexpr uint32_t idDKV = idesc_bf16(128, kHalf, false, true);  // dV, dK halves
      constexpr uint32_t idDQ = idesc_bf16(128, kQc, true, true);     // dQ^T half
      const uint64_t dKm = umma_desc_sw128(0, 16, 1024);               // K-major operands
      const uint64_t dMN_q = umma_desc_sw128(0, kQChunkC, 1024);       // MN-major, 64-row chunks
      const uint64_t dMN_k = umma_desc_sw128(0, kKChunkC, 1024);       // MN-major, 128-row chunks
      const uint32_t a_k = smem_u32(s.k[0]), a_v = smem_u32(s.v[0]), a_ds = smem_u32(s.ds);
      const uint32_t a_q = smem_u32(s.q[0][0]), a_do = smem_u32(s.dout[0][0]);
      constexpr uint32_t kStage = 2 * kQChunkC;
      // X^T (partial) = A B^T over this CTA's half of the head dim
      auto issue_t = [&](uint32_t col, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int ks = 0; ks < kHalf / 16; ++ks) {
          const uint32_t off_a = (ks >> 2) * kKChunkC + (ks & 3) * 32;
          const uint32_t off_b = (ks >> 2) * kQChunkC + (ks & 3) * 32;
          umma_ss(tbase + col, desc_at(dKm, a_base + off_a), desc_at(dKm, b_base + off_b), idST, ks > 0 ? 1u : 0u);
        }
      };
      auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
      bool ok = wait(&s.kv_full, 0) && wait(&s.q_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_t(kColSc, a_k, a_q);
        issue_t(kColDpc, a_v, a_do);
        umma_commit(&s.sdp_full);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it & 1;
        // dV[:, half] += P^T dO[:, half]; P^T is bf16 in tensor memory, q columns
        // 0-31 at column offset 0 and 32-63 at offset 48 (each half over its own S^T)
        if (!wait(&s.p_full, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kQc / 16; ++ks) {
          const uint32_t a_col = kColSc + (ks < 2 ? ks * 8 : 48 + (ks - 2) * 8);
          umma_ts(tbase + kColDvc, tbase + a_col, desc_at(dMN_q, a_do + st * kStage + ks * 2048), idDKV,
                  (it > 0 || ks > 0) ? 1u : 0u);
        }
        // dK[:, half] += dS^T Q[:, half] ; dQ^T[half] = K[:, half]^T dS^T
        if (!wait(&s.ds_full, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kQc / 16; ++ks)
          umma_ss(tbase + kColDkc, desc_at(dKm, a_ds + ks * 32), desc_at(dMN_q, a_q + st * kStage + ks * 2048), idDKV,
                  (it > 0 || ks > 0) ? 1u : 0u);
        if constexpr (kDq) {
          const int bq = it & 1;  // dQ^T tensor-memory buffer
          if (it >= 2 && !wait(&s.dq_empty[bq], ((it >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_ss(tbase + kColDqc + 64 * bq, desc_at(dMN_k, a_k + ks * 2048), desc_at(dMN_k, a_ds + ks * 2048),
                    idDQ, ks > 0 ? 1u : 0u);
          umma_commit(&s.dq_full[bq]);
        }
        umma_commit(&s.ds_empty);
        umma_commit(&s.q_empty[st]);
        if (it + 1 == n_it) umma_commit(&s.acc_full);
        // the next tile's partial S^T (over P^T, which the dV product above
        // read first) and dP^T (read by the P / dS warps before dS was formed)
        if (it + 1 < n_it) {
          if (!wait(&s.q_full[st ^ 1], ((it + 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_t(kColSc, a_k, a_q + (st ^ 1) * kStage);
          issue_t(kColDpc, a_v, a_do + (st ^ 1) * kStage);
          umma_commit(&s.sdp_full);
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
    // ------------------ exchange, P and dS (key rows; one half of the q columns)
    const int r = (warp & 3) * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int j = kt * kTile + r;  // K/V buffer row of this thread
    const int c0 = half * 32;      // first q column of this half
    const float sl2 = g.scale * 1.4426950408889634f;
    uint8_t* ds_row = s.ds + r * 128;
    const uint32_t xs_peer = peer_addr(s.xs, peer), xdp_peer = peer_addr(s.xdp, peer);
    const uint32_t xfull_peer = peer_addr(&s.x_full, peer), xempty_peer = peer_addr(&s.x_empty, peer);
    const uint8_t* xs_loc = reinterpret_cast<const uint8_t*>(s.xs);
    const uint8_t* xdp_loc = reinterpret_cast<const uint8_t*>(s.xdp);
    // rows [key, row_end) of the real rows attend this thread's key
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
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;
      int h, q0;
      decode(it, h, q0);
      uint64_t km = 0;  // dropout: keep bits of this key over the half's 32 q columns
      if constexpr (kDrop)
        km = key_keep_mask<4>(g, b, h, g.row_offset + q0 + c0, g.kv_offset + kt * kTile + (warp & 3) * 32, lane);
      if (!warp_wait(&s.q_full[st], (it >> 1) & 1, &s.abort_flag, vstatus) ||
          !warp_wait(&s.sdp_full, it & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[32], dr[32];  // this CTA's partial S^T and dP^T of the half's 32 q columns
      tmem_ld32(tbase + lane_off + kColSc + c0, sr);
      tmem_ld32(tbase + lane_off + kColDpc + c0, dr);
      tmem_wait_ld();
      // hand them to the peer, once it has read what it got for the previous tile
      if (it > 0 && !warp_wait_cluster(&s.x_empty, (it - 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t o = xoff(r, 8 * half + k);
        st_peer_v4(xs_peer + o, __uint_as_float(sr[4 * k]), __uint_as_float(sr[4 * k + 1]),
                   __uint_as_float(sr[4 * k + 2]), __uint_as_float(sr[4 * k + 3]));
        st_peer_v4(xdp_peer + o, __uint_as_float(dr[4 * k]), __uint_as_float(dr[4 * k + 1]),
                   __uint_as_float(dr[4 * k + 2]), __uint_as_float(dr[4 * k + 3]));
      }
      arrive_peer(xfull_peer);
      // the peer's partials complete S^T and dP^T
      if (!warp_wait_cluster(&s.x_full, it & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      float sv[32], dpv[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t o = xoff(r, 8 * half + k);
        const float4 a = *reinterpret_cast<const float4*>(xs_loc + o);
        const float4 d = *reinterpret_cast<const float4*>(xdp_loc + o);
        sv[4 * k] = __uint_as_float(sr[4 * k]) + a.x;
        sv[4 * k + 1] = __uint_as_float(sr[4 * k + 1]) + a.y;
        sv[4 * k + 2] = __uint_as_float(sr[4 * k + 2]) + a.z;
        sv[4 * k + 3] = __uint_as_float(sr[4 * k + 3]) + a.w;
        dpv[4 * k] = __uint_as_float(dr[4 * k]) + d.x;
        dpv[4 * k + 1] = __uint_as_float(dr[4 * k + 1]) + d.y;
        dpv[4 * k + 2] = __uint_as_float(dr[4 * k + 2]) + d.z;
        dpv[4 * k + 3] = __uint_as_float(dr[4 * k + 3]) + d.w;
      }
      arrive_peer(xempty_peer);  // this CTA's buffer is read: the peer may write the next tile's
      // q columns [c_lo, c_hi) of this tile attend the key (relative to c0)
      const int row0 = g.row_offset + q0;
      const int c_lo = max(0, key - row0) - c0;
      const int c_hi = min(min(kQc, n_real - q0), row_end - row0) - c0;
      float p[32];
      const float4* l4 = reinterpret_cast<const float4*>(s.lse2[st] + c0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l = l4[c4];
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * c4 + e;
          const float pe = fast_exp2(sv[c] * sl2 - lv[e]);
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
      tmem_st16(tbase + lane_off + kColSc + 48 * half, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);

      const float4* d4 = reinterpret_cast<const float4*>(s.delta[st] + c0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 dl = d4[c4];
        const int c = 4 * c4;
        float dp[4] = {dpv[c], dpv[c + 1], dpv[c + 2], dpv[c + 3]};
        if constexpr (kDrop) {
#pragma unroll
          for (int e = 0; e < 4; ++e) dp[e] = ((km >> (c + e)) & 1u) ? dp[e] : 0.f;
        }
        pk[2 * c4] = pack_bf16x2(p[c] * fmaf(dp[0], sc_dp, -dl.x), p[c + 1] * fmaf(dp[1], sc_dp, -dl.y));
        pk[2 * c4 + 1] = pack_bf16x2(p[c + 2] * fmaf(dp[2], sc_dp, -dl.z), p[c + 3] * fmaf(dp[3], sc_dp, -dl.w));
      }
      if (it > 0 && !warp_wait(&s.ds_empty, (it - 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      // this half's 64 B of the key row of dS^T, 128B-swizzled K-major layout
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int c16 = 4 * half + k4;
        *reinterpret_cast<uint4*>(ds_row + ((c16 ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&s.ds_full);
    }
    if (ok) {
      // this thread's dK / dV row: its half of this CTA's 128 columns
      if (!warp_wait(&s.acc_full, 0, &s.abort_flag, vstatus)) {
        ok = false;
      } else {
        tc_fence_after();
#pragma unroll 1
        for (int c = half * (kHalf / 2); c < (half + 1) * (kHalf / 2); c += 32) {
          uint32_t vv[32], kk[32];
          tmem_ld32(tbase + lane_off + kColDvc + c, vv);
          tmem_ld32(tbase + lane_off + kColDkc + c, kk);
          tmem_wait_ld();
          if (j < g.S_kv) {
            const float dvs = kDrop ? g.drop_scale : 1.0f;  // dropout: the keep scale of P^T
            const size_t off = kv_row(g, b, hk, j) * kDc + d0 + c;
            if (grads_bf16) {
              uint4* pv = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dv) + off);
              uint4* pkk = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dk) + off);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pv[e] = make_uint4(pack_bf16x2(__uint_as_float(vv[8 * e]) * dvs, __uint_as_float(vv[8 * e + 1]) * dvs),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 2]) * dvs, __uint_as_float(vv[8 * e + 3]) * dvs),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 4]) * dvs, __uint_as_float(vv[8 * e + 5]) * dvs),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 6]) * dvs, __uint_as_float(vv[8 * e + 7]) * dvs));
                pkk[e] = make_uint4(pack_bf16x2(__uint_as_float(kk[8 * e]), __uint_as_float(kk[8 * e + 1])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 2]), __uint_as_float(kk[8 * e + 3])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 4]), __uint_as_float(kk[8 * e + 5])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 6]), __uint_as_float(kk[8 * e + 7])));
              }
            } else {
              float4* pv = reinterpret_cast<float4*>(reinterpret_cast<float*>(dv) + off);
              float4* pkk = reinterpret_cast<float4*>(reinterpret_cast<float*>(dk) + off);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pv[e] = make_float4(__uint_as_float(vv[4 * e]) * dvs, __uint_as_float(vv[4 * e + 1]) * dvs,
                                    __uint_as_float(vv[4 * e + 2]) * dvs, __uint_as_float(vv[4 * e + 3]) * dvs);
                pkk[e] = make_float4(__uint_as_float(kk[4 * e]), __uint_as_float(kk[4 * e + 1]),
                                     __uint_as_float(kk[4 * e + 2]), __uint_as_float(kk[4 * e + 3]));  // pre-scaled
              }
            }
          }
        }
      }
    }
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    }
  } else if (kDq && warp >= 8 && warp < 12) {
    // ----------------------------------------------- dQ read-out (d rows)
    const int r = tid - 256;  // d index within this CTA's half == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      int h, q0;
      decode(it, h, q0);
      const int bq = it & 1;
      if (!warp_wait(&s.dq_full[bq], (it >> 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t qv[64];
      tmem_ld32(tbase + lane_off + kColDqc + 64 * bq, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
      tmem_ld32(tbase + lane_off + kColDqc + 64 * bq + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s.dq_empty[bq]);
      float* base = dq_acc + ((static_cast<size_t>(b) * g.Hq + h) * g.L) * kDc + d0 + r;
      const int cmax = min(kQc, n_real - q0);
      if (cmax >= kQc) {  // full tile: no per-value row check on the red stream
#pragma unroll
        for (int c = 0; c < kQc; ++c) red_add_c(base + static_cast<size_t>(q0 + c) * kDc, __uint_as_float(qv[c]));
      } else {
#pragma unroll
        for (int c = 0; c < kQc; ++c)
          if (c < cmax) red_add_c(base + static_cast<size_t>(q0 + c) * kDc, __uint_as_float(qv[c]));
      }
    }
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (run && warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // neither CTA leaves while its peer may still write into its shared memory
  cluster_sync_all();
}

}  // namespace

// K4h launch: clusters of two CTAs, one cluster per (K/V tile some local row
// can reach by position, kv head); the zero-fill kernel writes the dK / dV of
// the others. Without a dq accumulator (dq_acc null) the dq products are left out.
cudaError_t launch_bwd256c_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                                const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                                const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                                cudaStream_t st) {
  if (g.D != kDc) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Bwd256cSmem) + 1024;  // + 1 KB to align the swizzled tiles
  auto kern = g.drop_t ? (dq_acc ? bwd256c_kernel<true, true> : bwd256c_kernel<false, true>)
                       : (dq_acc ? bwd256c_kernel<true, false> : bwd256c_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int reach = kv_tiles_reachable(g);
  const long long grid = 2LL * g.B * (reach > 0 ? reach : 1) * g.Hkv;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreadsC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16,
      status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
