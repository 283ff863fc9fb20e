// K4e: backward of per-document causal attention for head dim 512.
//
// Reference (NeMo AutoModel API): gemma4_moe.cp_attention
// `_ffpa_varlen_backward_chunk` -- the backward of the head-dim-512 global
// layers from the saved (merged) out / lse. The arithmetic is that of the
// other head dims: with P = exp(scale q.k - lse) on allowed pairs and
// delta = rowsum(dout * out),
//   dV += P^T dO,  dP = dO V^T,  dS = P (dP - delta),
//   dK += scale dS^T Q,  dQ += scale dS K.
//
// Design (GB300). dK and dV of one 128-row K/V tile at D = 512 are 2 x 256 KB
// of fp32, twice the whole tensor memory, so the head dim of the outputs is
// split over four CTAs: CTA (item, kv head, slice c) owns columns
// [128 c, 128 c + 128) of dK, dV and dQ and keeps dK / dV in tensor memory
// over all the q tiles that attend its keys. Each of the four forms the whole
// S^T = K Q^T and dP^T = V dO^T (contractions over all 512 columns): its own
// slice of K and V stays in shared memory, the other six 64-column chunks of
// K, V, Q and dO stream through a two-slot ring (48 KB a slot; the four CTAs
// of a tile run side by side and read the same chunks, mostly from L2), and
// its slices of Q and dO sit in a stage that the output products read.
// The tensor-memory map is that of the D = 256 kernel:
//   S^T  [0, 64)   dP^T  [64, 128)   dQ^T  [128, 256) (two buffers)
//   dV   [256, 384)   dK  [384, 512)
//   warp 0  loads          warp 1  issues the MMAs       warp 2  owns the tensor memory
//   warps 4-7 and 12-15  P, dS (thread = key row; q columns 0-31 / 32-63)
//   warps 8-11  dQ read-out (thread = d row of the slice), red.global.add
// The tensor pipe runs 22 D FLOPs per allowed (row, key) pair against the
// 10 D counted: S^T and dP^T are formed once per slice.
// With attention dropout (kDrop) each P / dS warp draws its 32 keys' keep
// masks over the half's q columns (dropout.cuh): dropped weights are zeroed in
// P^T, dS = P (Z dP - delta), and dV is scaled by the keep scale when written.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {
namespace {

constexpr int kD5 = 512;
constexpr int kSlice = 128;               // output columns per CTA
constexpr int kNSlice = kD5 / kSlice;     // CTAs per (K/V tile, kv head)
constexpr int kRingSlots = 2;
constexpr int kStreamed = kD5 / 64 - 2;   // 64-column chunks through the ring per q tile
constexpr int kKChunkB = kTile * 128;     // 128 rows x 128 B
constexpr int kQChunkB = kBwdQ * 128;     // 64 rows x 128 B
constexpr int kThreads5 = 512;
constexpr int kZeroCtas5 = 152;  // CTAs that carry the zero-fill (the first wave on 152 SMs)
constexpr uint32_t kColS = 0, kColDp = 64, kColDq = 128, kColDv = 256, kColDk = 384;

struct RingSlot {  // chunk e of K, V (the K/V tile's rows) and of Q, dO (the q tile's rows)
  alignas(1024) uint8_t k[kKChunkB];
  alignas(1024) uint8_t v[kKChunkB];
  alignas(1024) uint8_t q[kQChunkB];
  alignas(1024) uint8_t dout[kQChunkB];
};

struct Bwd512Smem {
  alignas(1024) uint8_t kc[2][kKChunkB];   // this slice's two K chunks (resident)
  alignas(1024) uint8_t vc[2][kKChunkB];   // and V chunks
  alignas(1024) uint8_t qs[2][kQChunkB];   // this slice's Q chunks of the current q tile
  alignas(1024) uint8_t dos[2][kQChunkB];  // and dO chunks
  RingSlot ring[kRingSlots];               // the other six chunks, one per slot
  alignas(1024) uint8_t ds[kKChunkB];      // dS^T, 128 keys x 64 q, bf16, 128B-swizzled
  alignas(16) float lse2[2][kBwdQ];        // per q row: lse log2(e), by tile parity
  alignas(16) float delta[2][kBwdQ];       // per q row: scale * delta
  uint64_t kv_full, qs_full, qs_empty, r_full[kRingSlots], r_empty[kRingSlots];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full[2], dq_empty[2], acc_full, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, kt, q64_lo, nq64, n_real, skip, work, n_att;
};

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Chunk index (of the eight 64-column chunks) of the i-th streamed chunk of slice c.
__device__ __forceinline__ int streamed_chunk(int c, int i) { return i < 2 * c ? i : i + 2; }

// kDq: with the dq products (else dK / dV only, for the fixed-order dq pass).
template <bool kDq, bool kDrop>
__global__ void __launch_bounds__(kThreads5, 1)
    bwd512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                  const float* __restrict__ delta, float* __restrict__ dq_acc, void* __restrict__ dk,
                  void* __restrict__ dv, int grads_bf16, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw so the compiler keeps the shared address space
  Bwd512Smem& s = *reinterpret_cast<Bwd512Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = static_cast<int>(blockIdx.x) % kNSlice;
  const int hk = (static_cast<int>(blockIdx.x) / kNSlice) % g.Hkv;
  const int item = static_cast<int>(blockIdx.x) / kNSlice / g.Hkv;
  volatile int* vstatus = status;

  if (tid == 0) {
    // the attended K/V tiles lead the work list; the grid must cover them
    const int n_att = seg[g.off[BD_SEG_OFF_COUNTS] + 3];
    int work = 0;
    s.n_att = -1;
    if (n_att < 0 || n_att > g.B * g.nkt || n_att > static_cast<int>(gridDim.x) / (kNSlice * g.Hkv)) {
      atomicOr(status, BD_STATUS_BOUNDS);
    } else {
      work = item < n_att ? 1 : 0;
      s.n_att = n_att;
    }
    s.work = work;
  }
  __syncthreads();
  // dK / dV of the tiles no local row attends are zero. With at least a wave
  // of working CTAs, warps 2-3 of the first kZeroCtas5 of them write these
  // rows during their main loop (their tiles lead the longest-first list, so
  // these CTAs run longest); with fewer, every CTA of the grid takes a share,
  // the idle ones with all their threads.
  const int n_att_s = s.n_att;
  const int n_zw = n_att_s * g.Hkv * kNSlice >= kZeroCtas5 ? kZeroCtas5 : static_cast<int>(gridDim.x);
  if (!s.work) {
    if (n_att_s >= 0 && static_cast<int>(blockIdx.x) < n_zw)
      zero_unattended_kv(seg, g, n_att_s, static_cast<int>(blockIdx.x), n_zw, tid, kThreads5, dk, dv, grads_bf16,
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
    s.q64_lo = qlo / kBwdQ;
    s.nq64 = qhi > qlo ? (qhi - 1) / kBwdQ - qlo / kBwdQ + 1 : 0;
    s.n_real = n_real;
    s.skip = (!ok || *vstatus != 0) ? 1 : 0;
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    mbar_init(&s.qs_full, 1);
    mbar_init(&s.qs_empty, 1);
    for (int i = 0; i < kRingSlots; ++i) {
      mbar_init(&s.r_full[i], 1);
      mbar_init(&s.r_empty[i], 1);
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
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, kt = s.kt, q64_lo = s.q64_lo, nq64 = s.nq64, n_real = s.n_real;
  const int G = g.G;
  const int n_it = G * nq64;  // (query head of the group, 64-row q tile) steps
  // P / dS warpgroups: warps 4-7 (half 0, q columns 0-31) and 12-15 (half 1, 32-63)
  const bool is_pds = (warp >= 4 && warp < 8) || warp >= 12;
  const int half = warp >= 12 ? 1 : 0;

  if (warp == 2) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;

  auto decode = [&](int it, int& h, int& q0) {
    const int gq = it / nq64;
    h = hk * G + gq;
    q0 = (q64_lo + it - gq * nq64) * kBwdQ;
  };

  if (warp == 0) {
    // -------------------------------------------------------------- loads
    const int pl = b * g.Hkv + hk, krow = kt * kTile;
    const int kx = g.kv_tm ? pl : krow, ky = g.kv_tm ? krow : pl;  // K/V box origin (rows, planes)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_dout);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.kv_full, 4 * kKChunkB);
      for (int u = 0; u < 2; ++u) {
        tma_load_3d(s.kc[u], &tm_k, &s.kv_full, (2 * slice + u) * 64, kx, ky);
        tma_load_3d(s.vc[u], &tm_v, &s.kv_full, (2 * slice + u) * 64, kx, ky);
      }
    }
    int rc = 0, n_qs = 0;  // ring chunks and slice stages issued
    bool stopped = false;
    for (int it = 0; it < n_it && !stopped; ++it) {
      int h, q0;
      decode(it, h, q0);
      const int qpl = b * g.Hq + h;
      // the per-row values are fetched first so that their global-load latency
      // overlaps the waits below
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
      // the six streamed chunks, in the order the S^T / dP^T products use them
      if (lane == 0) {
        for (int i = 0; i < kStreamed; ++i, ++rc) {
          const int sl = rc % kRingSlots, e = streamed_chunk(slice, i);
          if (rc >= kRingSlots && !pipe_wait(&s.r_empty[sl], (rc / kRingSlots - 1) & 1, &s.abort_flag, vstatus)) {
            stopped = true;
            break;
          }
          mbar_arrive_expect_tx(&s.r_full[sl], 2 * kKChunkB + 2 * kQChunkB);
          tma_load_3d(s.ring[sl].k, &tm_k, &s.r_full[sl], e * 64, kx, ky);
          tma_load_3d(s.ring[sl].v, &tm_v, &s.r_full[sl], e * 64, kx, ky);
          tma_load_3d(s.ring[sl].q, &tm_q, &s.r_full[sl], e * 64, q0, qpl);
          tma_load_3d(s.ring[sl].dout, &tm_dout, &s.r_full[sl], e * 64, q0, qpl);
        }
      }
      stopped = __shfl_sync(0xffffffffu, stopped ? 1 : 0, 0) != 0;
      if (stopped) break;
      // this slice's Q / dO chunks, once the previous tile's output products are done;
      // their barrier also publishes the tile's row values (slot it & 1: tile it - 2's,
      // whose readers finished before the previous tile's dK product was issued)
      if (it > 0 && !warp_wait(&s.qs_empty, (it - 1) & 1, &s.abort_flag, vstatus)) {
        stopped = true;
        break;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s.lse2[it & 1][lane + 32 * e] = l2[e];
        s.delta[it & 1][lane + 32 * e] = dl[e];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.qs_full, 4 * kQChunkB);
        for (int u = 0; u < 2; ++u) {
          tma_load_3d(s.qs[u], &tm_q, &s.qs_full, (2 * slice + u) * 64, q0, qpl);
          tma_load_3d(s.dos[u], &tm_dout, &s.qs_full, (2 * slice + u) * 64, q0, qpl);
        }
      }
      ++n_qs;
    }
    if (lane == 0) {
      if (stopped) {
        s.abort_flag = 1;
        atomicOr(status, BD_STATUS_TIMEOUT);
      }
      // no copy into this CTA's shared memory may still be in flight at exit
      mbar_wait_drain(&s.kv_full, 0);
      if (n_qs > 0) mbar_wait_drain(&s.qs_full, (n_qs - 1) & 1);
      for (int x = (rc > kRingSlots ? rc - kRingSlots : 0); x < rc; ++x)
        mbar_wait_drain(&s.r_full[x % kRingSlots], (x / kRingSlots) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idST = idesc_bf16(128, kBwdQ, false, false);  // S^T, dP^T: both K-major
      constexpr uint32_t idDKV = idesc_bf16(128, kSlice, false, true); // dV, dK: Q / dO MN-major
      constexpr uint32_t idDQ = idesc_bf16(128, kBwdQ, true, true);    // dQ^T = K^T dS^T
      const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);          // K-major operands
      const uint64_t dMN_q = umma_desc_sw128(0, kQChunkB, 1024);       // MN-major, 64-row chunks
      const uint64_t dMN_k = umma_desc_sw128(0, kKChunkB, 1024);       // MN-major, 128-row chunks
      const uint32_t a_kc = smem_u32(s.kc[0]), a_vc = smem_u32(s.vc[0]), a_ds = smem_u32(s.ds);
      const uint32_t a_qs = smem_u32(s.qs[0]), a_dos = smem_u32(s.dos[0]);
      auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
      // X^T (+)= A B^T over one 64-column chunk (A: 128 key rows, B: 64 q rows)
      auto chunk = [&](uint32_t col, uint32_t a, uint32_t bb, bool first) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_ss(tbase + col, desc_at(dK_major, a + ks * 32), desc_at(dK_major, bb + ks * 32), idST,
                  (first && ks == 0) ? 0u : 1u);
      };
      bool ok = wait(&s.kv_full, 0);
      int rc = 0;
      for (int it = 0; ok && it < n_it; ++it) {
        // S^T and dP^T over the streamed chunks, then over this slice's own
        // (the previous tile's dV product has read P^T out of the S^T columns
        // and its dS was formed from dP^T before ds_full: both issued above)
        for (int i = 0; i < kStreamed; ++i, ++rc) {
          const int sl = rc % kRingSlots;
          if (!wait(&s.r_full[sl], (rc / kRingSlots) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          chunk(kColS, smem_u32(s.ring[sl].k), smem_u32(s.ring[sl].q), i == 0);
          chunk(kColDp, smem_u32(s.ring[sl].v), smem_u32(s.ring[sl].dout), i == 0);
          umma_commit(&s.r_empty[sl]);
        }
        if (!ok || !wait(&s.qs_full, it & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < 2; ++u) chunk(kColS, a_kc + u * kKChunkB, a_qs + u * kQChunkB, false);
        umma_commit(&s.s_full);
        for (int u = 0; u < 2; ++u) chunk(kColDp, a_vc + u * kKChunkB, a_dos + u * kQChunkB, false);
        umma_commit(&s.dp_full);
        // dV += P^T dO[:, slice]; P^T is bf16 in tensor memory, q columns 0-31 at
        // column offset 0 and 32-63 at offset 48 (each half writes over its own S^T)
        if (!wait(&s.p_full, it & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBwdQ / 16; ++ks) {
          const uint32_t a_col = kColS + (ks < 2 ? ks * 8 : 48 + (ks - 2) * 8);
          umma_ts(tbase + kColDv, tbase + a_col, desc_at(dMN_q, a_dos + ks * 2048), idDKV, (it > 0 || ks > 0) ? 1u : 0u);
        }
        // dK += dS^T Q[:, slice] ; dQ^T[slice] = K[:, slice]^T dS^T
        if (!wait(&s.ds_full, it & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBwdQ / 16; ++ks)
          umma_ss(tbase + kColDk, desc_at(dK_major, a_ds + ks * 32), desc_at(dMN_q, a_qs + ks * 2048), idDKV,
                  (it > 0 || ks > 0) ? 1u : 0u);
        if constexpr (kDq) {
          const int bq = it & 1;  // dQ^T tensor-memory buffer
          if (it >= 2 && !wait(&s.dq_empty[bq], ((it >> 1) - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_ss(tbase + kColDq + 64 * bq, desc_at(dMN_k, a_kc + ks * 2048), desc_at(dMN_k, a_ds + ks * 2048),
                    idDQ, ks > 0 ? 1u : 0u);
          umma_commit(&s.dq_full[bq]);
        }
        umma_commit(&s.ds_empty);
        umma_commit(&s.qs_empty);
        if (it == n_it - 1) umma_commit(&s.acc_full);
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
    // s (documents are contiguous runs) and, with a window, p - s < W: the rows
    // attending s are [s, min(doc_end(s), s + W)) of the real rows, doc_end(s)
    // found once from cu_q.
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
    const int row_end = min(doc_end, g.window > 0 ? key + g.window : 0x3fffffff);
    // dropout: scale * keep scale multiplies a kept dP (a dropped one is zero)
    const float sc_dp = kDrop ? g.scale * g.drop_scale : g.scale;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;  // slot of this tile's row values
      int h, q0;
      decode(it, h, q0);
      uint64_t km = 0;  // dropout: keep bits of this key over the half's 32 q columns
      if constexpr (kDrop)
        km = key_keep_mask<4>(g, b, h, g.row_offset + q0 + c0, g.kv_offset + kt * kTile + (warp & 3) * 32, lane);
      // the slice stage's barrier also publishes this tile's row values
      if (!warp_wait(&s.qs_full, it & 1, &s.abort_flag, vstatus) ||
          !warp_wait(&s.s_full, it & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(tbase + lane_off + kColS + c0, sr);
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
      tmem_st16(tbase + lane_off + kColS + 48 * half, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);

      if (!warp_wait(&s.dp_full, it & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(tbase + lane_off + kColDp + c0, sr);
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
      if (it > 0 && !warp_wait(&s.ds_empty, (it - 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
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
    }
    if (ok) {
      // this thread's dK / dV row: its half of the slice's columns
      if (!warp_wait(&s.acc_full, 0, &s.abort_flag, vstatus)) {
        ok = false;
      } else {
        tc_fence_after();
#pragma unroll 1
        for (int c = half * (kSlice / 2); c < (half + 1) * (kSlice / 2); c += 32) {
          uint32_t vv[32];
          tmem_ld32(tbase + lane_off + kColDv + c, vv);
          tmem_wait_ld();
          if constexpr (kDrop) {  // dropout: the keep scale of P^T
#pragma unroll
            for (int e = 0; e < 32; ++e) vv[e] = __float_as_uint(__uint_as_float(vv[e]) * g.drop_scale);
          }
          uint32_t kk[32];
          tmem_ld32(tbase + lane_off + kColDk + c, kk);
          tmem_wait_ld();
          if (j < g.S_kv) {
            const size_t off = kv_row(g, b, hk, j) * kD5 + slice * kSlice + c;
            if (grads_bf16) {
              uint4* pv = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dv) + off);
              uint4* pk4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dk) + off);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pv[e] = make_uint4(pack_bf16x2(__uint_as_float(vv[8 * e]), __uint_as_float(vv[8 * e + 1])),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 2]), __uint_as_float(vv[8 * e + 3])),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 4]), __uint_as_float(vv[8 * e + 5])),
                                   pack_bf16x2(__uint_as_float(vv[8 * e + 6]), __uint_as_float(vv[8 * e + 7])));
                pk4[e] = make_uint4(pack_bf16x2(__uint_as_float(kk[8 * e]), __uint_as_float(kk[8 * e + 1])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 2]), __uint_as_float(kk[8 * e + 3])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 4]), __uint_as_float(kk[8 * e + 5])),
                                    pack_bf16x2(__uint_as_float(kk[8 * e + 6]), __uint_as_float(kk[8 * e + 7])));
              }
            } else {
              uint4* pv = reinterpret_cast<uint4*>(reinterpret_cast<float*>(dv) + off);
              uint4* pk4 = reinterpret_cast<uint4*>(reinterpret_cast<float*>(dk) + off);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pv[e] = make_uint4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
                pk4[e] = make_uint4(kk[4 * e], kk[4 * e + 1], kk[4 * e + 2], kk[4 * e + 3]);  // dS was pre-scaled
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
  } else if (warp == 2 || warp == 3) {
    if (static_cast<int>(blockIdx.x) < n_zw)
      zero_unattended_kv(seg, g, n_att_s, static_cast<int>(blockIdx.x), n_zw, tid - 64, 64, dk, dv, grads_bf16, status);
  } else if (kDq && warp >= 8 && warp < 12) {
    // ----------------------------------------------- dQ read-out (d rows)
    const int r = tid - 256;  // d index within the slice == TMEM lane
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
      tmem_ld32(tbase + lane_off + kColDq + 64 * bq, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
      tmem_ld32(tbase + lane_off + kColDq + 64 * bq + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s.dq_empty[bq]);
      float* base = dq_acc + ((static_cast<size_t>(b) * g.Hq + h) * g.L) * kD5 + slice * kSlice + r;
      const int cmax = min(kBwdQ, n_real - q0);
      if (cmax >= kBwdQ) {  // full tile: no per-value row check on the red stream
#pragma unroll
        for (int c = 0; c < kBwdQ; ++c) red_add_f32(base + static_cast<size_t>(q0 + c) * kD5, __uint_as_float(qv[c]));
      } else {
#pragma unroll
        for (int c = 0; c < kBwdQ; ++c)
          if (c < cmax) red_add_f32(base + static_cast<size_t>(q0 + c) * kD5, __uint_as_float(qv[c]));
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

}  // namespace

// K4e launch: one CTA per (attended K/V tile, kv head, 128-column slice), the
// four slices of a tile adjacent in the grid; only tiles some local row can
// reach by position get working CTAs (the first of them also write the others' zeros).
// Without a dq accumulator (dq_acc null) the dq products are left out.
cudaError_t launch_bwd512_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                               const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                               const float* delta, float* dq_acc, void* dk, void* dv, int bf16, int32_t* status,
                               cudaStream_t st) {
  if (g.D != kD5) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Bwd512Smem) + 1024;  // + 1 KB to align the swizzled tiles
  auto kern = g.drop_t ? (dq_acc ? bwd512_kernel<true, true> : bwd512_kernel<false, true>)
                       : (dq_acc ? bwd512_kernel<true, false> : bwd512_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int reach = kv_tiles_reachable(g);
  const long long grid = static_cast<long long>(g.B) * (reach > 0 ? reach : 1) * g.Hkv * kNSlice;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads5), smem, st,
      mq, mdo, mk, mv, seg, g, lse, delta, dq_acc, dk, dv, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
