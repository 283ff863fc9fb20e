// K4g: dq of the backward in a fixed order for D = 512 -- deterministic (the
// pages' `_CP_FLASH_DETERMINISTIC`), the head-dim-512 counterpart of K4d / K4f.
// S (128 columns), dP (128) and the whole 128 x 512 dQ (512) would need 768
// tensor-memory columns, so dQ is split into two 256-column halves, one CTA
// each: CTA (q tile, query head, half) walks the q tile's K/V tiles in
// increasing order, forms the whole S = Q K^T and dP = dO V^T (contractions
// over all 512 columns), dS over S as in K4f, and accumulates its half
//   dQ[:, 256 half + 64c : + 64] += dS K[:, 256 half + 64c : + 64]   (TS form)
// in tensor memory, writing it once. Neither Q / dO (256 KB) nor a K/V tile
// fits in shared memory, so everything streams through a ring of 32 KB
// slots, per K/V tile in the order the products use it: (Q, K) chunk pairs
// for S, (dO, V) pairs for dP, then this half's K chunks for dQ.
//   warp 0   TMA: the chunk ring      warp 1  one thread issues the MMAs
//   warp 2   tensor memory            warps 4-7  thread = q row: P, dS, dq rows
// With attention dropout (kDrop) each row draws its keep mask of a K/V tile
// (dropout.cuh) before the tile's S and dP arrive: dS = P (Z dP - delta).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dq_stream.cuh"
#include "dropout.cuh"

namespace bd {

namespace {

constexpr int kD5 = 512;
constexpr int kChunks5 = kD5 / 64;       // 64-column chunks per row
constexpr int kHalfChunks = kChunks5 / 2;  // dQ chunks per CTA
constexpr int kChunkB5 = kTile * 128;    // 128 rows x 128 B
constexpr int kSlots5 = 6;               // ring slots
constexpr int kPerTile5 = 2 * kChunks5 + kHalfChunks;  // (Q, K), (dO, V), K
constexpr int kThreads5 = 256;
constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 256;

struct RingSlot5 {
  alignas(1024) uint8_t a[kChunkB5];  // q side: a Q or dO chunk
  alignas(1024) uint8_t b[kChunkB5];  // K/V side: a K or V chunk
};

struct Dq512Smem {
  RingSlot5 ring[kSlots5];
  uint64_t r_full[kSlots5], r_empty[kSlots5];
  uint64_t sdp_full;  // S and dP of the current tile are in tensor memory
  uint64_t ds_full;   // dS of the current tile is in tensor memory (128 arrivals)
  uint64_t dq_done;   // every dQ product is complete
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, qt, kt_lo, nk, n_real, skip;
};
static_assert(sizeof(Dq512Smem) + 1024 <= 232448, "shared memory per CTA");

template <bool kDrop>
__global__ void __launch_bounds__(kThreads5, 1)
    bwd_dq512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                     const float* __restrict__ delta, void* __restrict__ dq, int dq_bf16, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  Dq512Smem& s = *reinterpret_cast<Dq512Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = static_cast<int>(blockIdx.x) & 1;  // dQ columns [256 half, 256 half + 256)
  const int h = (static_cast<int>(blockIdx.x) >> 1) % g.Hq, hk = h / g.G;
  volatile int* vstatus = status;

  if (tid == 0) {
    const int item = (static_cast<int>(blockIdx.x) >> 1) / g.Hq;
    const int wi = seg[g.off[BD_SEG_OFF_FWD_WORK] + item];
    int ok = wi >= 0 && wi < g.B * g.nqt;
    const int b = ok ? wi / g.nqt : 0, qt = ok ? wi % g.nqt : 0;
    const int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
    ok = ok && hdr[kHdrMagic] == kSegMagic && hdr[kHdrRowOffset] == g.row_offset && hdr[kHdrL] == g.L &&
         hdr[kHdrKvOffset] == g.kv_offset && hdr[kHdrSkv] == g.S_kv && hdr[kHdrWindow] == g.window &&
         hdr[kHdrSfull] == g.S_full;
    const int n_real = hdr[BD_SEG_N_REAL];
    const int32_t* kr = seg + g.off[BD_SEG_OFF_QT_KRANGE] + (b * g.nqt + qt) * 2;
    const int kt_lo = kr[0], kt_hi = kr[1];
    const int nk = kt_hi >= kt_lo ? kt_hi - kt_lo + 1 : 0;
    ok = ok && n_real >= 0 && n_real <= g.L && (nk == 0 || (kt_lo >= 0 && kt_hi < g.nkt));
    if (!ok) atomicOr(status, BD_STATUS_BOUNDS);
    s.b = b;
    s.qt = qt;
    s.kt_lo = kt_lo;
    s.nk = nk;
    s.n_real = n_real;
    s.skip = (!ok || *vstatus != 0) ? 1 : 0;
    s.abort_flag = 0;
    for (int i = 0; i < kSlots5; ++i) {
      mbar_init(&s.r_full[i], 1);
      mbar_init(&s.r_empty[i], 1);
    }
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.ds_full, 128);
    mbar_init(&s.dq_done, 1);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, qt = s.qt, kt_lo = s.kt_lo, nk = s.nk, n_real = s.n_real;
  const size_t row0 = (static_cast<size_t>(b) * g.Hq + h) * g.L;  // dq / lse / delta row of local row 0
  const size_t elem = dq_bf16 ? 2 : 4;

  if (nk == 0) {  // no row of this q tile sees a key: this half of dq = 0
    if (tid >= 128) {
      const int i = qt * kTile + (tid - 128);
      if (i < g.L) {
        uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dq) + ((row0 + i) * kD5 + 256 * half) * elem);
        for (size_t c = 0; c < 256 * elem / 16; ++c) o4[c] = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  if (warp == 2) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_dout);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    const int pl = b * g.Hkv + hk, qpl = b * g.Hq + h, q0 = qt * kTile;
    int n = 0;  // ring chunks issued
    bool ok = true;
    for (int j = 0; ok && j < nk; ++j) {
      const int row = (kt_lo + j) * kTile;
      const int kx = g.kv_tm ? pl : row, ky = g.kv_tm ? row : pl;
      for (int u = 0; u < kPerTile5; ++u) {
        const int sl = n % kSlots5;
        if (n >= kSlots5 && !pipe_wait(&s.r_empty[sl], (n / kSlots5 - 1) & 1, &s.abort_flag, vstatus)) {
          ok = false;
          break;
        }
        if (u < 2 * kChunks5) {  // (Q, K) for S, then (dO, V) for dP
          const bool is_s = u < kChunks5;
          const int c = u % kChunks5;
          mbar_arrive_expect_tx(&s.r_full[sl], 2 * kChunkB5);
          tma_load_3d(s.ring[sl].a, is_s ? &tm_q : &tm_dout, &s.r_full[sl], c * 64, q0, qpl);
          tma_load_3d(s.ring[sl].b, is_s ? &tm_k : &tm_v, &s.r_full[sl], c * 64, kx, ky);
        } else {  // this half's K chunks for dQ
          const int c = kHalfChunks * half + (u - 2 * kChunks5);
          mbar_arrive_expect_tx(&s.r_full[sl], kChunkB5);
          tma_load_3d(s.ring[sl].b, &tm_k, &s.r_full[sl], c * 64, kx, ky);
        }
        ++n;
      }
    }
    if (!ok) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // no copy into this CTA's shared memory may still be in flight at exit
    for (int x = (n > kSlots5 ? n - kSlots5 : 0); x < n; ++x)
      mbar_wait_drain(&s.r_full[x % kSlots5], (x / kSlots5) & 1);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idX = idesc_bf16(128, 128, false, false);  // S, dP: both operands K-major
    constexpr uint32_t idDQ = idesc_bf16(128, 64, false, true);   // dQ chunk: dS from TMEM, K chunk MN-major
    const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);
    const uint64_t dMN = umma_desc_sw128(0, kChunkB5, 1024);
    auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
    int n = 0;  // ring chunks consumed
    // the slot of the next ring chunk, once it has landed
    auto next_chunk = [&](int& sl) -> bool {
      sl = n % kSlots5;
      if (!wait(&s.r_full[sl], (n / kSlots5) & 1)) return false;
      tc_fence_after();
      return true;
    };
    bool ok = true;
    for (int j = 0; ok && j < nk; ++j) {
      // S = Q K^T, then dP = dO V^T, over the eight chunks of the head dim (the
      // previous tile's dQ products, issued before, have read its dS out of
      // the S columns, and its dP was read before ds_full)
      for (int u = 0; u < 2 * kChunks5; ++u) {
        int sl;
        if (!next_chunk(sl)) {
          ok = false;
          break;
        }
        const int c = u % kChunks5;
        const uint32_t aa = smem_u32(s.ring[sl].a), bb = smem_u32(s.ring[sl].b);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_ss(tbase + (u < kChunks5 ? kColS : kColDp), desc_at(dK_major, aa + ks * 32),
                  desc_at(dK_major, bb + ks * 32), idX, (c > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.r_empty[sl]);
        ++n;
      }
      if (!ok) break;
      umma_commit(&s.sdp_full);
      // this half of dQ += dS K, chunk by chunk; dS is bf16 in the S columns
      if (!wait(&s.ds_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < kHalfChunks; ++c) {
        int sl;
        if (!next_chunk(sl)) {
          ok = false;
          break;
        }
        const uint32_t bb = smem_u32(s.ring[sl].b);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          umma_ts(tbase + kColDq + 64 * c, tbase + kColS + ks * 8, desc_at(dMN, bb + ks * 2048), idDQ,
                  (j > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.r_empty[sl]);
        ++n;
      }
    }
    if (ok) {
      umma_commit(&s.dq_done);
    } else {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    umma_commit(&s.mma_drain);
    mbar_wait_drain(&s.mma_drain, 0);
  } else if (warp >= 4) {
    // ------------------------------------------- P and dS (thread = q row)
    const int r = tid - 128;  // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int i = qt * kTile + r;
    const bool real = i < n_real;
    int jlo = 1, jhi = 0;  // allowed K/V buffer rows [jlo, jhi] of this row
    float nl2 = 0.f, ndl = 0.f;
    if (real) {
      const int p = g.row_offset + i;
      const int doc_start = seg[g.off[BD_SEG_OFF_ROW_LO] + b * g.L + i];
      jlo = row_lo_window(doc_start, p, g.window) - g.kv_offset;
      jhi = min(p - g.kv_offset, g.S_kv - 1);  // a K/V chunk may end before the row
      nl2 = lse[row0 + i] * -1.4426950408889634f;
      ndl = delta[row0 + i] * -g.scale;  // dS is formed pre-scaled: scale * P (dP - delta)
    }
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      uint32_t km[4] = {0u, 0u, 0u, 0u};  // dropout: keep bits of this row over the tile's 128 keys
      if constexpr (kDrop) row_keep_mask(g, b, h, g.row_offset + i, g.kv_offset + (kt_lo + j) * kTile, km);
      if (!warp_wait(&s.sdp_full, j & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int c0 = (kt_lo + j) * kTile;
      // a row sees all of this tile, none of it, or part of it
      const bool dead = !real || jhi < c0 || jlo > c0 + kTile - 1;
      const bool full = jlo <= c0 && c0 + kTile - 1 <= jhi;
      uint32_t pk[2][32];  // dS of keys [64 hf, 64 hf + 64), bf16 pairs
      dq_form_ds<kDrop>(tbase + lane_off + kColS, tbase + lane_off + kColDp, g.scale, nl2, ndl, dead, full, jlo - c0,
                        jhi - c0, pk, km, g.drop_scale);
      // dS over this row's S columns (read above): the A operand of the dQ products
      tmem_st32(tbase + lane_off + kColS, pk[0]);
      tmem_st32(tbase + lane_off + kColS + 32, pk[1]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.ds_full);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !warp_wait(&s.dq_done, 0, &s.abort_flag, vstatus)) ok = false;
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    } else {
      tc_fence_after();
      dq_store_cols(tbase + lane_off + kColDq, 256, dq, (row0 + i) * kD5 + 256 * half, dq_bf16, i < g.L);
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

// dq in a fixed order for D = 512 (q and dout maps with 128-row boxes): two
// CTAs per (q tile, query head), one per 256-column half.
cudaError_t launch_bwd_dq512(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                             const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                             const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st) {
  if (g.D != kD5) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Dq512Smem) + 1024;  // + 1 KB to align the swizzled tiles
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
  auto kern = g.drop_t ? bwd_dq512_kernel<true> : bwd_dq512_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * g.Hq * 2;  // (q tile, query head, half)
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads5), smem,
      st, mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
