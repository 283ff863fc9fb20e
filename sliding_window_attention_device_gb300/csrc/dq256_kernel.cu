// K4f: dq of the backward in a fixed order for D = 256 -- deterministic (the
// pages' `_CP_FLASH_DETERMINISTIC`, gemma4_moe.cp_local_ring backward), the
// head-dim-256 counterpart of K4d. One CTA owns a 128-row q tile of one query
// head and walks its K/V tiles in increasing order, accumulating dQ in tensor
// memory and writing it once:
//   S  = Q K^T, dP = dO V^T                      (TMEM cols [0,128), [128,256))
//   P  = 2^(scale log2(e) q.k - lse log2(e)) on the allowed keys, dS = P (scale
//        dP - scale delta), written as bf16 over S (cols [0,64))
//   dQ[:, 64c:64c+64] += dS K[:, 64c:64c+64]      (TMEM cols [256,512), TS form)
// Q and dO (128 KB) stay in shared memory; a K/V tile (128 KB at D = 256)
// does not fit beside them, so its 64-column chunks stream through a ring of
// 16 KB slots in the order the products use them: K (for S), V (for dP), then
// K again (for dQ, once dS is formed). The tensor pipe runs the products in
// issue order, so S of the next tile (issued after this tile's dQ products)
// never overwrites a dS they still read.
//   warp 0   TMA: Q and dO once, the chunk ring     warp 1  one thread issues the MMAs
//   warp 2   tensor memory                          warps 4-7  thread = q row: P, dS, dq rows
// With attention dropout (kDrop) each row draws its keep mask of a K/V tile
// (dropout.cuh) before the tile's S and dP arrive: dS = P (Z dP - delta).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dq_stream.cuh"
#include "dropout.cuh"

namespace bd {

namespace {

constexpr int kD256 = 256;
constexpr int kChunks256 = kD256 / 64;   // 64-column (128 B) chunks per row
constexpr int kChunkB256 = kTile * 128;  // 128 rows x 128 B
constexpr int kSlots256 = 6;             // ring slots
constexpr int kPerTile = 3 * kChunks256; // ring chunks per K/V tile: K, V, K
constexpr int kThreads256 = 256;
constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 256;

struct Dq256Smem {
  alignas(1024) uint8_t q[kChunks256][kChunkB256];
  alignas(1024) uint8_t dout[kChunks256][kChunkB256];
  alignas(1024) uint8_t ring[kSlots256][kChunkB256];
  uint64_t qd_full, r_full[kSlots256], r_empty[kSlots256];
  uint64_t sdp_full;  // S and dP of the current tile are in tensor memory
  uint64_t ds_full;   // dS of the current tile is in tensor memory (128 arrivals)
  uint64_t dq_done;   // every dQ product is complete
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, qt, kt_lo, nk, n_real, skip;
};
static_assert(sizeof(Dq256Smem) + 1024 <= 232448, "shared memory per CTA");

template <bool kDrop>
__global__ void __launch_bounds__(kThreads256, 1)
    bwd_dq256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                     const float* __restrict__ delta, void* __restrict__ dq, int dq_bf16, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  Dq256Smem& s = *reinterpret_cast<Dq256Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % g.Hq, hk = h / g.G;
  volatile int* vstatus = status;

  if (tid == 0) {
    const int item = blockIdx.x / g.Hq;
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
    mbar_init(&s.qd_full, 1);
    for (int i = 0; i < kSlots256; ++i) {
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

  if (nk == 0) {  // no row of this q tile sees a key: dq = 0
    if (tid >= 128) {
      const int i = qt * kTile + (tid - 128);
      if (i < g.L) {
        uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dq) + (row0 + i) * kD256 * elem);
        for (size_t c = 0; c < kD256 * elem / 16; ++c) o4[c] = make_uint4(0, 0, 0, 0);
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
    mbar_arrive_expect_tx(&s.qd_full, 2 * kChunks256 * kChunkB256);
    for (int c = 0; c < kChunks256; ++c) {
      tma_load_3d(s.q[c], &tm_q, &s.qd_full, c * 64, qt * kTile, b * g.Hq + h);
      tma_load_3d(s.dout[c], &tm_dout, &s.qd_full, c * 64, qt * kTile, b * g.Hq + h);
    }
    const int pl = b * g.Hkv + hk;
    int n = 0;  // ring chunks issued
    bool ok = true;
    for (int j = 0; ok && j < nk; ++j) {
      const int row = (kt_lo + j) * kTile;
      for (int u = 0; u < kPerTile; ++u) {  // K chunks, V chunks, K chunks again
        const int sl = n % kSlots256;
        if (n >= kSlots256 && !pipe_wait(&s.r_empty[sl], (n / kSlots256 - 1) & 1, &s.abort_flag, vstatus)) {
          ok = false;
          break;
        }
        const void* map = (u / kChunks256 == 1) ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
        mbar_arrive_expect_tx(&s.r_full[sl], kChunkB256);
        tma_load_3d(s.ring[sl], map, &s.r_full[sl], (u % kChunks256) * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
        ++n;
      }
    }
    if (!ok) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // no copy into this CTA's shared memory may still be in flight at exit
    mbar_wait_drain(&s.qd_full, 0);
    for (int x = (n > kSlots256 ? n - kSlots256 : 0); x < n; ++x)
      mbar_wait_drain(&s.r_full[x % kSlots256], (x / kSlots256) & 1);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idX = idesc_bf16(128, 128, false, false);  // S, dP: both operands K-major
    constexpr uint32_t idDQ = idesc_bf16(128, 64, false, true);   // dQ chunk: dS from TMEM, K chunk MN-major
    const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);
    const uint64_t dMN = umma_desc_sw128(0, kChunkB256, 1024);
    const uint32_t a_q = smem_u32(s.q[0]), a_do = smem_u32(s.dout[0]), a_ring = smem_u32(s.ring[0]);
    auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
    int n = 0;  // ring chunks consumed
    // the slot of the next ring chunk, once it has landed
    auto next_chunk = [&](int& sl) -> bool {
      sl = n % kSlots256;
      if (!wait(&s.r_full[sl], (n / kSlots256) & 1)) return false;
      tc_fence_after();
      return true;
    };
    bool ok = wait(&s.qd_full, 0);
    for (int j = 0; ok && j < nk; ++j) {
      // S = Q K^T, then dP = dO V^T, over the four chunks of the head dim (the
      // previous tile's dQ products, issued before, have read its dS out of
      // the S columns, and its dP was read before ds_full)
      for (int u = 0; u < 2 * kChunks256; ++u) {
        int sl;
        if (!next_chunk(sl)) {
          ok = false;
          break;
        }
        const int c = u % kChunks256;
        const bool is_s = u < kChunks256;
        const uint32_t aa = (is_s ? a_q : a_do) + c * kChunkB256, bb = a_ring + sl * kChunkB256;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_ss(tbase + (is_s ? kColS : kColDp), desc_at(dK_major, aa + ks * 32), desc_at(dK_major, bb + ks * 32),
                  idX, (c > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.r_empty[sl]);
        ++n;
      }
      if (!ok) break;
      umma_commit(&s.sdp_full);
      // dQ[:, 64c:64c+64] += dS K[:, 64c:64c+64]; dS is bf16 in the S columns
      if (!wait(&s.ds_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < kChunks256; ++c) {
        int sl;
        if (!next_chunk(sl)) {
          ok = false;
          break;
        }
        const uint32_t bb = a_ring + sl * kChunkB256;
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
      dq_store_cols(tbase + lane_off + kColDq, kD256, dq, (row0 + i) * kD256, dq_bf16, i < g.L);
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

// dq in a fixed order for D = 256 (q and dout maps with 128-row boxes).
cudaError_t launch_bwd_dq256(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                             const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                             const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st) {
  if (g.D != kD256) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Dq256Smem) + 1024;  // + 1 KB to align the swizzled tiles
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
  auto kern = g.drop_t ? bwd_dq256_kernel<true> : bwd_dq256_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * g.Hq;  // (q tile, query head)
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads256), smem,
      st, mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
