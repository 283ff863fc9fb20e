// K4d: dq of the backward in a fixed order -- deterministic (the pages'
// `_CP_FLASH_DETERMINISTIC`, gemma4_moe.cp_local_ring backward). The main
// backward kernel adds each K/V tile's dq share to an fp32 accumulator with
// atomic adds, whose order varies from run to run; here one CTA owns a
// 128-row q tile of one query head and walks its K/V tiles in increasing
// order, accumulating dQ in tensor memory and writing it once:
//   S  = Q K^T, dP = dO V^T                     (TMEM cols [0,128), [128,256))
//   P  = 2^(scale log2(e) q.k - lse log2(e)) on the allowed keys (the saved
//        lse: no running max), dS = P (scale dP - scale delta)  (bf16, smem)
//   dQ += dS K                                   (TMEM cols [256, 256 + D))
// With dK / dV from the main kernel (whose dK / dV already accumulate inside
// one CTA), the whole backward is bitwise reproducible.
//   warp 0   TMA: Q and dO once, K / V tiles through an NS-stage ring
//   warp 1   one thread issues the MMAs       warp 2  tensor memory
//   warps 4-7  thread = q row: P, dS, and the dq rows at the end
// D = 64 or 128 (S, dP and dQ fill 384 of the 512 tensor-memory columns);
// D = 256 and 512 stream K/V through a chunk ring (dq256_kernel.cu, dq512_kernel.cu).
// With attention dropout (kDrop) each row draws its keep mask of a K/V tile
// (dropout.cuh) before the tile's S and dP arrive: dS = P (Z dP - delta).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

namespace {

template <int D, int NS>
struct DqSmem {
  static constexpr int kChunks = D / 64;           // 64-column (128 B) chunks per row
  static constexpr int kChunkBytes = kTile * 128;  // 128 rows x 128 B
  alignas(1024) uint8_t q[kChunks][kChunkBytes];
  alignas(1024) uint8_t dout[kChunks][kChunkBytes];
  alignas(1024) uint8_t k[NS][kChunks][kChunkBytes];
  alignas(1024) uint8_t v[NS][kChunks][kChunkBytes];
  alignas(1024) uint8_t ds[2][kChunkBytes];  // dS: 128 q x 128 keys bf16, two 64-key chunks, K-major, 128B-swizzled
  uint64_t qd_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t sdp_full;   // S and dP of the current tile are in tensor memory
  uint64_t sdp_empty;  // ... and have been read (128 arrivals)
  uint64_t ds_full;    // dS of the current tile is in shared memory (128 arrivals)
  uint64_t ds_empty;   // the dQ product has read it
  uint64_t dq_done;    // every dQ product is complete
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, qt, kt_lo, nk, n_real, skip;
};

constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 256;
constexpr int kDqThreads = 256;

template <int D, int NS, bool kDrop>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dout,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const int32_t* __restrict__ seg, const Geom g, const float* __restrict__ lse,
                  const float* __restrict__ delta, void* __restrict__ dq, int dq_bf16, int32_t* status) {
  pdl_begin();
  using Smem = DqSmem<D, NS>;
  constexpr int kChunks = Smem::kChunks;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
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
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.qd_full, 1);
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.sdp_empty, 128);
    mbar_init(&s.ds_full, 128);
    mbar_init(&s.ds_empty, 1);
    mbar_init(&s.dq_done, 1);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, qt = s.qt, kt_lo = s.kt_lo, nk = s.nk, n_real = s.n_real;
  const size_t row0 = (static_cast<size_t>(b) * g.Hq + h) * g.L;  // dq / lse / delta row of local row 0

  if (nk == 0) {  // no row of this q tile sees a key: dq = 0
    if (tid >= 128) {
      const int i = qt * kTile + (tid - 128);
      if (i < g.L) {
        uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dq) + (row0 + i) * D * (dq_bf16 ? 2 : 4));
        for (int c = 0; c < D * (dq_bf16 ? 2 : 4) / 16; ++c) o4[c] = make_uint4(0, 0, 0, 0);
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
    mbar_arrive_expect_tx(&s.qd_full, 2 * kChunks * Smem::kChunkBytes);
    for (int c = 0; c < kChunks; ++c) {
      tma_load_3d(s.q[c], &tm_q, &s.qd_full, c * 64, qt * kTile, b * g.Hq + h);
      tma_load_3d(s.dout[c], &tm_dout, &s.qd_full, c * 64, qt * kTile, b * g.Hq + h);
    }
    int issued = 0;
    for (int j = 0; j < nk; ++j) {
      const int st = j % NS, n = j / NS;
      const int row = (kt_lo + j) * kTile, pl = b * g.Hkv + hk;
      if (j >= NS && !(pipe_wait(&s.k_empty[st], (n - 1) & 1, &s.abort_flag, vstatus) &&
                       pipe_wait(&s.v_empty[st], (n - 1) & 1, &s.abort_flag, vstatus)))
        break;
      mbar_arrive_expect_tx(&s.k_full[st], kChunks * Smem::kChunkBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_3d(s.k[st][c], &tm_k, &s.k_full[st], c * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      mbar_arrive_expect_tx(&s.v_full[st], kChunks * Smem::kChunkBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_3d(s.v[st][c], &tm_v, &s.v_full[st], c * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      ++issued;
    }
    if (issued < nk) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // no copy into this CTA's shared memory may still be in flight at exit
    mbar_wait_drain(&s.qd_full, 0);
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j) {
      mbar_wait_drain(&s.k_full[j % NS], (j / NS) & 1);
      mbar_wait_drain(&s.v_full[j % NS], (j / NS) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idX = idesc_bf16(128, 128, false, false);  // S, dP: both operands K-major
    constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);    // dQ: dS K-major, K (keys x d) MN-major
    const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);
    const uint64_t dMN = umma_desc_sw128(0, Smem::kChunkBytes, 1024);
    const uint32_t a_q = smem_u32(s.q[0]), a_do = smem_u32(s.dout[0]), a_ds = smem_u32(s.ds[0]);
    const uint32_t a_k = smem_u32(s.k[0][0]), a_v = smem_u32(s.v[0][0]);
    constexpr uint32_t kTileBytes = kChunks * Smem::kChunkBytes;
    // X = A B^T over the head dim (A: 128 q rows, B: 128 keys)
    auto issue_x = [&](uint32_t col, uint32_t aa, uint32_t bb) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks >> 2) * Smem::kChunkBytes + (ks & 3) * 32;
        umma_ss(tbase + col, desc_at(dK_major, aa + off), desc_at(dK_major, bb + off), idX, ks > 0 ? 1u : 0u);
      }
    };
    auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
    bool ok = wait(&s.qd_full, 0) && wait(&s.k_full[0], 0) && wait(&s.v_full[0], 0);
    if (ok) {
      tc_fence_after();
      issue_x(kColS, a_q, a_k);
      issue_x(kColDp, a_do, a_v);
      umma_commit(&s.sdp_full);
    }
    for (int j = 0; ok && j < nk; ++j) {
      const int st = j % NS;
      // S and dP of the next tile as soon as this tile's have been read out,
      // so that they run while the P / dS threads work on this one
      if (j + 1 < nk) {
        const int st1 = (j + 1) % NS, par1 = ((j + 1) / NS) & 1;
        if (!(wait(&s.sdp_empty, j & 1) && wait(&s.k_full[st1], par1) && wait(&s.v_full[st1], par1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_x(kColS, a_q, a_k + st1 * kTileBytes);
        issue_x(kColDp, a_do, a_v + st1 * kTileBytes);
        umma_commit(&s.sdp_full);
      }
      // dQ += dS K over this tile's 128 keys
      if (!wait(&s.ds_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks)
        umma_ss(tbase + kColDq, desc_at(dK_major, a_ds + (ks >> 2) * Smem::kChunkBytes + (ks & 3) * 32),
                desc_at(dMN, a_k + st * kTileBytes + ks * 2048), idDQ, (j > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&s.ds_empty);
      umma_commit(&s.k_empty[st]);
      umma_commit(&s.v_empty[st]);
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
    const float2 sl2 = make_float2(g.scale * 1.4426950408889634f, g.scale * 1.4426950408889634f);
    const float scd = kDrop ? g.scale * g.drop_scale : g.scale;  // dropout: a kept dP's factor
    const float2 sc = make_float2(scd, scd), nl2v = make_float2(nl2, nl2), ndlv = make_float2(ndl, ndl);
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      uint32_t km[4];  // dropout: keep bits of this row over the tile's 128 keys
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
      const int a_lo = jlo - c0, e_hi = jhi - c0;
      uint32_t pk[2][32];  // dS of keys [64 hf, 64 hf + 64), bf16 pairs
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[64], dr[64];
        tmem_ld32(tbase + lane_off + kColS + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tbase + lane_off + kColS + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tbase + lane_off + kColDp + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
        tmem_ld32(tbase + lane_off + kColDp + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
        tmem_wait_ld();
        tmem_regs_ready<64>(sr);
        tmem_regs_ready<64>(dr);
        if (hf == 1) {  // S and dP are read: the next tile's may go in
          tc_fence_before();
          mbar_arrive(&s.sdp_empty);
        }
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
      // the previous tile's dQ product must be done reading the dS buffer
      if (j > 0 && !warp_wait(&s.ds_empty, (j - 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint8_t* ds_row = s.ds[hf] + r * 128;  // this row of the 64-key chunk (128B swizzle)
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16)
          *reinterpret_cast<uint4*>(ds_row + ((c16 ^ (r & 7)) << 4)) =
              make_uint4(pk[hf][4 * c16], pk[hf][4 * c16 + 1], pk[hf][4 * c16 + 2], pk[hf][4 * c16 + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&s.ds_full);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !warp_wait(&s.dq_done, 0, &s.abort_flag, vstatus)) ok = false;
    if (!ok) {
      s.abort_flag = 1;
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    } else {
      tc_fence_after();
      const size_t row = row0 + i;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_off + kColDq + c, o);
        tmem_wait_ld();
        if (i < g.L) {
          if (dq_bf16) {
            uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dq) + row * D + c);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              d4[e] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * e]), __uint_as_float(o[8 * e + 1])),
                                 pack_bf16x2(__uint_as_float(o[8 * e + 2]), __uint_as_float(o[8 * e + 3])),
                                 pack_bf16x2(__uint_as_float(o[8 * e + 4]), __uint_as_float(o[8 * e + 5])),
                                 pack_bf16x2(__uint_as_float(o[8 * e + 6]), __uint_as_float(o[8 * e + 7])));
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(dq) + row * D + c);
#pragma unroll
            for (int e = 0; e < 8; ++e) d4[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, int NS>
cudaError_t launch_dq(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk, const CUtensorMap& mv,
                      const int32_t* seg, const Geom& g, const float* lse, const float* delta, void* dq, int bf16,
                      int32_t* status, cudaStream_t st) {
  const size_t smem = sizeof(DqSmem<D, NS>) + 1024;  // + 1 KB to align the swizzled tiles
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
  auto kern = g.drop_t ? bwd_dq_kernel<D, NS, true> : bwd_dq_kernel<D, NS, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * g.Hq;  // (q tile, query head)
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kDqThreads), smem, st, mq,
      mdo, mk, mv, seg, g, lse, delta, dq, bf16, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq256(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                             const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                             const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st);
cudaError_t launch_bwd_dq512(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                             const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                             const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st);

// dq in a fixed order for D = 64 / 128 / 256 / 512 (q and dout maps with 128-row boxes).
cudaError_t launch_bwd_dq(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                          const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                          const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st) {
  switch (g.D) {
    case 64: return launch_dq<64, 3>(mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status, st);
    case 128: return launch_dq<128, 2>(mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status, st);
    case 256: return launch_bwd_dq256(mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status, st);  // dq256_kernel.cu
    case 512: return launch_bwd_dq512(mq, mdo, mk, mv, seg, g, lse, delta, dq, bf16, status, st);  // dq512_kernel.cu
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bd
