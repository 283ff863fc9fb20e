// K3: forward of per-document causal attention for one CP query shard.
//
// What it computes (NeMo AutoModel API, blockdiag_cp.kernels
// `_cp_blockdiag_varlen`): for every real local row p, the softmax over the
// allowed keys [lo(p), p] (lo = max(doc_start, p - W + 1)) of scale * q.k,
// times V; LSE = natural-log sum-exp (gemma4_moe.cp_attention `_scatter_lse`:
// -inf on rows that take no part). Padding rows return zeros.
//
// Design (GB300): one CTA per (128-row q tile, pair of query heads of the same
// GQA group); the work list puts the q tiles with the most K/V tiles first.
//   warp 0      TMA producer: Q tiles once, then K and V tiles of the tile's
//               contiguous K/V range through an NS-stage ring (128B swizzle).
//   warp 1      one thread issues tcgen05.mma: S = Q K^T into TMEM, and
//               O += P V with P read from TMEM (the "TS" form).
//   warp 2      allocates / frees tensor memory.
//   warps 4..   one warpgroup per q tile: each thread owns one row; reads S
//               from TMEM, applies the mask only on partial tiles, keeps the
//               running max / sum in fp32, writes P (bf16) over S in TMEM,
//               rescales O only when the max grows by more than 2^8, and
//               finally normalises O and writes out / LSE: out is staged
//               as bf16 rows in the K ring (free once the head's last PV
//               product is done) and copied to global memory a whole row
//               per 16-byte lane group, so each warp store is one
//               contiguous 512-byte run instead of 32 scattered pieces.
// The two q tiles of a CTA share every K/V tile (same kv head), so the tensor
// core works on one while the other's softmax runs.
// With attention dropout (kDrop), each softmax thread draws its row's keep
// mask of a K/V tile before that tile's S arrives, zeroes the dropped weights
// of P (the row sum stays the undropped one) and folds the keep scale into the
// final normalisation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

template <int D, int NQ, int NS>
struct FwdSmem {
  static constexpr int kChunks = D / 64;         // 64-column (128 B) chunks per row
  static constexpr int kChunkBytes = kTile * 128;  // 128 rows x 128 B
  alignas(1024) uint8_t q[NQ][kChunks][kChunkBytes];
  alignas(1024) uint8_t k[NS][kChunks][kChunkBytes];
  alignas(1024) uint8_t v[NS][kChunks][kChunkBytes];
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[NQ], p_full[NQ], o_done[NQ];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  // work item, decoded by thread 0
  int b, qt, kt_lo, nk, n_real, skip;
};

template <int D, int NQ>
struct FwdTmem {
  __host__ __device__ static constexpr int kS(int qi) { return qi * 128; }
  __host__ __device__ static constexpr int kO(int qi) { return NQ * 128 + qi * D; }
  static constexpr int kUsed = NQ * (128 + D);
  static constexpr int kCols = kUsed <= 32 ? 32 : kUsed <= 64 ? 64 : kUsed <= 128 ? 128 : kUsed <= 256 ? 256 : 512;
  static_assert(kUsed <= 512, "tensor memory budget");
};

template <int D, int NQ, int NS, bool kMerge, bool kDrop>
__global__ void __launch_bounds__(128 + NQ * 128, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ seg, const Geom g,
               __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int32_t* status) {
  pdl_begin();
  using Smem = FwdSmem<D, NQ, NS>;
  using TM = FwdTmem<D, NQ>;
  constexpr int kChunks = Smem::kChunks;
  static_assert(sizeof(Smem::k) >= NQ * kTile * D * 2, "out staging fits the K ring");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw so the compiler keeps the shared address space
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pairs = g.Hq / NQ;
  const int pair = blockIdx.x % n_pairs;
  volatile int* vstatus = status;

  if (tid == 0) {
    const int item = blockIdx.x / n_pairs;
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
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_done[i], 1);
    }
    mbar_init(&s.q_full, 1);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
    if (!s.skip && nk > 0) {
      // the first copies go out now, ahead of the block barriers and the
      // tensor-memory allocation: Q of the heads and K / V of the first tiles
      const int h0e = pair * NQ, hke = h0e / g.G;
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.q_full, NQ * kChunks * Smem::kChunkBytes);
      for (int qi = 0; qi < NQ; ++qi)
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(s.q[qi][c], &tm_q, &s.q_full, c * 64, qt * kTile, b * g.Hq + h0e + qi);
      for (int j = 0; j < NS && j < nk; ++j) {
        const int row = (kt_lo + j) * kTile, pl = b * g.Hkv + hke;
        mbar_arrive_expect_tx(&s.k_full[j], kChunks * Smem::kChunkBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(s.k[j][c], &tm_k, &s.k_full[j], c * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
        mbar_arrive_expect_tx(&s.v_full[j], kChunks * Smem::kChunkBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(s.v[j][c], &tm_v, &s.v_full[j], c * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      }
    }
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, qt = s.qt, kt_lo = s.kt_lo, nk = s.nk, n_real = s.n_real;
  const int h0 = pair * NQ, hk = h0 / g.G;

  if (nk == 0) {
    // No row of this q tile sees a key: zeros and -inf (merging: a running
    // result is kept, an empty one set to zeros and -inf).
    if (tid >= 128) {
      const int qi = (tid - 128) >> 7, r = (tid - 128) & 127;
      const int i = qt * kTile + r;
      if (i < g.L) {
        const size_t row = (static_cast<size_t>(b) * g.Hq + h0 + qi) * g.L + i;
        if (!kMerge || lse[row] == -INFINITY) {
          uint4* o4 = reinterpret_cast<uint4*>(out + row * D);
          for (int c = 0; c < D / 8; ++c) o4[c] = make_uint4(0, 0, 0, 0);
          lse[row] = -INFINITY;
        }
      }
    }
    return;
  }

  if (warp == 2) {
    tmem_alloc(&s.tmem_base, TM::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // (Q and the first NS tiles were issued with the barrier set-up)
    int k_issued = nk < NS ? nk : NS, v_issued = k_issued;
    for (int j = k_issued; j < nk; ++j) {
      const int st = j % NS, n = j / NS;
      if (j >= NS && !pipe_wait(&s.k_empty[st], (n - 1) & 1, &s.abort_flag, vstatus))
        break;
      mbar_arrive_expect_tx(&s.k_full[st], kChunks * Smem::kChunkBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_3d(s.k[st][c], &tm_k, &s.k_full[st], c * 64, g.kv_tm ? b * g.Hkv + hk : (kt_lo + j) * kTile, g.kv_tm ? (kt_lo + j) * kTile : b * g.Hkv + hk);
      ++k_issued;
      if (j >= NS && !pipe_wait(&s.v_empty[st], (n - 1) & 1, &s.abort_flag, vstatus))
        break;
      mbar_arrive_expect_tx(&s.v_full[st], kChunks * Smem::kChunkBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_3d(s.v[st][c], &tm_v, &s.v_full[st], c * 64, g.kv_tm ? b * g.Hkv + hk : (kt_lo + j) * kTile, g.kv_tm ? (kt_lo + j) * kTile : b * g.Hkv + hk);
      ++v_issued;
    }
    if (v_issued < nk) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // make sure no copy into this CTA's shared memory is still in flight at exit
    mbar_wait_drain(&s.q_full, 0);
    for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j) mbar_wait_drain(&s.k_full[j % NS], (j / NS) & 1);
    for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j) mbar_wait_drain(&s.v_full[j % NS], (j / NS) & 1);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
    const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);                 // Q, K: K-major
    const uint64_t dMN = umma_desc_sw128(0, Smem::kChunkBytes, 1024);       // V: MN-major
    const uint32_t a_q = smem_u32(s.q[0][0]), a_k = smem_u32(s.k[0][0]), a_v = smem_u32(s.v[0][0]);
    constexpr uint32_t kTileBytes = kChunks * Smem::kChunkBytes;
    auto issue_s = [&](int qi, int st) {
      const uint32_t d = tbase + TM::kS(qi);
      const uint32_t qa = a_q + qi * kTileBytes, ka = a_k + st * kTileBytes;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks >> 2) * Smem::kChunkBytes + (ks & 3) * 32;
        umma_ss(d, desc_at(dK_major, qa + off), desc_at(dK_major, ka + off), idS, ks > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int qi, int st, bool acc) {
      const uint32_t d = tbase + TM::kO(qi);
      const uint32_t va = a_v + st * kTileBytes;
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks)
        umma_ts(d, tbase + TM::kS(qi) + ks * 8, desc_at(dMN, va + ks * 2048), idPV, (acc || ks > 0) ? 1u : 0u);
    };
    bool ok = pipe_wait(&s.q_full, 0, &s.abort_flag, vstatus) &&
              pipe_wait(&s.k_full[0], 0, &s.abort_flag, vstatus);
    if (ok) {
      tc_fence_after();
      for (int qi = 0; qi < NQ; ++qi) {
        issue_s(qi, 0);
        umma_commit(&s.s_full[qi]);
      }
      umma_commit(&s.k_empty[0]);
    }
    for (int j = 0; ok && j < nk; ++j) {
      const int st = j % NS;
      if (!pipe_wait(&s.v_full[st], (j / NS) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      for (int qi = 0; qi < NQ; ++qi) {
        if (!pipe_wait(&s.p_full[qi], j & 1, &s.abort_flag, vstatus)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(qi, st, j > 0);
        umma_commit(&s.o_done[qi]);
        if (j + 1 < nk) {
          const int st1 = (j + 1) % NS;
          if (qi == 0 &&
              !pipe_wait(&s.k_full[st1], ((j + 1) / NS) & 1, &s.abort_flag, vstatus)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(qi, st1);
          umma_commit(&s.s_full[qi]);
        }
      }
      if (!ok) break;
      umma_commit(&s.v_empty[st]);
      if (j + 1 < nk) umma_commit(&s.k_empty[(j + 1) % NS]);
    }
    if (!ok) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    umma_commit(&s.mma_drain);
    mbar_wait_drain(&s.mma_drain, 0);
  } else if (warp >= 4) {
    // ------------------------------------------------- softmax warpgroups
    const int qi = (warp - 4) >> 2;
    const int r = tid - 128 - qi * 128;          // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tbase + lane_off + TM::kS(qi);
    const uint32_t t_o = tbase + lane_off + TM::kO(qi);
    const int h = h0 + qi;
    const int i = qt * kTile + r;
    const bool real = i < n_real;
    int jlo = 1, jhi = 0;  // allowed K/V buffer rows [jlo, jhi] of this row
    if (real) {
      const int p = g.row_offset + i;
      const int doc_start = seg[g.off[BD_SEG_OFF_ROW_LO] + b * g.L + i];
      jlo = row_lo_window(doc_start, p, g.window) - g.kv_offset;
      jhi = min(p - g.kv_offset, g.S_kv - 1);  // a K/V chunk may end before the row
    }
    const float sl2 = g.scale * 1.4426950408889634f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      uint32_t km[4];  // dropout: keep bits of this row over the tile's 128 keys
      if constexpr (kDrop) row_keep_mask(g, b, h, g.row_offset + i, g.kv_offset + (kt_lo + j) * kTile, km);
      if (!warp_wait(&s.s_full[qi], j & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S in two halves: the second half's load is in flight while the first
      // half's max is formed
      uint32_t xr[128];
      tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&xr[0]));
      tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[32]));
      tmem_wait_ld();
      tmem_regs_ready<64>(&xr[0]);
      tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&xr[64]));
      tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&xr[96]));
      const int c0 = (kt_lo + j) * kTile;
      // a row either sees the whole tile, none of it (another document, or a
      // padding row), or part of it (the diagonal / document-start tiles); only
      // a warp with a partly seen row needs the per-element mask
      const bool dead = jhi < c0 || jlo > c0 + kTile - 1;
      const bool unmasked = __all_sync(0xffffffffu, dead || (jlo <= c0 && c0 + kTile - 1 <= jhi));
      const int a_lo = jlo - c0, e_hi = jhi - c0;
      float x[128];  // raw scores, -inf where masked
      float mx[8];   // eight independent 16-column maxima (short dependency chains)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        if (hf == 1) {
          tmem_wait_ld();
          tmem_regs_ready<64>(&xr[64]);
        }
        if (unmasked) {
#pragma unroll
          for (int c = 64 * hf; c < 64 * hf + 64; ++c) x[c] = __uint_as_float(xr[c]);
        } else {
#pragma unroll
          for (int c = 64 * hf; c < 64 * hf + 64; ++c) x[c] = (c >= a_lo && c <= e_hi) ? __uint_as_float(xr[c]) : -INFINITY;
        }
#pragma unroll
        for (int k = 4 * hf; k < 4 * hf + 4; ++k) {
          float a = fmax3(x[16 * k], x[16 * k + 1], x[16 * k + 2]);
#pragma unroll
          for (int c = 16 * k + 3; c < 16 * k + 15; c += 2) a = fmax3(a, x[c], x[c + 1]);
          mx[k] = fmaxf(a, x[16 * k + 15]);
        }
      }
      float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      tmax = dead ? -INFINITY : tmax * sl2;  // the scale is positive: the max of the scaled scores
      const float m_new = fmaxf(m, tmax);
      const bool need = m_new > m + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_exp2(m - m_new) : 1.0f;
        if (need) {
          l *= alpha;
          m = m_new;
        }
        if (j > 0) {
          if (!warp_wait(&s.o_done[qi], (j - 1) & 1, &s.abort_flag, vstatus)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
            const float2 av = make_float2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), av);
              o[e] = __float_as_uint(v.x);
              o[e + 1] = __float_as_uint(v.y);
            }
            tmem_st32(t_o + c, o);
          }
          tmem_wait_st();
        }
      }
      // exponent offset; -inf on a row that sees nothing of this tile, so P = 0
      const float nmm = dead ? -INFINITY : (m == -INFINITY) ? 0.f : -m;
      // two-wide fp32 FMA and add (one instruction per pair of columns): the
      // exponent scale * log2(e) * score - max, and the row sum in four pairs
      // of partial sums
      const float2 sl2v = make_float2(sl2, sl2), nmmv = make_float2(nmm, nmm);
      float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float2 ex = __ffma2_rn(make_float2(x[2 * c], x[2 * c + 1]), sl2v, nmmv);
        const float p0 = fast_exp2(ex.x), p1 = fast_exp2(ex.y);
        rs2[c & 3] = __fadd2_rn(rs2[c & 3], make_float2(p0, p1));
        if constexpr (kDrop) {
          const uint32_t kb = km[c >> 4] >> ((2 * c) & 31);
          pk[c] = pack_bf16x2((kb & 1u) ? p0 : 0.f, (kb & 2u) ? p1 : 0.f);
        } else {
          pk[c] = pack_bf16x2(p0, p1);
        }
      }
      const float2 r01 = __fadd2_rn(rs2[0], rs2[1]), r23 = __fadd2_rn(rs2[2], rs2[3]);
      const float2 r = __fadd2_rn(r01, r23);
      const float rs = r.x + r.y;
      l += rs;
      tmem_st32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full[qi]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !warp_wait(&s.o_done[qi], (nk - 1) & 1, &s.abort_flag, vstatus)) ok = false;
    if (!ok) s.abort_flag = 1;
    // the warpgroup's four warps take the same path below (it has a barrier)
    ok = named_bar_and(1 + qi, 128, ok);
    if (!ok) {
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    } else {
      tc_fence_after();
      float inv = l > 0.f ? (kDrop ? g.drop_scale : 1.0f) / l : 0.f;
      float lse_v = (real && l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
      uint4* o4 = reinterpret_cast<uint4*>(out + row * D);
      // merging into a running (out, lse): log-sum-exp weights of the two sides;
      // an empty side (lse -inf) has weight 0 and its out is not read
      float w_old = 0.f;
      bool store = i < g.L;
      if (kMerge && store) {
        const float lse_o = lse[row];
        if (lse_v == -INFINITY) {
          store = lse_o == -INFINITY;  // nothing new: keep a running result, zero an empty one
        } else if (lse_o != -INFINITY) {
          const float mx = fmaxf(lse_o, lse_v);
          const float ea = expf(lse_o - mx), eb = expf(lse_v - mx), tot = ea + eb;
          w_old = ea / tot;
          inv *= eb / tot;
          lse_v = mx + logf(tot);
        }
      }
      if constexpr (kMerge) {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c, o);
          tmem_wait_ld();
          if (store) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float v[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(o[8 * e + k]) * inv;
              if (kMerge && w_old != 0.f) {
                const uint4 old = o4[c / 8 + e];
                const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&ow[k]);
                  v[2 * k] = fmaf(w_old, __low2float(h2), v[2 * k]);
                  v[2 * k + 1] = fmaf(w_old, __high2float(h2), v[2 * k + 1]);
                }
              }
              uint4 w;
              w.x = pack_bf16x2(v[0], v[1]);
              w.y = pack_bf16x2(v[2], v[3]);
              w.z = pack_bf16x2(v[4], v[5]);
              w.w = pack_bf16x2(v[6], v[7]);
              o4[c / 8 + e] = w;
            }
          }
        }
      } else {
        // O (bf16) of this head into the K ring, which every S product of
        // this CTA has finished reading once this head's last PV is done:
        // row r at r * 2D bytes, 16-byte piece c at slot c ^ (r & 7)
        uint8_t* stg = &s.k[0][0][0] + qi * (kTile * D * 2);
        uint32_t oa[D];  // all of O's row, one wait
#pragma unroll
        for (int c = 0; c < D; c += 32) tmem_ld32(t_o + c, *reinterpret_cast<uint32_t(*)[32]>(&oa[c]));
        tmem_wait_ld();
        tmem_regs_ready<D>(oa);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          const uint32_t* o = oa + c;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            const int piece = c / 8 + e;
            *reinterpret_cast<uint4*>(stg + r * (D * 2) + ((piece ^ (r & 7)) << 4)) = w;
          }
        }
        named_bar_sync(1 + qi, 128);
        // whole rows to global memory: a warp instruction writes 512
        // contiguous bytes (2 rows at D = 128, 4 at D = 64)
        constexpr int kPieces = D / 8, kRows = 32 / kPieces;
        const int pc = lane % kPieces;
        __nv_bfloat16* obase = out + (static_cast<size_t>(b) * g.Hq + h) * g.L * D;
#pragma unroll 4
        for (int k2 = 0; k2 < 32 / kRows; ++k2) {
          const int rr = (warp & 3) * 32 + k2 * kRows + lane / kPieces;
          const int gi = qt * kTile + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * (D * 2) + ((pc ^ (rr & 7)) << 4));
          if (gi < g.L) reinterpret_cast<uint4*>(obase + static_cast<size_t>(gi) * D)[pc] = w;
        }
      }
      if (store) lse[row] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, TM::kCols);
  }
}

template <int D, int NQ, int NS>
static cudaError_t launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                              const int32_t* seg, const Geom& g, __nv_bfloat16* out, float* lse, int32_t* status,
                              int merge, cudaStream_t st) {
  const size_t smem = sizeof(FwdSmem<D, NQ, NS>) + 1024;  // + 1 KB to align the swizzled tiles
  auto kern = g.drop_t ? (merge ? fwd_kernel<D, NQ, NS, true, true> : fwd_kernel<D, NQ, NS, false, true>)
                       : (merge ? fwd_kernel<D, NQ, NS, true, false> : fwd_kernel<D, NQ, NS, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * (g.Hq / NQ);
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(128 + NQ * 128), smem, st, mq,
      mk, mv, seg, g, out, lse, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_fwd256(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                          const Geom& g, void* out, float* lse, int32_t* status, int merge, cudaStream_t st);

// Two query heads of one GQA group per CTA when the group size is even and
// D <= 128 (tensor memory: 2 x (128 + D) columns); one otherwise. D = 256 has
// its own kernel with K / V streamed in halves (fwd256_kernel.cu).
cudaError_t launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                       const Geom& g, void* out, float* lse, int32_t* status, int merge, cudaStream_t st) {
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const bool pairs = (g.G % 2) == 0;
  switch (g.D) {
    case 64:
      return pairs ? launch_one<64, 2, 3>(mq, mk, mv, seg, g, o, lse, status, merge, st)
                   : launch_one<64, 1, 3>(mq, mk, mv, seg, g, o, lse, status, merge, st);
    case 128:
      return pairs ? launch_one<128, 2, 2>(mq, mk, mv, seg, g, o, lse, status, merge, st)
                   : launch_one<128, 1, 2>(mq, mk, mv, seg, g, o, lse, status, merge, st);
    case 256:
      return launch_fwd256(mq, mk, mv, seg, g, out, lse, status, merge, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace bd
