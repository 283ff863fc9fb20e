// K3b: forward for head dim 512 (the Gemma4 full-attention layers,
// gemma4_moe.cp_attention / cp_local_ring: D = 512 global layers). Same result
// as K3 -- the softmax over the allowed keys, out and lse -- with the head dim
// split: Q (128 x 512) stays in shared memory; K streams through a ring of
// 64-column chunks (the S = Q K^T product takes 32 k-steps); O is produced in
// two 256-column halves, one per pass over the K/V tiles, because S plus the
// whole fp32 O would need 640 tensor-memory columns:
//   pass 0: online softmax as in K3, O[:, 0:256] += P V[:, 0:256], normalised
//           and written with lse at the end of the pass;
//   pass 1: S recomputed, P = 2^(scale log2(e) s - lse log2(e)) -- already
//           normalised, no running max -- and O[:, 256:512] += P V[:, 256:512].
// S is double-buffered (step t in buffer t & 1), so the next step's S = Q K^T
// runs while the softmax works on this one.
//   warp 0   TMA: Q once, K chunks through a 2-slot ring (K one step ahead of V),
//            a V half per tile
//   warp 1   one thread issues the MMAs      warp 2  tensor memory
//   warps 4-7  thread = q row: softmax, P (bf16 over S in tensor memory), out
// With attention dropout (kDrop) each row draws its keep mask of a tile (in
// both passes) before the tile's S arrives, zeroes the dropped weights of the
// P it hands to the PV products (the row sum stays the undropped one) and
// folds the keep scale into the scale of each O half.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

namespace {

constexpr int kD512 = 512;
constexpr int kQChunks = kD512 / 64;        // 8 chunks of 64 columns
constexpr int kChunkB = kTile * 128;        // 128 rows x 128 B
constexpr int kKSlots = 2;                  // K chunk ring
constexpr int kVChunks = 4;                 // one 256-column half of V
constexpr uint32_t kColS = 0, kColO = 256;  // S / P: two 128-column buffers; O half: 256 columns
constexpr int kThreads512 = 256;

struct Fwd512Smem {
  alignas(1024) uint8_t q[kQChunks][kChunkB];
  alignas(1024) uint8_t k[kKSlots][kChunkB];
  alignas(1024) uint8_t v[kVChunks][kChunkB];
  uint64_t q_full, k_full[kKSlots], k_empty[kKSlots], v_full, v_empty;
  // per S buffer, so that each has at most one phase outstanding when waited
  // on: step t's S completes only after step t - 2's PV product
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, qt, kt_lo, nk, n_real, skip;
};

// kMerge: merge this K/V chunk's result into the running (out, lse) instead
// of writing it (log-sum-exp weights, as the merge kernel).
template <bool kMerge, bool kDrop>
__global__ void __launch_bounds__(kThreads512, 1)
    fwd512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ seg, const Geom g,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  Fwd512Smem& s =
      *reinterpret_cast<Fwd512Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
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
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    mbar_init(&s.v_full, 1);
    mbar_init(&s.v_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_done[i], 1);
    }
    mbar_init(&s.o_free, 128);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s.skip) return;
  const int b = s.b, qt = s.qt, kt_lo = s.kt_lo, nk = s.nk, n_real = s.n_real;

  if (nk == 0) {  // no row of this q tile sees a key: zeros and -inf
    if (tid >= 128) {
      const int i = qt * kTile + (tid - 128);
      if (i < g.L) {
        const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
        if (!kMerge || lse[row] == -INFINITY) {  // merging: a running result is kept
          uint4* o4 = reinterpret_cast<uint4*>(out + row * kD512);
          for (int c = 0; c < kD512 / 8; ++c) o4[c] = make_uint4(0, 0, 0, 0);
          lse[row] = -INFINITY;
        }
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
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    mbar_arrive_expect_tx(&s.q_full, kQChunks * kChunkB);
    for (int c = 0; c < kQChunks; ++c) tma_load_3d(s.q[c], &tm_q, &s.q_full, c * 64, qt * kTile, b * g.Hq + h);
    const int pl = b * g.Hkv + hk;
    const int total = 2 * nk;  // (pass, tile) steps
    int kc = 0, vt = 0;        // K chunks and V halves issued
    bool stop = false;
    // K of step u (8 chunks through the ring)
    auto load_k = [&](int u) {
      const int row = (kt_lo + u % nk) * kTile;
      for (int c = 0; c < kQChunks; ++c, ++kc) {
        const int slot = kc % kKSlots;
        if (kc >= kKSlots && !pipe_wait(&s.k_empty[slot], (kc / kKSlots - 1) & 1, &s.abort_flag, vstatus))
          return false;
        mbar_arrive_expect_tx(&s.k_full[slot], kChunkB);
        tma_load_3d(s.k[slot], &tm_k, &s.k_full[slot], c * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      }
      return true;
    };
    // K runs one step ahead of V, in the order the MMAs use them: S(0), S(1),
    // PV(0), S(2), PV(1), ...
    for (int t = 0; t < total && !stop; ++t) {
      if ((t == 0 && !load_k(0)) || (t + 1 < total && !load_k(t + 1))) {
        stop = true;
        break;
      }
      if (vt > 0 && !pipe_wait(&s.v_empty, (vt - 1) & 1, &s.abort_flag, vstatus)) {
        stop = true;
        break;
      }
      const int row = (kt_lo + t % nk) * kTile, p = t / nk;
      mbar_arrive_expect_tx(&s.v_full, kVChunks * kChunkB);
      for (int c = 0; c < kVChunks; ++c)
        tma_load_3d(s.v[c], &tm_v, &s.v_full, (kVChunks * p + c) * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      ++vt;
    }
    if (stop) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // no copy into this CTA's shared memory may still be in flight at exit
    mbar_wait_drain(&s.q_full, 0);
    for (int x = (kc > kKSlots ? kc - kKSlots : 0); x < kc; ++x) mbar_wait_drain(&s.k_full[x % kKSlots], (x / kKSlots) & 1);
    if (vt > 0) mbar_wait_drain(&s.v_full, (vt - 1) & 1);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16(128, 128, false, false);   // S = Q K^T: both K-major
    constexpr uint32_t idPV = idesc_bf16(128, 256, false, true);   // O half += P V half: V MN-major
    const uint64_t dK_major = umma_desc_sw128(0, 16, 1024);
    const uint64_t dMN = umma_desc_sw128(0, kChunkB, 1024);          // 16 KB between 64-column chunks
    const uint32_t a_q = smem_u32(s.q[0]), a_k = smem_u32(s.k[0]), a_v = smem_u32(s.v[0]);
    auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
    const int total = 2 * nk;  // (pass, tile) steps
    int kc = 0;                // K chunks consumed
    // S(u) = Q K^T over the 8 head-dim chunks into buffer u & 1
    auto issue_s = [&](int u) {
      const uint32_t d = tbase + kColS + (u & 1) * 128;
      for (int c = 0; c < kQChunks; ++c, ++kc) {
        const int slot = kc % kKSlots;
        if (!wait(&s.k_full[slot], (kc / kKSlots) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_ss(d, desc_at(dK_major, a_q + c * kChunkB + ks * 32), desc_at(dK_major, a_k + slot * kChunkB + ks * 32),
                  idS, (c > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.k_empty[slot]);
      }
      umma_commit(&s.s_full[u & 1]);
      return true;
    };
    bool ok = wait(&s.q_full, 0) && issue_s(0) && (total < 2 || issue_s(1));
    for (int t = 0; ok && t < total; ++t) {
      const int p = t / nk, j = t - p * nk;
      // O half += P V half (pass 1 starts once pass 0's O has been read out)
      if (!wait(&s.p_full[t & 1], (t >> 1) & 1) || !wait(&s.v_full, t & 1) ||
          (p == 1 && j == 0 && !wait(&s.o_free, 0))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks)
        umma_ts(tbase + kColO, tbase + kColS + (t & 1) * 128 + ks * 8, desc_at(dMN, a_v + ks * 2048), idPV,
                (j > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&s.v_empty);
      umma_commit(&s.o_done[t & 1]);
      // S two steps on goes into the buffer this PV product reads (issued after it)
      if (t + 2 < total && !issue_s(t + 2)) {
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
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax (thread = row)
    const int r = tid - 128;  // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_o = tbase + lane_off + kColO;
    const int i = qt * kTile + r;
    const bool real = i < n_real;
    int jlo = 1, jhi = 0;  // allowed K/V buffer rows [jlo, jhi] of this row
    if (real) {
      const int p = g.row_offset + i;
      const int doc_start = seg[g.off[BD_SEG_OFF_ROW_LO] + b * g.L + i];
      jlo = row_lo_window(doc_start, p, g.window) - g.kv_offset;
      jhi = min(p - g.kv_offset, g.S_kv - 1);
    }
    const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
    const float sl2 = g.scale * 1.4426950408889634f;
    float m = -INFINITY, l = 0.f, nl2 = 0.f;  // nl2: -lse log2(e), pass 1
    // what the epilogues write: out = w_new * (this chunk's normalised O)
    // + w_old * (the running out) when merging; nothing for a row whose chunk
    // result is empty while its running result is not
    bool store = false;
    float w_old = 0.f, w_new = 1.f;
    bool ok = true, empty = true;             // empty: the row sees no key at all
    int t = 0;
    for (int p = 0; p < 2 && ok; ++p) {
      for (int j = 0; j < nk; ++j, ++t) {
        uint32_t km[4];  // dropout: keep bits of this row over the tile's 128 keys
        if constexpr (kDrop) row_keep_mask(g, b, h, g.row_offset + i, g.kv_offset + (kt_lo + j) * kTile, km);
        if (!warp_wait(&s.s_full[t & 1], (t >> 1) & 1, &s.abort_flag, vstatus)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_s = tbase + lane_off + kColS + (t & 1) * 128;  // this step's S buffer
        uint32_t xr[128];
        tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&xr[0]));
        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[32]));
        tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&xr[64]));
        tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&xr[96]));
        tmem_wait_ld();
        tmem_regs_ready<128>(xr);
        const int c0 = (kt_lo + j) * kTile;
        const bool dead = jhi < c0 || jlo > c0 + kTile - 1;
        const bool full = jlo <= c0 && c0 + kTile - 1 <= jhi;
        const int a_lo = jlo - c0, e_hi = jhi - c0;
        float nmm;  // exponent offset
        if (p == 0) {
          float tmax = -INFINITY;
          if (!dead) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (full || (c >= a_lo && c <= e_hi)) tmax = fmaxf(tmax, __uint_as_float(xr[c]));
            tmax *= sl2;
          }
          const float m_new = fmaxf(m, tmax);
          const bool need = m_new > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? fast_exp2(m - m_new) : 1.0f;
            if (need) {
              l *= alpha;
              m = m_new;
            }
            if (j > 0) {  // rescale the running O once its last product is done
              if (!warp_wait(&s.o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, &s.abort_flag, vstatus)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const float2 av = make_float2(alpha, alpha);
#pragma unroll 1
              for (int c = 0; c < 256; c += 32) {
                uint32_t o[32];
                tmem_ld32(t_o + c, o);
                tmem_wait_ld();
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
          nmm = (m == -INFINITY) ? 0.f : -m;
        } else {
          nmm = nl2;
        }
        const bool zero = dead || (p == 1 && empty);
        const float2 sl2v = make_float2(sl2, sl2), nmmv = make_float2(nmm, nmm);
        float2 rs2 = make_float2(0.f, 0.f);
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 ex = __ffma2_rn(make_float2(__uint_as_float(xr[2 * c]), __uint_as_float(xr[2 * c + 1])), sl2v, nmmv);
          float p0 = fast_exp2(ex.x), p1 = fast_exp2(ex.y);
          if (zero) {
            p0 = 0.f;
            p1 = 0.f;
          } else if (!full) {
            p0 = (2 * c >= a_lo && 2 * c <= e_hi) ? p0 : 0.f;
            p1 = (2 * c + 1 >= a_lo && 2 * c + 1 <= e_hi) ? p1 : 0.f;
          }
          rs2 = __fadd2_rn(rs2, make_float2(p0, p1));
          if constexpr (kDrop) {
            const uint32_t kb = km[c >> 4] >> ((2 * c) & 31);
            pk[c] = pack_bf16x2((kb & 1u) ? p0 : 0.f, (kb & 2u) ? p1 : 0.f);
          } else {
            pk[c] = pack_bf16x2(p0, p1);
          }
        }
        if (p == 0) l += rs2.x + rs2.y;
        tmem_st32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[t & 1]);
      }
      ok = __all_sync(0xffffffffu, ok);
      // end of the pass: this half of O, once its last product is done
      // (PV products complete in order: the last one's completion covers the rest)
      if (ok && !warp_wait(&s.o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, &s.abort_flag, vstatus)) ok = false;
      if (!ok) break;
      tc_fence_after();
      const float dscale = kDrop ? g.drop_scale : 1.0f;  // dropout: the keep scale of P
      float scale_o = w_new * dscale;  // pass 1: P was already normalised
      if (p == 0) {
        empty = !(real && l > 0.f);
        float lse_v = empty ? -INFINITY : (m + __log2f(l)) * 0.6931471805599453f;
        nl2 = empty ? 0.f : -(m + __log2f(l));  // -lse log2(e) of this chunk
        store = i < g.L;
        if (kMerge && store) {
          const float lse_o = lse[row];
          if (lse_v == -INFINITY) {
            store = lse_o == -INFINITY;  // nothing new: keep a running result, zero an empty one
          } else if (lse_o != -INFINITY) {
            const float mx = fmaxf(lse_o, lse_v);
            const float ea = expf(lse_o - mx), eb = expf(lse_v - mx), tot = ea + eb;
            w_old = ea / tot;
            w_new = eb / tot;
            lse_v = mx + logf(tot);
          }
        }
        if (store) lse[row] = lse_v;
        scale_o = empty ? 0.f : w_new * dscale / l;
      }
      uint4* o4 = reinterpret_cast<uint4*>(out + row * kD512 + 256 * p);
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t o[32];
        tmem_ld32(t_o + c, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (p == 1 && empty) ? 0.f : __uint_as_float(o[8 * e + k]) * scale_o;
            if (kMerge && w_old != 0.f) {  // an empty running side is not read
              const uint4 old = o4[c / 8 + e];
              const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&ow[k]);
                v[2 * k] = fmaf(w_old, __low2float(h2), v[2 * k]);
                v[2 * k + 1] = fmaf(w_old, __high2float(h2), v[2 * k + 1]);
              }
            }
            o4[c / 8 + e] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                       pack_bf16x2(v[6], v[7]));
          }
        }
      }
      if (p == 0) {  // the O columns may take pass 1's products
        tc_fence_before();
        mbar_arrive(&s.o_free);
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

// Forward for D = 512 (q, k, v maps with 64 x 128 boxes); `merge`: merged into
// the running (out, lse).
cudaError_t launch_fwd512(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                          const Geom& g, void* out, float* lse, int32_t* status, bool merge, cudaStream_t st) {
  if (g.D != kD512) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Fwd512Smem) + 1024;  // + 1 KB to align the swizzled tiles
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
  auto kern = g.drop_t ? (merge ? fwd512_kernel<true, true> : fwd512_kernel<false, true>)
                       : (merge ? fwd512_kernel<true, false> : fwd512_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * g.Hq;  // (q tile, query head)
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads512), smem,
      st, mq, mk, mv, seg, g, static_cast<__nv_bfloat16*>(out), lse, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
