// K3c: forward for head dim 256 (the Gemma4 sliding-window layers of
// gemma4_moe.cp_local_ring: bottom-right causal plus a left window over the
// concatenated neighbourhood, D = 256). Same result as K3: for every real
// local row p the softmax over its allowed keys [lo(p), p] of scale * q.k,
// times V, and LSE = m + log(l); padding rows return zeros and -inf.
//
// Design (GB300): one CTA per (128-row q tile, query head), 256 threads.
// Q (128 x 256, 64 KB) stays in shared memory. K and V stream through one
// ring of five 32 KB slots, each slot holding one 128-column half of a K or V
// tile (two 64-column chunks, 128B-swizzled), in the order the MMAs consume
// them: K(0), K(1), then per tile t: V(t), K(t+2). S is double-buffered in
// tensor memory (tile t in buffer t & 1), so S(t+1) = Q K(t+1)^T runs while
// the softmax works on tile t; O (256 fp32 columns) takes two N = 128
// products per tile, one per V half, with P read from tensor memory.
//   tensor memory  [0,128) S / P of even tiles, [128,256) of odd tiles,
//                  [256,512) O
//   warp 0  TMA producer        warp 1  one thread issues tcgen05.mma
//   warp 2  tensor memory       warps 4-7  softmax, thread = q row
// The softmax is K3's: online max / sum in fp32, the mask only on tiles a row
// sees partly, O rescaled only when the running max grows by more than 2^8.
// With attention dropout (kDrop) each row draws its keep mask of a tile before
// the tile's S arrives and zeroes the dropped weights of P; the keep scale is
// folded into the final normalisation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "dropout.cuh"
#include "pipeline.cuh"

namespace bd {

namespace {

constexpr int kD256 = 256;
constexpr int kQChunks256 = kD256 / 64;  // 64-column chunks of a row
constexpr int kChunkB256 = kTile * 128;  // 128 rows x 128 B
constexpr int kSlots256 = 5;             // ring slots, each a 128-column half of K or V
constexpr uint32_t kColS256 = 0, kColO256 = 256;
constexpr int kThreadsF256 = 256;

struct Fwd256Smem {
  alignas(1024) uint8_t q[kQChunks256][kChunkB256];
  alignas(1024) uint8_t ring[kSlots256][2][kChunkB256];
  uint64_t q_full, full[kSlots256], empty[kSlots256];
  // per S buffer, so each has at most one phase outstanding when waited on:
  // tile t's S is issued only after tile t - 2's PV products
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int b, qt, kt_lo, nk, n_real, skip;
};
static_assert(sizeof(Fwd256Smem) + 1024 <= 232448, "shared memory per CTA");
static_assert(2 * 2 * kChunkB256 >= kTile * kD256 * 2, "out staging fits ring slots 0-1");

// kMerge: merge this K/V chunk's result into the running (out, lse) instead
// of writing it (log-sum-exp weights, as the merge kernel).
template <bool kMerge, bool kDrop>
__global__ void __launch_bounds__(kThreadsF256, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ seg, const Geom g,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  Fwd256Smem& s = *reinterpret_cast<Fwd256Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
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
    for (int i = 0; i < kSlots256; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_done[i], 1);
    }
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
    if (!s.skip && nk > 0) {
      // the first copies go out now, ahead of the block barriers and the
      // tensor-memory allocation: Q, then the halves of K(0) and K(1) into
      // ring slots 0-3 (units 0-3 of the producer's order)
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&s.q_full, kQChunks256 * kChunkB256);
      for (int c = 0; c < kQChunks256; ++c) tma_load_3d(s.q[c], &tm_q, &s.q_full, c * 64, qt * kTile, b * g.Hq + h);
      const int pl = b * g.Hkv + hk;
      for (int x = 0; x < (nk < 2 ? 2 : 4); ++x) {
        const int row = (kt_lo + (x >> 1)) * kTile, half = x & 1;
        mbar_arrive_expect_tx(&s.full[x], 2 * kChunkB256);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(s.ring[x][c], &tm_k, &s.full[x], (2 * half + c) * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      }
    }
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
          uint4* o4 = reinterpret_cast<uint4*>(out + row * kD256);
          for (int c = 0; c < kD256 / 8; ++c) o4[c] = make_uint4(0, 0, 0, 0);
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
    // (Q and the halves of K(0), K(1) were issued with the barrier set-up)
    const int pl = b * g.Hkv + hk;
    int u = nk < 2 ? 2 : 4;  // ring units issued
    // one half of tile t of K or V into the next slot
    auto load_half = [&](const CUtensorMap* map, int t, int half) {
      const int slot = u % kSlots256;
      if (u >= kSlots256 && !pipe_wait(&s.empty[slot], (u / kSlots256 - 1) & 1, &s.abort_flag, vstatus))
        return false;
      mbar_arrive_expect_tx(&s.full[slot], 2 * kChunkB256);
      const int row = (kt_lo + t) * kTile;
      for (int c = 0; c < 2; ++c)
        tma_load_3d(s.ring[slot][c], map, &s.full[slot], (2 * half + c) * 64, g.kv_tm ? pl : row, g.kv_tm ? row : pl);
      ++u;
      return true;
    };
    auto load_tile = [&](const CUtensorMap* map, int t) { return load_half(map, t, 0) && load_half(map, t, 1); };
    bool ok = true;
    for (int t = 0; ok && t < nk; ++t) ok = load_tile(&tm_v, t) && (t + 2 >= nk || load_tile(&tm_k, t + 2));
    if (!ok) {
      s.abort_flag = 1;
      atomicOr(status, BD_STATUS_TIMEOUT);
    }
    // no copy into this CTA's shared memory may still be in flight at exit
    mbar_wait_drain(&s.q_full, 0);
    for (int x = (u > kSlots256 ? u - kSlots256 : 0); x < u; ++x)
      mbar_wait_drain(&s.full[x % kSlots256], (x / kSlots256) & 1);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16(128, 128, false, false);   // S = Q K^T: both K-major
    constexpr uint32_t idPV = idesc_bf16(128, 128, false, true);   // O half += P V half: V MN-major
    const uint64_t dKm = umma_desc_sw128(0, 16, 1024);
    const uint64_t dMN = umma_desc_sw128(0, kChunkB256, 1024);      // 16 KB between a half's two chunks
    const uint32_t a_q = smem_u32(s.q[0]), a_ring = smem_u32(s.ring[0][0]);
    auto wait = [&](uint64_t* bar, uint32_t par) { return pipe_wait(bar, par, &s.abort_flag, vstatus); };
    int u = 0;  // ring units consumed
    auto take = [&]() {
      const int slot = u % kSlots256;
      if (!wait(&s.full[slot], (u / kSlots256) & 1)) return -1;
      tc_fence_after();
      return slot;
    };
    // S(t) = Q K(t)^T into buffer t & 1: two halves of the head dim, 8 k-steps each
    auto issue_s = [&](int t) {
      const uint32_t d = tbase + kColS256 + (t & 1) * 128;
      for (int hf = 0; hf < 2; ++hf) {
        const int slot = take();
        if (slot < 0) return false;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_ss(d, desc_at(dKm, a_q + (2 * hf + c) * kChunkB256 + ks * 32),
                    desc_at(dKm, a_ring + slot * 2 * kChunkB256 + c * kChunkB256 + ks * 32), idS,
                    (hf | c | ks) ? 1u : 0u);
        umma_commit(&s.empty[slot]);
        ++u;
      }
      umma_commit(&s.s_full[t & 1]);
      return true;
    };
    // O[:, 128 hf : 128 hf + 128] += P(t) V(t)[:, half hf], P from tensor memory
    auto issue_pv = [&](int t) {
      for (int hf = 0; hf < 2; ++hf) {
        const int slot = take();
        if (slot < 0) return false;
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          umma_ts(tbase + kColO256 + hf * 128, tbase + kColS256 + (t & 1) * 128 + ks * 8,
                  desc_at(dMN, a_ring + slot * 2 * kChunkB256 + ks * 2048), idPV, (t > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&s.empty[slot]);
        ++u;
      }
      umma_commit(&s.o_done[t & 1]);
      return true;
    };
    bool ok = wait(&s.q_full, 0) && issue_s(0) && (nk < 2 || issue_s(1));
    for (int t = 0; ok && t < nk; ++t) {
      if (!wait(&s.p_full[t & 1], (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S two tiles on goes into the buffer this PV product reads (issued after it)
      ok = issue_pv(t) && (t + 2 >= nk || issue_s(t + 2));
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
    const uint32_t t_o = tbase + lane_off + kColO256;
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
    for (int t = 0; t < nk; ++t) {
      uint32_t km[4];  // dropout: keep bits of this row over the tile's 128 keys
      if constexpr (kDrop) row_keep_mask(g, b, h, g.row_offset + i, g.kv_offset + (kt_lo + t) * kTile, km);
      if (!warp_wait(&s.s_full[t & 1], (t >> 1) & 1, &s.abort_flag, vstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_s = tbase + lane_off + kColS256 + (t & 1) * 128;  // this tile's S buffer
      // S in two halves: the second half's load is in flight while the first
      // half's max is formed
      uint32_t xr[128];
      tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&xr[0]));
      tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[32]));
      tmem_wait_ld();
      tmem_regs_ready<64>(&xr[0]);
      tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&xr[64]));
      tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&xr[96]));
      const int c0 = (kt_lo + t) * kTile;
      // a row either sees the whole tile, none of it, or part of it; only a
      // warp with a partly seen row needs the per-element mask
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
        if (t > 0) {  // rescale the running O once the last PV products are done
          if (!warp_wait(&s.o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, &s.abort_flag, vstatus)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD256; c += 32) {
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
      const float2 rsum = __fadd2_rn(r01, r23);
      l += rsum.x + rsum.y;
      tmem_st32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full[t & 1]);
    }
    ok = __all_sync(0xffffffffu, ok);
    // the last tile's PV products complete after every earlier one
    if (ok && !warp_wait(&s.o_done[(nk - 1) & 1], ((nk - 1) >> 1) & 1, &s.abort_flag, vstatus)) ok = false;
    if (!ok) s.abort_flag = 1;
    // the four softmax warps take the same path below (it has a barrier)
    ok = named_bar_and(1, 128, ok);
    if (!ok) {
      if (lane == 0) atomicOr(status, BD_STATUS_TIMEOUT);
    } else {
      tc_fence_after();
      float inv = l > 0.f ? (kDrop ? g.drop_scale : 1.0f) / l : 0.f;
      float lse_v = (real && l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      const size_t row = (static_cast<size_t>(b) * g.Hq + h) * g.L + i;
      uint4* o4 = reinterpret_cast<uint4*>(out + row * kD256);
      // merging into a running (out, lse): log-sum-exp weights of the two sides;
      // an empty side (lse -inf) has weight 0 and its out is not read
      float w_old = 0.f;
      bool store = i < g.L;
      if (kMerge && store) {
        const float lse_o = lse[row];
        if (lse_v == -INFINITY) {
          store = lse_o == -INFINITY;  // nothing new: keep a running result, zero an empty one
        } else if (lse_o != -INFINITY) {
          const float mxl = fmaxf(lse_o, lse_v);
          const float ea = expf(lse_o - mxl), eb = expf(lse_v - mxl), tot = ea + eb;
          w_old = ea / tot;
          inv *= eb / tot;
          lse_v = mxl + logf(tot);
        }
      }
      if constexpr (kMerge) {
#pragma unroll 1
        for (int c = 0; c < kD256; c += 32) {
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
              o4[c / 8 + e] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                         pack_bf16x2(v[6], v[7]));
            }
          }
        }
      } else {
        // out (bf16) staged in ring slots 0-1, which no copy or product uses
        // once the last tile's PV products are done: row r at 512 r bytes,
        // 16-byte piece c at slot c ^ (r & 7); then one 512-byte row per warp
        // store instead of 32 scattered 16-byte pieces
        uint8_t* stg = &s.ring[0][0][0];
#pragma unroll 1
        for (int c = 0; c < kD256; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int piece = c / 8 + e;
            *reinterpret_cast<uint4*>(stg + r * (kD256 * 2) + ((piece ^ (r & 7)) << 4)) =
                make_uint4(pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
          }
        }
        named_bar_sync(1, 128);
        __nv_bfloat16* obase = out + (static_cast<size_t>(b) * g.Hq + h) * g.L * kD256;
#pragma unroll 4
        for (int k2 = 0; k2 < 32; ++k2) {
          const int rr = (warp & 3) * 32 + k2;
          const int gi = qt * kTile + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * (kD256 * 2) + ((lane ^ (rr & 7)) << 4));
          if (gi < g.L) reinterpret_cast<uint4*>(obase + static_cast<size_t>(gi) * kD256)[lane] = w;
        }
      }
      if (store) lse[row] = lse_v;
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

// Forward for D = 256 (q, k, v maps with 64 x 128 boxes); `merge`: merged into
// the running (out, lse).
cudaError_t launch_fwd256(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                          const Geom& g, void* out, float* lse, int32_t* status, int merge, cudaStream_t st) {
  if (g.D != kD256) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Fwd256Smem) + 1024;  // + 1 KB to align the swizzled tiles
  int dev = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
  auto kern = g.drop_t ? (merge ? fwd256_kernel<true, true> : fwd256_kernel<false, true>)
                       : (merge ? fwd256_kernel<true, false> : fwd256_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(g.B) * g.nqt * g.Hq;  // (q tile, query head)
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (const cudaError_t le = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsF256), smem, st, mq,
      mk, mv, seg, g, static_cast<__nv_bfloat16*>(out), lse, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
