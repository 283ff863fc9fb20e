// Internal definitions shared by the bdattn kernels and host code.
#pragma once

#include <cstdint>
#include <utility>
#include "bdattn.h"  // include/ is on the include path

namespace bd {

constexpr int kTile = 128;          // q rows / K-V rows per tile (forward, classification)
constexpr int kBwdQ = 64;           // q rows per backward iteration
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // pipeline wait limit (2 s)
constexpr int kAbortBits = BD_STATUS_TIMEOUT;      // other CTAs' errors that end a wait early

// Geometry as the kernels see it (scale resolved, table offsets computed).
struct Geom {
  int B, Hq, Hkv, D, G;
  int S_full, L, row_offset, kv_offset, S_kv, window;
  float scale;
  int kv_tm;                      // k, v, dk, dv token-major: [S_kv][B][Hkv][D]
  uint32_t drop_t;                // dropout: keep iff a pair's 16-bit draw >= drop_t; 0: no dropout
  float drop_scale;               // dropout: factor of a kept weight, 2^16 / (2^16 - drop_t)
  uint32_t seed_lo, seed_hi;      // dropout: Philox key
  int nqt, nkt, nkw;              // 128-row q tiles, 128-row K/V tiles, bitmap words per q tile
  int off[BD_SEG_NOFF];           // word offsets of the table regions
};

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int align4(int x) { return (x + 3) & ~3; }

// Table layout: each region starts on a 16-byte boundary.
__host__ __device__ inline void seg_layout(int B, int L, int S_kv, int* off, int* nqt, int* nkt, int* nkw) {
  *nqt = cdiv(L, kTile);
  *nkt = cdiv(S_kv, kTile);
  *nkw = cdiv(*nkt, 32);
  int o = 0;
  off[BD_SEG_OFF_HDR] = o;        o = align4(o + B * BD_SEG_HDR_WORDS);
  off[BD_SEG_OFF_CU_Q] = o;       o = align4(o + B * (L + 1));
  off[BD_SEG_OFF_CU_K] = o;       o = align4(o + B * (L + 1));
  off[BD_SEG_OFF_ROW_LO] = o;     o = align4(o + B * L);
  off[BD_SEG_OFF_QT_KRANGE] = o;  o = align4(o + B * (*nqt) * 2);
  off[BD_SEG_OFF_KT_QRANGE] = o;  o = align4(o + B * (*nkt) * 2);
  off[BD_SEG_OFF_FULL_BITS] = o;  o = align4(o + B * (*nqt) * (*nkw));
  off[BD_SEG_OFF_FWD_WORK] = o;   o = align4(o + B * (*nqt));
  off[BD_SEG_OFF_BWD_WORK] = o;   o = align4(o + B * (*nkt));
  off[BD_SEG_OFF_COUNTS] = o;     o = align4(o + 8);
  off[BD_SEG_OFF_TOTAL] = o;
}

// Row index of (batch row b, kv head hk, K/V buffer row j) in k, v, dk, dv.
__host__ __device__ inline size_t kv_row(const Geom& g, int b, int hk, int j) {
  return g.kv_tm ? (static_cast<size_t>(j) * g.B + b) * g.Hkv + hk
                 : (static_cast<size_t>(b) * g.Hkv + hk) * g.S_kv + j;
}

// Exchange plan layout (BD_PLAN_OFF_* regions, each on a 16-byte boundary).
// Returns the total words, or -1 when a size is out of range.
constexpr int kPlanMagic = 0x62647870;  // "bdxp"
constexpr int kPlanMaxRanks = 1024;
__host__ __device__ inline long long plan_layout(int B, int W, int L, int* off) {
  if (B < 1 || W < 1 || L < 1 || W > kPlanMaxRanks) return -1;
  if (static_cast<long long>(W) * L > 0x7fffffffLL || static_cast<long long>(B) * W > (1 << 24)) return -1;
  long long o = 0;
  long long sz[BD_PLAN_OFF_TOTAL] = {BD_PLAN_HDR_WORDS, W, W, W, W, static_cast<long long>(W) * W, W, W, W, W,
                                     static_cast<long long>(W) * L, 2LL * B * W};
  for (int i = 0; i < BD_PLAN_OFF_TOTAL; ++i) {
    off[i] = static_cast<int>(o);
    o = (o + sz[i] + 3) & ~3LL;
    if (o > 0x7fffffffLL) return -1;
  }
  off[BD_PLAN_OFF_TOTAL] = static_cast<int>(o);
  return o;
}

// Header words that record the geometry the table was built for.
constexpr int kHdrRowOffset = 16, kHdrL = 17, kHdrKvOffset = 18, kHdrSkv = 19, kHdrWindow = 20,
              kHdrSfull = 21, kHdrMagic = 22,
              kHdrKvChunk = 23;  // 1: table built for one K/V chunk (no K/V range requirement)
constexpr int kSegMagic = 0x62646174;  // "bdat"

// The allowed key interval [lo, hi] (global positions) of a real local row i:
// hi = p, lo = max(doc_start, p - W + 1).
__device__ __forceinline__ int row_lo_window(int doc_start, int p, int window) {
  return (window > 0 && p - window + 1 > doc_start) ? p - window + 1 : doc_start;
}

// Number of 128-row K/V tiles some local row can attend by position alone:
// a row p in [row_offset, row_offset + L) attends keys s <= p and, with a
// window W, s > p - W. Every tile the segment table marks as attended lies in
// this range, so a backward grid of B x this many tiles covers them all.
__host__ __device__ inline int kv_tiles_reachable(const Geom& g) {
  const long long hi = static_cast<long long>(g.row_offset) + g.L - 1 - g.kv_offset;
  const long long lo = g.window > 0 ? static_cast<long long>(g.row_offset) - g.window + 1 - g.kv_offset : 0;
  const long long a = lo > 0 ? lo : 0;
  const long long e = hi < g.S_kv - 1 ? hi : static_cast<long long>(g.S_kv) - 1;
  return e < a ? 0 : static_cast<int>(e / kTile - a / kTile + 1);
}

#ifdef __CUDACC__
// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization and starts with pdl_begin(): it waits
// (griddepcontrol.wait) until the grids before it in the stream have completed
// and their memory is visible -- so it touches no global memory before that --
// and then lets the next grid launch (griddepcontrol.launch_dependents). A
// dependent grid launches only once every CTA of this one has started, so its
// CTAs take only resources this grid leaves free; what it gains is that its
// CTAs are already resident when this grid ends, instead of launching then.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class... Exp, class... Act>
inline cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Act&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

// Zero dK / dV rows of the K/V tiles no local row attends. The backward work
// list holds the n_att attended tiles first; the (position, kv head) pairs of
// the rest, x = (z - n_att) * Hkv + hk, are taken by writer w of n_w as
// x = w, w + n_w, ...; threads t = 0..nthr-1 share each tile. The stores are
// marked streaming (evict-first) as nothing reads these lines again soon.
__device__ inline void zero_unattended_kv(const int32_t* seg, const Geom& g, int n_att, int w, int n_w, int t, int nthr,
                                          void* dk, void* dv, int grads_bf16, int32_t* status) {
  const int n_items = g.B * g.nkt;
  const long long n_pairs = static_cast<long long>(n_items - n_att) * g.Hkv;
  const size_t row_bytes = static_cast<size_t>(g.D) * (grads_bf16 ? 2 : 4);  // a multiple of 16
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (long long x = w; x < n_pairs; x += n_w) {
    const int z = n_att + static_cast<int>(x / g.Hkv), hk = static_cast<int>(x % g.Hkv);
    const int wi = seg[g.off[BD_SEG_OFF_BWD_WORK] + z];
    if (wi < 0 || wi >= n_items) {
      if (t == 0) atomicOr(status, BD_STATUS_BOUNDS);
      continue;
    }
    const int b = wi / g.nkt, r0 = (wi % g.nkt) * kTile;
    const int r1 = r0 + kTile < g.S_kv ? r0 + kTile : g.S_kv;
    const size_t vpr = row_bytes / 16;  // 16-byte pieces per row
    const size_t n16 = static_cast<size_t>(r1 - r0) * vpr;
    uint4* pk = static_cast<uint4*>(dk);
    uint4* pv = static_cast<uint4*>(dv);
    if (!g.kv_tm) {  // the tile's rows are contiguous
      const size_t off = kv_row(g, b, hk, r0) * vpr;
      for (size_t i = t; i < n16; i += nthr) {
        __stcs(pk + off + i, zero);
        __stcs(pv + off + i, zero);
      }
    } else {  // token-major: one row of this kv head per token
      for (size_t i = t; i < n16; i += nthr) {
        const size_t off = kv_row(g, b, hk, r0 + static_cast<int>(i / vpr)) * vpr + i % vpr;
        __stcs(pk + off, zero);
        __stcs(pv + off, zero);
      }
    }
  }
}
#endif

}  // namespace bd
