// Internal definitions shared by the bdattn kernels and host code.
#pragma once

#include <cstdint>
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

// Header words that record the geometry the table was built for.
constexpr int kHdrRowOffset = 16, kHdrL = 17, kHdrKvOffset = 18, kHdrSkv = 19, kHdrWindow = 20,
              kHdrSfull = 21, kHdrMagic = 22;
constexpr int kSegMagic = 0x62646174;  // "bdat"

// The allowed key interval [lo, hi] (global positions) of a real local row i:
// hi = p, lo = max(doc_start, p - W + 1).
__device__ __forceinline__ int row_lo_window(int doc_start, int p, int window) {
  return (window > 0 && p - window + 1 > doc_start) ? p - window + 1 : doc_start;
}

}  // namespace bd
