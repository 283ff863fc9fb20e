// K1 (segmentation) and K2 (128x128 tile classification) of the block-diagonal
// CP attention path.
//
// K1 follows blockdiag_cp.kernels `_cp_blockdiag_varlen` / `_varlen_seg_for_rank`
// (NeMo AutoModel API): padding is a contiguous tail so the real local rows
// are a prefix [0, n_real); one varlen segment per document the local rows
// touch, q segment = its local rows, k segment = [doc_start, last local q + 1).
// Only the first segment can start before the shard (the straddle), so its
// document start is found by scanning left; every later segment starts inside
// the shard. The reference builds this on the host after a .tolist() copy;
// here one CTA per batch row builds it on the device with warp ballots and a
// block scan, so no host synchronisation is needed.
//
// K2 marks every (128-row q tile, 128-row K/V tile) as full, partial or empty.
// A real row p may attend the keys [lo(p), p] with lo(p) = max(doc_start(p),
// p - W + 1); lo and hi are non-decreasing in p, so the non-empty K/V tiles
// of a q tile form one contiguous range, and so do the q rows of a K/V tile.
// The forward and backward kernels only visit those ranges (empty tiles are
// never loaded) and mask only the partial tiles.
#include <climits>
#include <cstdint>

#include "common.cuh"

namespace bd {

namespace {

struct MinOp { __device__ int operator()(int a, int b) const { return a < b ? a : b; } };
struct MaxOp { __device__ int operator()(int a, int b) const { return a > b ? a : b; } };
struct OrOp  { __device__ int operator()(int a, int b) const { return a | b; } };
struct AddOp { __device__ int operator()(int a, int b) const { return a + b; } };

// Every thread of the block gets the reduction of `v`.
template <class Op>
__device__ int block_reduce(int v, Op op, int* s_red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) s_red[w] = v;
  __syncthreads();
  v = s_red[lane < nw ? lane : 0];
#pragma unroll
  for (int o = 16; o; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exclusive prefix sum of `v` over the block; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* s_red, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) s_red[w] = incl;
  __syncthreads();
  int wpre = 0, tot = 0;
  for (int x = 0; x < nw; ++x) {
    const int t = s_red[x];
    if (x < w) wpre += t;
    tot += t;
  }
  *total = tot;
  return wpre + incl - v;
}

}  // namespace

// One CTA per batch row.
__global__ void __launch_bounds__(1024) seg_build_kernel(const int32_t* __restrict__ doc, Geom g,
                                                         int32_t* __restrict__ seg, int32_t* status, int kv_chunk) {
  pdl_begin();
  __shared__ int s_red[32];
  const int b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
  const int ro = g.row_offset, L = g.L;
  const int32_t* row = doc + static_cast<size_t>(b) * g.S_full;
  int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
  int32_t* cu_q = seg + g.off[BD_SEG_OFF_CU_Q] + b * (L + 1);
  int32_t* cu_k = seg + g.off[BD_SEG_OFF_CU_K] + b * (L + 1);
  int32_t* rowlo = seg + g.off[BD_SEG_OFF_ROW_LO] + b * L;

  // Layout over the whole row: ids >= 0, no document after padding.
  int bad = 0;
#pragma unroll 8
  for (int p = tid; p < g.S_full; p += nthr) {
    const int c = row[p];
    if (c < 0 || (p > 0 && c != 0 && row[p - 1] == 0)) bad = 1;
  }
  bad = block_reduce(bad, OrOp(), s_red);

  // n_real: the first padding row of the shard (L if none).
  int first_pad = L;
  for (int i = tid; i < L; i += nthr)
    if (row[ro + i] == 0) {
      first_pad = i;
      break;
    }
  const int n_real = block_reduce(first_pad, MinOp(), s_red);

  // Segment starts: local row 0 and every row whose id differs from the previous
  // one, compacted in order with a ballot + block scan.
  int n_seg = 0;
  for (int c0 = 0; c0 < n_real; c0 += nthr) {
    const int i = c0 + tid;
    const int f = (i < n_real) && (i == 0 || row[ro + i] != row[ro + i - 1]);
    int tot;
    const int pos = block_exclusive_scan(f, s_red, &tot);
    if (f) cu_q[n_seg + pos] = i;
    n_seg += tot;
  }

  // Document start of the first segment: scan left from the shard start.
  int s_first = ro;
  if (n_real > 0) {
    const int id0 = row[ro];
    int found = -1;
    for (int c1 = ro; c1 > 0; c1 -= nthr) {
      const int p = c1 - 1 - tid;
      const int f = (p >= 0 && row[p] != id0) ? p : -1;
      const int m = block_reduce(f, MaxOp(), s_red);
      if (m >= 0) {
        found = m;
        break;
      }
    }
    s_first = found + 1;
  }
  if (tid == 0) cu_q[n_seg] = n_real;
  __syncthreads();  // cu_q visible to the whole block

  // Each local document id must not occur before its own run. Fast path: ids
  // increase from segment to segment and the first one exceeds every id before
  // the straddle. Otherwise check every segment exactly.
  if (n_seg > 0) {
    int m0 = INT_MIN;
#pragma unroll 8
    for (int p = tid; p < s_first; p += nthr) m0 = max(m0, row[p]);
    m0 = block_reduce(m0, MaxOp(), s_red);
    int fast_ok = 1;
    for (int k = tid; k < n_seg; k += nthr) {
      const int idk = row[ro + cu_q[k]];
      const int prev = (k == 0) ? m0 : row[ro + cu_q[k - 1]];
      if (!(idk > prev)) fast_ok = 0;
    }
    fast_ok = block_reduce(fast_ok, MinOp(), s_red);
    if (!fast_ok) {
      int dup = 0;
      for (int k = 0; k < n_seg && !dup; ++k) {
        const int idk = row[ro + cu_q[k]];
        const int st = (k == 0) ? s_first : ro + cu_q[k];
        int hit = 0;
        for (int p = tid; p < st; p += nthr)
          if (row[p] == idk) {
            hit = 1;
            break;
          }
        dup = block_reduce(hit, OrOp(), s_red);
      }
      bad |= dup;
    }
  }

  // Document start of every local row (-1 on padding rows).
  for (int i = tid; i < L; i += nthr) {
    int v = -1;
    if (i < n_real) {
      int lo = 0, hi = n_seg - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_q[mid] <= i) lo = mid; else hi = mid - 1;
      }
      v = (lo == 0) ? s_first : ro + cu_q[lo];
    }
    rowlo[i] = v;
  }

  // cu_k and the maxima.
  const int real_end = ro + n_real;
  int mq = 0, mk = 0, mt = 0;
  for (int k = tid; k < n_seg; k += nthr) {
    const int q0 = cu_q[k], q1 = cu_q[k + 1];
    const int st = (k == 0) ? s_first : ro + q0;
    cu_k[k] = st - s_first;
    const int sq = q1 - q0, sk = ro + q1 - st;
    mq = max(mq, sq);
    mk = max(mk, sk);
    if (k >= 1) mt = max(mt, sq);
  }
  mq = block_reduce(mq, MaxOp(), s_red);
  mk = block_reduce(mk, MaxOp(), s_red);
  mt = block_reduce(mt, MaxOp(), s_red);

  if (tid == 0) {
    cu_k[n_seg] = real_end - s_first;
    const int need_lo = n_real > 0 ? row_lo_window(s_first, ro, g.window) : ro;
    // a chunk of the K/V range need not hold every key the rows may attend
    const int kv_bad = !kv_chunk && n_real > 0 && (need_lo < g.kv_offset || real_end > g.kv_offset + g.S_kv);
    const int row_status = (bad ? BD_STATUS_LAYOUT : 0) | (kv_bad ? BD_STATUS_KV_RANGE : 0);
    hdr[BD_SEG_N_REAL] = n_real;
    hdr[BD_SEG_N_SEG] = n_seg;
    hdr[BD_SEG_S_FIRST] = s_first;
    hdr[BD_SEG_REAL_END] = real_end;
    hdr[BD_SEG_MAX_Q] = mq;
    hdr[BD_SEG_MAX_K] = mk;
    hdr[BD_SEG_FIRST_Q] = n_seg >= 1 ? cu_q[1] : 0;
    hdr[BD_SEG_FIRST_K] = n_seg >= 2 ? ro + cu_q[1] - s_first : (n_seg == 1 ? real_end - s_first : 0);
    hdr[BD_SEG_MAX_TAIL] = mt;
    hdr[BD_SEG_KV_NEED_LO] = need_lo;
    hdr[BD_SEG_ROW_STATUS] = row_status;
    for (int x = 11; x < kHdrRowOffset; ++x) hdr[x] = 0;
    hdr[kHdrRowOffset] = ro;
    hdr[kHdrL] = L;
    hdr[kHdrKvOffset] = g.kv_offset;
    hdr[kHdrSkv] = g.S_kv;
    hdr[kHdrWindow] = g.window;
    hdr[kHdrSfull] = g.S_full;
    hdr[kHdrKvChunk] = kv_chunk;
    hdr[kHdrMagic] = kSegMagic;
    for (int x = kHdrKvChunk + 1; x < BD_SEG_HDR_WORDS; ++x) hdr[x] = 0;
    if (row_status) atomicOr(status, row_status);
  }
}

// A single CTA classifies every tile of every batch row and builds the two
// longest-first work lists. Dynamic shared memory: (nbins) ints of histogram.
__global__ void __launch_bounds__(1024) classify_kernel(Geom g, int32_t* __restrict__ seg, int nbins) {
  pdl_begin();
  extern __shared__ int s_hist[];
  __shared__ int s_red[32];
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int ro = g.row_offset, L = g.L, W = g.window;
  int n_full = 0, n_part = 0, n_kv_att = 0;

  for (int b = 0; b < g.B; ++b) {
    const int32_t* hdr = seg + g.off[BD_SEG_OFF_HDR] + b * BD_SEG_HDR_WORDS;
    const int32_t* rowlo = seg + g.off[BD_SEG_OFF_ROW_LO] + b * L;
    int32_t* qk = seg + g.off[BD_SEG_OFF_QT_KRANGE] + b * g.nqt * 2;
    int32_t* kq = seg + g.off[BD_SEG_OFF_KT_QRANGE] + b * g.nkt * 2;
    int32_t* bits = seg + g.off[BD_SEG_OFF_FULL_BITS] + b * g.nqt * g.nkw;
    const int n_real = hdr[BD_SEG_N_REAL];

    // Per q tile: the range of K/V tiles and which of them are full.
    for (int qt = tid; qt < g.nqt; qt += nthr) {
      const int first = qt * kTile;
      int kt_lo = 0, kt_hi = -1;
      for (int w = 0; w < g.nkw; ++w) bits[qt * g.nkw + w] = 0;
      if (first < n_real) {
        const int last = min(first + kTile - 1, n_real - 1);
        const int j_lo = max(row_lo_window(rowlo[first], ro + first, W) - g.kv_offset, 0);
        const int j_hi = min(ro + last - g.kv_offset, g.S_kv - 1);
        if (j_lo <= j_hi) {
          kt_lo = j_lo / kTile;
          kt_hi = j_hi / kTile;
          const bool all_real = first + kTile - 1 < n_real;
          const int lo_last = row_lo_window(rowlo[last], ro + last, W);
          const int hi_first = ro + first;
          uint32_t word = 0;
          int cur_w = kt_lo >> 5;
          for (int kt = kt_lo; kt <= kt_hi; ++kt) {
            if ((kt >> 5) != cur_w) {
              bits[qt * g.nkw + cur_w] = static_cast<int32_t>(word);
              word = 0;
              cur_w = kt >> 5;
            }
            const int s0 = g.kv_offset + kt * kTile;
            const bool full = all_real && lo_last <= s0 && s0 + kTile - 1 <= hi_first &&
                              kt * kTile + kTile - 1 < g.S_kv;
            if (full) {
              word |= 1u << (kt & 31);
              ++n_full;
            } else {
              ++n_part;
            }
          }
          bits[qt * g.nkw + cur_w] = static_cast<int32_t>(word);
        }
      }
      qk[2 * qt] = kt_lo;
      qk[2 * qt + 1] = kt_hi;
    }

    // Per K/V tile: the local q rows whose allowed interval meets it.
    for (int kt = tid; kt < g.nkt; kt += nthr) {
      const int s_lo = g.kv_offset + kt * kTile;
      const int s_hi = g.kv_offset + min(kt * kTile + kTile - 1, g.S_kv - 1);
      const int i_begin = max(0, s_lo - ro);
      // first row in [i_begin, n_real) whose lo exceeds s_hi
      int a = i_begin, e = n_real;
      while (a < e) {
        const int mid = (a + e) >> 1;
        if (row_lo_window(rowlo[mid], ro + mid, W) > s_hi) e = mid; else a = mid + 1;
      }
      const int i_end = a;
      kq[2 * kt] = (i_begin < i_end) ? i_begin : 0;
      kq[2 * kt + 1] = (i_begin < i_end) ? i_end : 0;
      n_kv_att += i_begin < i_end ? 1 : 0;
    }
  }
  n_full = block_reduce(n_full, AddOp(), s_red);
  n_part = block_reduce(n_part, AddOp(), s_red);
  n_kv_att = block_reduce(n_kv_att, AddOp(), s_red);
  if (tid == 0) {
    int32_t* counts = seg + g.off[BD_SEG_OFF_COUNTS];
    counts[0] = n_full;
    counts[1] = n_part;
    counts[2] = g.B * g.nqt * g.nkt - n_full - n_part;
    counts[3] = n_kv_att;  // these K/V tiles lead the backward work list
    for (int x = 4; x < 8; ++x) counts[x] = 0;
  }
  __syncthreads();  // ranges written above are read below by other threads

  // Longest-first work lists (counting sort on the work estimate, descending).
  for (int list = 0; list < 2; ++list) {
    const int n_items = list == 0 ? g.B * g.nqt : g.B * g.nkt;
    int32_t* out = seg + g.off[list == 0 ? BD_SEG_OFF_FWD_WORK : BD_SEG_OFF_BWD_WORK];
    for (int x = tid; x < nbins; x += nthr) s_hist[x] = 0;
    __syncthreads();
    auto key_of = [&](int item) -> int {
      int key;
      if (list == 0) {
        const int32_t* qk = seg + g.off[BD_SEG_OFF_QT_KRANGE] + item * 2;
        key = qk[1] >= qk[0] ? qk[1] - qk[0] + 1 : 0;
      } else {
        const int32_t* kq = seg + g.off[BD_SEG_OFF_KT_QRANGE] + item * 2;
        key = kq[1] > kq[0] ? (kq[1] - 1) / kBwdQ - kq[0] / kBwdQ + 1 : 0;
      }
      return min(key, nbins - 1);
    };
    for (int it = tid; it < n_items; it += nthr) atomicAdd(&s_hist[nbins - 1 - key_of(it)], 1);
    __syncthreads();
    // exclusive scan of the histogram, in chunks of blockDim
    int carry = 0;
    for (int c0 = 0; c0 < nbins; c0 += nthr) {
      const int x = c0 + tid;
      const int v = x < nbins ? s_hist[x] : 0;
      int tot;
      const int ex = block_exclusive_scan(v, s_red, &tot);
      __syncthreads();
      if (x < nbins) s_hist[x] = carry + ex;
      carry += tot;
      __syncthreads();
    }
    for (int it = tid; it < n_items; it += nthr) {
      const int pos = atomicAdd(&s_hist[nbins - 1 - key_of(it)], 1);
      out[pos] = it;
    }
    __syncthreads();
  }
}

cudaError_t launch_seg_build(const int32_t* doc, const Geom& g, int32_t* seg, int32_t* status, cudaStream_t st,
                             int kv_chunk) {
  if (const cudaError_t le = launch_pdl(seg_build_kernel, dim3(g.B), dim3(1024), 0, st, doc, g, seg, status, kv_chunk);
      le != cudaSuccess) return le;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // histogram bins of the work-list sort (48 KB of shared memory at most)
  int nbins = (g.nkt > cdiv(g.L, kBwdQ) ? g.nkt : cdiv(g.L, kBwdQ)) + 1;
  if (nbins > 12288) nbins = 12288;
  if (const cudaError_t le = launch_pdl(classify_kernel, dim3(1), dim3(1024), static_cast<size_t>(nbins) * 4, st, g,
      seg, nbins); le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace bd
