/*
 * Plain fp64 CPU oracle for per-document causal (block-diagonal) attention of
 * one context-parallel query shard against a K/V range.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call this code:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * it. It shares no code, header or table with the CUDA library.
 *
 * Sources (NVIDIA NeMo AutoModel API pages):
 *  [K.mask]    blockdiag_cp.kernels, `_cp_blockdiag_mask`: a query attends a key
 *              iff they share a document, neither is padding, and the key is
 *              causally visible; the diagonal is always allowed.
 *  [K.varlen]  blockdiag_cp.kernels, `_cp_blockdiag_varlen`: equal to mask +
 *              SDPA on real query rows; padding is a contiguous tail; one
 *              segment per document the local rows touch, q segment = the
 *              local rows of that document, k segment = [doc_start,
 *              last_local_q+1); padding query rows are returned as zeros.
 *  [K.seg]     blockdiag_cp.kernels, `_varlen_seg_for_rank` and
 *              `precompute_blockdiag_varlen_meta` (cu_seqlens per rank,
 *              {"n_real": 0} for an all-padding shard).
 *  [E.halo]    blockdiag_cp.exchange, left-halo plan: the K/V range a rank
 *              needs is [s_first, real_end).
 *  [R.fa]      gemma4_moe.cp_local_ring, module text: the sliding layer is a
 *              bottom-right causal attention with a left window.
 *  [A.lse]     gemma4_moe.cp_attention, `_scatter_lse`: LSE is -inf on rows
 *              that take no part.
 *  [K.drop]    blockdiag_cp.kernels, `_cp_blockdiag_varlen`, argument
 *              `dropout_p` (the chance that an attention weight is dropped); the same argument
 *              on the FlashAttention varlen helpers and ring-attention
 *              functions of gemma4_moe.cp_attention. Read as inverted
 *              dropout on the attention probabilities: each allowed P_ps is
 *              kept with probability 1 - p and scaled by the inverse of that
 *              probability, the LSE stays that of the undropped softmax.
 *  [Philox]    J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
 *              random numbers: as easy as 1, 2, 3", SC'11: the counter-based
 *              generator Philox-4x32-10 that draws the keep decisions.
 *
 * The window is read as p - s < W (W <= 0: no window). The LSE is the natural
 * logarithm. GQA maps query head h to kv head h / (Hq / Hkv).
 *
 * Floating point: inputs arrive as fp64 (the Python side widens the bf16
 * inputs exactly); every sum, exp and log is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int B, Hq, Hkv, D;
  int S_full;     /* length of each doc_ids row (full padded sequence) */
  int L;          /* local query rows */
  int row_offset; /* global position of local row 0 */
  int kv_offset;  /* global position of K/V buffer row 0 */
  int S_kv;       /* K/V buffer rows */
  int window;     /* <= 0: none */
  double scale;
  double dropout_p;            /* [K.drop] probability of dropping an attention weight; 0: none */
  uint32_t seed_lo, seed_hi;   /* [Philox] key of the dropout stream */
} og_geom;

/* Error codes returned by the oracle entry points. */
enum { OG_OK = 0, OG_ERR_ARG = -1, OG_ERR_EMPTY_ROW = -2, OG_ERR_NOMEM = -3 };

/* ---------------------------------------------------------------- mask --- */

/* [K.mask] with the sliding window added on the non-diagonal clause. */
static int og_allowed(const int32_t* doc_row, int p, int s, int window) {
  if (s == p) return 1;
  const int dp = doc_row[p];
  if (dp == 0 || dp != doc_row[s]) return 0;
  if (s > p) return 0;
  if (window > 0 && p - s >= window) return 0;
  return 1;
}

/* ------------------------------------------------------------- dropout --- */

/* [Philox] Philox-4x32 with R = 10 rounds. The state is four 32-bit words
 * (the counter) and the key two 32-bit words. One round multiplies words 0
 * and 2 by the round multipliers M0 = 0xD2511F53 and M1 = 0xCD9E8D57 (full
 * 64-bit products) and forms the new state
 *   ( hi(M1 x2) ^ x1 ^ k0,  lo(M1 x2),  hi(M0 x0) ^ x3 ^ k1,  lo(M0 x0) );
 * between rounds the key is bumped by the Weyl constants W0 = 0x9E3779B9
 * (golden ratio) and W1 = 0xBB67AE85 (sqrt(3) - 1). The first round uses the
 * key as given. */
static void og_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * x0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    const uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
    const uint32_t y1 = (uint32_t)p1;
    const uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
    const uint32_t y3 = (uint32_t)p0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* Test hook: n independent evaluations, ctr[n][4], key[n][2] -> out[n][4]. */
int og_philox(const uint32_t* ctr, const uint32_t* key, int n, uint32_t* out) {
  if (n < 0 || (n > 0 && (!ctr || !key || !out))) return OG_ERR_ARG;
  for (int i = 0; i < n; ++i) og_philox4x32_10(ctr + 4 * i, key + 2 * i, out + 4 * i);
  return OG_OK;
}

/* Keep threshold on a 16-bit uniform: T = round(p * 2^16). A weight is kept
 * iff its 16-bit draw u >= T, i.e. with probability (2^16 - T) / 2^16. */
static uint32_t og_drop_threshold(double p) { return (uint32_t)floor(p * 65536.0 + 0.5); }

/* Scale of a kept weight: the inverse of the keep probability. */
static double og_drop_scale(const og_geom* g) {
  const uint32_t T = og_drop_threshold(g->dropout_p);
  return 65536.0 / (double)(65536u - T);
}

/* The 16-bit draw of the pair (query head h, query position p, key position s)
 * of batch row b: one Philox call covers eight consecutive key positions of
 * one query row; counter = (s / 8, p, h, b), key = (seed_lo, seed_hi); key s
 * takes the 16-bit piece s mod 8 of the 128-bit output (word (s mod 8) / 2,
 * low half for even s, high half for odd s). Positions are global. */
static uint32_t og_drop_u16(const og_geom* g, int b, int h, int p, int s) {
  const uint32_t ctr[4] = {(uint32_t)s >> 3, (uint32_t)p, (uint32_t)h, (uint32_t)b};
  const uint32_t key[2] = {g->seed_lo, g->seed_hi};
  uint32_t r[4];
  og_philox4x32_10(ctr, key, r);
  const uint32_t w = r[(s & 7) >> 1];
  return (s & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* Multiplier of P_ps in the output: 0 (dropped), the keep scale (kept), or 1
 * without dropout. */
static double og_drop_factor(const og_geom* g, int b, int h, int p, int s) {
  if (g->dropout_p <= 0.0) return 1.0;
  return og_drop_u16(g, b, h, p, s) >= og_drop_threshold(g->dropout_p) ? og_drop_scale(g) : 0.0;
}

static int og_geom_ok(const og_geom* g) {
  if (!g || g->B <= 0 || g->Hq <= 0 || g->Hkv <= 0 || g->D <= 0) return 0;
  if (!(g->dropout_p >= 0.0 && g->dropout_p < 1.0) || og_drop_threshold(g->dropout_p) > 65535u) return 0;
  if (g->Hq % g->Hkv) return 0;
  if (g->L < 0 || g->S_kv < 0 || g->S_full <= 0) return 0;
  if (g->row_offset < 0 || g->row_offset + g->L > g->S_full) return 0;
  if (g->kv_offset < 0 || g->kv_offset + g->S_kv > g->S_full) return 0;
  return 1;
}

/* Dense allow-mask [B][L][S_kv] (bytes 0/1), exactly as [K.mask] builds it
 * (including the padding rows' self-edge). */
int og_mask(const int32_t* doc, const og_geom* g, uint8_t* mask) {
  if (!og_geom_ok(g) || !doc || !mask) return OG_ERR_ARG;
  for (int b = 0; b < g->B; ++b) {
    const int32_t* row = doc + (size_t)b * g->S_full;
    for (int i = 0; i < g->L; ++i)
      for (int j = 0; j < g->S_kv; ++j)
        mask[((size_t)b * g->L + i) * g->S_kv + j] =
            (uint8_t)og_allowed(row, g->row_offset + i, g->kv_offset + j, g->window);
  }
  return OG_OK;
}

/* Number of allowed (query, key) pairs over real query rows, padding rows'
 * self-edges excluded: the unmasked work of the attention. */
int64_t og_pairs(const int32_t* doc, const og_geom* g) {
  if (!og_geom_ok(g) || !doc) return -1;
  int64_t total = 0;
  for (int b = 0; b < g->B; ++b) {
    const int32_t* row = doc + (size_t)b * g->S_full;
    int64_t sub = 0;
#pragma omp parallel for reduction(+ : sub) schedule(dynamic, 16)
    for (int i = 0; i < g->L; ++i) {
      const int p = g->row_offset + i;
      if (row[p] == 0) continue;
      for (int j = 0; j < g->S_kv; ++j) sub += og_allowed(row, p, g->kv_offset + j, g->window);
    }
    total += sub;
  }
  return total;
}

/* ------------------------------------------------------------ segments --- */

/* Per batch row output block of og_segments (int32):
 *   [0] n_real   [1] n_seg   [2] s_first  [3] real_end  [4] max_q  [5] max_k
 *   [6] first_q  [7] first_k [8] max_tail [9] kv_need_lo
 *   [10] layout_error (0/1)  [11] kv_range_error (0/1)
 *   [16 .. 16+L]        cu_q[0..n_seg]
 *   [16+L+1 .. 16+2L+1] cu_k[0..n_seg]
 * Stride per row: 16 + 2 * (L + 1). */
enum { OG_SEG_HDR = 16 };

int og_seg_stride(int L) { return OG_SEG_HDR + 2 * (L + 1); }

/* [K.varlen] + [K.seg]: walk the local rows once; a new segment starts at
 * local row 0 and wherever the document id changes; each segment's document
 * start is found by scanning left from its first row while the id is equal
 * (which can cross into earlier shards: the straddle). */
int og_segments(const int32_t* doc, const og_geom* g, int32_t* out) {
  if (!og_geom_ok(g) || !doc || !out) return OG_ERR_ARG;
  const int L = g->L, stride = og_seg_stride(L);
  for (int b = 0; b < g->B; ++b) {
    const int32_t* row = doc + (size_t)b * g->S_full;
    int32_t* o = out + (size_t)b * stride;
    int32_t* cu_q = o + OG_SEG_HDR;
    int32_t* cu_k = cu_q + (L + 1);
    memset(o, 0, sizeof(int32_t) * (size_t)stride);

    int n_real = L;
    for (int i = 0; i < L; ++i)
      if (row[g->row_offset + i] == 0) {
        n_real = i;
        break;
      }
    int n_seg = 0;
    for (int i = 0; i < n_real; ++i)
      if (i == 0 || row[g->row_offset + i] != row[g->row_offset + i - 1]) cu_q[n_seg++] = i;
    cu_q[n_seg] = n_real;

    int s_first = g->row_offset;
    int layout_err = 0;
    int max_q = 0, max_k = 0, max_tail = 0;
    for (int k = 0; k < n_seg; ++k) {
      const int id = row[g->row_offset + cu_q[k]];
      int start = g->row_offset + cu_q[k];
      while (start > 0 && row[start - 1] == id) --start;
      if (k == 0) s_first = start;
      cu_k[k] = start; /* made relative to s_first below */
      const int sq = cu_q[k + 1] - cu_q[k];
      const int sk = g->row_offset + cu_q[k + 1] - start;
      if (sq > max_q) max_q = sq;
      if (sk > max_k) max_k = sk;
      if (k >= 1 && sq > max_tail) max_tail = sq;
      /* the id must not occur before its own run */
      for (int s = 0; s < start; ++s)
        if (row[s] == id) {
          layout_err = 1;
          break;
        }
    }
    const int real_end = g->row_offset + n_real;
    for (int k = 0; k < n_seg; ++k) cu_k[k] -= s_first;
    cu_k[n_seg] = real_end - s_first;

    /* padding only as a tail, ids non-negative, over the whole row */
    for (int s = 0; s < g->S_full; ++s) {
      if (row[s] < 0) layout_err = 1;
      if (s > 0 && row[s - 1] == 0 && row[s] != 0) layout_err = 1;
    }

    /* lowest key any real local row may attend: min over rows of
     * max(doc_start(p), p - W + 1) */
    int need_lo = real_end;
    for (int k = 0; k < n_seg; ++k) {
      for (int i = cu_q[k]; i < cu_q[k + 1]; ++i) {
        const int p = g->row_offset + i;
        int lo = s_first + cu_k[k];
        if (g->window > 0 && p - g->window + 1 > lo) lo = p - g->window + 1;
        if (lo < need_lo) need_lo = lo;
      }
    }
    if (n_seg == 0) need_lo = g->row_offset;
    int kv_err = 0;
    if (n_real > 0 && (need_lo < g->kv_offset || real_end > g->kv_offset + g->S_kv)) kv_err = 1;

    o[0] = n_real;
    o[1] = n_seg;
    o[2] = s_first;
    o[3] = real_end;
    o[4] = max_q;
    o[5] = max_k;
    o[6] = n_seg >= 1 ? cu_q[1] : 0;
    o[7] = n_seg >= 1 ? cu_k[1] : 0;
    o[8] = max_tail;
    o[9] = need_lo;
    o[10] = layout_err;
    o[11] = kv_err;
  }
  return OG_OK;
}

/* ------------------------------------------------------------- forward --- */

static double og_dot(const double* a, const double* b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

/* One query row: softmax(scale * q k^T + mask) v over the allowed keys.
 * Padding rows give out = 0, lse = -inf ([K.varlen], [A.lse]).
 * xbuf: scratch of S_kv doubles. Returns 0, or OG_ERR_EMPTY_ROW when a real
 * row has no allowed key inside the K/V buffer. */
static int og_fwd_row(const double* q, const double* k, const double* v, const int32_t* doc,
                      const og_geom* g, int b, int h, int i, double* out_row, double* lse_out,
                      double* xbuf) {
  const int D = g->D, G = g->Hq / g->Hkv, hk = h / G;
  const int32_t* row = doc + (size_t)b * g->S_full;
  const int p = g->row_offset + i;
  if (row[p] == 0) {
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    *lse_out = -INFINITY;
    return OG_OK;
  }
  const double* qr = q + (((size_t)b * g->Hq + h) * g->L + i) * D;
  const double* kb = k + ((size_t)b * g->Hkv + hk) * (size_t)g->S_kv * D;
  const double* vb = v + ((size_t)b * g->Hkv + hk) * (size_t)g->S_kv * D;
  double m = -INFINITY;
  for (int j = 0; j < g->S_kv; ++j) {
    if (og_allowed(row, p, g->kv_offset + j, g->window)) {
      xbuf[j] = g->scale * og_dot(qr, kb + (size_t)j * D, D);
      if (xbuf[j] > m) m = xbuf[j];
    } else {
      xbuf[j] = -INFINITY;
    }
  }
  if (m == -INFINITY) return OG_ERR_EMPTY_ROW;
  double l = 0.0;
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  for (int j = 0; j < g->S_kv; ++j) {
    if (xbuf[j] == -INFINITY) continue;
    const double w = exp(xbuf[j] - m);
    l += w;  /* [K.drop] the softmax normaliser is the undropped one */
    const double wz = w * og_drop_factor(g, b, h, p, g->kv_offset + j);
    const double* vr = vb + (size_t)j * D;
    for (int d = 0; d < D; ++d) out_row[d] += wz * vr[d];
  }
  for (int d = 0; d < D; ++d) out_row[d] /= l;
  *lse_out = m + log(l);
  return OG_OK;
}

/* Forward for a list of rows sel[n][3] = (b, h, i).
 * q: [B][Hq][L][D], k, v: [B][Hkv][S_kv][D]; out: [n][D], lse: [n]. */
int og_fwd_rows(const double* q, const double* k, const double* v, const int32_t* doc, const og_geom* g,
                const int32_t* sel, int n, double* out, double* lse) {
  if (!og_geom_ok(g) || !q || !k || !v || !doc || !sel || !out || !lse) return OG_ERR_ARG;
  int err = OG_OK;
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(g->S_kv > 0 ? g->S_kv : 1));
    if (!xbuf) {
#pragma omp atomic write
      err = OG_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int t = 0; t < n; ++t) {
        const int b = sel[3 * t], h = sel[3 * t + 1], i = sel[3 * t + 2];
        if (b < 0 || b >= g->B || h < 0 || h >= g->Hq || i < 0 || i >= g->L) {
#pragma omp atomic write
          err = OG_ERR_ARG;
          continue;
        }
        const int r = og_fwd_row(q, k, v, doc, g, b, h, i, out + (size_t)t * g->D, lse + t, xbuf);
        if (r != OG_OK) {
#pragma omp atomic write
          err = r;
        }
      }
      free(xbuf);
    }
  }
  return err;
}

/* Forward of one K/V chunk (the keys of the K/V buffer only) for rows
 * sel[n][3]: the softmax over the allowed keys that lie in the chunk. A real
 * row with no allowed key in the chunk gets out = 0 and lse = -inf, the
 * identity of the log-sum-exp merge of chunk results (gemma4_moe.cp_local_ring
 * per-chunk forward and `-inf`-safe merge). */
int og_fwd_rows_chunk(const double* q, const double* k, const double* v, const int32_t* doc, const og_geom* g,
                      const int32_t* sel, int n, double* out, double* lse) {
  if (!og_geom_ok(g) || !q || !k || !v || !doc || !sel || !out || !lse) return OG_ERR_ARG;
  int err = OG_OK;
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(g->S_kv > 0 ? g->S_kv : 1));
    if (!xbuf) {
#pragma omp atomic write
      err = OG_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int t = 0; t < n; ++t) {
        const int b = sel[3 * t], h = sel[3 * t + 1], i = sel[3 * t + 2];
        if (b < 0 || b >= g->B || h < 0 || h >= g->Hq || i < 0 || i >= g->L) {
#pragma omp atomic write
          err = OG_ERR_ARG;
          continue;
        }
        double* o = out + (size_t)t * g->D;
        int r = og_fwd_row(q, k, v, doc, g, b, h, i, o, lse + t, xbuf);
        if (r == OG_ERR_EMPTY_ROW) {
          for (int d = 0; d < g->D; ++d) o[d] = 0.0;
          lse[t] = -INFINITY;
          r = OG_OK;
        }
        if (r != OG_OK) {
#pragma omp atomic write
          err = r;
        }
      }
      free(xbuf);
    }
  }
  return err;
}

/* ------------------------------------------------------------ backward --- */

/* Analytic backward of the loss sum(out * dout) for selected query rows
 * (dq) and selected keys (dk, dv summed over the query heads of the key's
 * GQA group):
 *   P_ps  = exp(scale q_p.k_s - lse_p)         (allowed pairs, real rows)
 *   Z_ps  = dropout factor (0 or the keep scale; 1 without dropout)
 *   delta = dout_p . out_p                      (out = sum_s P Z v)
 *   dS_ps = P_ps (Z_ps dout_p . v_s - delta_p)
 *   dq_p  = scale sum_s dS_ps k_s
 *   dk_s  = scale sum_p dS_ps q_p ,  dv_s = sum_p P_ps Z_ps dout_p
 * Padding query rows contribute nothing and get dq = 0 ([K.varlen]).
 *
 * rows[nr][3] = (b, h, i) -> dq[nr][D]
 * keys[nk][3] = (b, hk, j) -> dk[nk][D], dv[nk][D]
 * The forward of every row that a selected key receives from is recomputed
 * here (out, lse, delta), so the cost grows with the selected keys' fan-in. */
int og_bwd(const double* q, const double* k, const double* v, const double* dout, const int32_t* doc,
           const og_geom* g, const int32_t* rows, int nr, const int32_t* keys, int nk, double* dq, double* dk,
           double* dv) {
  if (!og_geom_ok(g) || !q || !k || !v || !dout || !doc) return OG_ERR_ARG;
  if ((nr > 0 && (!rows || !dq)) || (nk > 0 && (!keys || !dk || !dv))) return OG_ERR_ARG;
  const int B = g->B, Hq = g->Hq, L = g->L, D = g->D, G = g->Hq / g->Hkv;
  const size_t nrows = (size_t)B * Hq * L;
  uint8_t* need = (uint8_t*)calloc(nrows, 1);
  double* lse_all = (double*)malloc(sizeof(double) * nrows);
  double* delta_all = (double*)malloc(sizeof(double) * nrows);
  if (!need || !lse_all || !delta_all) {
    free(need);
    free(lse_all);
    free(delta_all);
    return OG_ERR_NOMEM;
  }
  int err = OG_OK;
  /* rows whose forward statistics are needed */
  for (int t = 0; t < nr; ++t) {
    const int b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= L) {
      err = OG_ERR_ARG;
      break;
    }
    need[((size_t)b * Hq + h) * L + i] = 1;
  }
  for (int t = 0; t < nk && err == OG_OK; ++t) {
    const int b = keys[3 * t], hk = keys[3 * t + 1], j = keys[3 * t + 2];
    if (b < 0 || b >= B || hk < 0 || hk >= g->Hkv || j < 0 || j >= g->S_kv) {
      err = OG_ERR_ARG;
      break;
    }
    const int32_t* row = doc + (size_t)b * g->S_full;
    for (int i = 0; i < L; ++i) {
      const int p = g->row_offset + i;
      if (row[p] == 0 || !og_allowed(row, p, g->kv_offset + j, g->window)) continue;
      for (int gg = 0; gg < G; ++gg) need[((size_t)b * Hq + hk * G + gg) * L + i] = 1;
    }
  }
  if (err != OG_OK) goto done;

  /* forward statistics of the needed rows */
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(g->S_kv > 0 ? g->S_kv : 1));
    double* orow = (double*)malloc(sizeof(double) * (size_t)D);
    if (!xbuf || !orow) {
#pragma omp atomic write
      err = OG_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (long long r = 0; r < (long long)nrows; ++r) {
        if (!need[r]) continue;
        const int i = (int)(r % L), h = (int)((r / L) % Hq), b = (int)(r / ((size_t)L * Hq));
        double lse;
        const int e = og_fwd_row(q, k, v, doc, g, b, h, i, orow, &lse, xbuf);
        if (e != OG_OK) {
#pragma omp atomic write
          err = e;
          continue;
        }
        lse_all[r] = lse;
        delta_all[r] = og_dot(dout + (size_t)r * D, orow, D);
      }
    }
    free(xbuf);
    free(orow);
  }
  if (err != OG_OK) goto done;

  /* dq for the selected rows */
#pragma omp parallel for schedule(dynamic, 4)
  for (int t = 0; t < nr; ++t) {
    const int b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
    const int hk = h / G, p = g->row_offset + i;
    const size_t r = ((size_t)b * Hq + h) * L + i;
    double* dqr = dq + (size_t)t * D;
    for (int d = 0; d < D; ++d) dqr[d] = 0.0;
    const int32_t* row = doc + (size_t)b * g->S_full;
    if (row[p] == 0) continue;
    const double* qr = q + r * D;
    const double* dor = dout + r * D;
    const double* kb = k + ((size_t)b * g->Hkv + hk) * (size_t)g->S_kv * D;
    const double* vb = v + ((size_t)b * g->Hkv + hk) * (size_t)g->S_kv * D;
    for (int j = 0; j < g->S_kv; ++j) {
      if (!og_allowed(row, p, g->kv_offset + j, g->window)) continue;
      const double* kr = kb + (size_t)j * D;
      const double P = exp(g->scale * og_dot(qr, kr, D) - lse_all[r]);
      const double Z = og_drop_factor(g, b, h, p, g->kv_offset + j);
      const double dS = P * (Z * og_dot(dor, vb + (size_t)j * D, D) - delta_all[r]);
      for (int d = 0; d < D; ++d) dqr[d] += g->scale * dS * kr[d];
    }
  }

  /* dk, dv for the selected keys */
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < nk; ++t) {
    const int b = keys[3 * t], hk = keys[3 * t + 1], j = keys[3 * t + 2];
    const int s = g->kv_offset + j;
    double* dkr = dk + (size_t)t * D;
    double* dvr = dv + (size_t)t * D;
    for (int d = 0; d < D; ++d) dkr[d] = dvr[d] = 0.0;
    const int32_t* row = doc + (size_t)b * g->S_full;
    const double* kr = k + (((size_t)b * g->Hkv + hk) * g->S_kv + j) * D;
    const double* vr = v + (((size_t)b * g->Hkv + hk) * g->S_kv + j) * D;
    for (int gg = 0; gg < G; ++gg) {
      const int h = hk * G + gg;
      for (int i = 0; i < L; ++i) {
        const int p = g->row_offset + i;
        if (row[p] == 0 || !og_allowed(row, p, s, g->window)) continue;
        const size_t r = ((size_t)b * Hq + h) * L + i;
        const double* qr = q + r * D;
        const double* dor = dout + r * D;
        const double P = exp(g->scale * og_dot(qr, kr, D) - lse_all[r]);
        const double Z = og_drop_factor(g, b, h, p, s);
        const double dS = P * (Z * og_dot(dor, vr, D) - delta_all[r]);
        for (int d = 0; d < D; ++d) {
          dvr[d] += P * Z * dor[d];
          dkr[d] += g->scale * dS * qr[d];
        }
      }
    }
  }

done:
  free(need);
  free(lse_all);
  free(delta_all);
  return err;
}

/* Test hook: the dropout factor Z of every (local row i, K/V buffer row j) for
 * batch row b and query head h, [L][S_kv], whether or not the pair is allowed
 * (1 everywhere without dropout). */
int og_dropout_factors(const og_geom* g, int b, int h, double* z) {
  if (!og_geom_ok(g) || !z || b < 0 || b >= g->B || h < 0 || h >= g->Hq) return OG_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 16)
  for (int i = 0; i < g->L; ++i)
    for (int j = 0; j < g->S_kv; ++j)
      z[(size_t)i * g->S_kv + j] = og_drop_factor(g, b, h, g->row_offset + i, g->kv_offset + j);
  return OG_OK;
}
