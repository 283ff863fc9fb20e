/*
 * bdattn -- per-document causal (block-diagonal) attention for one
 * context-parallel query shard, forward and backward, on GB300 (sm_103a).
 *
 * What is computed (NVIDIA NeMo AutoModel API pages):
 *  - blockdiag_cp.kernels, `_cp_blockdiag_mask`: a local query row at global
 *    position p may attend key position s iff both carry the same document id,
 *    neither is padding (id 0), and s <= p; the diagonal is always allowed.
 *  - gemma4_moe.cp_local_ring (module text): the sliding layer adds a left
 *    window on top of bottom-right causal; here a window W > 0 also requires
 *    p - s < W.
 *  - blockdiag_cp.kernels, `_cp_blockdiag_varlen`: the result equals mask +
 *    softmax attention on real query rows; padding is a contiguous tail so the
 *    real local rows are a prefix; padding query rows are returned as zeros.
 *    One varlen segment per document the local rows touch: q segment = the
 *    local rows of that document, k segment = [doc_start, last_local_q + 1).
 *  - blockdiag_cp.kernels, `precompute_blockdiag_varlen_meta`: the
 *    segmentation is built once per step, with no host synchronisation.
 *
 * Geometry of a virtual context-parallel rank r of cp_size ranks:
 *   local query rows are global positions [row_offset, row_offset + L)
 *   (row_offset = r * L); the K/V buffer holds global positions
 *   [kv_offset, kv_offset + S_kv) and must contain [s_first, real_end) of
 *   every batch row (the left-halo plan's needed range, blockdiag_cp.exchange).
 *
 * Layouts (all contiguous, row-major):
 *   doc_ids  int32 [B, S_full]        0 = padding, > 0 = document id
 *   q, dout  bf16  [B, Hq,  L,    D]
 *   k, v     bf16  [B, Hkv, S_kv, D]  query head h reads kv head h / (Hq/Hkv)
 *                                     ([S_kv, B, Hkv, D] with kv_layout = BD_KV_SBHD)
 *   out      bf16  [B, Hq,  L,    D]
 *   lse      fp32  [B, Hq,  L]        natural-log sum-exp; -inf on padding rows
 *   dq       fp32 or bf16 [B, Hq, L, D]
 *   dk, dv   fp32 or bf16 [B, Hkv, S_kv, D]   summed over each GQA group (k's layout)
 * D must be 64, 128, 256 or 512 (512: the head-dim-512 global layers of
 * gemma4_moe.cp_attention). All device pointers are caller-owned and must be
 * 16-byte aligned. The library allocates no device memory and never
 * synchronises the stream; every entry point only enqueues work on `stream`.
 *
 * Errors:
 *   - return value: BD_OK, or an argument / CUDA error found on the host
 *     before or at launch (nothing, or nothing further, is enqueued);
 *   - *status (one device int32, zero it before the first call of a step):
 *     kernels OR BD_STATUS_* bits into it. When a bit is set, later kernels
 *     skip their work (their outputs are left unwritten) instead of faulting.
 */
#ifndef BDATTN_H
#define BDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef void* bd_stream_t;

typedef struct {
  int B;          /* batch rows */
  int Hq;         /* query heads */
  int Hkv;        /* key/value heads; Hq % Hkv == 0 */
  int D;          /* head dim: 64, 128, 256 or 512 */
  int S_full;     /* length of each doc_ids row (full padded sequence) */
  int L;          /* local query rows */
  int row_offset; /* global position of local row 0 */
  int kv_offset;  /* global position of K/V buffer row 0 */
  int S_kv;       /* K/V buffer rows */
  int window;     /* left window W (> 0: also require p - s < W); <= 0: none */
  float scale;    /* softmax scale; <= 0 means D^-0.5 */
  int kv_layout;  /* layout of k, v, dk, dv: BD_KV_BHSD (0) or BD_KV_SBHD (1) */
  float dropout_p;  /* chance of dropping an attention weight, 0 <= p < 1 (0: none); see below */
  uint32_t seed_lo; /* dropout seed: low and high 32 bits (the Philox key) */
  uint32_t seed_hi;
} bd_geom;

/* Attention dropout (blockdiag_cp.kernels, `_cp_blockdiag_varlen` argument
 * `dropout_p`, the chance that an attention weight is dropped). Inverted dropout on the
 * softmax probabilities: out_p = sum_s P_ps Z_ps v_s with Z_ps = 0 (dropped)
 * or 2^16 / (2^16 - T) (kept); the LSE is that of the undropped softmax, and
 * the backward takes the same Z (dV = sum_p P Z dO, dS = P (Z dP - delta)).
 * The decision of the pair (query head h, global query position p, global key
 * position s) of batch row b: Philox-4x32-10 (Salmon et al., SC'11) with
 * counter (s / 8, p, h, b) and key (seed_lo, seed_hi) gives eight 16-bit draws,
 * key s taking draw s mod 8 (word (s mod 8) / 2; low half for even s); the pair
 * is kept iff its draw u >= T = round(dropout_p * 2^16). Decisions depend on
 * global positions only, so K/V chunks, shards and buffer offsets agree.
 * Every forward and backward entry point takes dropout, at every head dim;
 * they return BD_ERR_ARG for dropout_p outside [0, 1) or rounding to
 * T = 2^16. A forward and the backward of the same step must use the same
 * dropout_p and seed. */

/* K/V layouts. BD_KV_SBHD is token-major, [S_kv][B][Hkv][D]: the receive
 * buffer of the needed-only all-to-all-v (pieces in source order make the
 * needed range), read in place; dk / dv are then written token-major too,
 * ready to be sent back and index-added by bd_attn_needed_scatter_add. */
#define BD_KV_BHSD 0
#define BD_KV_SBHD 1

/* Host return codes. */
#define BD_OK 0
#define BD_ERR_ARG 1         /* invalid argument; nothing enqueued */
#define BD_ERR_CUDA 2        /* a CUDA runtime/driver call failed */
#define BD_ERR_UNSUPPORTED 3 /* device is not a Blackwell sm_10x part */

/* Device status bits (OR-ed into *status). */
#define BD_STATUS_LAYOUT 0x1   /* a doc id < 0, a document after padding, or a
                                  local document id that also occurs before its
                                  own run (ids must form one contiguous run) */
#define BD_STATUS_KV_RANGE 0x2 /* K/V buffer misses part of [need_lo, real_end) */
#define BD_STATUS_BOUNDS 0x4   /* segment table inconsistent with the geometry */
#define BD_STATUS_TIMEOUT 0x8  /* a pipeline wait exceeded its time limit */

/* Gradient output dtypes for bd_attn_bwd. */
#define BD_DTYPE_F32 0
#define BD_DTYPE_BF16 1

/* Segment-table field indices within each batch row's header (int32). */
#define BD_SEG_N_REAL 0
#define BD_SEG_N_SEG 1
#define BD_SEG_S_FIRST 2
#define BD_SEG_REAL_END 3
#define BD_SEG_MAX_Q 4
#define BD_SEG_MAX_K 5
#define BD_SEG_FIRST_Q 6
#define BD_SEG_FIRST_K 7
#define BD_SEG_MAX_TAIL 8
#define BD_SEG_KV_NEED_LO 9
#define BD_SEG_ROW_STATUS 10
#define BD_SEG_HDR_WORDS 32

/* Word offsets of the regions of the segment table (see bd_attn_seg_layout). */
#define BD_SEG_OFF_HDR 0        /* [B][32]       per-row header */
#define BD_SEG_OFF_CU_Q 1       /* [B][L+1]      cu_q: segment starts (local rows), n_real last */
#define BD_SEG_OFF_CU_K 2       /* [B][L+1]      cu_k: k segment starts - s_first, real_end - s_first last */
#define BD_SEG_OFF_ROW_LO 3     /* [B][L]        doc start (global) of each local row, -1 on padding */
#define BD_SEG_OFF_QT_KRANGE 4  /* [B][nqt][2]   per 128-row q tile: first, last 128-row K/V tile (last < first: none) */
#define BD_SEG_OFF_KT_QRANGE 5  /* [B][nkt][2]   per 128-row K/V tile: first, end (exclusive) local q row attending it */
#define BD_SEG_OFF_FULL_BITS 6  /* [B][nqt][nkw] bit kt set: tile (qt, kt) is entirely allowed */
#define BD_SEG_OFF_FWD_WORK 7   /* [B*nqt]       q tiles (b*nqt+qt), most K/V tiles first */
#define BD_SEG_OFF_BWD_WORK 8   /* [B*nkt]       K/V tiles (b*nkt+kt), most q rows first */
#define BD_SEG_OFF_COUNTS 9     /* [8]           0: full tiles, 1: partial tiles, 2: empty tiles,
                                                 3: K/V tiles some local row attends (the first
                                                    entries of the backward work list) */
#define BD_SEG_OFF_TOTAL 10     /* total words */
#define BD_SEG_NOFF 11

/* Size in bytes of the segment table for this geometry (0 if invalid). */
size_t bd_attn_seg_bytes(const bd_geom* g);

/* Word offsets of the table regions, BD_SEG_NOFF entries; also writes
 * offsets[BD_SEG_NOFF..BD_SEG_NOFF+2] = nqt, nkt, nkw. Returns BD_OK or
 * BD_ERR_ARG. Host only; reads no device memory. */
int bd_attn_seg_layout(const bd_geom* g, int32_t* offsets /* >= BD_SEG_NOFF + 3 */);

/* Step 1 (per step, shared by every layer): build the varlen segmentation
 * of the local shard and the 128x128 tile classification.
 * Reads doc_ids [B, S_full] (device). Writes the segment table `seg`
 * (device, bd_attn_seg_bytes(g) bytes, caller-owned) and ORs LAYOUT /
 * KV_RANGE bits into *status (device). Reference: blockdiag_cp.kernels,
 * `_varlen_seg_for_rank` / `precompute_blockdiag_varlen_meta`; the needed
 * K/V range from blockdiag_cp.exchange. Segment fields per batch row:
 * n_real, n_seg, s_first, real_end, cu_q, cu_k, max_q, max_k (bit-exact
 * with the definition), first_q = cu_q[1], first_k = cu_k[1], max_tail =
 * largest q segment after the first; an all-padding shard has n_real =
 * n_seg = 0 and s_first = real_end = row_offset. */
int bd_attn_seg_build(const int32_t* doc_ids, const bd_geom* g, void* seg, int32_t* status, bd_stream_t stream);

/* The same table for one chunk of the K/V range (gemma4_moe.cp_local_ring:
 * the per-step forward over the K/V chunk a ring step holds). The K/V buffer
 * [kv_offset, kv_offset + S_kv) need not contain every key the local rows may
 * attend, so KV_RANGE is never set; bd_attn_fwd then gives each row the
 * softmax over its allowed keys inside the chunk, with out = 0 and lse = -inf
 * for a row that has none, and bd_attn_bwd_main (with the merged out / lse
 * of all chunks, through bd_attn_bwd_prep) adds the chunk's share of dq and
 * writes the chunk's dk / dv. Merge chunk forwards with bd_attn_merge. */
int bd_attn_seg_build_chunk(const int32_t* doc_ids, const bd_geom* g, void* seg, int32_t* status,
                            bd_stream_t stream);

/* The forward over one K/V chunk merged into a running result in its
 * epilogue (gemma4_moe.cp_local_ring: per-chunk forward and -inf-safe
 * merge, fused): out / lse hold the running result on entry -- from
 * bd_attn_fwd over the first chunk or from earlier calls of this one -- and
 * the merge of it with this chunk's forward on return, by the same rule as
 * bd_attn_merge, in fp32 before the one rounding of out to bf16. A row the
 * chunk gives nothing keeps its running result; a row empty on both sides
 * gets out = 0, lse = -inf; an empty running side's out is not read.
 * Arguments, table and errors as bd_attn_fwd. */
int bd_attn_fwd_merge(const void* q, const void* k, const void* v, const void* seg, const bd_geom* g, void* out,
                      float* lse, int32_t* status, bd_stream_t stream);

/* Log-sum-exp merge of a chunk's forward result into a running one, in place
 * (gemma4_moe.cp_local_ring: -inf-safe online softmax merge):
 *   lse = log(exp(lse) + exp(lse_chunk)),
 *   out = exp(lse_old - lse) out + exp(lse_chunk - lse) out_chunk,
 * in fp32 per element. A side with lse = -inf has weight 0 whatever its out
 * holds, so a running result may start as lse = -inf with any out; a row
 * empty on both sides stays out = 0, lse = -inf.
 * out, out_chunk: bf16 [B,Hq,L,D], 16-byte aligned; lse, lse_chunk: fp32
 * [B,Hq,L]. Device pointers, caller-owned; BD_ERR_ARG for null or misaligned
 * pointers. Does nothing if *status is already nonzero. */
int bd_attn_merge(void* out, float* lse, const void* out_chunk, const float* lse_chunk, const bd_geom* g,
                  int32_t* status, bd_stream_t stream);

/* Step 2: forward. out = softmax(scale * q k^T + mask) v per query row,
 * lse = natural-log sum of exp(scale * q.k) over the allowed keys.
 * Padding rows: out = 0, lse = -inf. Needs the table from
 * bd_attn_seg_build with the same geometry. Reference:
 * blockdiag_cp.kernels, `_cp_blockdiag_varlen`; LSE convention from
 * gemma4_moe.cp_attention, `_scatter_lse`. */
int bd_attn_fwd(const void* q, const void* k, const void* v, const void* seg, const bd_geom* g, void* out,
                float* lse, int32_t* status, bd_stream_t stream);

/* Scratch bytes bd_attn_bwd needs in `workspace` (device, caller-owned):
 * an fp32 dq accumulator [B,Hq,L,D] and delta = rowsum(dout*out) [B,Hq,L]. */
size_t bd_attn_bwd_workspace_bytes(const bd_geom* g);

/* Step 3: backward of sum(out * dout) from the saved out and lse (no forward
 * recompute). dq [B,Hq,L,D]; dk, dv [B,Hkv,S_kv,D] summed over the Hq/Hkv
 * query heads of each group (the all-gather's reduce-scatter(SUM) over
 * ranks is left to the caller). Padding rows give dq = 0 and contribute
 * nothing; K/V rows no query attends get 0. grad_dtype: BD_DTYPE_F32 or
 * BD_DTYPE_BF16 (for all three gradients). Reference: gemma4_moe.
 * cp_local_ring, `sliding_ring_compute_fa_bwd`; blockdiag_cp.exchange,
 * `_AllGatherSeqDiff` (sum semantics). */
int bd_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* seg, const bd_geom* g, int grad_dtype, void* dq, void* dk, void* dv, void* workspace,
                int32_t* status, bd_stream_t stream);

/* The same backward with bitwise reproducible results (the pages'
 * `_CP_FLASH_DETERMINISTIC`): dk / dv as bd_attn_bwd (they accumulate inside
 * one CTA), and dq from a separate pass in which one CTA per 128-row q tile and
 * query head walks its K/V tiles in increasing order, recomputing S and dP and
 * accumulating dQ in tensor memory -- no atomic additions anywhere. Same
 * arguments and results as bd_attn_bwd (workspace: the same size, holding
 * delta); any head dim (at D = 256 the dq pass streams each K/V tile's K
 * twice, for S and for dQ; at D = 512 two CTAs per q tile and query head each
 * form S and dP for one 256-column half of dq). Three launches: delta,
 * dK / dV (with the zero rows of unattended K/V tiles), dq. */
int bd_attn_bwd_deterministic(const void* dout, const void* q, const void* k, const void* v, const void* out,
                              const float* lse, const void* seg, const bd_geom* g, int grad_dtype, void* dq,
                              void* dk, void* dv, void* workspace, int32_t* status, bd_stream_t stream);

/* The three stages bd_attn_bwd runs, one kernel each, for callers that want
 * to schedule or time them separately (same arguments, same rules):
 *  _prep:     delta[B,Hq,L] = rowsum(dout * out) in fp32 and a zeroed fp32 dq
 *             accumulator, both in `workspace`;
 *  _main:     dk, dv (written in full) and the dq accumulation (of the final,
 *             scaled gradient) in `workspace`;
 *  _finalize: dq = accumulator, converted to grad_dtype.
 * They must run in this order on one stream with the same workspace. With the
 * K/V range split into chunks (bd_attn_seg_build_chunk), run _prep once with
 * the merged out, then _main once per chunk (that chunk's geometry, table,
 * k, v, dk, dv and the merged lse; B, Hq, Hkv, D, S_full, L, row_offset and
 * window as in _prep), then _finalize: dq is the sum over the chunks. */
int bd_attn_bwd_prep(const void* dout, const void* out, const bd_geom* g, void* workspace, int32_t* status,
                     bd_stream_t stream);
int bd_attn_bwd_main(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                     const void* seg, const bd_geom* g, int grad_dtype, void* dk, void* dv, void* workspace,
                     int32_t* status, bd_stream_t stream);
int bd_attn_bwd_finalize(const bd_geom* g, int grad_dtype, void* dq, void* workspace, int32_t* status,
                         bd_stream_t stream);

/* The same backward with the fp32 dq output as its own accumulator, in two
 * stages and without a finalize pass (bd_attn_bwd takes this path when
 * grad_dtype is BD_DTYPE_F32):
 *  _prep_dq: delta in `workspace` (whose accumulator part is not used) and
 *            dq [B,Hq,L,D] fp32 set to zero;
 *  _main_dq: dk, dv in grad_dtype as bd_attn_bwd_main, and dq += scale * dS K
 *            for every attended tile, so dq holds the final gradient when the
 *            kernel ends.
 * dq must be 16-byte aligned fp32 device memory (BD_ERR_ARG otherwise, or for
 * a null dq); run _prep_dq then _main_dq on one stream with the same dq and
 * workspace. */
int bd_attn_bwd_prep_dq(const void* dout, const void* out, const bd_geom* g, void* workspace, float* dq,
                        int32_t* status, bd_stream_t stream);
int bd_attn_bwd_main_dq(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                        const void* seg, const bd_geom* g, int grad_dtype, float* dq, void* dk, void* dv,
                        void* workspace, int32_t* status, bd_stream_t stream);

/* Allocation-free backward. Same arguments and results as bd_attn_bwd
 * except that there is no `workspace`: the dq accumulator and delta live in
 * one static scratch array of BD_NOALLOC_SCRATCH_BYTES per GPU, part of the
 * library's device code and held until the process exits. It is for callers
 * that can hand the library their inputs and outputs but cannot allocate
 * device memory at call time -- for example a host that reserved its whole
 * memory budget up front, or a plugin whose framework forbids allocations
 * outside its own allocator -- so it calls no cudaMalloc, cudaFree or
 * allocating routine. The paper pages have no counterpart; this is a
 * deployment convenience.
 *  - Returns BD_ERR_SCRATCH_TOO_SMALL (nothing enqueued) when
 *    bd_attn_bwd_workspace_bytes(g) exceeds BD_NOALLOC_SCRATCH_BYTES.
 *  - Set-up: the first call on each device (with that device current) looks
 *    up the array's device address (cudaGetSymbolAddress). Under CUDA's lazy
 *    module loading (the default) that is also when the driver loads the
 *    library's code holding the array and so takes its device memory; with
 *    CUDA_MODULE_LOADING=EAGER it is taken when the context is created. A
 *    caller that reserves its memory budget up front should therefore do the
 *    set-up first: a call with every pointer argument NULL (g included) does
 *    only the set-up of the current device, enqueues nothing and returns
 *    BD_OK. Make the set-up before any stream capture. If the array cannot be
 *    placed, the call returns BD_ERR_NOALLOC_SETUP.
 *  - Every call on a device shares the one array, and each call starts by
 *    zeroing the part it accumulates into. Calls whose kernels overlap on the
 *    GPU (other streams, other host threads) race on it: serialise them. */
#define BD_NOALLOC_SCRATCH_BYTES (16u << 20)
#define BD_ERR_SCRATCH_TOO_SMALL 4
#define BD_ERR_NOALLOC_SETUP 5
int bd_attn_bwd_noalloc(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* seg, const bd_geom* g, int grad_dtype, void* dq, void* dk,
                        void* dv, int32_t* status, bd_stream_t stream);

/* ---- K/V exchange plans (blockdiag_cp.exchange) --------------------------
 *
 * The global left-halo plan and the needed-only all-to-all-v split plan,
 * computed on the device from the replicated doc ids with no host
 * synchronisation, and the sender's local halves of the needed-only exchange
 * (`_NeededKVExchange`): the gather of the send buffer and the index-add of
 * the returned gradients. The collective that moves the buffers between GPUs
 * is not part of this library.
 *
 * The sequence of S_full positions splits into cp_size equal chunks of
 * L = S_full / cp_size; rank r owns [r*L, (r+1)*L). Rank r needs the K/V
 * range [s_first_r, real_end_r): real_end_r = r*L + its real local rows,
 * s_first_r = the first position of the run of equal ids holding r*L (the
 * straddle of its first document). With B > 1 the range covers every batch
 * row's range (rows whose local rows are all padding do not count); a rank
 * with no real row at all needs nothing: s_first = real_end = r*L.
 *   back_r = r*L - s_first_r;  use_halo = (back_r <= L for every rank);
 *   halo_size = max_r back_r   (the uniform-size neighbour exchange; rank r
 *                               keeps the last back_r tokens it receives);
 *   counts[src][dst] = |[src*L, (src+1)*L) intersect [s_first_dst, real_end_dst)|;
 *   for this plan's rank:  in_splits[dst] = counts[rank][dst] (send counts),
 *   out_splits[src] = counts[src][rank] (receive counts), send_off / recv_off
 *   their exclusive prefix sums, and send_index = the local positions
 *   (0..L-1) of the send buffer's tokens, destination by destination, each
 *   destination's piece in increasing position. The receiver's pieces, in
 *   source order, make its needed range.
 *
 * The plan is an int32 array (device, caller-owned, 16-byte aligned) of
 * bd_attn_plan_bytes(B, cp_size, L) bytes, regions at the word offsets that
 * bd_attn_plan_layout returns (BD_PLAN_OFF_* order). */
#define BD_PLAN_HDR_WORDS 16
#define BD_PLAN_MAGIC 0        /* header word: 0x62647870 once built */
#define BD_PLAN_CP_SIZE 1
#define BD_PLAN_L 2
#define BD_PLAN_RANK 3
#define BD_PLAN_B 4
#define BD_PLAN_USE_HALO 5
#define BD_PLAN_HALO_SIZE 6
#define BD_PLAN_TOTAL_SEND 7   /* sum of in_splits = send buffer tokens */
#define BD_PLAN_TOTAL_RECV 8   /* sum of out_splits = real_end_rank - s_first_rank */

#define BD_PLAN_OFF_HDR 0         /* [16]          header */
#define BD_PLAN_OFF_S_FIRST 1     /* [cp_size]     s_first of every rank */
#define BD_PLAN_OFF_REAL_END 2    /* [cp_size]     real_end of every rank */
#define BD_PLAN_OFF_BACK 3        /* [cp_size]     back_r (= halo tokens rank r receives from r - 1) */
#define BD_PLAN_OFF_HALO_SEND 4   /* [cp_size]     halo tokens rank r sends to r + 1 (= back_{r+1}; 0 for the last) */
#define BD_PLAN_OFF_COUNTS 5      /* [cp_size][cp_size]  counts[src][dst] */
#define BD_PLAN_OFF_IN_SPLITS 6   /* [cp_size]     this rank's per-destination send counts */
#define BD_PLAN_OFF_OUT_SPLITS 7  /* [cp_size]     this rank's per-source receive counts */
#define BD_PLAN_OFF_SEND_OFF 8    /* [cp_size]     exclusive prefix sums of in_splits */
#define BD_PLAN_OFF_RECV_OFF 9    /* [cp_size]     exclusive prefix sums of out_splits */
#define BD_PLAN_OFF_SEND_INDEX 10 /* [cp_size * L] send_index (first TOTAL_SEND entries) */
#define BD_PLAN_OFF_ROW_RANGE 11  /* [B][cp_size][2]  scratch of the build */
#define BD_PLAN_OFF_TOTAL 12      /* total words */
#define BD_PLAN_NOFF 13

/* Bytes of a plan (0 for an invalid size: B, cp_size or L < 1, cp_size >
 * 1024, or cp_size * L beyond 2^31 - 1). */
size_t bd_attn_plan_bytes(int B, int cp_size, int L);
/* Word offsets of the plan's regions into offsets[BD_PLAN_NOFF]. */
int bd_attn_plan_layout(int B, int cp_size, int L, int32_t* offsets);

/* Build the plan of rank `rank` from doc_ids int32 [B, S_full] (device).
 * S_full must be a multiple of cp_size. Two kernels: per (rank, batch row)
 * the real rows and the run start, then the plan. Sets BD_STATUS_LAYOUT (and
 * still writes the plan) for a negative id or a real id after padding
 * inside a chunk. BD_ERR_ARG for a null or misaligned pointer, an invalid
 * size or rank. */
int bd_attn_exchange_plan(const int32_t* doc_ids, int B, int S_full, int cp_size, int rank, void* plan,
                          int32_t* status, bd_stream_t stream);

/* Forward of the needed-only exchange on the sender: the send buffer
 * send[j][b][c][:] = x_local[b][c][send_index[j]][:] for j < TOTAL_SEND, in
 * the token-major layout [max_rows][B][C][D] so that each destination's piece
 * is one contiguous block (starting at token send_off[dst]). x_local is
 * [B][C][L][D]; dtype BD_DTYPE_BF16 or BD_DTYPE_F32; D * element size a
 * multiple of 16 bytes. The token count is read from the plan on the device:
 * when it exceeds max_rows, BD_STATUS_BOUNDS is set and nothing is written
 * (max_rows = cp_size * L always suffices). Does nothing if *status is
 * already nonzero. B and L must match the plan's (else BD_STATUS_BOUNDS). */
int bd_attn_needed_gather(const void* x_local, const void* plan, int B, int C, int L, int D, int dtype, void* send,
                          int max_rows, int32_t* status, bd_stream_t stream);

/* Backward of the needed-only exchange on the sender (the index-add): the
 * gradients of the send buffer, grad_send [max_rows][B][C][D] (first
 * TOTAL_SEND tokens used), summed onto their source tokens:
 * grad_local[b][c][t][:] = sum over destinations whose piece holds t, in
 * destination order, of that token's gradient, accumulated in fp32; 0 for a
 * token no destination needs. grad_local [B][C][L][D] is written in full.
 * Deterministic. Same dtype, size and status rules as bd_attn_needed_gather. */
int bd_attn_needed_scatter_add(const void* grad_send, const void* plan, int B, int C, int L, int D, int dtype,
                               void* grad_local, int max_rows, int32_t* status, bd_stream_t stream);

/* Human-readable text for a host return code. */
const char* bd_attn_strerror(int code);

/* Test hook for the bounded waits: launches one CTA that waits on an
 * mbarrier nobody arrives on, with the given limit in nanoseconds, and ORs
 * BD_STATUS_TIMEOUT into *status when the wait gives up. */
int bd_attn_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, bd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BDATTN_H */
