"""Oracle of the K/V exchange plans of block-diagonal context parallelism.

TEST INFRASTRUCTURE ONLY (as the rest of this package): the tests and the
CPU legs of ``bench.py`` use it; the product path never imports it.

What it computes follows the NeMo AutoModel page ``blockdiag_cp.exchange``:
  * the global left-halo exchange plan: for every rank r the contiguous K/V
    range ``[s_first_r, real_end_r)`` it needs (the straddle of its first
    document, owned by lower ranks, plus its own real rows), the straddle
    length ``back_r = r*L - s_first_r``, and ``use_halo`` when every
    straddle fits in the left neighbour (``back_r <= L`` for all ranks);
    the halo exchange is uniform-size, so it moves ``max_r back_r`` tokens
    and each receiver keeps the last ``back_r`` of them;
  * the per-(src, dst) split sizes and the local gather index of the general
    needed-only all-to-all-v: source s sends destination r the part of its
    chunk ``[s*L, (s+1)*L)`` inside r's needed range, once per destination;
    the receiver's pieces, in source order, make its needed range;
  * ``_NeededKVExchange``: forward gathers the send buffer from the local
    chunk with the gather index; backward index-adds the per-destination
    gradients back onto the source tokens.

Readings where the page is silent: a rank whose rows are all padding needs
nothing (``s_first = real_end = r*L``, ``back = 0``); with several batch rows
the exchange moves the same positions of every row, so a rank's range is the
smallest range covering every row's range (rows without real local rows do
not count); padding is one tail per row and a document one run of equal
non-zero ids -- a negative id, or a real id after padding, is a layout error.

Plain loops over positions; nothing here is shared with the attention oracle
or the CUDA library.
"""
from __future__ import annotations

import numpy as np


def row_range(doc_row, r: int, L: int) -> tuple[int, int, bool]:
    """(s_first, real_end, layout_error) of rank r's chunk in one batch row.

    real_end = r*L + the number of real (non-zero id) local rows; s_first =
    the first position of the run of equal ids holding position r*L (scan left
    while the id repeats). No real local row: (r*L, r*L)."""
    lo = r * L
    n_real, bad, seen_pad = 0, False, False
    for i in range(L):
        d = int(doc_row[lo + i])
        if d < 0:
            bad = True
        if d == 0:
            seen_pad = True
        else:
            if seen_pad:
                bad = True
            n_real += 1
    if n_real == 0:
        return lo, lo, bad
    s = lo
    while s > 0 and int(doc_row[s - 1]) == int(doc_row[lo]):
        s -= 1
    return s, lo + n_real, bad


def plan(doc_ids, cp_size: int) -> dict:
    """The global plan every rank derives from the replicated doc ids [B, S]."""
    doc = np.asarray(doc_ids).reshape(-1, np.asarray(doc_ids).shape[-1])
    B, S = doc.shape
    if cp_size <= 0 or S % cp_size:
        raise ValueError("the sequence must split into cp_size equal chunks")
    L = S // cp_size
    s_first, real_end, layout_error = [], [], False
    for r in range(cp_size):
        lo_r, hi_r, any_real = None, None, False
        for b in range(B):
            s, e, bad = row_range(doc[b], r, L)
            layout_error = layout_error or bad
            if e > r * L:  # this row has real local rows
                any_real = True
                lo_r = s if lo_r is None else min(lo_r, s)
                hi_r = e if hi_r is None else max(hi_r, e)
        if not any_real:
            lo_r = hi_r = r * L
        s_first.append(lo_r)
        real_end.append(hi_r)
    back = [r * L - s_first[r] for r in range(cp_size)]
    counts = [[0] * cp_size for _ in range(cp_size)]  # counts[src][dst]
    for src in range(cp_size):
        for dst in range(cp_size):
            a = max(src * L, s_first[dst])
            e = min((src + 1) * L, real_end[dst])
            counts[src][dst] = max(0, e - a)
    return dict(cp_size=cp_size, L=L, B=B, S=S, s_first=s_first, real_end=real_end, back=back,
                use_halo=all(x <= L for x in back), halo_size=max(back),
                halo_recv=list(back), halo_send=[back[r + 1] if r + 1 < cp_size else 0 for r in range(cp_size)],
                counts=counts, layout_error=layout_error)


def a2a_split(p: dict, rank: int) -> tuple[list, list, list]:
    """(in_splits, out_splits, send_index) of one rank: per-destination send
    counts, per-source receive counts, and the local positions (0..L-1) of the
    send buffer's tokens, destination by destination."""
    W, L = p["cp_size"], p["L"]
    in_splits = [p["counts"][rank][dst] for dst in range(W)]
    out_splits = [p["counts"][src][rank] for src in range(W)]
    send_index = []
    for dst in range(W):
        a = max(rank * L, p["s_first"][dst])
        e = min((rank + 1) * L, p["real_end"][dst])
        for pos in range(a, e):
            send_index.append(pos - rank * L)
    return in_splits, out_splits, send_index


def gather(x_local, send_index):
    """Forward of the needed-only exchange on the sender: x_local [B, C, L, D]
    -> send buffer [B, C, len(send_index), D], token j = x_local[:, :, send_index[j]]."""
    x = np.asarray(x_local)
    out = np.zeros(x.shape[:2] + (len(send_index),) + x.shape[3:], dtype=x.dtype)
    for j, t in enumerate(send_index):
        out[:, :, j] = x[:, :, t]
    return out


def scatter_add(grad_send, send_index, L: int):
    """Backward on the sender: grad_send [B, C, len(send_index), D] index-added
    into zeros [B, C, L, D] at send_index (fp64)."""
    g = np.asarray(grad_send, dtype=np.float64)
    out = np.zeros(g.shape[:2] + (L,) + g.shape[3:], dtype=np.float64)
    for j, t in enumerate(send_index):
        out[:, :, t] += g[:, :, j]
    return out
