"""fp64 CPU oracle for per-document causal attention of one context-parallel shard.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only users. The product path (the CUDA
library and its Python binding) never imports this package, and this package
imports nothing from the product.

What it computes follows the NeMo AutoModel API pages:
  * ``blockdiag_cp.kernels._cp_blockdiag_mask`` -- the dense allow-mask
    (same document, neither padding, key causally visible, diagonal allowed);
  * ``blockdiag_cp.kernels._cp_blockdiag_varlen`` -- mask + SDPA on real query
    rows, padding query rows returned as zeros;
  * ``blockdiag_cp.kernels._varlen_seg_for_rank`` /
    ``precompute_blockdiag_varlen_meta`` -- the per-rank varlen segmentation;
  * ``gemma4_moe.cp_local_ring`` (module text) -- bottom-right causal plus a
    left window for the sliding layer, read as ``p - s < window``; the
    per-chunk forward over a part of the keys and the ``-inf``-safe online
    softmax merge of chunk results (``fwd_chunk``, ``merge``);
  * ``blockdiag_cp.kernels._cp_blockdiag_varlen(..., dropout_p)`` -- attention
    dropout, read as inverted dropout on the attention probabilities with the
    keep decisions drawn by Philox-4x32-10 (Salmon et al., SC'11) from a
    counter of (key position / 8, query position, query head, batch row).

Every attention function here is a plain loop in ``bdattn_oracle.c`` (fp64,
OpenMP over independent rows); ``merge`` is its formula written out in numpy.
The rest of this module only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bdattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SEG_HDR = 16
SEG_FIELDS = ("n_real", "n_seg", "s_first", "real_end", "max_q", "max_k", "first_q", "first_k",
              "max_tail", "kv_need_lo", "layout_error", "kv_range_error")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP). Returns the library path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("S_full", ctypes.c_int), ("L", ctypes.c_int), ("row_offset", ctypes.c_int),
                ("kv_offset", ctypes.c_int), ("S_kv", ctypes.c_int), ("window", ctypes.c_int),
                ("scale", ctypes.c_double), ("dropout_p", ctypes.c_double), ("seed_lo", ctypes.c_uint32),
                ("seed_hi", ctypes.c_uint32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            G = ctypes.POINTER(Geom)
            lib.og_mask.argtypes = [P, G, P]
            lib.og_mask.restype = ctypes.c_int
            lib.og_pairs.argtypes = [P, G]
            lib.og_pairs.restype = ctypes.c_int64
            lib.og_seg_stride.argtypes = [ctypes.c_int]
            lib.og_seg_stride.restype = ctypes.c_int
            lib.og_segments.argtypes = [P, G, P]
            lib.og_segments.restype = ctypes.c_int
            lib.og_fwd_rows.argtypes = [P, P, P, P, G, P, ctypes.c_int, P, P]
            lib.og_fwd_rows.restype = ctypes.c_int
            lib.og_fwd_rows_chunk.argtypes = [P, P, P, P, G, P, ctypes.c_int, P, P]
            lib.og_fwd_rows_chunk.restype = ctypes.c_int
            lib.og_bwd.argtypes = [P, P, P, P, P, G, P, ctypes.c_int, P, ctypes.c_int, P, P, P]
            lib.og_bwd.restype = ctypes.c_int
            lib.og_philox.argtypes = [P, P, ctypes.c_int, P]
            lib.og_philox.restype = ctypes.c_int
            lib.og_dropout_factors.argtypes = [G, ctypes.c_int, ctypes.c_int, P]
            lib.og_dropout_factors.restype = ctypes.c_int
            _lib = lib
    return _lib


def geom(B, Hq, Hkv, D, S_full, L, row_offset, kv_offset, S_kv, window=0, scale=None, dropout_p=0.0,
         seed=0) -> Geom:
    """Geometry of one shard; dropout_p > 0 turns on attention dropout drawn
    from the 64-bit `seed` (Philox key = low, high 32 bits)."""
    if scale is None or scale <= 0:
        scale = float(D) ** -0.5
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return Geom(int(B), int(Hq), int(Hkv), int(D), int(S_full), int(L), int(row_offset), int(kv_offset),
                int(S_kv), int(window), float(scale), float(dropout_p), seed & 0xFFFFFFFF, seed >> 32)


def philox(ctr, key) -> np.ndarray:
    """Philox-4x32-10 (Salmon et al., SC'11): ctr [n, 4], key [n, 2] uint32 ->
    [n, 4] uint32, one independent evaluation per row."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(-1, 4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(-1, 2))
    assert c.shape[0] == k.shape[0]
    out = np.zeros_like(c)
    _check(_load().og_philox(_ptr(c), _ptr(k), c.shape[0], _ptr(out)), "philox")
    return out


def dropout_factors(g: Geom, b: int, h: int) -> np.ndarray:
    """[L, S_kv] dropout factor of every (local row, K/V buffer row) pair of batch
    row b, query head h: 0 (dropped) or the keep scale; all 1 without dropout."""
    z = np.zeros((g.L, g.S_kv), dtype=np.float64)
    _check(_load().og_dropout_factors(ctypes.byref(g), int(b), int(h), _ptr(z)), "dropout_factors")
    return z


def _f64(x) -> np.ndarray:
    """Widen to a C-contiguous float64 numpy array (bf16 -> f64 is exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def mask(doc_ids, g: Geom) -> np.ndarray:
    """Dense [B, L, S_kv] allow-mask (bool) exactly as the mask page defines it."""
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    out = np.zeros((g.B, g.L, g.S_kv), dtype=np.uint8)
    _check(_load().og_mask(_ptr(doc), ctypes.byref(g), _ptr(out)), "mask")
    return out.astype(bool)


def pairs(doc_ids, g: Geom) -> int:
    """Allowed (query, key) pairs over real query rows (no padding self-edges)."""
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    n = _load().og_pairs(_ptr(doc), ctypes.byref(g))
    if n < 0:
        raise RuntimeError("oracle pairs: bad geometry")
    return int(n)


def segments(doc_ids, g: Geom) -> list[dict]:
    """Per batch row: the varlen segmentation (bit-exact fields + cu_q/cu_k)."""
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    lib = _load()
    stride = lib.og_seg_stride(g.L)
    out = np.zeros((g.B, stride), dtype=np.int32)
    _check(lib.og_segments(_ptr(doc), ctypes.byref(g), _ptr(out)), "segments")
    res = []
    for b in range(g.B):
        o = out[b]
        d = {name: int(o[i]) for i, name in enumerate(SEG_FIELDS)}
        n = d["n_seg"]
        d["cu_q"] = o[SEG_HDR:SEG_HDR + n + 1].copy()
        d["cu_k"] = o[SEG_HDR + g.L + 1:SEG_HDR + g.L + 1 + n + 1].copy()
        res.append(d)
    return res


def _all_rows(g: Geom) -> np.ndarray:
    b, h, i = np.meshgrid(np.arange(g.B), np.arange(g.Hq), np.arange(g.L), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int32)


def _all_keys(g: Geom) -> np.ndarray:
    b, h, j = np.meshgrid(np.arange(g.B), np.arange(g.Hkv), np.arange(g.S_kv), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), j.ravel()], axis=1).astype(np.int32)


def fwd(q, k, v, doc_ids, g: Geom, rows=None):
    """Forward. rows=None: every (b, h, i); returns out [B,Hq,L,D], lse [B,Hq,L].
    rows=[(b,h,i),...]: returns out [n,D], lse [n]."""
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    assert qd.shape == (g.B, g.Hq, g.L, g.D) and kd.shape == (g.B, g.Hkv, g.S_kv, g.D) == vd.shape
    full = rows is None
    sel = _all_rows(g) if full else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = sel.shape[0]
    out = np.zeros((n, g.D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    _check(_load().og_fwd_rows(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(doc), ctypes.byref(g), _ptr(sel), n,
                               _ptr(out), _ptr(lse)), "fwd")
    if full:
        return out.reshape(g.B, g.Hq, g.L, g.D), lse.reshape(g.B, g.Hq, g.L)
    return out, lse


def fwd_chunk(q, k, v, doc_ids, g: Geom, rows=None):
    """Forward over one K/V chunk: the K/V buffer [kv_offset, kv_offset + S_kv)
    holds only part of the keys the rows may attend. Each row gets the softmax
    over its allowed keys inside the chunk; a real row with none gets out = 0,
    lse = -inf. Same shapes as fwd()."""
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    assert qd.shape == (g.B, g.Hq, g.L, g.D) and kd.shape == (g.B, g.Hkv, g.S_kv, g.D) == vd.shape
    full = rows is None
    sel = _all_rows(g) if full else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = sel.shape[0]
    out = np.zeros((n, g.D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    _check(_load().og_fwd_rows_chunk(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(doc), ctypes.byref(g), _ptr(sel), n,
                                     _ptr(out), _ptr(lse)), "fwd_chunk")
    if full:
        return out.reshape(g.B, g.Hq, g.L, g.D), lse.reshape(g.B, g.Hq, g.L)
    return out, lse


def merge(out_a, lse_a, out_b, lse_b):
    """Log-sum-exp merge of two chunk results (gemma4_moe.cp_local_ring: online
    softmax merge of per-chunk (out, lse), safe when either or both are -inf):
        lse = log(exp(lse_a) + exp(lse_b))
        out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b
    A row with both lse = -inf gets out = 0, lse = -inf. fp64."""
    oa, ob = np.asarray(out_a, np.float64), np.asarray(out_b, np.float64)
    la, lb = np.asarray(lse_a, np.float64), np.asarray(lse_b, np.float64)
    m = np.maximum(la, lb)
    both_empty = np.isneginf(m)
    ms = np.where(both_empty, 0.0, m)
    ea, eb = np.exp(la - ms), np.exp(lb - ms)  # exp(-inf) = 0 for an empty side
    tot = ea + eb
    lse = np.where(both_empty, -np.inf, ms + np.log(np.where(both_empty, 1.0, tot)))
    wa = np.where(both_empty, 0.0, ea / np.where(both_empty, 1.0, tot))
    wb = np.where(both_empty, 0.0, eb / np.where(both_empty, 1.0, tot))
    out = wa[..., None] * oa + wb[..., None] * ob
    return out, lse


def bwd(q, k, v, dout, doc_ids, g: Geom, rows=None, keys=None, full=None):
    """Backward of sum(out * dout).

    full=True (or rows and keys both None): returns dq [B,Hq,L,D], dk, dv
    [B,Hkv,S_kv,D]. Otherwise rows=[(b,h,i)] -> dq [nr,D] and keys=[(b,hk,j)]
    -> dk, dv [nk,D] (either list may be empty)."""
    qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
    doc = _i32(doc_ids).reshape(g.B, g.S_full)
    if full is None:
        full = rows is None and keys is None
    if full:
        rs, ks = _all_rows(g), _all_keys(g)
    else:
        rs = np.ascontiguousarray(np.asarray(rows if rows is not None else [], dtype=np.int32).reshape(-1, 3))
        ks = np.ascontiguousarray(np.asarray(keys if keys is not None else [], dtype=np.int32).reshape(-1, 3))
    nr, nk = rs.shape[0], ks.shape[0]
    dq = np.zeros((max(nr, 1), g.D), dtype=np.float64)
    dk = np.zeros((max(nk, 1), g.D), dtype=np.float64)
    dv = np.zeros((max(nk, 1), g.D), dtype=np.float64)
    _check(_load().og_bwd(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dod), _ptr(doc), ctypes.byref(g), _ptr(rs), nr,
                          _ptr(ks), nk, _ptr(dq), _ptr(dk), _ptr(dv)), "bwd")
    dq, dk, dv = dq[:nr], dk[:nk], dv[:nk]
    if full:
        return (dq.reshape(g.B, g.Hq, g.L, g.D), dk.reshape(g.B, g.Hkv, g.S_kv, g.D),
                dv.reshape(g.B, g.Hkv, g.S_kv, g.D))
    return dq, dk, dv
