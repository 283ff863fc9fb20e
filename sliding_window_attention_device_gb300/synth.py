"""Seeded synthetic inputs shaped like the NeMo AutoModel block-diagonal CP workloads.

This module draws document layouts and bf16 tensors and nothing else: it holds
none of the attention arithmetic (no masks, segments or softmax), so the CUDA
path and the fp64 oracle can both be fed from it.

Recipe (fixed so every run and every machine draws the same thing):
  * ``numpy.random.Generator(PCG64(seed))`` draws the document layout of batch
    rows 0..B-1 in order. "Packed until S minus a padding tail": draw the tail
    length T first, append documents while the packed length is below S - T,
    cut the last document so it ends exactly at S - T, then pad with id 0.
    Document ids are 1, 2, 3, ... along each row; padding is 0.
  * K and V cover the full padded sequence: ``torch.Generator('cpu')`` seeded
    with ``seed * 1000 + 1`` (K) and ``seed * 1000 + 2`` (V) draws
    [B, Hkv, S, D] ~ N(0, 1) in fp32, rounded to bf16. A shard's K/V buffer is
    a slice of these rows.
  * Q and dO of query shard r are drawn per shard (seeds ``seed * 1000 + 10 +
    2 r`` and ``seed * 1000 + 11 + 2 r``) as [B, Hq, L, D] ~ N(0, 1) rounded to
    bf16; the full-sequence Q is the concatenation of the shards' draws.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "doc_layout", "kv_rows", "q_shard", "dout_shard"]


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    B: int
    Hq: int
    Hkv: int
    D: int
    S: int          # full padded sequence length
    cp_size: int    # virtual context-parallel world size; L = S / cp_size
    layout: tuple   # document-length recipe, see doc_layout()
    window: int = 0
    ranks: tuple = ()
    kv: str = "full"  # "full": [0, S); "prefix": [0, (r+1) L); "needed": [s_first, real_end)
    notes: str = ""

    @property
    def L(self) -> int:
        return self.S // self.cp_size

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def prefix_kv(self, r: int) -> tuple[int, int]:
        """(kv_offset, S_kv) for the "full" and "prefix" K/V rules."""
        if self.kv == "full":
            return 0, self.S
        if self.kv == "prefix":
            return 0, (r + 1) * self.L
        raise ValueError("the needed-range rule depends on the segmentation; compute it from the doc ids")


WORKLOADS = {
    "C1": Workload("C1", "tiny block-diagonal shard", B=1, Hq=2, Hkv=1, D=64, S=256, cp_size=4,
                   layout=("explicit", (100, 90, 50), 16), window=0, ranks=(2,), kv="full"),
    "C2": Workload("C2", "packed multi-doc block-diagonal, 32K", B=2, Hq=32, Hkv=8, D=128, S=32768, cp_size=8,
                   layout=("lognormal", 2048.0, 1.0, 64, 16384, 511), window=0, ranks=tuple(range(8)),
                   kv="full"),
    "C3": Workload("C3", "Gemma4-style sliding layer, window 1024", B=1, Hq=16, Hkv=8, D=256, S=65536,
                   cp_size=8, layout=("uniform", 512, 16384, 511), window=1024, ranks=tuple(range(8)),
                   kv="prefix"),
    "C4": Workload("C4", "single long document spanning all shards", B=1, Hq=64, Hkv=8, D=128, S=131072,
                   cp_size=16, layout=("single",), window=0, ranks=(15, 7), kv="prefix"),
    "C5": Workload("C5", "many short docs, needed-range K/V", B=4, Hq=32, Hkv=4, D=128, S=65536, cp_size=8,
                   layout=("uniform", 128, 4096, 0), window=0, ranks=tuple(range(8)), kv="needed"),
    "C5w4096": Workload("C5w4096", "many short docs, needed-range K/V, window 4096", B=4, Hq=32, Hkv=4, D=128,
                        S=65536, cp_size=8, layout=("uniform", 128, 4096, 0), window=4096,
                        ranks=tuple(range(8)), kv="needed"),
    "G512": Workload("G512", "Gemma4-style global layer, head dim 512", B=1, Hq=16, Hkv=4, D=512,
                     S=32768, cp_size=8, layout=("uniform", 512, 16384, 511), window=0, ranks=tuple(range(8)),
                     kv="prefix"),
    "C5w512": Workload("C5w512", "many short docs, needed-range K/V, window 512", B=4, Hq=32, Hkv=4, D=128,
                       S=65536, cp_size=8, layout=("uniform", 128, 4096, 0), window=512,
                       ranks=tuple(range(8)), kv="needed"),
}


def _pack_row(rng: np.random.Generator, S: int, tail: int, draw) -> np.ndarray:
    ids = np.zeros(S, dtype=np.int32)
    end = S - tail
    pos, doc = 0, 1
    while pos < end:
        n = int(draw())
        n = max(1, min(n, end - pos))
        ids[pos:pos + n] = doc
        pos += n
        doc += 1
    return ids


def doc_layout(layout: tuple, B: int, S: int, seed: int = 0) -> np.ndarray:
    """Document ids [B, S] (int32; 0 = padding) for one of the layout recipes:

    ("explicit", lengths, pad)                 the given lengths, then `pad` zeros
    ("lognormal", median, sigma, lo, hi, tmax) lengths round(lognormal) clipped to [lo, hi],
                                               tail T ~ U{0..tmax}
    ("uniform", lo, hi, tmax)                  lengths ~ U{lo..hi}, tail T ~ U{0..tmax}
    ("single",)                                one document over the whole row, no padding
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    kind = layout[0]
    rows = []
    for _ in range(B):
        if kind == "explicit":
            lengths, pad = layout[1], layout[2]
            ids = np.zeros(S, dtype=np.int32)
            pos = 0
            for d, n in enumerate(lengths, start=1):
                ids[pos:pos + n] = d
                pos += n
            assert pos + pad == S, "explicit layout must fill the row"
        elif kind == "lognormal":
            median, sigma, lo, hi, tmax = layout[1:]
            tail = int(rng.integers(0, tmax + 1))
            mu = float(np.log(median))
            ids = _pack_row(rng, S, tail,
                            lambda: int(round(float(np.clip(rng.lognormal(mu, sigma), lo, hi)))))
        elif kind == "uniform":
            lo, hi, tmax = layout[1:]
            tail = int(rng.integers(0, tmax + 1)) if tmax > 0 else 0
            ids = _pack_row(rng, S, tail, lambda: int(rng.integers(lo, hi + 1)))
        elif kind == "single":
            ids = np.ones(S, dtype=np.int32)
        else:
            raise ValueError(f"unknown layout {kind!r}")
        rows.append(ids)
    return np.stack(rows, axis=0)


def _randn_bf16(shape, seed: int):
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def kv_rows(w: Workload, seed: int = 0, lo: int = 0, hi: int | None = None):
    """bf16 K and V rows [lo, hi) of the full sequence: each [B, Hkv, hi-lo, D]."""
    hi = w.S if hi is None else hi
    k = _randn_bf16((w.B, w.Hkv, w.S, w.D), seed * 1000 + 1)[:, :, lo:hi].contiguous()
    v = _randn_bf16((w.B, w.Hkv, w.S, w.D), seed * 1000 + 2)[:, :, lo:hi].contiguous()
    return k, v


def q_shard(w: Workload, r: int, seed: int = 0):
    """bf16 queries of shard r: [B, Hq, L, D]."""
    return _randn_bf16((w.B, w.Hq, w.L, w.D), seed * 1000 + 10 + 2 * r)


def dout_shard(w: Workload, r: int, seed: int = 0):
    """bf16 output gradient of shard r: [B, Hq, L, D]."""
    return _randn_bf16((w.B, w.Hq, w.L, w.D), seed * 1000 + 11 + 2 * r)
