#!/usr/bin/env python
"""Benchmark of per-document causal (block-diagonal) CP attention, forward + backward.

Metric: fwd+bwd TFLOP/s counting only unmasked FLOPs (4*D per allowed
(query, key) pair per query head forward, 10*D backward), and the fraction of
the GB300's measured dense BF16 peak, on one GPU.

Workload (default): the packed multi-document 32K shard set -- B=2, Hq=32,
Hkv=8, D=128, S=32768 split into 8 virtual context-parallel ranks (L=4096),
K/V = the full sequence. One step runs the whole path for every rank:
segmentation + tile classification, forward, backward (prep, main, dq
finalize). Inputs are resident in HBM before the timed region; K/V (268 MB)
exceed the 129 MB L2, so no flush is needed between steps.

With --kv-chunks ring, each shard's K/V arrives in per-rank pieces as in a
ring step: a forward per piece merged into the shard's (out, lse) in the
forward's epilogue, then one backward main per piece with the merged out /
lse. --kv-chunks ring-merge does the merges with the separate log-sum-exp
merge kernel and adds its HBM roofline to the line. The FLOP count is the
same as the unchunked step's.

With --exchange, the line is instead the sender side of the needed-only
K/V exchange for every rank of the workload: the exchange plan built from the
device doc ids, the gather of K and V into the send buffers and the index-add
of the returned dK / dV, in algorithmic GB/s against the HBM roofline.

With --gpus N (torchrun), each GPU runs an independent replica with its own
seed (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sliding_window_attention_device_gb300 import synth  # noqa: E402

METRIC = "fwd+bwd TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 peak, 1 GPU"
UNIT = "TFLOP/s"

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the backward main
# kernel, the mean over the 8 launches (one per shard) of one bench step, from
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` (see profiles/);
# valid only for the kernel sources whose hash is recorded here.
# the backward main-stage kernel of each head dim
BWD_KERNEL = {64: "bwd128_kernel<64>", 128: "bwd128_kernel<128>", 256: "bwd_kernel<256>",
              512: "bwd512_kernel (four CTAs per K/V tile, one per 128-column slice)"}
# the fixed-order dq pass of each head dim above 128
DQ_KERNEL = {256: "bwd_dq256_kernel", 512: "bwd_dq512_kernel (two CTAs per q tile, one per 256-column half)"}
TRAFFIC = {"kernel": "bwd128_kernel<128>", "workload": "C2", "source_sha256": "197ab565abf9f318", "bytes_per_launch": 1.60883e9}


# ------------------------------------------------------------------ workload
def doc_starts(row: np.ndarray) -> np.ndarray:
    """Global start position of the run each position belongs to."""
    n = row.shape[0]
    change = np.ones(n, bool)
    change[1:] = row[1:] != row[:-1]
    return np.maximum.accumulate(np.where(change, np.arange(n), 0))


def pairs_closed_form(doc: np.ndarray, row_offset: int, L: int, window: int) -> int:
    """Allowed (query, key) pairs over real local rows: each real row p attends
    [max(doc_start(p), p - W + 1), p], so it contributes p - lo + 1 keys."""
    total = 0
    for b in range(doc.shape[0]):
        st = doc_starts(doc[b])
        p = row_offset + np.arange(L)
        lo = st[p]
        if window > 0:
            lo = np.maximum(lo, p - window + 1)
        real = doc[b, p] != 0
        total += int(((p - lo + 1) * real).sum())
    return total


def needed_range(doc: np.ndarray, row_offset: int, L: int) -> tuple[int, int]:
    """[min_b s_first, max_b real_end) of a shard (the needed-only K/V range)."""
    lo, hi = None, None
    for b in range(doc.shape[0]):
        p = row_offset + np.arange(L)
        real = doc[b, p] != 0
        n_real = int(np.argmin(real)) if not real.all() else L
        if n_real == 0:
            continue
        s_first = int(doc_starts(doc[b])[row_offset])
        lo = s_first if lo is None else min(lo, s_first)
        hi = row_offset + n_real if hi is None else max(hi, row_offset + n_real)
    if lo is None:
        return row_offset, 1
    return lo, hi - lo


def shard_plan(w: synth.Workload, doc: np.ndarray):
    plan = []
    for r in w.ranks:
        ro = r * w.L
        if w.kv == "needed":
            kvo, skv = needed_range(doc, ro, w.L)
        else:
            kvo, skv = w.prefix_kv(r)
        plan.append(dict(r=r, row_offset=ro, kv_offset=kvo, S_kv=skv,
                         pairs=pairs_closed_form(doc, ro, w.L, w.window)))
    return plan


# ------------------------------------------------------------------- helpers
def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(source="measured", bf16_tflops=d.get("bf16_tflops"),
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), hbm_gbs=d.get("hbm_gbs"))
    return dict(source="fallback", bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, hbm_gbs=6800.0)


def choose_peak(peaks: dict, clocks: dict) -> tuple[float, str]:
    """The bf16 denominator that matches the clock record of the timed region:
    the burst figure (a GEMM timed alone at full clock) when the median SM
    clock sat at its maximum and the power cap never engaged, else the
    sustained one (a GEMM held for seconds under the power cap)."""
    burst, sust = peaks.get("bf16_tflops"), peaks.get("bf16_tflops_sustained")
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    at_max = sm is not None and bool(smax) and sm >= 0.99 * smax
    if burst and (at_max and not capped or not sust):
        return float(burst), f"{peaks['source']} bf16_tflops (burst: median SM clock at its maximum, no power cap)"
    return float(sust), f"{peaks['source']} bf16_tflops_sustained (SM clock below its maximum or power-capped)"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def kernel_source_sha() -> str:
    """Hash of the sources the D = 128 backward main kernel is built from."""
    h = hashlib.sha256()
    for f in ("bwd128_kernel.cu", "common.cuh", "pipeline.cuh", "sm100_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "sliding_window_attention_device_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------- multi-rank bookkeeping
def rank_seed(seed: int, rank: int) -> int:
    """Each rank's replica draws its own inputs (weak scaling: independent problems)."""
    return seed + rank


def allreduce_max(x: float, device, world: int) -> float:
    """The slowest rank's time: the job is done when every rank is."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: the FLOPs every rank did in one step over the step time."""
    return world * flop_per_rank / (ms_per_step * 1e-3) / 1e12


# --------------------------------------------------------------- our path
class Replica:
    """Device-resident inputs / outputs of every shard of the workload."""

    def __init__(self, w: synth.Workload, seed: int, dev: torch.device, grad_dtype, ranks=None,
                 deterministic=False, fwd_only=False):
        from sliding_window_attention_device_gb300 import bdattn
        self.bd, self.w, self.dev, self.grad_dtype = bdattn, w, dev, grad_dtype
        self.deterministic = deterministic  # dq by the fixed-order pass: bitwise reproducible
        self.fwd_only = fwd_only  # segments and forward only
        self.doc_np = synth.doc_layout(w.layout, w.B, w.S, seed)
        self.plan = [sh for sh in shard_plan(w, self.doc_np) if ranks is None or sh["r"] in ranks]
        self.doc = torch.from_numpy(self.doc_np).to(dev)
        k, v = synth.kv_rows(w, seed)
        self.k_full, self.v_full = k.to(dev), v.to(dev)
        self.status = bdattn.new_status(dev)
        self.shards = []
        ws = 0
        for sh in self.plan:
            g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, sh["row_offset"], sh["kv_offset"], sh["S_kv"], w.window)
            a, b = sh["kv_offset"], sh["kv_offset"] + sh["S_kv"]
            k_sh = self.k_full if (a, b) == (0, w.S) else self.k_full[:, :, a:b].contiguous()
            v_sh = self.v_full if (a, b) == (0, w.S) else self.v_full[:, :, a:b].contiguous()
            d = dict(g=g, pairs=sh["pairs"], k=k_sh, v=v_sh,
                     q=synth.q_shard(w, sh["r"], seed).to(dev), do=synth.dout_shard(w, sh["r"], seed).to(dev),
                     seg=torch.empty(bdattn.seg_bytes(g) // 4, dtype=torch.int32, device=dev),
                     out=torch.empty(w.B, w.Hq, w.L, w.D, dtype=torch.bfloat16, device=dev),
                     lse=torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev),
                     dq=torch.empty(w.B, w.Hq, w.L, w.D, dtype=grad_dtype, device=dev),
                     dk=torch.empty(w.B, w.Hkv, sh["S_kv"], w.D, dtype=grad_dtype, device=dev),
                     dv=torch.empty(w.B, w.Hkv, sh["S_kv"], w.D, dtype=grad_dtype, device=dev))
            ws = max(ws, bdattn.bwd_workspace_bytes(g))
            self.shards.append(d)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        # per shard: segment build + classification, forward, backward prep,
        # backward main (which also writes the zero dK / dV of unattended
        # tiles), and (bf16 gradients only) the dq finalize; fp32 dq is
        # accumulated in place
        self.launches_per_step = (5 if grad_dtype == torch.float32 else 6) * len(self.shards)
        if deterministic:  # delta, dK / dV, dq: one more launch per shard than the fp32 path
            self.launches_per_step = 6 * len(self.shards)
        if fwd_only:  # segment build, classification, forward
            self.launches_per_step = 3 * len(self.shards)

    def flops(self) -> tuple[float, float, float]:
        D, Hq = self.w.D, self.w.Hq
        pairs = sum(s["pairs"] for s in self.shards)
        if self.fwd_only:
            return 4.0 * D * Hq * pairs, 4.0 * D * Hq * pairs, 0.0
        return 14.0 * D * Hq * pairs, 4.0 * D * Hq * pairs, 10.0 * D * Hq * pairs

    def run_shard(self, i, ev=None):
        """The whole path for shard i on the current stream: segments, forward, backward."""
        bd = self.bd
        s = self.shards[i]
        g = s["g"]
        ws = self.workspace[:bd.bwd_workspace_bytes(g)]
        bd.bd_attn_seg_build(self.doc, g, seg=s["seg"], status=self.status)
        if ev is not None:
            ev["fwd"][i][0].record()
        bd.bd_attn_fwd(s["q"], s["k"], s["v"], s["seg"], g, self.status, out=s["out"], lse=s["lse"])
        if ev is not None:
            ev["fwd"][i][1].record()
        if self.fwd_only:
            return
        if self.deterministic:
            if ev is not None:
                ev["bwd"][i][0].record()
            bd.bd_attn_bwd_deterministic(s["do"], s["q"], s["k"], s["v"], s["out"], s["lse"], s["seg"], g,
                                         self.status, grad_dtype=s["dq"].dtype, dq=s["dq"], dk=s["dk"], dv=s["dv"],
                                         workspace=ws)
            if ev is not None:
                ev["bwd"][i][1].record()
            return
        direct = s["dq"].dtype == torch.float32  # fp32 dq is its own accumulator: no finalize
        if direct:
            bd.bd_attn_bwd_prep_dq(s["do"], s["out"], g, self.status, ws, s["dq"])
        else:
            bd.bd_attn_bwd_prep(s["do"], s["out"], g, self.status, ws)
        if ev is not None:
            ev["bwd"][i][0].record()
        if direct:
            bd.bd_attn_bwd_main_dq(s["do"], s["q"], s["k"], s["v"], s["lse"], s["seg"], g, self.status, ws,
                                   s["dq"], s["dk"], s["dv"])
        else:
            bd.bd_attn_bwd_main(s["do"], s["q"], s["k"], s["v"], s["lse"], s["seg"], g, self.status, ws,
                                s["dk"], s["dv"])
        if ev is not None:
            ev["bwd"][i][1].record()
        if not direct:
            bd.bd_attn_bwd_finalize(g, self.status, ws, s["dq"])

    def step(self, ev=None):
        for i in range(len(self.shards)):
            self.run_shard(i, ev)


class RingChunkReplica(Replica):
    """The same shards with K/V arriving in pieces, as one ring step at a time
    (gemma4_moe.cp_local_ring, the ring forward loop: per step the K/V block of
    one context-parallel rank, a varlen forward over it returning (out, lse),
    the -inf-safe merge, and a per-chunk backward with the merged out / lse).
    A shard's K/V range is cut at the ranks' boundaries [j L, (j+1) L); blocks
    owned by a rank after the shard's own are skipped, as the loop skips them
    (no local row reaches a later position), and so are blocks wholly before
    every local row's sliding window. Each chunk has its own table,
    contiguous K / V and dK / dV; the first chunk's forward writes the shard's
    out / lse, the others go through a scratch (out, lse) and the merge kernel."""

    def __init__(self, w: synth.Workload, seed: int, dev: torch.device, grad_dtype, ranks=None, fused=True):
        super().__init__(w, seed, dev, grad_dtype, ranks)
        bd = self.bd
        self.fused = fused  # merge in the forward's epilogue (else: forward to scratch + merge kernel)
        kv_cache = {}
        self.launches_per_step = 0
        for s, sh in zip(self.shards, self.plan):
            lo, hi = sh["kv_offset"], sh["kv_offset"] + sh["S_kv"]
            chunks = []
            for j in range(sh["r"] + 1):
                a, b = max(lo, j * w.L), min(hi, (j + 1) * w.L)
                if b <= a or (w.window > 0 and b <= sh["row_offset"] - w.window + 1):
                    continue  # empty, or wholly before every local row's window
                if (a, b) not in kv_cache:
                    kv_cache[(a, b)] = (self.k_full[:, :, a:b].contiguous(), self.v_full[:, :, a:b].contiguous())
                g = bd.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, sh["row_offset"], a, b - a, w.window)
                k, v = kv_cache[(a, b)]
                chunks.append(dict(g=g, k=k, v=v, seg=torch.empty(bd.seg_bytes(g) // 4, dtype=torch.int32, device=dev),
                                   dk=torch.empty(w.B, w.Hkv, b - a, w.D, dtype=grad_dtype, device=dev),
                                   dv=torch.empty(w.B, w.Hkv, b - a, w.D, dtype=grad_dtype, device=dev)))
            if not chunks:
                raise ValueError(f"shard r={sh['r']}: no K/V chunk")
            s["chunks"] = chunks
            n = len(chunks)
            # per chunk: table build + classification, forward, backward main;
            # per merge one launch unless fused; per shard the backward prep
            # (and the dq finalize for bf16 gradients)
            self.launches_per_step += (4 * n + (0 if fused else n - 1) + 1 +
                                       (0 if grad_dtype == torch.float32 else 1))
        self.n_merges = sum(len(s["chunks"]) - 1 for s in self.shards)
        self.kv_chunk_bytes = sum(k.numel() * 2 + v.numel() * 2 for k, v in kv_cache.values())
        self.out_c = torch.empty(w.B, w.Hq, w.L, w.D, dtype=torch.bfloat16, device=dev)
        self.lse_c = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)

    def merge_bytes(self) -> float:
        """Algorithmic bytes of one merge launch: read both (out, lse), write one."""
        w = self.w
        rows = w.B * w.Hq * w.L
        return 3.0 * rows * (w.D * 2 + 4)

    def run_shard(self, i, ev=None):
        bd = self.bd
        s = self.shards[i]
        ws = self.workspace[:bd.bwd_workspace_bytes(s["g"])]
        for c in s["chunks"]:
            bd.bd_attn_seg_build_chunk(self.doc, c["g"], seg=c["seg"], status=self.status)
        if ev is not None:
            ev["fwd"][i][0].record()
        for n, c in enumerate(s["chunks"]):
            if n == 0:
                bd.bd_attn_fwd(s["q"], c["k"], c["v"], c["seg"], c["g"], self.status, out=s["out"], lse=s["lse"])
                continue
            if self.fused:
                bd.bd_attn_fwd_merge(s["q"], c["k"], c["v"], c["seg"], c["g"], self.status, s["out"], s["lse"])
                continue
            bd.bd_attn_fwd(s["q"], c["k"], c["v"], c["seg"], c["g"], self.status, out=self.out_c, lse=self.lse_c)
            if ev is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            bd.bd_attn_merge(s["out"], s["lse"], self.out_c, self.lse_c, c["g"], self.status)
            if ev is not None:
                e1.record()
                ev["merge"].append((e0, e1))
        if ev is not None:
            ev["fwd"][i][1].record()
        direct = s["dq"].dtype == torch.float32
        if direct:
            bd.bd_attn_bwd_prep_dq(s["do"], s["out"], s["g"], self.status, ws, s["dq"])
        else:
            bd.bd_attn_bwd_prep(s["do"], s["out"], s["g"], self.status, ws)
        if ev is not None:
            ev["bwd"][i][0].record()
        for c in s["chunks"]:
            if direct:
                bd.bd_attn_bwd_main_dq(s["do"], s["q"], c["k"], c["v"], s["lse"], c["seg"], c["g"], self.status,
                                       ws, s["dq"], c["dk"], c["dv"])
            else:
                bd.bd_attn_bwd_main(s["do"], s["q"], c["k"], c["v"], s["lse"], c["seg"], c["g"], self.status, ws,
                                    c["dk"], c["dv"])
        if ev is not None:
            ev["bwd"][i][1].record()
        if not direct:
            bd.bd_attn_bwd_finalize(s["g"], self.status, ws, s["dq"])


def run_exchange(args, local_rank: int) -> dict:
    """The sender side of the needed-only K/V exchange for every virtual rank of
    the workload (blockdiag_cp.exchange: the exchange plan from the device doc
    ids, `_NeededKVExchange` forward gather of K and V into the token-major send
    buffer, and its backward index-add of the returned dK / dV): one step runs
    all four for every rank. Inputs resident in HBM; the collective between
    GPUs is not part of it."""
    from sliding_window_attention_device_gb300 import bdattn as bd
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.config]
    W, L = w.cp_size, w.L
    doc_np = synth.doc_layout(w.layout, w.B, w.S, args.seed)
    doc = torch.from_numpy(doc_np).to(dev)
    k, v = synth.kv_rows(w, args.seed)
    k, v = k.to(dev), v.to(dev)
    status = bd.new_status(dev)
    # the send-buffer sizes come from the plans, read back once before timing
    plans = [bd.bd_attn_exchange_plan(doc, W, r, status=status)[0] for r in range(W)]
    p = bd.read_plan(plans[0], w.B, W, L)
    ranks = []
    for r in range(W):
        n = sum(p["counts"][r])
        gen = torch.Generator(device=dev).manual_seed(args.seed * 100 + r)
        ranks.append(dict(
            plan=plans[r], n=n,
            k=k[:, :, r * L:(r + 1) * L].contiguous(), v=v[:, :, r * L:(r + 1) * L].contiguous(),
            sk=torch.empty((max(n, 1), w.B, w.Hkv, w.D), dtype=torch.bfloat16, device=dev),
            sv=torch.empty((max(n, 1), w.B, w.Hkv, w.D), dtype=torch.bfloat16, device=dev),
            gk=torch.rand((max(n, 1), w.B, w.Hkv, w.D), generator=gen, device=dev),
            gv=torch.rand((max(n, 1), w.B, w.Hkv, w.D), generator=gen, device=dev),
            dk=torch.empty((w.B, w.Hkv, L, w.D), dtype=torch.float32, device=dev),
            dv=torch.empty((w.B, w.Hkv, L, w.D), dtype=torch.float32, device=dev)))
    del k, v
    kinds = ("plan", "gather", "scatter_add")

    def phase(kind):
        for i, s in enumerate(ranks):
            if kind == "plan":
                bd.bd_attn_exchange_plan(doc, W, i, plan=s["plan"], status=status)
            elif kind == "gather":
                bd.bd_attn_needed_gather(s["k"], s["plan"], s["sk"], status)
                bd.bd_attn_needed_gather(s["v"], s["plan"], s["sv"], status)
            else:
                bd.bd_attn_needed_scatter_add(s["gk"], s["plan"], s["dk"], status)
                bd.bd_attn_needed_scatter_add(s["gv"], s["plan"], s["dv"], status)

    # Each phase (every rank's plans, gathers or index-adds) is one CUDA graph:
    # the launches are small enough that issuing them one by one from Python
    # would leave the GPU waiting on the host.
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            for kd in kinds:
                phase(kd)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} after warm-up")
    graphs = {}
    for kd in kinds:
        graphs[kd] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[kd]):
            phase(kd)
    for _ in range(args.warmup):
        for kd in kinds:
            graphs[kd].replay()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(str(local_rank)) as clk:
        torch.cuda.synchronize()
        start.record()
        for m in events:
            m[0].record()
            for j, kd in enumerate(kinds):
                graphs[kd].replay()
                m[j + 1].record()
        stop.record()
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the timed region")
    ms = start.elapsed_time(stop)
    kind_ms = {kd: sum(m[j].elapsed_time(m[j + 1]) for m in events) for j, kd in enumerate(kinds)}
    row = w.B * w.Hkv * w.D  # elements per token
    sent = sum(s["n"] for s in ranks)
    # algorithmic bytes per step: the gathers read each local chunk once and write
    # the send buffers (K and V, bf16); the index-adds read the returned fp32
    # gradients and write the local dK / dV once
    gather_bytes = 2 * (W * L * row * 2 + sent * row * 2)
    scatter_bytes = 2 * (sent * row * 4 + W * L * row * 4)
    peaks = read_peaks()
    steps = args.steps

    def roof(kind, nbytes):
        t = kind_ms[kind] * 1e-3 / steps
        return {"kernel": kind, "bound": "hbm", "achieved": round(nbytes / t / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(nbytes / t / 1e9 / peaks["hbm_gbs"], 4), "bytes_per_step": nbytes,
                "ms_per_step": round(kind_ms[kind] / steps, 4), "launches_per_step": 2 * W}

    value = (gather_bytes + scatter_bytes) / (ms * 1e-3 / steps) / 1e9
    return {
        "metric": "needed-only K/V exchange, sender side (plan + gather + index-add), algorithmic GB/s, 1 GPU",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms / steps, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 K/V, f32 gradients", "data": "synthetic",
        "config": {"workload": f"{w.key}: {w.title}", "B": w.B, "Hkv": w.Hkv, "D": w.D, "S": w.S, "cp_size": W,
                   "L": L, "use_halo": bool(p["use_halo"]), "halo_size": p["halo_size"], "tokens_sent": sent,
                   "seed": args.seed, "l2": "send buffers and gradients of all ranks exceed L2 together; no flush"},
        "plan_us_per_rank": round(kind_ms["plan"] * 1e3 / (steps * W), 2),
        "roofline": roof("gather", gather_bytes), "roofline_index_add": roof("scatter_add", scatter_bytes),
        "gpu_launches": 6 * W * steps, "launch": "one CUDA graph per phase (plans, gathers, index-adds of every rank)",
        "clocks": clk.summary(),
    }


def smi_index(local_rank: int) -> str:
    visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return visible[local_rank].strip() if local_rank < len(visible) else str(local_rank)


def timed_steps(rep, steps: int, warmup: int, world: int, local_rank: int) -> dict:
    """W untimed warm-up steps, then exactly `steps` steps between two CUDA events on
    the launching stream, bracketed by a barrier and a synchronize on both sides,
    with per-shard forward / backward events and the SM clocks sampled meanwhile."""
    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(warmup):
        rep.step()
    torch.cuda.synchronize()
    if int(rep.status.item()) != 0:
        raise RuntimeError(f"device status {int(rep.status.item()):#x} after warm-up")
    n = len(rep.shards)
    ev_steps = [{"fwd": [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)],
                 "bwd": [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)],
                 "merge": []}
                for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(smi_index(local_rank)) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for k in range(steps):
            rep.step(ev_steps[k])
        stop.record()
        torch.cuda.synchronize()
        barrier()
    clocks = clk.summary()
    if int(rep.status.item()) != 0:
        raise RuntimeError(f"device status {int(rep.status.item()):#x} in the timed region")
    fwd_only = getattr(rep, "fwd_only", False)
    return {
        "ms": start.elapsed_time(stop),
        "fwd_ms": sum(e["fwd"][i][0].elapsed_time(e["fwd"][i][1]) for e in ev_steps for i in range(n)),
        "bwd_ms": 0.0 if fwd_only else sum(e["bwd"][i][0].elapsed_time(e["bwd"][i][1])
                                           for e in ev_steps for i in range(n)),
        "merge_ms": sum(a.elapsed_time(b) for e in ev_steps for a, b in e["merge"]),
        "n_merge": sum(len(e["merge"]) for e in ev_steps),
        "clocks": clocks,
    }


# the other workloads timed in the same run as the headline (few steps each)
OTHER_CONFIGS = (("C3", None), ("C4", {15}), ("C5w512", None), ("G512", None))


def run_other_configs(args, dev, local_rank: int, peaks: dict) -> dict:
    """fwd+bwd throughput of the other workloads, same fields and timing rules as
    the headline line (CUDA events, inputs resident, clock record per workload)."""
    res = {}
    grad_dtype = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    steps, warmup = max(3, min(args.steps, 5)), 3
    for key, ranks in OTHER_CONFIGS:
        w = synth.WORKLOADS[key]
        rep = Replica(w, args.seed, dev, grad_dtype, ranks)
        total_flop, fwd_flop, bwd_flop = rep.flops()
        t = timed_steps(rep, steps, warmup, 1, local_rank)
        ms_per_step = t["ms"] / steps
        value = total_flop / (ms_per_step * 1e-3) / 1e12
        bwd_tf = bwd_flop * steps / (t["bwd_ms"] * 1e-3) / 1e12
        peak, src = choose_peak(peaks, t["clocks"])
        res[key] = {
            "workload": f"{w.key}: {w.title}", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "S": w.S,
            "cp_size": w.cp_size, "L": w.L, "window": w.window, "kv": w.kv, "ranks": [s["r"] for s in rep.plan],
            "pairs": sum(s["pairs"] for s in rep.shards), "value": round(value, 2), "unit": UNIT,
            "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 4),
            "tokens_per_s": round(w.B * w.L * len(rep.shards) / (ms_per_step * 1e-3), 1),
            "fwd_tflops": round(fwd_flop * steps / (t["fwd_ms"] * 1e-3) / 1e12, 2),
            "bwd_main_tflops": round(bwd_tf, 2), "peak": peak, "peak_source": src,
            "frac": round(value / peak, 4),
            "frac_of_burst": round(value / peaks["bf16_tflops"], 4) if peaks.get("bf16_tflops") else None,
            "frac_of_sustained": (round(value / peaks["bf16_tflops_sustained"], 4)
                                  if peaks.get("bf16_tflops_sustained") else None),
            "gpu_launches": rep.launches_per_step * steps, "clocks": t["clocks"],
        }
        del rep
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank: int, world: int, local_rank: int):
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.config]
    grad_dtype = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    ranks = None if args.shards is None else {int(x) for x in args.shards.split(",")}
    chunked = args.kv_chunks in ("ring", "ring-merge")
    if chunked:
        rep = RingChunkReplica(w, rank_seed(args.seed, rank), dev, grad_dtype, ranks, fused=args.kv_chunks == "ring")
    else:
        rep = Replica(w, rank_seed(args.seed, rank), dev, grad_dtype, ranks, deterministic=args.deterministic,
                      fwd_only=args.fwd_only)
    total_flop, fwd_flop, bwd_flop = rep.flops()
    t = timed_steps(rep, args.steps, args.warmup, world, local_rank)
    clocks = t["clocks"]
    ms, fwd_ms, bwd_ms, merge_ms, n_merge = t["ms"], t["fwd_ms"], t["bwd_ms"], t["merge_ms"], t["n_merge"]
    fwd_only = getattr(rep, "fwd_only", False)
    ms = allreduce_max(ms, dev, world)
    ms_per_step = ms / args.steps

    e2e = None
    if not args.no_e2e and not chunked and not fwd_only:
        e2e = run_e2e(rep, args, total_flop, world, ms_per_step)

    if rank != 0:
        return None
    peaks = read_peaks()
    value = job_tflops(total_flop, ms_per_step, world)
    bwd_achieved = bwd_flop * args.steps / (bwd_ms * 1e-3) / 1e12 if bwd_ms > 0 else 0.0
    peak, peak_source = choose_peak(peaks, clocks)
    burst, sust = peaks.get("bf16_tflops"), peaks.get("bf16_tflops_sustained")
    fracs = lambda a: {"frac_of_burst": round(a / burst, 4) if burst else None,
                       "frac_of_sustained": round(a / sust, 4) if sust else None}
    traffic = None
    if (TRAFFIC["bytes_per_launch"] and TRAFFIC["source_sha256"] == kernel_source_sha() and not chunked
            and w.key == TRAFFIC["workload"] and not getattr(rep, "deterministic", False)):
        traffic = TRAFFIC["bytes_per_launch"]  # measured per whole-shard launch, not per chunk
    n_bwd = sum(len(s["chunks"]) for s in rep.shards) if chunked else len(rep.shards)
    fwd_kernel_ms = fwd_ms - merge_ms  # the forward region less its merges
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.key}: {w.title}", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "S": w.S,
                   "cp_size": w.cp_size, "L": w.L, "ranks": [s["r"] for s in rep.plan], "window": w.window, "kv": w.kv,
                   "grad_dtype": args.grad_dtype, "l2": "inputs larger than L2 (K/V 268 MB), no flush",
                   "pairs": sum(s["pairs"] for s in rep.shards), "seed": args.seed,
                   "backward": "deterministic (fixed-order dq pass)" if getattr(rep, "deterministic", False)
                   else "dq by fp32 atomic additions",
                   "kv_chunks": (f"{args.kv_chunks}: K/V cut at the cp ranks' boundaries, owners after the shard "
                                 f"skipped, {n_bwd} chunks, {rep.n_merges} merges per step, "
                                 + ("in the forward's epilogue" if rep.fused else "by the merge kernel"))
                                if chunked else "none"},
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "peak": peak, "peak_source": peak_source, **fracs(value / world),
        "tokens_per_s": round(world * w.B * w.L * len(rep.shards) / (ms_per_step * 1e-3), 1),
        "fwd_tflops": round(fwd_flop * args.steps / (fwd_kernel_ms * 1e-3) / 1e12, 2),
        "bwd_main_tflops": round(bwd_achieved, 2),
        "roofline": {"kernel": (f"backward: delta, {BWD_KERNEL[w.D]} without dq, "
                                f"{DQ_KERNEL.get(w.D, f'bwd_dq_kernel<{w.D}>')}"
                                if getattr(rep, "deterministic", False) else
                                f"{BWD_KERNEL[w.D]} (backward main stage, zero dK/dV of unattended tiles included)"),
                     "bound": "tensor", "achieved": round(bwd_achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(bwd_achieved / peak, 4),
                     **fracs(bwd_achieved), "peak_source": peak_source,
                     "traffic": traffic,
                     "flops_per_launch": bwd_flop / n_bwd,
                     "avg_launch_ms": round(bwd_ms / (args.steps * n_bwd), 4)},
        "gpu_launches": rep.launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if fwd_only:
        fwd_s = fwd_ms * 1e-3 / (args.steps * len(rep.shards))
        fwd_achieved = fwd_flop / len(rep.shards) / fwd_s / 1e12
        line["metric"] = "fwd TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 peak, 1 GPU"
        line["e2e_note"] = "forward only: the end-to-end timing covers the whole path"
        line["roofline"] = {"kernel": f"fwd{'512' if w.D == 512 else ''}_kernel (forward, D {w.D})", "bound": "tensor",
                            "achieved": round(fwd_achieved, 2), "peak": peak, "unit": "TFLOP/s",
                            "frac": round(fwd_achieved / peak, 4), **fracs(fwd_achieved),
                            "peak_source": peak_source,
                            "traffic": None, "flops_per_launch": fwd_flop / len(rep.shards),
                            "avg_launch_ms": round(fwd_s * 1e3, 4)}
        del line["bwd_main_tflops"]
    if chunked:
        line["e2e_note"] = "end-to-end timing is taken on the unchunked path only"
        if n_merge:
            merge_s = merge_ms * 1e-3 / n_merge
            achieved = rep.merge_bytes() / merge_s / 1e9
            line["merge_roofline"] = {
                "kernel": f"merge_kernel<{w.D}>", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": f"{peaks['source']} hbm_gbs", "bytes_per_launch": rep.merge_bytes(),
                "avg_launch_ms": round(merge_ms / n_merge, 4), "launches": n_merge,
                "share_of_step": round(merge_ms / ms, 4)}
    if world == 1 and args.configs and not chunked and not fwd_only and not getattr(rep, "deterministic", False):
        del rep
        torch.cuda.empty_cache()
        line["configs"] = run_other_configs(args, dev, local_rank, peaks)
    return line


def e2e_bound_ms(device_ms: float, h2d_bytes: float, d2h_bytes: float, h2d_gbs: float, d2h_gbs: float) -> float:
    """Lower bound on an end-to-end step whose copies overlap the kernels: the
    device step, or either direction's bytes at its measured link rate."""
    return max(device_ms, h2d_bytes / (h2d_gbs * 1e9) * 1e3, d2h_bytes / (d2h_gbs * 1e9) * 1e3)


def run_e2e(rep: Replica, args, total_flop: float, world: int, device_ms: float) -> dict:
    """Same step through the C ABI with host buffers: pinned host inputs copied in
    and every output copied back inside the timed region. As a user would run it,
    the copies overlap the kernels: one stream brings each shard's inputs in ahead
    of the compute stream, another copies each shard's outputs out while the next
    shard computes; events keep every buffer from being overwritten while in use."""
    dev = rep.dev
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
    h_doc = pin(rep.doc)
    h_k, h_v = pin(rep.k_full), pin(rep.v_full)
    h_in = [(pin(s["q"]), pin(s["do"])) for s in rep.shards]
    h_out = [{n: torch.empty(s[n].shape, dtype=s[n].dtype, pin_memory=True) for n in ("out", "lse", "dq", "dk", "dv")}
             for s in rep.shards]
    full_kv = all(s["k"].data_ptr() == rep.k_full.data_ptr() for s in rep.shards)
    h2d = h_doc.numel() * 4 + h_k.numel() * 2 + h_v.numel() * 2 + sum(a.numel() * 2 + b.numel() * 2 for a, b in h_in)
    d2h = sum(sum(t.numel() * t.element_size() for t in o.values()) for o in h_out)

    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = len(rep.shards)
    ev_in = [torch.cuda.Event() for _ in range(n)]    # shard i inputs (and the shared ones) landed
    ev_done = [torch.cuda.Event() for _ in range(n)]  # shard i computed: inputs free, outputs ready
    ev_out = [torch.cuda.Event() for _ in range(n)]   # shard i outputs copied out: outputs free
    state = {"first": True}

    def step():
        first = state["first"]
        with torch.cuda.stream(s_in):
            if not first:  # the previous step's last shard still reads doc / K / V
                s_in.wait_event(ev_done[n - 1])
            rep.doc.copy_(h_doc, non_blocking=True)
            rep.k_full.copy_(h_k, non_blocking=True)
            rep.v_full.copy_(h_v, non_blocking=True)
            for i, (s, (hq, hd)) in enumerate(zip(rep.shards, h_in)):
                if not first:
                    s_in.wait_event(ev_done[i])
                s["q"].copy_(hq, non_blocking=True)
                s["do"].copy_(hd, non_blocking=True)
                ev_in[i].record(s_in)
        for i, s in enumerate(rep.shards):
            comp.wait_event(ev_in[i])
            if not first:
                comp.wait_event(ev_out[i])
            if not full_kv:
                a = s["g"].kv_offset
                s["k"].copy_(rep.k_full[:, :, a:a + s["g"].S_kv])
                s["v"].copy_(rep.v_full[:, :, a:a + s["g"].S_kv])
            rep.run_shard(i)
            ev_done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                for name, t in h_out[i].items():
                    t.copy_(s[name], non_blocking=True)
                ev_out[i].record(s_out)
        state["first"] = False

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    steps = max(1, args.steps // 2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for _ in range(steps):
        step()
    comp.wait_event(ev_out[n - 1])  # the last read-back ends the timed region
    t1.record(comp)
    torch.cuda.synchronize()
    if int(rep.status.item()) != 0:
        raise RuntimeError(f"device status {int(rep.status.item()):#x} in the end-to-end run")
    ms = allreduce_max(t0.elapsed_time(t1) / steps, dev, world)
    # the host link on its own, after the timed region: the largest output copied
    # out and the largest input copied in, three times each
    def link_gbs(dst, src, stream):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)  # warm-up
            a.record(stream)
            for _ in range(3):
                dst.copy_(src, non_blocking=True)
            b.record(stream)
        torch.cuda.synchronize()
        return 3 * src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
    big = max(((h_out[i][nm], s[nm]) for i, s in enumerate(rep.shards) for nm in h_out[i]),
              key=lambda p: p[1].numel() * p[1].element_size())
    bw_d2h = link_gbs(big[0], big[1], s_out)
    bw_h2d = link_gbs(rep.k_full, h_k, s_in)
    bound = e2e_bound_ms(device_ms, h2d, d2h, bw_h2d, bw_d2h)
    return {"value": round(job_tflops(total_flop, ms, world), 2), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "copies": "pinned host buffers, overlapped with the kernels on two copy streams",
            "link_gbs": {"h2d": round(bw_h2d, 1), "d2h": round(bw_d2h, 1)},
            "bound_ms": round(bound, 3), "frac_of_bound": round(bound / ms, 4),
            "bound_note": "max of the device step and each direction's bytes over its measured link rate"}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(w: synth.Workload, seed: int, n_heads: int = 4, rank_index: int = 3):
    """fp64 oracle forward + backward on a bounded slice of the workload: batch row 0,
    the first `n_heads` query heads (whole GQA groups when n_heads >= Hq/Hkv), every
    local row of one shard."""
    import oracle
    doc = synth.doc_layout(w.layout, w.B, w.S, seed)
    plan = shard_plan(w, doc)
    sh = plan[min(rank_index, len(plan) - 1)]
    n_heads = max(1, min(n_heads, w.Hq))
    n_kv = 1 if n_heads <= w.G else -(-n_heads // w.G)
    if n_heads > w.G:
        n_heads = n_kv * w.G
    k, v = synth.kv_rows(w, seed, sh["kv_offset"], sh["kv_offset"] + sh["S_kv"])
    q = synth.q_shard(w, sh["r"], seed)[:1, :n_heads]
    do = synth.dout_shard(w, sh["r"], seed)[:1, :n_heads]
    g = oracle.geom(1, n_heads, n_kv, w.D, w.S, w.L, sh["row_offset"], sh["kv_offset"], sh["S_kv"], w.window)
    args = (q, k[:1, :n_kv], v[:1, :n_kv], do, doc[:1], g)
    flop = 14.0 * w.D * n_heads * pairs_closed_form(doc[:1], sh["row_offset"], w.L, w.window)
    desc = (f"{w.key} shard r={sh['r']}: batch row 0, query heads 0..{n_heads - 1} ({n_kv} kv groups), "
            f"all {w.L} local rows, fwd + full bwd (dq, dk, dv)")
    return args, flop, desc


def time_oracle(args_tuple):
    import oracle
    q, k, v, do, doc, g = args_tuple
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, doc, g)
    oracle.bwd(q, k, v, do, doc, g)
    return time.perf_counter() - t0


def cpu_cores() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    if n and n.isdigit():
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(w: synth.Workload, seed: int, n_heads: int) -> dict:
    args, flop, desc = oracle_sample(w, seed, n_heads=n_heads)
    secs = time_oracle(args)
    return {"value": round(flop / secs / 1e12, 6), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": desc, "seconds": round(secs, 2)}


def run_reference(args, rank: int, world: int):
    """The oracle as the reference arm: each step is a bounded sample of the workload
    on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.config]
    sample_args, flop, desc = oracle_sample(w, args.seed, n_heads=1)
    for _ in range(args.warmup):
        time_oracle(sample_args)
    secs = [time_oracle(sample_args) for _ in range(args.steps)]
    ms = 1e3 * sum(secs) / len(secs)
    value = flop / (ms * 1e-3) / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.key}: {w.title}", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "S": w.S,
                       "cp_size": w.cp_size, "L": w.L, "window": w.window, "kv": w.kv, "seed": args.seed},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="C2", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--grad-dtype", choices=("f32", "bf16"), default="f32")
    ap.add_argument("--shards", default=None, help="comma-separated cp ranks to run (default: all of the workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fwd-only", action="store_true",
                    help="segments and forward only")
    ap.add_argument("--deterministic", action="store_true",
                    help="bitwise reproducible backward (dq by a fixed-order pass instead of atomic additions)")
    ap.add_argument("--exchange", action="store_true",
                    help="time the sender side of the needed-only K/V exchange (plan, gather, index-add) instead")
    ap.add_argument("--kv-chunks", choices=("none", "ring", "ring-merge"), default="none",
                    help="ring: each shard's K/V in per-rank chunks, each chunk's forward merged in its epilogue, "
                         "backward per chunk; ring-merge: the same with the separate merge kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", action=argparse.BooleanOptionalAction, default=True,
                    help="also time C3, C4 (rank 15), C5w512 and G512 (a few steps each) into the line's "
                         "'configs' block (single GPU, default workload path only)")
    ap.add_argument("--cpu-heads", type=int, default=None,
                    help="query heads of batch row 0 in the oracle's timed CPU-baseline slice "
                         "(default: about 10-30 s of CPU work; 8 for head dim 512, else 32)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 must be launched with torchrun (one process per GPU)")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from sliding_window_attention_device_gb300 import build as _build
    _build.build()
    if args.exchange:
        if rank == 0:
            print(json.dumps(run_exchange(args, local_rank)), flush=True)
        return
    try:
        line = run_ours(args, rank, world, local_rank)
        if line is not None:
            if world == 1 and not args.no_cpu_baseline:
                wk = synth.WORKLOADS[args.config]
                heads = args.cpu_heads if args.cpu_heads is not None else (8 if wk.D >= 512 else 32)
                line["cpu_baseline"] = cpu_baseline(wk, args.seed, heads)
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
