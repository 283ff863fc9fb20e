"""Shared helpers for the parity tests: seeded cases, the GPU path through the
C ABI, and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sliding_window_attention_device_gb300 import synth

MAX_ABS = 2e-2      # out / dq / dk / dv vs the fp64 oracle (bf16 inputs, fp32 accumulation)
MEAN_ABS = 2e-3
LSE_ABS = 1e-3      # lse on real rows


def needed_kv(doc: np.ndarray, w: synth.Workload, r: int) -> tuple[int, int]:
    """[min_b s_first, max_b real_end) from the oracle's segmentation."""
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, r * w.L, 0, w.S, w.window)
    segs = oracle.segments(doc, g)
    lo = min(s["s_first"] for s in segs)
    hi = max(s["real_end"] for s in segs)
    if hi <= lo:
        return r * w.L, 1
    return lo, hi - lo


def make_case(w: synth.Workload, r: int, seed: int = 0, kv: tuple[int, int] | None = None) -> dict:
    doc = synth.doc_layout(w.layout, w.B, w.S, seed)
    if kv is None:
        kv = needed_kv(doc, w, r) if w.kv == "needed" else w.prefix_kv(r)
    kv_offset, S_kv = kv
    k, v = synth.kv_rows(w, seed, kv_offset, kv_offset + S_kv)
    return dict(w=w, r=r, doc=doc, q=synth.q_shard(w, r, seed), k=k, v=v, do=synth.dout_shard(w, r, seed),
                row_offset=r * w.L, kv_offset=kv_offset, S_kv=S_kv, window=w.window)


def oracle_geom(c: dict):
    w = c["w"]
    return oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], c["window"],
                       dropout_p=c.get("dropout_p", 0.0), seed=c.get("drop_seed", 0))


def gpu_geom(c: dict):
    from sliding_window_attention_device_gb300 import bdattn
    w = c["w"]
    return bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], c["window"],
                       dropout_p=c.get("dropout_p", 0.0), seed=c.get("drop_seed", 0))


def run_gpu(c: dict, grad_dtype=torch.float32, bwd: bool = True) -> dict:
    from sliding_window_attention_device_gb300 import bdattn
    dev = torch.device("cuda")
    g = gpu_geom(c)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    seg, status = bdattn.bd_attn_seg_build(doc, g)
    w = c["w"]
    out = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.B, w.Hq, w.L), float("nan"), dtype=torch.float32, device=dev)
    out, lse = bdattn.bd_attn_fwd(q, k, v, seg, g, status, out=out, lse=lse)
    res = dict(g=g, seg=seg, status=status, out=out, lse=lse)
    if bwd:
        # NaN-filled outputs: an element the kernels leave unwritten fails the finiteness checks
        dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=grad_dtype, device=dev)
        dk = torch.full((w.B, w.Hkv, c["S_kv"], w.D), float("nan"), dtype=grad_dtype, device=dev)
        dv = torch.full_like(dk, float("nan"))
        dq, dk, dv = bdattn.bd_attn_bwd(do, q, k, v, out, lse, seg, g, status, grad_dtype=grad_dtype,
                                        dq=dq, dk=dk, dv=dv)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    res["status_word"] = int(status.item())
    return res


def assert_close(name: str, got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    d = np.abs(got - ref)
    mx, mn = float(d.max(initial=0.0)), float(d.mean()) if d.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, f"{name}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    return mx, mn


def assert_lse(got, ref, real_mask):
    got = got.detach().double().cpu().numpy()
    assert np.isneginf(got[~real_mask]).all(), "lse must be -inf on padding rows"
    d = np.abs(got[real_mask] - ref[real_mask])
    assert np.isfinite(got[real_mask]).all()
    assert d.max(initial=0.0) <= LSE_ABS, f"lse max-abs {d.max():.3e}"


def real_rows(c: dict) -> np.ndarray:
    """[B, Hq, L] bool: the query row is a real (non-padding) token."""
    w = c["w"]
    ro = c["row_offset"]
    r = c["doc"][:, ro:ro + w.L] != 0
    return np.repeat(r[:, None, :], w.Hq, axis=1)


# bf16 gradients: the fp32 result rounded once to bf16 (relative error <= 2^-8,
# half a unit in the last of bf16's 8 significant bits) on top of the fp32
# accumulation error the parity bar already covers
BF16_REL = 2.0 ** -8


def assert_close_bf16(name: str, got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, rel=BF16_REL):
    """Element-wise |got - ref| <= max_abs + rel |ref|; mean-abs over the whole
    tensor <= mean_abs + rel mean |ref|."""
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    d = np.abs(got - ref)
    bound = max_abs + rel * np.abs(ref)
    worst = int(np.argmax(d - bound)) if d.size else 0
    assert (d <= bound).all(), (f"{name}: |err| {d.flat[worst]:.3e} > {bound.flat[worst]:.3e} "
                                f"at {np.unravel_index(worst, d.shape)} (ref {ref.flat[worst]:.4f})")
    if d.size:
        assert d.mean() <= mean_abs + rel * np.abs(ref).mean(), f"{name}: mean-abs {d.mean():.3e}"
    return float(d.max(initial=0.0)), float(d.mean()) if d.size else 0.0
