"""Attention dropout on the GPU against the fp64 oracle, element by element.

blockdiag_cp.kernels `_cp_blockdiag_varlen` takes `dropout_p`, the chance that
an attention weight is dropped. Both sides draw the keep decision of every (query head,
query position, key position) pair from Philox-4x32-10 with the counter
(key / 8, query, head, batch row) and the seed, each from its own code; so
out, lse, dq, dk and dv must agree within the parity bar for the same p and
seed, as without dropout. The cases cover head dims 64 / 128 / 256 / 512, K/V
buffers that start at a position that is not a multiple of 8 (the decisions
follow global positions), windows, GQA groups of 1 to 4, both gradient dtypes,
the fixed-order (deterministic) backward, K/V in chunks (forwards merged in
the forward's epilogue, the per-chunk backward with the merged out / lse) at
head dims 64 to 512, and token-major K/V read in place.

Tolerance: the parity bar times the keep scale 2^16 / (2^16 - T). Every term
a dropout run adds is an undropped term times Z <= that scale, and the terms
the GPU rounds to bf16 before its tensor-core products (dS, for dK and dQ)
carry that factor, so their rounding errors do too: x1.11 at p = 0.1, x2 at
p = 0.5.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (MAX_ABS, MEAN_ABS, assert_close, assert_close_bf16, assert_lse, make_case, oracle_geom,
                     real_rows, run_gpu)
from sliding_window_attention_device_gb300 import bdattn, synth

pytestmark = pytest.mark.gpu


def W(key, B, Hq, Hkv, D, S, cp, layout, window=0, kv="full"):
    return synth.Workload(key, key, B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, cp_size=cp, layout=layout, window=window,
                          ranks=tuple(range(cp)), kv=kv)


CASES = [
    ("d128_g2", W("a", 2, 4, 2, 128, 1280, 4, ("uniform", 20, 300, 40)), 2),
    ("d128_g4_needed", W("b", 2, 8, 2, 128, 1536, 4, ("uniform", 37, 501, 0), kv="needed"), 3),
    ("d64_g1_window", W("c", 1, 3, 3, 64, 1024, 2, ("uniform", 50, 400, 70), window=100), 1),
    ("d256_g2_window", W("d", 1, 4, 2, 256, 1280, 4, ("uniform", 100, 600, 30), window=150, kv="prefix"), 3),
    ("d256_g1_needed", W("e", 2, 2, 2, 256, 1024, 4, ("uniform", 37, 501, 0), kv="needed"), 2),
    ("d512_g2_needed", W("k", 1, 4, 2, 512, 1024, 4, ("uniform", 37, 501, 0), kv="needed"), 3),
    ("d512_g1_window", W("l", 1, 2, 2, 512, 1024, 2, ("uniform", 40, 300, 10), window=90), 1),
]


def _case(w, r, p, seed):
    c = make_case(w, r, seed=r + 7)
    c["dropout_p"], c["drop_seed"] = p, seed
    return c


def _bar(p):
    """(max-abs, mean-abs) for dropout probability p: the parity bar times the
    keep scale."""
    t = int(np.floor(p * 65536 + 0.5))
    k = 65536.0 / (65536 - t)
    return MAX_ABS * k, MEAN_ABS * k


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("name,w,r", CASES, ids=[c[0] for c in CASES])
def test_dropout_fwd_bwd_parity(name, w, r, p):
    c = _case(w, r, p, seed=0x5EED_0000_0000_0000 + r)
    if w.kv == "needed":  # these cases start their K/V buffer off the 8-key grid of the draws
        assert c["kv_offset"] % 8 != 0, c["kv_offset"]
    g = oracle_geom(c)
    out, lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], g)
    dq, dk, dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], g)
    real = real_rows(c)
    mx, mn = _bar(p)
    for gd in (torch.float32, torch.bfloat16):
        res = run_gpu(c, grad_dtype=gd)
        assert res["status_word"] == 0, f"status {res['status_word']:#x}"
        assert_close(f"{name} p{p} out", res["out"], out, mx, mn)
        assert_lse(res["lse"], lse, real)
        close = assert_close if gd == torch.float32 else assert_close_bf16
        close(f"{name} p{p} dq {gd}", res["dq"], dq, mx, mn)
        close(f"{name} p{p} dk {gd}", res["dk"], dk, mx, mn)
        close(f"{name} p{p} dv {gd}", res["dv"], dv, mx, mn)


def test_dropout_changes_the_result_and_follows_the_seed():
    w = CASES[0][1]
    base = run_gpu(_case(w, 2, 0.0, 0))
    a = run_gpu(_case(w, 2, 0.5, 1))
    b = run_gpu(_case(w, 2, 0.5, 1))
    c = run_gpu(_case(w, 2, 0.5, 2))
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["dk"], b["dk"])
    assert not torch.equal(a["out"], c["out"])
    assert not torch.equal(a["out"], base["out"])
    assert torch.equal(a["lse"], base["lse"])  # the normaliser is the undropped softmax's


@pytest.mark.parametrize("name", ["d128_g4_needed", "d256_g2_window", "d512_g2_needed"])
def test_dropout_deterministic_backward(name):
    w, r = next((c[1], c[2]) for c in CASES if c[0] == name)
    c = _case(w, r, 0.3, 99)
    res = run_gpu(c)
    g = oracle_geom(c)
    dq, dk, dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], g)
    dev = torch.device("cuda")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    got = [bdattn.bd_attn_bwd_deterministic(do, q, k, v, res["out"], res["lse"], res["seg"], res["g"],
                                            res["status"]) for _ in range(2)]
    torch.cuda.synchronize()
    assert int(res["status"].item()) == 0
    for t0, t1 in zip(*got):
        assert torch.equal(t0, t1)  # bitwise reproducible
    mx, mn = _bar(0.3)
    assert_close(f"{name} det dq", got[0][0], dq, mx, mn)
    assert_close(f"{name} det dk", got[0][1], dk, mx, mn)
    assert_close(f"{name} det dv", got[0][2], dv, mx, mn)
    assert torch.equal(got[0][1], res["dk"]) and torch.equal(got[0][2], res["dv"])


@pytest.mark.parametrize("D", [128, 512])
def test_dropout_chunked_forward_merge(D):
    """K/V in three chunks, each merged into the running (out, lse) in the
    forward's epilogue, equals the oracle's one-piece dropout forward."""
    w = W("f", 1, 4, 2, D, 1536, 4, ("uniform", 40, 900, 20))
    r = 3
    c = _case(w, r, 0.25, 1234)
    g = oracle_geom(c)
    out_ref, lse_ref = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], g)
    dev = torch.device("cuda")
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q = c["q"].to(dev)
    status = bdattn.new_status(dev)
    out = torch.empty(w.B, w.Hq, w.L, w.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)
    cuts = (0, 301, 777, w.S)  # chunk starts off the 8-key grid
    for n in range(3):
        a, e = cuts[n], cuts[n + 1]
        gc = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, r * w.L, a, e - a, dropout_p=0.25, seed=1234)
        segc, _ = bdattn.bd_attn_seg_build_chunk(doc, gc, status=status)
        kc, vc = c["k"][:, :, a:e].contiguous().to(dev), c["v"][:, :, a:e].contiguous().to(dev)
        if n == 0:
            bdattn.bd_attn_fwd(q, kc, vc, segc, gc, status, out=out, lse=lse)
        else:
            bdattn.bd_attn_fwd_merge(q, kc, vc, segc, gc, status, out, lse)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close("chunked dropout out", out, out_ref, *_bar(0.25))
    assert_lse(lse, lse_ref, real_rows(c))


@pytest.mark.parametrize("D,window", [(64, 200), (128, 0), (256, 0), (512, 150)])
def test_dropout_chunked_backward(D, window):
    """The backward over K/V in three chunks (a ring step): per-chunk forwards
    merged in the forward's epilogue, prep once with the merged out, one
    backward main per chunk (dq accumulating, dk / dv per chunk), finalize --
    equals the oracle's one-piece dropout backward. The chunks start off the
    8-key grid of the draws, so each one's decisions come from global key
    positions."""
    w = W("g", 1, 4, 2, D, 1536, 4, ("uniform", 40, 900, 20), window=window)
    r, p, seed = 3, 0.2, 0xC0FFEE
    c = _case(w, r, p, seed)
    g_ref = oracle_geom(c)
    out_ref, lse_ref = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], g_ref)
    dq_ref, dk_ref, dv_ref = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], g_ref)
    dev = torch.device("cuda")
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, do = c["q"].to(dev), c["do"].to(dev)
    status = bdattn.new_status(dev)
    out = torch.empty(w.B, w.Hq, w.L, w.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)
    cuts = (0, 301, 777, w.S)
    chunks = []
    for n in range(3):
        a, e = cuts[n], cuts[n + 1]
        gc = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, r * w.L, a, e - a, window, dropout_p=p, seed=seed)
        segc, _ = bdattn.bd_attn_seg_build_chunk(doc, gc, status=status)
        kc, vc = c["k"][:, :, a:e].contiguous().to(dev), c["v"][:, :, a:e].contiguous().to(dev)
        if n == 0:
            bdattn.bd_attn_fwd(q, kc, vc, segc, gc, status, out=out, lse=lse)
        else:
            bdattn.bd_attn_fwd_merge(q, kc, vc, segc, gc, status, out, lse)
        chunks.append((gc, segc, kc, vc))
    g_full = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, r * w.L, 0, w.S, window, dropout_p=p, seed=seed)
    ws = torch.empty(bdattn.bwd_workspace_bytes(g_full), dtype=torch.uint8, device=dev)
    dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.float32, device=dev)
    bdattn.bd_attn_bwd_prep(do, out, g_full, status, ws)
    dks, dvs = [], []
    for gc, segc, kc, vc in chunks:
        dk = torch.full((w.B, w.Hkv, gc.S_kv, w.D), float("nan"), dtype=torch.float32, device=dev)
        dv = torch.full_like(dk, float("nan"))
        bdattn.bd_attn_bwd_main(do, q, kc, vc, lse, segc, gc, status, ws, dk, dv)
        dks.append(dk)
        dvs.append(dv)
    bdattn.bd_attn_bwd_finalize(g_full, status, ws, dq)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    mx, mn = _bar(p)
    assert_close(f"D{D} chunked dropout out", out, out_ref, mx, mn)
    assert_lse(lse, lse_ref, real_rows(c))
    assert_close(f"D{D} chunked dropout dq", dq, dq_ref, mx, mn)
    assert_close(f"D{D} chunked dropout dk", torch.cat(dks, dim=2), dk_ref, mx, mn)
    assert_close(f"D{D} chunked dropout dv", torch.cat(dvs, dim=2), dv_ref, mx, mn)


def _run_layout(c, layout):
    """Forward and backward with K/V (and dK / dV) in the given layout; the
    gradients come back head-major."""
    w, dev = c["w"], torch.device("cuda")
    g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], w.window,
                    kv_layout=layout, dropout_p=c["dropout_p"], seed=c["drop_seed"])
    tm = layout == bdattn.KV_SBHD
    to = (lambda t: t.permute(2, 0, 1, 3).contiguous()) if tm else (lambda t: t)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, do = c["q"].to(dev), c["do"].to(dev)
    k, v = to(c["k"]).to(dev), to(c["v"]).to(dev)
    seg, status = bdattn.bd_attn_seg_build(doc, g)
    out, lse = bdattn.bd_attn_fwd(q, k, v, seg, g, status)
    dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.float32, device=dev)
    dk = torch.full(bdattn.kv_shape(g), float("nan"), dtype=torch.float32, device=dev)
    dv = torch.full_like(dk, float("nan"))
    bdattn.bd_attn_bwd(do, q, k, v, out, lse, seg, g, status, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    back = (lambda t: t.permute(1, 2, 0, 3)) if tm else (lambda t: t)
    return dict(out=out.cpu(), lse=lse.cpu(), dq=dq.cpu(), dk=back(dk).cpu(), dv=back(dv).cpu())


@pytest.mark.parametrize("name", ["d128_g4_needed", "d256_g1_needed", "d512_g2_needed", "d64_g1_window"])
def test_dropout_token_major(name):
    """Token-major K/V (the receive buffer of the needed-only exchange, read in
    place) under dropout: out, lse, dk and dv bit-equal to the head-major run,
    and every output within the dropout bar of the oracle."""
    w, r = next((x[1], x[2]) for x in CASES if x[0] == name)
    c = _case(w, r, 0.3, 0xABCDEF0123)
    a = _run_layout(c, bdattn.KV_BHSD)
    t = _run_layout(c, bdattn.KV_SBHD)
    assert torch.equal(a["out"], t["out"]) and torch.equal(a["lse"], t["lse"])
    assert torch.equal(a["dk"], t["dk"]) and torch.equal(a["dv"], t["dv"])
    g = oracle_geom(c)
    out, lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], g)
    dq, dk, dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], g)
    mx, mn = _bar(0.3)
    assert_close(f"{name} token-major dropout out", t["out"], out, mx, mn)
    assert_lse(t["lse"], lse, real_rows(c))
    assert_close(f"{name} token-major dropout dq", t["dq"], dq, mx, mn)
    assert_close(f"{name} token-major dropout dk", t["dk"], dk, mx, mn)
    assert_close(f"{name} token-major dropout dv", t["dv"], dv, mx, mn)
