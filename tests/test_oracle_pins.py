"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a fact the pages or the mathematics fix:
the hand-worked segmentation example, per-document unsharded causal attention
computed by torch's own SDPA (fp64) and autograd, central finite differences,
closed forms, and the invariants the pages state (CP == non-CP, dK/dV summed
over ranks, needed range == full range, window >= S == causal).
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sliding_window_attention_device_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _runs(row):
    """(start, end, id) of each maximal run of equal ids."""
    out, s = [], 0
    for p in range(1, len(row) + 1):
        if p == len(row) or row[p] != row[s]:
            out.append((s, p, int(row[s])))
            s = p
    return out


def _tiny(layout=("explicit", (10, 20, 5, 21), 8), B=1, Hq=4, Hkv=2, D=8, S=64, cp=4, window=0, seed=0):
    w = synth.Workload("T", "tiny", B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, cp_size=cp, layout=layout, window=window)
    doc = synth.doc_layout(layout, B, S, seed)
    k, v = synth.kv_rows(w, seed)
    qs = [synth.q_shard(w, r, seed) for r in range(cp)]
    ds = [synth.dout_shard(w, r, seed) for r in range(cp)]
    return w, doc, torch.cat(qs, 2), k, v, torch.cat(ds, 2)


def _per_doc_reference(w, doc, q_full, k, v, dout_full, window=0):
    """Unsharded per-document causal attention with torch SDPA (fp64) and autograd.
    Returns out, lse over all S rows plus dq over all rows and dk, dv (fp64)."""
    G = w.Hq // w.Hkv
    out = torch.zeros(w.B, w.Hq, w.S, w.D, dtype=torch.float64)
    lse = torch.full((w.B, w.Hq, w.S), float("-inf"), dtype=torch.float64)
    dq = torch.zeros_like(out)
    dk = torch.zeros(w.B, w.Hkv, w.S, w.D, dtype=torch.float64)
    dv = torch.zeros_like(dk)
    scale = w.D ** -0.5
    for b in range(w.B):
        for (a, e, did) in _runs(doc[b]):
            if did == 0:
                continue
            n = e - a
            qq = q_full[b:b + 1, :, a:e].double().clone().requires_grad_(True)
            kk = k[b:b + 1, :, a:e].double().repeat_interleave(G, dim=1).clone().requires_grad_(True)
            vv = v[b:b + 1, :, a:e].double().repeat_interleave(G, dim=1).clone().requires_grad_(True)
            if window > 0:
                ones = torch.ones(n, n, dtype=torch.bool)
                band = torch.tril(ones) & torch.triu(ones, diagonal=-(window - 1))
                o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=band, scale=scale)
                sc = torch.where(band, (qq @ kk.transpose(-1, -2)) * scale, float("-inf"))
            else:
                o = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
                causal = torch.tril(torch.ones(n, n, dtype=torch.bool))
                sc = torch.where(causal, (qq @ kk.transpose(-1, -2)) * scale, float("-inf"))
            (o * dout_full[b:b + 1, :, a:e].double()).sum().backward()
            out[b, :, a:e] = o[0].detach()
            lse[b, :, a:e] = torch.logsumexp(sc, dim=-1)[0].detach()
            dq[b, :, a:e] = qq.grad[0]
            dk[b, :, a:e] = kk.grad[0].view(w.Hkv, G, n, w.D).sum(1)
            dv[b, :, a:e] = vv.grad[0].view(w.Hkv, G, n, w.D).sum(1)
    return out, lse, dq, dk, dv


# --------------------------------------------------------------------------- segmentation


def test_worked_example_segments():
    gold = json.load(open(os.path.join(GOLDEN, "worked_example_c1.json")))
    lay = gold["layout"]
    doc = synth.doc_layout(("explicit", tuple(lay["lengths"]), lay["pad"]), 1, lay["S"])
    L = lay["L"]
    for r, exp in gold["ranks"].items():
        r = int(r)
        g = oracle.geom(1, 2, 1, 64, lay["S"], L, r * L, 0, lay["S"])
        seg = oracle.segments(doc, g)[0]
        for key in ("n_real", "n_seg", "s_first", "real_end", "max_q", "max_k", "first_q", "first_k", "max_tail"):
            assert seg[key] == exp[key], (r, key, seg[key], exp[key])
        assert seg["cu_q"].tolist() == exp["cu_q"]
        assert seg["cu_k"].tolist() == exp["cu_k"]
        assert seg["layout_error"] == 0 and seg["kv_range_error"] == 0
        assert oracle.pairs(doc, g) == exp["pairs"]


def _random_layouts():
    cases = []
    for seed in range(6):
        cases.append((("uniform", 3, 40, 12), 2, 160, seed))
    cases.append((("single",), 1, 160, 0))
    cases.append((("explicit", (1, 1, 1, 50, 1, 70, 4), 32), 1, 160, 0))
    return cases


@pytest.mark.parametrize("layout,B,S,seed", _random_layouts())
def test_segments_reconstruct_dense_mask(layout, B, S, seed):
    """Bottom-right causal segments reproduce the page's dense mask on real rows, and
    only the first local segment can have more keys than queries."""
    doc = synth.doc_layout(layout, B, S, seed)
    cp = 4
    L = S // cp
    for r in range(cp):
        g = oracle.geom(B, 1, 1, 8, S, L, r * L, 0, S)
        segs = oracle.segments(doc, g)
        m = oracle.mask(doc, g)
        for b in range(B):
            seg = segs[b]
            n_real = seg["n_real"]
            # real rows are a prefix; padding rows keep only their self-edge
            for i in range(n_real, L):
                row = m[b, i]
                assert row.sum() == 1 and row[r * L + i]
            rebuilt = np.zeros((L, S), dtype=bool)
            for kk in range(seg["n_seg"]):
                q0, q1 = seg["cu_q"][kk], seg["cu_q"][kk + 1]
                k0 = seg["s_first"] + seg["cu_k"][kk]
                k1 = seg["s_first"] + seg["cu_k"][kk + 1]
                sq, sk = q1 - q0, k1 - k0
                assert sk >= sq
                if kk > 0:
                    assert sk == sq
                for a in range(sq):
                    for c in range(sk):
                        if c <= a + (sk - sq):  # bottom-right aligned causal
                            rebuilt[q0 + a, k0 + c] = True
            assert (rebuilt[:n_real] == m[b, :n_real]).all()
            assert seg["real_end"] == r * L + n_real


def test_segment_errors_fire():
    S, L = 64, 16
    good = np.array([[1] * 20 + [2] * 30 + [0] * 14], dtype=np.int32)
    g = oracle.geom(1, 1, 1, 8, S, L, 16, 0, S)
    s = oracle.segments(good, g)[0]
    assert s["layout_error"] == 0 and s["kv_range_error"] == 0
    bad = good.copy()
    bad[0, 60] = 3  # a document after padding
    assert oracle.segments(bad, g)[0]["layout_error"] == 1
    reuse = np.array([[1] * 10 + [2] * 10 + [1] * 30 + [0] * 14], dtype=np.int32)  # id 1 in two runs
    g2 = oracle.geom(1, 1, 1, 8, S, L, 32, 0, S)
    assert oracle.segments(reuse, g2)[0]["layout_error"] == 1
    neg = good.copy()
    neg[0, 3] = -1
    assert oracle.segments(neg, g)[0]["layout_error"] == 1
    # the K/V buffer must cover [s_first, real_end)
    g3 = oracle.geom(1, 1, 1, 8, S, L, 16, 4, 40)
    assert oracle.segments(good, g3)[0]["kv_range_error"] == 1
    g4 = oracle.geom(1, 1, 1, 8, S, L, 16, 0, 31)
    assert oracle.segments(good, g4)[0]["kv_range_error"] == 1
    # a window narrows the needed range: rows 16..31 with W=4 need keys from 13
    g5 = oracle.geom(1, 1, 1, 8, S, L, 16, 13, 19, window=4)
    s5 = oracle.segments(good, g5)[0]
    assert s5["kv_need_lo"] == 13 and s5["kv_range_error"] == 0
    # all-padding shard
    g6 = oracle.geom(1, 1, 1, 8, S, L, 48, 0, S)
    s6 = oracle.segments(good, g6)[0]
    assert s6["n_real"] == 2 and s6["n_seg"] == 1
    allpad = np.array([[1] * 20 + [0] * 44], dtype=np.int32)
    s7 = oracle.segments(allpad, g6)[0]
    assert s7["n_real"] == 0 and s7["n_seg"] == 0 and s7["s_first"] == 48 and s7["real_end"] == 48
    assert s7["kv_range_error"] == 0


# --------------------------------------------------------------------------- forward / backward


@pytest.mark.parametrize("window", [0, 7])
def test_fwd_bwd_match_per_document_sdpa(window):
    """CP shard results == unsharded per-document causal attention (torch fp64 SDPA +
    autograd), restricted to the shard's rows; dK/dV summed over the GQA group and
    over the ranks' contributions."""
    w, doc, q_full, k, v, dout_full = _tiny(window=window)
    out_ref, lse_ref, dq_ref, dk_ref, dv_ref = _per_doc_reference(w, doc, q_full, k, v, dout_full, window)
    L = w.L
    dk_sum = np.zeros((w.B, w.Hkv, w.S, w.D))
    dv_sum = np.zeros_like(dk_sum)
    for r in range(w.cp_size):
        g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, window)
        q = q_full[:, :, r * L:(r + 1) * L]
        do = dout_full[:, :, r * L:(r + 1) * L]
        out, lse = oracle.fwd(q, k, v, doc, g)
        real = torch.from_numpy(doc[:, r * L:(r + 1) * L] != 0)[:, None, :].expand(w.B, w.Hq, L)
        o_ref = out_ref[:, :, r * L:(r + 1) * L]
        np.testing.assert_allclose(out, torch.where(real[..., None], o_ref, 0).numpy(), atol=1e-12, rtol=0)
        l_ref = lse_ref[:, :, r * L:(r + 1) * L]
        assert np.isneginf(lse[~real.numpy()]).all()
        np.testing.assert_allclose(lse[real.numpy()], l_ref[real].numpy(), atol=1e-12, rtol=0)
        dq, dk, dv = oracle.bwd(q, k, v, do, doc, g)
        np.testing.assert_allclose(dq, torch.where(real[..., None], dq_ref[:, :, r * L:(r + 1) * L], 0).numpy(),
                                   atol=1e-11, rtol=0)
        dk_sum += dk
        dv_sum += dv
    # dK/dV: the reduce-scatter(SUM) semantics of the all-gather exchange
    np.testing.assert_allclose(dk_sum, dk_ref.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv_sum, dv_ref.numpy(), atol=1e-11, rtol=0)


def test_fwd_equals_dense_mask_softmax():
    """The oracle's per-row predicate equals mask + softmax with the page's dense mask
    (numpy softmax over the materialised [B,1,L,S] mask) on real rows."""
    w, doc, q_full, k, v, _ = _tiny(layout=("uniform", 3, 30, 6), B=2, S=96, cp=3, seed=3)
    L = w.L
    for r in range(w.cp_size):
        g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S)
        q = q_full[:, :, r * L:(r + 1) * L]
        out, _ = oracle.fwd(q, k, v, doc, g)
        m = oracle.mask(doc, g)
        G = w.Hq // w.Hkv
        kr = k.double().numpy().repeat(G, axis=1)
        vr = v.double().numpy().repeat(G, axis=1)
        sc = np.einsum("bhid,bhjd->bhij", q.double().numpy(), kr) * w.D ** -0.5
        sc = np.where(m[:, None], sc, -np.inf)
        p = np.exp(sc - sc.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        dense = np.einsum("bhij,bhjd->bhid", p, vr)
        real = (doc[:, r * L:(r + 1) * L] != 0)[:, None, :, None]
        np.testing.assert_allclose(out, np.where(real, dense, 0.0), atol=1e-12, rtol=0)


def test_finite_differences():
    """Analytic backward == central differences of sum(out * dout) (fp64, h = 1e-6)."""
    w = synth.Workload("T", "fd", B=1, Hq=2, Hkv=1, D=4, S=16, cp_size=2, layout=("explicit", (5, 7), 4), window=3)
    doc = synth.doc_layout(w.layout, 1, 16)
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 8, 4))
    k = rng.standard_normal((1, 1, 16, 4))
    v = rng.standard_normal((1, 1, 16, 4))
    do = rng.standard_normal((1, 2, 8, 4))
    g = oracle.geom(1, 2, 1, 4, 16, 8, 8, 0, 16, window=3)

    def loss(qq, kk, vv):
        out, _ = oracle.fwd(qq, kk, vv, doc, g)
        return float((out * do).sum())

    dq, dk, dv = oracle.bwd(q, k, v, do, doc, g)
    h = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = plus
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = minus
            lm = loss(args["q"], args["k"], args["v"])
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_closed_forms():
    """First row of a document: out = v_start, lse = scale q.k; a length-1 document has
    dq = 0; W = 1 gives out_p = v_p; padding rows give 0 / -inf / 0."""
    w, doc, q_full, k, v, dout_full = _tiny(layout=("explicit", (1, 9, 14, 1, 7), 0), S=32, cp=2)
    L = w.L
    scale = w.D ** -0.5
    G = w.Hq // w.Hkv
    for r in range(2):
        g = oracle.geom(1, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S)
        q = q_full[:, :, r * L:(r + 1) * L]
        out, lse = oracle.fwd(q, k, v, doc, g)
        dq, _, _ = oracle.bwd(q, k, v, dout_full[:, :, r * L:(r + 1) * L], doc, g)
        for (a, e, did) in _runs(doc[0]):
            if not (r * L <= a < (r + 1) * L):
                continue
            i = a - r * L
            for h in range(w.Hq):
                np.testing.assert_array_equal(out[0, h, i], v[0, h // G, a].double().numpy())
                exp_lse = scale * float((q[0, h, i].double() * k[0, h // G, a].double()).sum())
                assert abs(lse[0, h, i] - exp_lse) < 1e-12
                if e - a == 1:
                    assert np.abs(dq[0, h, i]).max() == 0.0
        g1 = oracle.geom(1, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, window=1)
        out1, _ = oracle.fwd(q, k, v, doc, g1)
        for i in range(L):
            for h in range(w.Hq):
                np.testing.assert_array_equal(out1[0, h, i], v[0, h // G, r * L + i].double().numpy())
    # padding rows
    w2, doc2, q2, k2, v2, d2 = _tiny()
    g2 = oracle.geom(1, w2.Hq, w2.Hkv, w2.D, w2.S, w2.L, 3 * w2.L, 0, w2.S)
    out, lse = oracle.fwd(q2[:, :, 48:], k2, v2, doc2, g2)
    dq, _, _ = oracle.bwd(q2[:, :, 48:], k2, v2, d2[:, :, 48:], doc2, g2)
    pad = doc2[0, 48:] == 0
    assert pad.sum() == 8
    assert (out[0][:, pad] == 0).all() and np.isneginf(lse[0][:, pad]).all() and (dq[0][:, pad] == 0).all()


def test_window_at_least_S_is_causal_and_needed_range_equals_full():
    w, doc, q_full, k, v, dout_full = _tiny(layout=("uniform", 4, 30, 5), B=2, S=96, cp=3, seed=5)
    L = w.L
    for r in range(w.cp_size):
        q = q_full[:, :, r * L:(r + 1) * L]
        do = dout_full[:, :, r * L:(r + 1) * L]
        g0 = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, 0)
        gW = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, w.S)
        o0, l0 = oracle.fwd(q, k, v, doc, g0)
        oW, lW = oracle.fwd(q, k, v, doc, gW)
        np.testing.assert_array_equal(o0, oW)
        np.testing.assert_array_equal(l0, lW)
        r0 = oracle.bwd(q, k, v, do, doc, g0)
        rW = oracle.bwd(q, k, v, do, doc, gW)
        for a, b in zip(r0, rW):
            np.testing.assert_array_equal(a, b)
        # needed range [min s_first, max real_end)
        segs = oracle.segments(doc, g0)
        lo = min(s["s_first"] for s in segs)
        hi = max(s["real_end"] for s in segs)
        if hi <= lo:
            continue
        gN = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, lo, hi - lo, 0)
        assert all(s["kv_range_error"] == 0 for s in oracle.segments(doc, gN))
        oN, lN = oracle.fwd(q, k[:, :, lo:hi], v[:, :, lo:hi], doc, gN)
        np.testing.assert_allclose(oN, o0, atol=1e-13, rtol=0)
        dqN, dkN, dvN = oracle.bwd(q, k[:, :, lo:hi], v[:, :, lo:hi], do, doc, gN)
        np.testing.assert_allclose(dqN, r0[0], atol=1e-13, rtol=0)
        np.testing.assert_allclose(dkN, r0[1][:, :, lo:hi], atol=1e-13, rtol=0)
        assert np.abs(r0[1][:, :, :lo]).max(initial=0) == 0 and np.abs(r0[1][:, :, hi:]).max(initial=0) == 0
        np.testing.assert_allclose(dvN, r0[2][:, :, lo:hi], atol=1e-13, rtol=0)


def test_no_fully_masked_real_row():
    w, doc, q_full, k, v, _ = _tiny(layout=("uniform", 1, 12, 9), B=2, S=96, cp=4, seed=11, window=2)
    L = w.L
    for r in range(w.cp_size):
        g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, 2)
        _, lse = oracle.fwd(q_full[:, :, r * L:(r + 1) * L], k, v, doc, g)
        real = (doc[:, r * L:(r + 1) * L] != 0)[:, None, :].repeat(w.Hq, 1)
        assert np.isfinite(lse[real]).all()
        assert np.isneginf(lse[~real]).all()


def test_sampled_rows_and_keys_match_full():
    w, doc, q_full, k, v, dout_full = _tiny(layout=("uniform", 3, 25, 7), B=2, S=96, cp=3, seed=2)
    L = w.L
    r = 1
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S)
    q = q_full[:, :, r * L:(r + 1) * L]
    do = dout_full[:, :, r * L:(r + 1) * L]
    out, lse = oracle.fwd(q, k, v, doc, g)
    dq, dk, dv = oracle.bwd(q, k, v, do, doc, g)
    rows = [(1, 3, 5), (0, 0, 31), (1, 2, 17)]
    keys = [(0, 1, 40), (1, 0, 63), (1, 1, 2)]
    o_s, l_s = oracle.fwd(q, k, v, doc, g, rows=rows)
    dq_s, dk_s, dv_s = oracle.bwd(q, k, v, do, doc, g, rows=rows, keys=keys)
    for t, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o_s[t], out[b, h, i])
        assert l_s[t] == lse[b, h, i]
        np.testing.assert_allclose(dq_s[t], dq[b, h, i], atol=1e-14, rtol=0)
    for t, (b, hk, j) in enumerate(keys):
        np.testing.assert_allclose(dk_s[t], dk[b, hk, j], atol=1e-14, rtol=0)
        np.testing.assert_allclose(dv_s[t], dv[b, hk, j], atol=1e-14, rtol=0)
