"""Token-major K/V (kv_layout = BD_KV_SBHD: k, v, dk, dv as [S_kv, B, Hkv, D],
the receive buffer of the needed-only all-to-all-v, blockdiag_cp.exchange
`_NeededKVExchange`) on the GPU:

  * the same inputs in either layout give the same out and lse bit for bit
    and the same dk / dv bit for bit (both are formed inside one CTA), and dq
    within the parity tolerance (its fp32 additions run in no fixed order),
    all against the oracle too;
  * the whole needed-only exchange emulated on one GPU: every source gathers
    its send buffer, each rank assembles its receive buffer (pieces in source
    order; torch.cat stands in for the collective) and runs attention on it in
    place, its dk / dv go back by the reverse split and are index-added at
    their sources -- the result equals the oracle's all-gather sum.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import LSE_ABS, assert_close, make_case, oracle_geom
from oracle import exchange as ox
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu

W_ = synth.Workload
CASES = [
    ("d128_g2_ragged", W_("ta", "token-major, D 128, ragged", B=2, Hq=4, Hkv=2, D=128, S=1280, cp_size=4,
                          layout=("uniform", 20, 300, 40)), 2),
    ("d64_window", W_("tb", "token-major, D 64, window 100", B=1, Hq=3, Hkv=3, D=64, S=1024, cp_size=2,
                      layout=("uniform", 50, 400, 70), window=100), 1),
    ("d256_window", W_("tc", "token-major, D 256, window 150", B=1, Hq=4, Hkv=2, D=256, S=1280, cp_size=4,
                       layout=("uniform", 100, 600, 30), window=150, kv="prefix"), 3),
]


def _run(c, layout, grad_dtype=torch.float32):
    from sliding_window_attention_device_gb300 import bdattn
    w, dev = c["w"], torch.device("cuda")
    g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], w.window,
                    kv_layout=layout)
    tm = layout == bdattn.KV_SBHD
    to = (lambda t: t.permute(2, 0, 1, 3).contiguous()) if tm else (lambda t: t)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, do = c["q"].to(dev), c["do"].to(dev)
    k, v = to(c["k"]).to(dev), to(c["v"]).to(dev)
    seg, status = bdattn.bd_attn_seg_build(doc, g)
    out = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.B, w.Hq, w.L), float("nan"), dtype=torch.float32, device=dev)
    bdattn.bd_attn_fwd(q, k, v, seg, g, status, out=out, lse=lse)
    dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=grad_dtype, device=dev)
    dk = torch.full(bdattn.kv_shape(g), float("nan"), dtype=grad_dtype, device=dev)
    dv = torch.full_like(dk, float("nan"))
    bdattn.bd_attn_bwd(do, q, k, v, out, lse, seg, g, status, grad_dtype=grad_dtype, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    back = (lambda t: t.permute(1, 2, 0, 3)) if tm else (lambda t: t)
    return dict(out=out.cpu(), lse=lse.cpu(), dq=dq.cpu(), dk=back(dk).cpu(), dv=back(dv).cpu())


@pytest.mark.parametrize("name,w,r", CASES, ids=[x[0] for x in CASES])
def test_token_major_matches_head_major(name, w, r):
    from sliding_window_attention_device_gb300 import bdattn
    c = make_case(w, r)
    a = _run(c, bdattn.KV_BHSD)
    t = _run(c, bdattn.KV_SBHD)
    assert torch.equal(a["out"], t["out"]) and torch.equal(a["lse"], t["lse"])
    assert torch.equal(a["dk"], t["dk"]) and torch.equal(a["dv"], t["dv"])
    ref_dq, ref_dk, ref_dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], oracle_geom(c))
    assert_close(f"{name} token-major dq", t["dq"], ref_dq)
    assert_close(f"{name} token-major dk", t["dk"], ref_dk)
    assert_close(f"{name} token-major dv", t["dv"], ref_dv)
    ref_out, ref_lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], oracle_geom(c))
    assert_close(f"{name} token-major out", t["out"], ref_out)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(t["lse"].numpy()), fin)
    assert np.abs(t["lse"].double().numpy()[fin] - ref_lse[fin]).max(initial=0.0) <= LSE_ABS


def test_token_major_bf16_gradients():
    from sliding_window_attention_device_gb300 import bdattn
    c = make_case(CASES[0][1], CASES[0][2])
    a = _run(c, bdattn.KV_BHSD, torch.bfloat16)
    t = _run(c, bdattn.KV_SBHD, torch.bfloat16)
    assert torch.equal(a["dk"], t["dk"]) and torch.equal(a["dv"], t["dv"])
    assert torch.isfinite(t["dq"].float()).all()


def test_needed_only_exchange_end_to_end():
    """Every rank attends its needed range delivered by the emulated
    all-to-all-v, read in place token-major; dk / dv return to their sources
    and are index-added: the per-rank out / dq and the summed dk / dv equal the
    oracle run on the full sequence (the all-gather path, reduce-scatter sum)."""
    from sliding_window_attention_device_gb300 import bdattn
    w = W_("te", "needed-only exchange, 4 ranks", B=2, Hq=4, Hkv=2, D=128, S=1024, cp_size=4,
           layout=("uniform", 100, 700, 30))
    dev = torch.device("cuda")
    W, L = w.cp_size, w.L
    doc_np = synth.doc_layout(w.layout, w.B, w.S, 0)
    p = ox.plan(doc_np, W)
    assert not p["use_halo"]  # a document spans more than two ranks: the general exchange
    doc = torch.from_numpy(doc_np).to(dev)
    k_full, v_full = synth.kv_rows(w, 0)
    kd, vd = k_full.to(dev), v_full.to(dev)
    status = bdattn.new_status(dev)
    plans = [bdattn.bd_attn_exchange_plan(doc, W, r, status=status)[0] for r in range(W)]
    sends = []
    for s in range(W):
        sk = torch.empty((W * L, w.B, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
        sv = torch.empty_like(sk)
        bdattn.bd_attn_needed_gather(kd[:, :, s * L:(s + 1) * L].contiguous(), plans[s], sk, status)
        bdattn.bd_attn_needed_gather(vd[:, :, s * L:(s + 1) * L].contiguous(), plans[s], sv, status)
        sends.append((sk, sv))
    send_off = [[sum(p["counts"][s][:r]) for r in range(W)] for s in range(W)]
    back_k = [[None] * W for _ in range(W)]  # back_k[s][r]: rank r's dk rows for source s's tokens
    back_v = [[None] * W for _ in range(W)]
    ref_dk = np.zeros((w.B, w.Hkv, w.S, w.D))
    ref_dv = np.zeros_like(ref_dk)
    for r in range(W):
        lo, hi = p["s_first"][r], p["real_end"][r]
        pieces = [(s, send_off[s][r], p["counts"][s][r]) for s in range(W)]
        rk = torch.cat([sends[s][0][o:o + n] for s, o, n in pieces])  # the receive buffer, token-major
        rv = torch.cat([sends[s][1][o:o + n] for s, o, n in pieces])
        assert rk.shape[0] == hi - lo and torch.equal(rk, kd[:, :, lo:hi].permute(2, 0, 1, 3))
        g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, lo, hi - lo, 0, kv_layout=bdattn.KV_SBHD)
        seg, _ = bdattn.bd_attn_seg_build(doc, g, status=status)
        q = synth.q_shard(w, r, 0).to(dev)
        do = synth.dout_shard(w, r, 0).to(dev)
        out, lse = bdattn.bd_attn_fwd(q, rk, rv, seg, g, status)
        dq, dk, dv = bdattn.bd_attn_bwd(do, q, rk, rv, out, lse, seg, g, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        og = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, L, r * L, 0, w.S, 0)
        q_c, do_c = synth.q_shard(w, r, 0), synth.dout_shard(w, r, 0)
        ref_out, _ = oracle.fwd(q_c, k_full, v_full, doc_np, og)
        rdq, rdk, rdv = oracle.bwd(q_c, k_full, v_full, do_c, doc_np, og)
        assert_close(f"rank {r} out", out, ref_out)
        assert_close(f"rank {r} dq", dq, rdq)
        ref_dk += rdk
        ref_dv += rdv
        off = 0
        for s, _, n in pieces:  # the reverse split: each source's rows, in source order
            back_k[s][r] = dk[off:off + n]
            back_v[s][r] = dv[off:off + n]
            off += n
    got_dk, got_dv = [], []
    for s in range(W):
        gk = torch.zeros((W * L, w.B, w.Hkv, w.D), dtype=torch.float32, device=dev)
        gv = torch.zeros_like(gk)
        n = sum(p["counts"][s])
        gk[:n] = torch.cat([back_k[s][r] for r in range(W)])  # destinations in order: the send layout
        gv[:n] = torch.cat([back_v[s][r] for r in range(W)])
        lk = torch.full((w.B, w.Hkv, L, w.D), float("nan"), dtype=torch.float32, device=dev)
        lv = torch.full_like(lk, float("nan"))
        bdattn.bd_attn_needed_scatter_add(gk, plans[s], lk, status)
        bdattn.bd_attn_needed_scatter_add(gv, plans[s], lv, status)
        got_dk.append(lk)
        got_dv.append(lv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close("exchanged dk", torch.cat(got_dk, dim=2), ref_dk)
    assert_close("exchanged dv", torch.cat(got_dv, dim=2), ref_dv)
