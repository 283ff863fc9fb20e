"""Head dim 512 (the Gemma4 global layers: gemma4_moe.cp_attention, D = 512
full-attention layers, `_ffpa_varlen_forward_chunk` / `_ffpa_varlen_backward_chunk`)
on the GPU against the oracle:

  * the split-D forward (Q resident, K streamed in 64-column chunks, O in two
    256-column passes) through bd_attn_fwd;
  * the backward through bd_attn_bwd (dK / dV / dQ columns split over four
    CTAs per K/V tile, S and dP formed in each): fp32 and bf16 gradients;
  * several q tiles with a ragged tail, GQA, a window, token-major K/V, and
    sampled rows / keys of the full-size workload.
  * the bitwise reproducible backward (two-half fixed-order dq pass).
(Chunked K/V with merges at D = 512 is covered with the other head dims in
the chunked-path tests.)"""
import numpy as np
import pytest
import torch

import oracle
from helpers import LSE_ABS, assert_close, make_case, oracle_geom, real_rows
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu

W_ = synth.Workload
CASES = [
    ("g2_ragged", W_("ga", "D 512, GQA 2, ragged", B=2, Hq=4, Hkv=2, D=512, S=1280, cp_size=4,
                     layout=("uniform", 20, 500, 40)), 2, 0),
    ("g1_window", W_("gb", "D 512, window 200", B=1, Hq=2, Hkv=2, D=512, S=1024, cp_size=2,
                     layout=("uniform", 100, 900, 30), window=200), 1, 0),
    ("g4_token_major", W_("gc", "D 512, GQA 4, token-major", B=1, Hq=4, Hkv=1, D=512, S=768, cp_size=3,
                          layout=("uniform", 64, 700, 10), kv="prefix"), 2, 1),
]


def _fwd(c, layout):
    from sliding_window_attention_device_gb300 import bdattn
    w, dev = c["w"], torch.device("cuda")
    g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], w.window,
                    kv_layout=layout)
    to = (lambda t: t.permute(2, 0, 1, 3).contiguous()) if layout else (lambda t: t)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, k, v = c["q"].to(dev), to(c["k"]).to(dev), to(c["v"]).to(dev)
    seg, status = bdattn.bd_attn_seg_build(doc, g)
    out = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.B, w.Hq, w.L), float("nan"), dtype=torch.float32, device=dev)
    bdattn.bd_attn_fwd(q, k, v, seg, g, status, out=out, lse=lse)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return g, seg, status, out, lse, (q, k, v, doc)


@pytest.mark.parametrize("name,w,r,layout", CASES, ids=[x[0] for x in CASES])
def test_d512_forward(name, w, r, layout):
    c = make_case(w, r)
    _, _, _, out, lse, _ = _fwd(c, layout)
    ref_out, ref_lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], oracle_geom(c))
    assert_close(f"{name} out", out, ref_out)
    real = real_rows(c)
    got = lse.double().cpu().numpy()
    assert np.isneginf(got[~real]).all()
    assert np.abs(got[real] - ref_lse[real]).max(initial=0.0) <= LSE_ABS


def _bwd(c, g, seg, status, out, lse, qkv, layout, grad_dtype=torch.float32):
    from sliding_window_attention_device_gb300 import bdattn
    q, k, v, _ = qkv
    w, dev = c["w"], q.device
    dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=grad_dtype, device=dev)
    dk = torch.full(bdattn.kv_shape(g), float("nan"), dtype=grad_dtype, device=dev)
    dv = torch.full_like(dk, float("nan"))
    bdattn.bd_attn_bwd(c["do"].to(dev), q, k, v, out, lse, seg, g, status, grad_dtype=grad_dtype, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    back = (lambda t: t.permute(1, 2, 0, 3)) if layout else (lambda t: t)
    return dq.cpu(), back(dk).cpu(), back(dv).cpu()


@pytest.mark.parametrize("name,w,r,layout", CASES, ids=[x[0] for x in CASES])
def test_d512_backward(name, w, r, layout):
    c = make_case(w, r)
    g, seg, status, out, lse, qkv = _fwd(c, layout)
    dq, dk, dv = _bwd(c, g, seg, status, out, lse, qkv, layout)
    rdq, rdk, rdv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], oracle_geom(c))
    assert_close(f"{name} dq", dq, rdq)
    assert_close(f"{name} dk", dk, rdk)
    assert_close(f"{name} dv", dv, rdv)


def test_d512_backward_bf16_gradients():
    c = make_case(CASES[0][1], CASES[0][2])
    g, seg, status, out, lse, qkv = _fwd(c, 0)
    f = _bwd(c, g, seg, status, out, lse, qkv, 0)
    h = _bwd(c, g, seg, status, out, lse, qkv, 0, torch.bfloat16)
    for a, b_, n in zip(h, f, ("dq", "dk", "dv")):
        assert torch.isfinite(a.float()).all(), n
        tol = 2.0 ** -7 * max(1.0, b_.abs().max().item())
        assert (a.float() - b_).abs().max().item() <= tol, n


@pytest.mark.parametrize("name,w,r,layout", CASES, ids=[x[0] for x in CASES])
def test_d512_deterministic(name, w, r, layout):
    """The bitwise reproducible backward at D = 512 (dK / dV from the main
    kernel without its dq products, dq from the two-half fixed-order pass):
    two runs agree bit for bit, dK / dV equal the atomic backward's, and all
    three match the oracle."""
    from sliding_window_attention_device_gb300 import bdattn
    c = make_case(w, r)
    g, seg, status, out, lse, qkv = _fwd(c, layout)
    q, k, v, _ = qkv
    runs = []
    for _ in range(2):
        dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.float32, device=q.device)
        dk = torch.full(bdattn.kv_shape(g), float("nan"), dtype=torch.float32, device=q.device)
        dv = torch.full_like(dk, float("nan"))
        bdattn.bd_attn_bwd_deterministic(c["do"].to(q.device), q, k, v, out, lse, seg, g, status, dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        back = (lambda t: t.permute(1, 2, 0, 3)) if layout else (lambda t: t)  # token-major: to [B, Hkv, S_kv, D]
        runs.append((dq.cpu(), back(dk).cpu(), back(dv).cpu()))
    for x, y, n in zip(runs[0], runs[1], ("dq", "dk", "dv")):
        assert torch.equal(x, y), f"{name}: {n} differs between two runs"
    adq, adk, adv = _bwd(c, g, seg, status, out, lse, qkv, layout)
    assert torch.equal(runs[0][1], adk) and torch.equal(runs[0][2], adv)
    rdq, rdk, rdv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], oracle_geom(c))
    assert_close(f"{name} deterministic dq", runs[0][0], rdq)
    assert_close(f"{name} deterministic dk", runs[0][1], rdk)
    assert_close(f"{name} deterministic dv", runs[0][2], rdv)


@pytest.mark.slow
def test_d512_full_size_sampled():
    w = synth.WORKLOADS["G512"]
    rng = np.random.default_rng(5)
    for r in (3, 7):
        c = make_case(w, r, seed=0)
        _, _, _, out, lse, _ = _fwd(c, 0)
        out, lse = out.float().cpu(), lse.cpu()
        rows = sorted({(0, int(rng.integers(w.Hq)), int(i)) for i in rng.integers(0, w.L, 40)})
        ref_out, ref_lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], oracle_geom(c), rows=rows)
        for t, (b, h, i) in enumerate(rows):
            d = np.abs(out[b, h, i].numpy() - ref_out[t])
            assert d.max() <= 2e-2, (r, b, h, i, d.max())
            if np.isfinite(ref_lse[t]):
                assert abs(float(lse[b, h, i]) - ref_lse[t]) <= LSE_ABS


@pytest.mark.slow
def test_d512_backward_full_size_sampled():
    from test_gpu_full import _check, _oracle_sampled, _pick
    w = synth.WORKLOADS["G512"]
    r = 5
    c = make_case(w, r, seed=0)
    g, seg, status, out, lse, qkv = _fwd(c, 0)
    dq, dk, dv = _bwd(c, g, seg, status, out, lse, qkv, 0)
    rows, keys = _pick(c, np.random.default_rng(31))
    ref_rows, ref_keys = _oracle_sampled(c, rows, keys)
    for (bb, h, i), (_, _, dq_ref) in ref_rows.items():
        _check(f"G512 r{r} dq[{bb},{h},{i}]", dq[bb, h, i].numpy(), dq_ref)
    for (bb, hk, j), (dk_ref, dv_ref) in ref_keys.items():
        _check(f"G512 r{r} dk[{bb},{hk},{j}]", dk[bb, hk, j].numpy(), dk_ref)
        _check(f"G512 r{r} dv[{bb},{hk},{j}]", dv[bb, hk, j].numpy(), dv_ref)
