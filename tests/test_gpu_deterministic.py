"""The bitwise reproducible backward (the pages' `_CP_FLASH_DETERMINISTIC`;
bd_attn_bwd_deterministic: dk / dv from the main kernel without its dq
products, dq from the fixed-order pass) on the GPU:

  * two runs give identical dq, dk and dv, bit for bit;
  * dk / dv equal those of the atomic-add backward bit for bit (the same
    arithmetic), and dq matches it within the parity tolerance;
  * dq, dk, dv match the oracle (windows, ragged tails, D = 64 / 128 / 256,
    GQA, token-major K/V, bf16 gradients, and sampled rows of full-size
    workloads).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, make_case, oracle_geom
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu

W_ = synth.Workload
CASES = [
    ("d128_g2_ragged", W_("da", "deterministic, D 128, ragged", B=2, Hq=4, Hkv=2, D=128, S=1280, cp_size=4,
                          layout=("uniform", 20, 300, 40)), 2, 0),
    ("d64_g3_window", W_("db", "deterministic, D 64, window 100", B=1, Hq=3, Hkv=1, D=64, S=1024, cp_size=2,
                         layout=("uniform", 50, 400, 70), window=100), 1, 0),
    ("d128_window_prefix_tm", W_("dc", "deterministic, D 128, window 150, token-major", B=1, Hq=4, Hkv=2, D=128,
                                 S=1280, cp_size=4, layout=("uniform", 100, 600, 30), window=150, kv="prefix"), 3, 1),
    ("d256_g2_window", W_("dd", "deterministic, D 256, window 300", B=1, Hq=4, Hkv=2, D=256, S=1280, cp_size=4,
                          layout=("uniform", 100, 600, 30), window=300, kv="prefix"), 3, 0),
    ("d256_ragged_tm", W_("de", "deterministic, D 256, ragged, token-major", B=2, Hq=2, Hkv=1, D=256, S=1024,
                          cp_size=4, layout=("uniform", 20, 300, 40)), 2, 1),
]


def _inputs(c, layout):
    from sliding_window_attention_device_gb300 import bdattn
    w, dev = c["w"], torch.device("cuda")
    g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], w.window,
                    kv_layout=layout)
    to = (lambda t: t.permute(2, 0, 1, 3).contiguous()) if layout else (lambda t: t)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, do = c["q"].to(dev), c["do"].to(dev)
    k, v = to(c["k"]).to(dev), to(c["v"]).to(dev)
    seg, status = bdattn.bd_attn_seg_build(doc, g)
    out, lse = bdattn.bd_attn_fwd(q, k, v, seg, g, status)
    return g, q, k, v, do, out, lse, seg, status


def _bwd(fn, g, q, k, v, do, out, lse, seg, status, grad_dtype=torch.float32):
    from sliding_window_attention_device_gb300 import bdattn
    dev = q.device
    dq = torch.full((g.B, g.Hq, g.L, g.D), float("nan"), dtype=grad_dtype, device=dev)
    dk = torch.full(bdattn.kv_shape(g), float("nan"), dtype=grad_dtype, device=dev)
    dv = torch.full_like(dk, float("nan"))
    fn(do, q, k, v, out, lse, seg, g, status, grad_dtype=grad_dtype, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dq, dk, dv


@pytest.mark.parametrize("name,w,r,layout", CASES, ids=[x[0] for x in CASES])
def test_deterministic_backward(name, w, r, layout):
    from sliding_window_attention_device_gb300 import bdattn
    c = make_case(w, r)
    args = _inputs(c, layout)
    a = _bwd(bdattn.bd_attn_bwd_deterministic, *args)
    b = _bwd(bdattn.bd_attn_bwd_deterministic, *args)
    for x, y, n in zip(a, b, ("dq", "dk", "dv")):
        assert torch.equal(x, y), f"{name}: {n} differs between two runs"
    ref = _bwd(bdattn.bd_attn_bwd, *args)
    assert torch.equal(a[1], ref[1]) and torch.equal(a[2], ref[2])
    assert_close(f"{name} dq vs atomic", a[0], ref[0].cpu())
    back = (lambda t: t.permute(1, 2, 0, 3)) if layout else (lambda t: t)
    rdq, rdk, rdv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], oracle_geom(c))
    assert_close(f"{name} dq", a[0], rdq)
    assert_close(f"{name} dk", back(a[1]), rdk)
    assert_close(f"{name} dv", back(a[2]), rdv)


def test_deterministic_bf16_gradients():
    from sliding_window_attention_device_gb300 import bdattn
    c = make_case(CASES[0][1], CASES[0][2])
    args = _inputs(c, 0)
    a = _bwd(bdattn.bd_attn_bwd_deterministic, *args, grad_dtype=torch.bfloat16)
    b = _bwd(bdattn.bd_attn_bwd_deterministic, *args, grad_dtype=torch.bfloat16)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    f = _bwd(bdattn.bd_attn_bwd_deterministic, *args)
    assert (a[0].float() - f[0].float()).abs().max().item() <= 2.0 ** -7 * max(1.0, f[0].abs().max().item())


@pytest.mark.slow
@pytest.mark.parametrize("key,r", [("C2", 4), ("C5w512", 3), ("C3", 7)])
def test_deterministic_full_size_sampled(key, r):
    from sliding_window_attention_device_gb300 import bdattn
    from test_gpu_full import _check, _oracle_sampled, _pick
    w = synth.WORKLOADS[key]
    c = make_case(w, r, seed=0)
    args = _inputs(c, 0)
    a = _bwd(bdattn.bd_attn_bwd_deterministic, *args)
    b = _bwd(bdattn.bd_attn_bwd_deterministic, *args)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    rows, keys = _pick(c, np.random.default_rng(77))
    ref_rows, ref_keys = _oracle_sampled(c, rows, keys)
    dq, dk, dv = (t.cpu() for t in a)
    for (bb, h, i), (_, _, dq_ref) in ref_rows.items():
        _check(f"{key} r{r} dq[{bb},{h},{i}]", dq[bb, h, i].numpy(), dq_ref)
    for (bb, hk, j), (dk_ref, dv_ref) in ref_keys.items():
        _check(f"{key} r{r} dk[{bb},{hk},{j}]", dk[bb, hk, j].numpy(), dk_ref)
        _check(f"{key} r{r} dv[{bb},{hk},{j}]", dv[bb, hk, j].numpy(), dv_ref)
