"""Exchange plans and the needed-only exchange's local halves on the GPU
(blockdiag_cp.exchange: the left-halo plan, the all-to-all-v split plan,
`_NeededKVExchange` forward gather / backward index-add) through the C ABI,
against the oracle (oracle/exchange.py): plans bit-exact for every rank of
every named workload and of random layouts, the gather bit-exact, the
index-add within fp32 rounding, and the receivers' pieces assembling each
rank's needed range exactly."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import exchange as ex
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "exchange_plans.json")


def _gpu_plans(doc: np.ndarray, W: int):
    from sliding_window_attention_device_gb300 import bdattn
    d = torch.from_numpy(np.ascontiguousarray(doc, dtype=np.int32)).cuda()
    status = bdattn.new_status(d.device)
    out = []
    for r in range(W):
        plan, _ = bdattn.bd_attn_exchange_plan(d, W, r, status=status)
        out.append(plan)
    torch.cuda.synchronize()
    B, S = doc.shape
    return [bdattn.read_plan(p, B, W, S // W) for p in out], int(status.item()), out


def _check_plans(doc, W, got, status, layout_ok=True):
    p = ex.plan(doc, W)
    assert p["layout_error"] == (not layout_ok)
    from sliding_window_attention_device_gb300 import bdattn
    assert bool(status & bdattn.STATUS_LAYOUT) == p["layout_error"]
    for r, g in enumerate(got):
        assert g["magic"] == bdattn.PLAN_MAGIC and g["cp_size"] == W and g["rank"] == r and g["L"] == p["L"]
        for k in ("s_first", "real_end", "back", "counts"):
            assert g[k] == p[k], (r, k)
        assert g["use_halo"] == int(p["use_halo"]) and g["halo_size"] == p["halo_size"]
        assert g["halo_send"] == p["halo_send"]
        ins, outs, idx = ex.a2a_split(p, r)
        assert g["in_splits"] == ins and g["out_splits"] == outs
        assert g["send_off"] == [sum(ins[:d]) for d in range(W)]
        assert g["recv_off"] == [sum(outs[:s]) for s in range(W)]
        assert g["total_send"] == len(idx) and g["total_recv"] == sum(outs)
        assert g["send_index"] == idx, r


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"][:24])
def test_plan_golden(case):
    doc = np.stack([np.concatenate([np.full(n, d, np.int32) for d, n in runs]) for runs in case["doc_runs"]])
    got, status, _ = _gpu_plans(doc, case["cp_size"])
    assert status == 0
    _check_plans(doc, case["cp_size"], got, status)
    assert got[0]["s_first"] == case["s_first"] and got[0]["back"] == case["back"]


@pytest.mark.parametrize("key", ["C1", "C2", "C3", "C4", "C5"])
def test_plan_named_workloads(key):
    w = synth.WORKLOADS[key]
    doc = synth.doc_layout(w.layout, w.B, w.S, 0)
    got, status, _ = _gpu_plans(doc, w.cp_size)
    assert status == 0
    _check_plans(doc, w.cp_size, got, status)


@pytest.mark.parametrize("seed,layout,B,S,W", [
    (1, ("uniform", 1, 40, 30), 3, 384, 8),
    (2, ("lognormal", 300.0, 1.5, 1, 5000, 700), 2, 8192, 4),
    (3, ("uniform", 3000, 9000, 0), 1, 24576, 6),
    (4, ("uniform", 1, 3, 0), 2, 96, 32),
    (5, ("single",), 4, 9000, 3),
])
def test_plan_random_layouts(seed, layout, B, S, W):
    doc = synth.doc_layout(layout, B, S, seed)
    got, status, _ = _gpu_plans(doc, W)
    _check_plans(doc, W, got, status)


def test_plan_all_padding_ranks_and_layout_error():
    doc = np.zeros((2, 64), np.int32)
    doc[0, :20] = 1
    doc[1, :5] = 7
    doc[1, 5:9] = 8
    got, status, _ = _gpu_plans(doc, 4)
    assert status == 0
    _check_plans(doc, 4, got, status)
    bad = doc.copy()
    bad[0, 40] = 3  # a real id after padding inside rank 2's chunk
    got, status, _ = _gpu_plans(bad, 4)
    _check_plans(bad, 4, got, status, layout_ok=False)


def _x(shape, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("C,D", [(3, 64), (2, 128), (1, 256)])
def test_gather_and_scatter_add_match_the_oracle(dtype, C, D):
    from sliding_window_attention_device_gb300 import bdattn
    doc = synth.doc_layout(("uniform", 5, 400, 50), 2, 1024, 11)
    W = 4
    L = 1024 // W
    _, status, plans = _gpu_plans(doc, W)
    assert status == 0
    p = ex.plan(doc, W)
    st = bdattn.new_status("cuda")
    for r in range(W):
        ins, _, idx = ex.a2a_split(p, r)
        x = _x((2, C, L, D), dtype, 100 + r)
        send = torch.full((W * L, 2, C, D), float("nan"), dtype=dtype, device="cuda")
        bdattn.bd_attn_needed_gather(x.cuda(), plans[r], send, st)
        gs = _x((W * L, 2, C, D), dtype, 200 + r)
        gs[len(idx):] = float("nan")  # rows past the send count must be ignored
        gl = torch.full((2, C, L, D), float("nan"), dtype=dtype, device="cuda")
        bdattn.bd_attn_needed_scatter_add(gs.cuda(), plans[r], gl, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        n = len(idx)
        ref = ex.gather(x.float().numpy(), idx)  # [B, C, n, D]
        got = send[:n].float().cpu().permute(1, 2, 0, 3).numpy()
        assert np.array_equal(got, ref), r
        assert torch.isnan(send[n:].float()).all()
        ref_g = ex.scatter_add(gs[:n].double().permute(1, 2, 0, 3).numpy(), idx, L)
        tol = 1e-5 if dtype == torch.float32 else 2e-2
        got_g = gl.double().cpu().numpy()
        assert np.isfinite(got_g).all()
        np.testing.assert_allclose(got_g, ref_g, rtol=tol, atol=tol)


@pytest.mark.parametrize("key", ["C4", "C5"])
def test_receivers_assemble_their_needed_range(key):
    """Full size, every rank: gather K from each source's chunk, hand each
    destination its piece in source order, and the result is exactly K over
    the destination's needed range; the index-add of those pieces' all-ones
    gradients counts how many ranks need each token."""
    from sliding_window_attention_device_gb300 import bdattn
    w = synth.WORKLOADS[key]
    doc = synth.doc_layout(w.layout, w.B, w.S, 0)
    W, L = w.cp_size, w.L
    k, _ = synth.kv_rows(w, 0)
    k = k.cuda()
    _, status, plans = _gpu_plans(doc, W)
    assert status == 0
    p = ex.plan(doc, W)
    st = bdattn.new_status("cuda")
    sends = []
    for s in range(W):
        send = torch.empty((W * L, w.B, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
        bdattn.bd_attn_needed_gather(k[:, :, s * L:(s + 1) * L].contiguous(), plans[s], send, st)
        sends.append(send)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    need = np.zeros(w.S, np.int64)
    for r in range(W):
        need[p["s_first"][r]:p["real_end"][r]] += 1
        pieces = []
        for s in range(W):
            off = sum(p["counts"][s][:r])
            pieces.append(sends[s][off:off + p["counts"][s][r]])
        got = torch.cat(pieces, 0).permute(1, 2, 0, 3)
        assert torch.equal(got, k[:, :, p["s_first"][r]:p["real_end"][r]]), r
    for s in range(W):
        ones = torch.ones((W * L, w.B, 1, 4), dtype=torch.float32, device="cuda")
        gl = torch.empty((w.B, 1, L, 4), dtype=torch.float32, device="cuda")
        bdattn.bd_attn_needed_scatter_add(ones, plans[s], gl, st)
        torch.cuda.synchronize()
        want = torch.from_numpy(need[s * L:(s + 1) * L].astype(np.float32))
        assert torch.equal(gl[0, 0, :, 0].cpu(), want), s


def test_send_buffer_too_small_sets_bounds():
    from sliding_window_attention_device_gb300 import bdattn
    doc = np.ones((1, 256), np.int32)  # one document: rank 0 sends its chunk to all 4 ranks
    _, status, plans = _gpu_plans(doc, 4)
    st = bdattn.new_status("cuda")
    x = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    send = torch.full((100, 1, 1, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    bdattn.bd_attn_needed_gather(x, plans[0], send, st)
    torch.cuda.synchronize()
    assert int(st.item()) == bdattn.STATUS_BOUNDS
    assert (send == 7.0).all()
