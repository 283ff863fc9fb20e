"""Forward / backward parity of the CUDA path against the fp64 oracle, element by
element, at sizes the oracle finishes in seconds: several 128-row tiles, ragged
q and K/V tails, odd and even GQA groups, D = 64 / 128 / 256 / 512, windows,
K/V sub-ranges, all-padding shards and length-1 documents."""
import numpy as np
import pytest
import torch

import oracle
from helpers import MAX_ABS, MEAN_ABS, assert_close, assert_lse, make_case, oracle_geom, real_rows, run_gpu
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu


def W(key, B, Hq, Hkv, D, S, cp, layout, window=0, kv="full"):
    return synth.Workload(key, key, B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, cp_size=cp, layout=layout, window=window,
                          ranks=tuple(range(cp)), kv=kv)


CASES = [
    # name, workload, ranks
    ("C1", synth.WORKLOADS["C1"], (2,)),
    ("C1_all_ranks", synth.WORKLOADS["C1"], (0, 1, 3)),
    ("d128_g2_ragged", W("a", 2, 4, 2, 128, 1280, 4, ("uniform", 20, 300, 40)), (0, 1, 2, 3)),
    ("d128_g3_needed", W("b", 2, 6, 2, 128, 1536, 4, ("uniform", 30, 500, 0), kv="needed"), (1, 3)),
    ("d64_g1_window", W("c", 1, 3, 3, 64, 1024, 2, ("uniform", 50, 400, 70), window=100), (0, 1)),
    ("d256_g2_window", W("d", 1, 4, 2, 256, 1280, 4, ("uniform", 100, 600, 30), window=150, kv="prefix"), (1, 3)),
    ("d256_g1", W("e", 1, 2, 2, 256, 768, 2, ("uniform", 100, 400, 10)), (0, 1)),
    ("d128_single_doc", W("f", 1, 4, 1, 128, 1536, 4, ("single",)), (0, 3)),
    ("d128_len1_docs", W("g", 1, 2, 1, 128, 640, 2, ("uniform", 1, 3, 17)), (0, 1)),
    ("d128_window1", W("h", 1, 2, 1, 128, 512, 2, ("uniform", 30, 200, 5), window=1), (1,)),
    ("d64_g4_big_window", W("i", 2, 8, 2, 64, 1024, 4, ("uniform", 60, 500, 90), window=100000), (1, 2)),
    ("d128_all_pad_shard", W("j", 1, 2, 1, 128, 1024, 4, ("explicit", (300, 200), 524)), (2, 3, 1)),
    ("d512_g2_needed", W("k", 1, 4, 2, 512, 1024, 4, ("uniform", 30, 400, 20), kv="needed"), (1, 3)),
    ("d512_len1_docs", W("l", 1, 2, 1, 512, 640, 2, ("uniform", 1, 3, 17)), (0,)),
    ("d512_window1", W("m", 1, 2, 1, 512, 512, 2, ("uniform", 30, 200, 5), window=1), (1,)),
    ("d512_all_pad_shard", W("n", 1, 2, 1, 512, 1024, 4, ("explicit", (300, 200), 524)), (2, 3)),
    ("d256_len1_docs", W("o", 1, 2, 1, 256, 640, 2, ("uniform", 1, 3, 17)), (0,)),
    ("d256_window1", W("p", 1, 2, 1, 256, 512, 2, ("uniform", 30, 200, 5), window=1), (1,)),
    ("d256_all_pad_shard", W("q", 1, 2, 1, 256, 1024, 4, ("explicit", (300, 200), 524)), (2, 3)),
]


def _oracle_full(c):
    g = oracle_geom(c)
    out, lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], g)
    dq, dk, dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], g)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("name,w,ranks", CASES, ids=[c[0] for c in CASES])
def test_fwd_bwd_parity(name, w, ranks):
    for r in ranks:
        c = make_case(w, r, seed=r + 1)
        res = run_gpu(c)
        assert res["status_word"] == 0, f"status {res['status_word']:#x}"
        out, lse, dq, dk, dv = _oracle_full(c)
        real = real_rows(c)
        assert_close(f"{name} r{r} out", res["out"], out)
        assert_lse(res["lse"], lse, real)
        assert_close(f"{name} r{r} dq", res["dq"], dq)
        assert_close(f"{name} r{r} dk", res["dk"], dk)
        assert_close(f"{name} r{r} dv", res["dv"], dv)
        # padding rows: exact zeros
        pad = ~real
        assert (res["out"].float().cpu().numpy()[pad] == 0).all()
        assert (res["dq"].cpu().numpy()[pad] == 0).all()


def test_bf16_gradients_track_fp32():
    w = W("k", 2, 4, 2, 128, 1280, 4, ("uniform", 20, 300, 40))
    c = make_case(w, 2, seed=9)
    r32 = run_gpu(c, grad_dtype=torch.float32)
    r16 = run_gpu(c, grad_dtype=torch.bfloat16)
    assert r32["status_word"] == 0 and r16["status_word"] == 0
    for n in ("dq", "dk", "dv"):
        a, b = r32[n].double(), r16[n].double()
        # bf16 output rounding only: |b - a| <= 2^-8 |a| (+ tiny absolute slack)
        assert ((b - a).abs() <= a.abs() * 2 ** -8 + 1e-30).all(), n


def test_repeat_calls_are_consistent():
    """The same inputs give the same forward bits every call; the dq atomics may
    reorder additions but stay within rounding."""
    w = W("l", 1, 4, 2, 128, 1024, 2, ("uniform", 50, 700, 20))
    c = make_case(w, 1, seed=4)
    a, b = run_gpu(c), run_gpu(c)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])
    assert torch.equal(a["dk"], b["dk"]) and torch.equal(a["dv"], b["dv"])
    assert (a["dq"] - b["dq"]).abs().max().item() < 1e-4


def test_cp_union_equals_unsharded():
    """Concatenating every rank's output gives the cp_size = 1 result; dK / dV of the
    full K/V summed over ranks equal the unsharded dK / dV (the all-gather's
    reduce-scatter sum)."""
    w4 = W("m", 1, 4, 2, 128, 1024, 4, ("uniform", 40, 400, 30))
    w1 = W("m", 1, 4, 2, 128, 1024, 1, ("uniform", 40, 400, 30))
    seed = 5
    full = make_case(w1, 0, seed=seed)
    full["q"] = torch.cat([synth.q_shard(w4, r, seed) for r in range(4)], 2)
    full["do"] = torch.cat([synth.dout_shard(w4, r, seed) for r in range(4)], 2)
    ref = run_gpu(full)
    outs, dks, dvs = [], 0, 0
    for r in range(4):
        res = run_gpu(make_case(w4, r, seed=seed))
        outs.append(res["out"].float())
        dks = dks + res["dk"]
        dvs = dvs + res["dv"]
    torch.testing.assert_close(torch.cat(outs, 2), ref["out"].float(), atol=2e-2, rtol=0)
    torch.testing.assert_close(dks, ref["dk"], atol=2e-2, rtol=0)
    torch.testing.assert_close(dvs, ref["dv"], atol=2e-2, rtol=0)


@pytest.mark.parametrize("name", ["d128_g2_ragged", "d256_g2_window"])
def test_direct_fp32_dq_matches_workspace_accumulator(name):
    """bd_attn_bwd_prep_dq / _main_dq (fp32 dq as its own accumulator) give the
    same gradients as prep / main / finalize through the workspace."""
    from sliding_window_attention_device_gb300 import bdattn
    w, ranks = next((c[1], c[2]) for c in CASES if c[0] == name)
    c = make_case(w, ranks[-1])
    res = run_gpu(c, bwd=False)
    g, seg, status = res["g"], res["seg"], res["status"]
    dev = torch.device("cuda")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    ws = torch.empty(bdattn.bwd_workspace_bytes(g), dtype=torch.uint8, device=dev)
    out = {}
    for mode in ("workspace", "direct"):
        dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.float32, device=dev)
        dk = torch.full((w.B, w.Hkv, c["S_kv"], w.D), float("nan"), dtype=torch.float32, device=dev)
        dv = torch.full_like(dk, float("nan"))
        if mode == "workspace":
            bdattn.bd_attn_bwd_prep(do, res["out"], g, status, ws)
            bdattn.bd_attn_bwd_main(do, q, k, v, res["lse"], seg, g, status, ws, dk, dv)
            bdattn.bd_attn_bwd_finalize(g, status, ws, dq)
        else:
            bdattn.bd_attn_bwd_prep_dq(do, res["out"], g, status, ws, dq)
            bdattn.bd_attn_bwd_main_dq(do, q, k, v, res["lse"], seg, g, status, ws, dq, dk, dv)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        out[mode] = (dq.cpu(), dk.cpu(), dv.cpu())
    (dq0, dk0, dv0), (dq1, dk1, dv1) = out["workspace"], out["direct"]
    assert torch.isfinite(dq1).all()
    torch.testing.assert_close(dq1, dq0, rtol=1e-4, atol=1e-5)
    assert torch.equal(dk1, dk0) and torch.equal(dv1, dv0)
