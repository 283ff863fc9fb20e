"""Full-size workloads compared with the fp64 oracle element by element, on whole
tensors: every local row and every key of the listed ranks, restricted to the
listed kv-head groups. A group is one kv head and its Hq/Hkv query heads; the
attention never mixes groups, so the oracle runs each group on its own. For a
group, out, lse and dq of its query heads and dk, dv of its kv head are compared
in full (no sampling, no fan-in budget: the keys every query of a long document
attends are included), with mean-abs over the whole compared tensor, padding
rows and unattended keys included.

The GPU runs the whole shard (all heads) exactly as the benchmark does. Both
gradient modes are checked against the same oracle result: fp32 gradients at
the parity bar (max-abs 2e-2, mean-abs 2e-3), bf16 gradients at that bar plus
bf16's rounding, 2^-8 of the reference value.

Passage: blockdiag_cp.kernels, `_cp_blockdiag_varlen` -- the result equals the
`_cp_blockdiag_mask` allow-mask plus softmax attention on real query rows.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, assert_close_bf16, assert_lse, make_case, run_gpu
from sliding_window_attention_device_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# one document deep enough that each early dK / dV tile sums many products, as
# in C4 (whose oracle would take minutes): 16 q tiles x 8 query heads = 128
# 128x128 tile products into each of the first K/V tiles, against 128 K/V tiles
DEEP = {
    "deep16k": synth.Workload("deep16k", "one 16K document, cp 8", B=1, Hq=8, Hkv=1, D=128, S=16384, cp_size=8,
                              layout=("single",), ranks=(7,), kv="prefix"),
}

# (workload, rank, kv groups)
SUBSETS = [("C2", 0, (0, 7)), ("C2", 4, (0, 7)), ("C2", 7, (0, 7)), ("C3", 7, (0, 7)), ("C5", 3, (0,)),
           ("C5w512", 3, (0,)), ("deep16k", 7, (0,)), ("G512", 5, (0,))]


def _workload(key):
    return DEEP[key] if key in DEEP else synth.WORKLOADS[key]


def _group_oracle(c, hk):
    """fp64 oracle for kv group hk on the whole shard: out, lse, dq [B, G, L, ...],
    dk, dv [B, S_kv, D]."""
    w = c["w"]
    G = w.G
    sl = slice(hk * G, (hk + 1) * G)
    g = oracle.geom(w.B, G, 1, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], c["window"])
    q, do = c["q"][:, sl], c["do"][:, sl]
    k, v = c["k"][:, hk:hk + 1], c["v"][:, hk:hk + 1]
    out, lse = oracle.fwd(q, k, v, c["doc"], g)
    dq, dk, dv = oracle.bwd(q, k, v, do, c["doc"], g)
    return out, lse, dq, dk[:, 0], dv[:, 0]


@pytest.mark.parametrize("key,r,groups", SUBSETS, ids=[f"{k}_r{r}" for k, r, _ in SUBSETS])
def test_full_size_group_subsets(key, r, groups):
    w = _workload(key)
    c = make_case(w, r, seed=0)
    res = {torch.float32: run_gpu(c, grad_dtype=torch.float32), torch.bfloat16: run_gpu(c, grad_dtype=torch.bfloat16)}
    for dt, rr in res.items():
        assert rr["status_word"] == 0, f"{key} r{r} {dt}: status {rr['status_word']:#x}"
    # the forward does not depend on the gradient dtype
    assert torch.equal(res[torch.float32]["out"], res[torch.bfloat16]["out"])
    ro = c["row_offset"]
    real = np.repeat((c["doc"][:, ro:ro + w.L] != 0)[:, None, :], w.G, axis=1)
    for hk in groups:
        sl = slice(hk * w.G, (hk + 1) * w.G)
        out, lse, dq, dk, dv = _group_oracle(c, hk)
        tag = f"{key} r{r} group {hk}"
        r32 = res[torch.float32]
        assert_close(f"{tag} out", r32["out"][:, sl], out)
        assert_lse(r32["lse"][:, sl], lse, real)
        pad = ~real
        assert (r32["out"][:, sl].float().cpu().numpy()[pad] == 0).all(), f"{tag}: padding rows of out not zero"
        for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
            idx = (slice(None), sl) if name == "dq" else (slice(None), hk)
            assert_close(f"{tag} {name} (fp32)", r32[name][idx], ref)
            assert_close_bf16(f"{tag} {name} (bf16)", res[torch.bfloat16][name][idx], ref)
        assert (r32["dq"][:, sl].cpu().numpy()[pad] == 0).all(), f"{tag}: padding rows of dq not zero"
    del res
    torch.cuda.empty_cache()
