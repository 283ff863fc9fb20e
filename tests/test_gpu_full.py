"""Full-size workloads through the same calls the benchmark times, checked on
sampled outputs the oracle computes one by one (query rows: out, lse, dq; keys
with a bounded fan-in: dk, dv) and by identities that hold at any size:
sum_s dV[s] = sum over attending rows of dO (each row of P sums to one)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import LSE_ABS, MAX_ABS, MEAN_ABS, make_case, run_gpu
from sliding_window_attention_device_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _row_lo(c):
    """Global doc start (window applied) of every local row; -1 on padding."""
    w, ro, L, W = c["w"], c["row_offset"], c["w"].L, c["window"]
    out = np.full((w.B, L), -1, np.int64)
    for b in range(w.B):
        d = c["doc"][b]
        starts = np.zeros(w.S, np.int64)
        change = np.ones(w.S, bool)
        change[1:] = d[1:] != d[:-1]
        idx = np.where(change, np.arange(w.S), 0)
        starts = np.maximum.accumulate(idx)
        p = ro + np.arange(L)
        lo = starts[p]
        if W > 0:
            lo = np.maximum(lo, p - W + 1)
        out[b] = np.where(d[p] != 0, lo, -1)
    return out


def _pick(c, rng, n_rows=48, n_keys=24, budget=4e6):
    w, ro, L = c["w"], c["row_offset"], c["w"].L
    rows = set()
    for i in (0, 1, 127, 128, L - 1):
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.Hq)), i))
    while len(rows) < n_rows:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(L))))
    lo = _row_lo(c)
    keys = []
    cands = [(int(rng.integers(w.B)), int(rng.integers(c["S_kv"]))) for _ in range(400)]
    tail = [(b, j) for b in range(w.B) for j in range(max(0, ro + L - c["kv_offset"] - 48), ro + L - c["kv_offset"])
            if 0 <= j < c["S_kv"]]
    rng.shuffle(tail)
    for b, j in tail[:100] + cands:
        s = c["kv_offset"] + j
        p = ro + np.arange(L)
        att = (lo[b] >= 0) & (lo[b] <= s) & (p >= s)
        cost = float(((p - lo[b] + 1) * att).sum()) * w.G
        if cost <= budget:
            keys.append((b, int(rng.integers(w.Hkv)), j))
        if len(keys) >= n_keys:
            break
    return sorted(rows), keys


def _oracle_sampled(c, rows, keys):
    w = c["w"]
    G = w.G
    res_rows, res_keys = {}, {}
    groups = {}
    for (b, h, i) in rows:
        groups.setdefault((b, h // G), ([], []))[0].append((b, h, i))
    for (b, hk, j) in keys:
        groups.setdefault((b, hk), ([], []))[1].append((b, hk, j))
    for (b, hk), (rs, ks) in groups.items():
        sl = slice(hk * G, (hk + 1) * G)
        q, do = c["q"][b:b + 1, sl], c["do"][b:b + 1, sl]
        k, v = c["k"][b:b + 1, hk:hk + 1], c["v"][b:b + 1, hk:hk + 1]
        g = oracle.geom(1, G, 1, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], c["window"])
        lr = [(0, h - hk * G, i) for (_, h, i) in rs]
        lk = [(0, 0, j) for (_, _, j) in ks]
        if lr:
            out, lse = oracle.fwd(q, k, v, c["doc"][b:b + 1], g, rows=lr)
        dq, dk, dv = oracle.bwd(q, k, v, do, c["doc"][b:b + 1], g, rows=lr, keys=lk)
        for t, key in enumerate(rs):
            res_rows[key] = (out[t], lse[t], dq[t])
        for t, key in enumerate(ks):
            res_keys[key] = (dk[t], dv[t])
    return res_rows, res_keys


def _check(name, got, ref):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    assert np.isfinite(np.asarray(got, np.float64)).all(), name
    assert d.max(initial=0) <= MAX_ABS and d.mean() <= MEAN_ABS, f"{name}: max {d.max():.3e} mean {d.mean():.3e}"


@pytest.mark.parametrize("key", ["C2", "C3", "C4", "C5", "C5w4096", "C5w512"])
def test_full_size_sampled(key):
    w = synth.WORKLOADS[key]
    rng = np.random.default_rng(123)
    for r in w.ranks:
        c = make_case(w, r, seed=0)
        res = run_gpu(c)
        assert res["status_word"] == 0, f"{key} r{r}: status {res['status_word']:#x}"
        rows, keys = _pick(c, rng)
        ref_rows, ref_keys = _oracle_sampled(c, rows, keys)
        out = res["out"].float().cpu()
        lse = res["lse"].cpu()
        dq = res["dq"].cpu()
        for (b, h, i), (o_ref, l_ref, dq_ref) in ref_rows.items():
            _check(f"{key} r{r} out[{b},{h},{i}]", out[b, h, i].numpy(), o_ref)
            _check(f"{key} r{r} dq[{b},{h},{i}]", dq[b, h, i].numpy(), dq_ref)
            if np.isneginf(l_ref):
                assert torch.isneginf(lse[b, h, i])
            else:
                assert abs(float(lse[b, h, i]) - l_ref) <= LSE_ABS, (key, r, b, h, i, float(lse[b, h, i]), l_ref)
        dk, dv = res["dk"].cpu(), res["dv"].cpu()
        for (b, hk, j), (dk_ref, dv_ref) in ref_keys.items():
            _check(f"{key} r{r} dk[{b},{hk},{j}]", dk[b, hk, j].numpy(), dk_ref)
            _check(f"{key} r{r} dv[{b},{hk},{j}]", dv[b, hk, j].numpy(), dv_ref)
        # identity: sum_s dV[s] == sum over real rows of the group's dO
        real = torch.from_numpy(c["doc"][:, c["row_offset"]:c["row_offset"] + w.L] != 0).cuda()
        do = c["do"].cuda().double() * real[:, None, :, None]
        lhs = res["dv"].double().sum(2)
        rhs = do.view(w.B, w.Hkv, w.G, w.L, w.D).sum((2, 3))
        rel = ((lhs - rhs).norm() / rhs.norm().clamp_min(1e-30)).item()
        assert rel < 1e-2, f"{key} r{r}: sum dV identity rel err {rel:.3e}"
        del res
        torch.cuda.empty_cache()
