"""Pins of the oracle's attention dropout against things other than itself.

The pages expose `dropout_p` (blockdiag_cp.kernels `_cp_blockdiag_varlen`),
the chance that an attention weight is dropped, and say no more. The oracle reads it as
inverted dropout on the attention probabilities, with the keep decisions drawn
by Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) from a counter of
(key position / 8, query position, query head, batch row) and a 64-bit seed:
a 16-bit draw u per pair, kept iff u >= T = round(p 2^16), kept weights scaled
by 2^16 / (2^16 - T).

Pins:
  * the generator equals Triton's Philox-4x32 with 10 rounds (the library's
    CPU interpreter) on random counters and keys;
  * a probability that rounds to T = 0 gives exactly the dropout-free results;
  * the keep rate over many pairs matches (2^16 - T) / 2^16 within a binomial
    bound, and every counter field and both key words change the decisions;
  * the forward equals the dense formula out = (softmax(masked scores) * Z) V
    with the same factors Z, and the LSE is the undropped one;
  * central finite differences of sum(out * dout) under a fixed seed;
  * the average over many seeds approaches the dropout-free output (E[Z] = 1);
  * a K/V range cut into chunks and merged gives the unchunked result (the
    decisions depend on global positions only).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from sliding_window_attention_device_gb300 import synth


def _triton_philox(ctr: np.ndarray, seeds: np.ndarray) -> np.ndarray:
    """Triton's Philox (tl.philox, 10 rounds) in its CPU interpreter, in a child
    process (tests/philox_triton_ref.py). The key of row i is
    (seeds[i] & 0xffffffff, seeds[i] >> 32)."""
    pytest.importorskip("triton")
    env = dict(os.environ, TRITON_INTERPRET="1")
    req = json.dumps({"ctr": ctr.astype(np.int64).tolist(), "seed": [int(x) for x in seeds]})
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(__file__), "philox_triton_ref.py")],
                       input=req, capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return np.asarray(json.loads(r.stdout)["out"], dtype=np.uint64).astype(np.uint32)


def test_philox_equals_triton_interpreter():
    rng = np.random.Generator(np.random.PCG64(11))
    n = 48
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    seeds = rng.integers(0, 2 ** 63, size=n, dtype=np.uint64) * 2 + rng.integers(0, 2, size=n, dtype=np.uint64)
    ctr[0] = 0
    seeds[0] = 0
    ctr[1] = 0xFFFFFFFF
    seeds[1] = 0xFFFFFFFFFFFFFFFF
    key = np.stack([seeds & 0xFFFFFFFF, seeds >> np.uint64(32)], axis=1).astype(np.uint32)
    got = oracle.philox(ctr, key)
    ref = _triton_philox(ctr, seeds)
    np.testing.assert_array_equal(got, ref)


def _case(layout=("uniform", 5, 40, 6), B=2, Hq=4, Hkv=2, D=8, S=128, cp=2, r=1, window=0, seed=0):
    w = synth.Workload("T", "dropout", B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, cp_size=cp, layout=layout, window=window)
    doc = synth.doc_layout(layout, B, S, seed)
    k, v = synth.kv_rows(w, seed)
    return w, doc, synth.q_shard(w, r, seed), k, v, synth.dout_shard(w, r, seed), r * w.L


def test_probability_rounding_to_zero_is_exactly_no_dropout():
    w, doc, q, k, v, do, ro = _case()
    g0 = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S)
    gt = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S, dropout_p=1e-6, seed=5)  # T = 0
    a = oracle.fwd(q, k, v, doc, g0) + oracle.bwd(q, k, v, do, doc, g0)
    b = oracle.fwd(q, k, v, doc, gt) + oracle.bwd(q, k, v, do, doc, gt)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_keep_rate_and_counter_fields(p):
    g = oracle.geom(2, 4, 2, 8, 4096, 512, 1024, 700, 2048, dropout_p=p, seed=0x1234_5678_9ABC_DEF0)
    T = int(np.floor(p * 65536 + 0.5))
    scale = 65536.0 / (65536 - T)
    z = oracle.dropout_factors(g, 1, 3)
    assert set(np.unique(z)) <= {0.0, scale}
    n = z.size
    kept = int((z > 0).sum())
    q = (65536 - T) / 65536
    sd = np.sqrt(n * q * (1 - q))
    assert abs(kept - n * q) < 5 * sd, (kept, n * q, sd)
    # every counter field and both key words enter the decisions
    others = [oracle.dropout_factors(g, 0, 3), oracle.dropout_factors(g, 1, 2),
              oracle.dropout_factors(oracle.geom(2, 4, 2, 8, 4096, 512, 1024, 700, 2048, dropout_p=p,
                                                 seed=0x1234_5678_9ABC_DEF1), 1, 3),
              oracle.dropout_factors(oracle.geom(2, 4, 2, 8, 4096, 512, 1024, 700, 2048, dropout_p=p,
                                                 seed=0x1234_5679_9ABC_DEF0), 1, 3)]
    for o in others:
        assert (o != z).mean() > 0.5 * 2 * q * (1 - q)
    # shifting the query row or the key by one position (same buffer) changes them too
    assert (z[1:] != z[:-1]).mean() > 0.5 * 2 * q * (1 - q)
    assert (z[:, 1:] != z[:, :-1]).mean() > 0.5 * 2 * q * (1 - q)
    # the decisions follow global positions: another K/V buffer start and
    # another shard geometry give the same factors at the same (p, s)
    g2 = oracle.geom(2, 4, 2, 8, 4096, 256, 1280, 900, 1000, dropout_p=p, seed=0x1234_5678_9ABC_DEF0)
    z2 = oracle.dropout_factors(g2, 1, 3)
    np.testing.assert_array_equal(z2, z[256:512, 200:1200])


@pytest.mark.parametrize("window", [0, 9])
def test_forward_equals_dense_formula(window):
    w, doc, q, k, v, _, ro = _case(window=window)
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S, window=window, dropout_p=0.3, seed=77)
    g0 = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S, window=window)
    out, lse = oracle.fwd(q, k, v, doc, g)
    _, lse0 = oracle.fwd(q, k, v, doc, g0)
    np.testing.assert_array_equal(lse, lse0)  # the softmax normaliser is the undropped one
    m = oracle.mask(doc, g)
    G = w.G
    kr = k.double().numpy().repeat(G, axis=1)
    vr = v.double().numpy().repeat(G, axis=1)
    sc = np.einsum("bhid,bhjd->bhij", q.double().numpy(), kr) * w.D ** -0.5
    sc = np.where(m[:, None], sc, -np.inf)
    p = np.exp(sc - sc.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    z = np.stack([np.stack([oracle.dropout_factors(g, b, h) for h in range(w.Hq)]) for b in range(w.B)])
    assert (z == 0).any() and (z > 1).any()
    dense = np.einsum("bhij,bhjd->bhid", p * z, vr)
    real = (doc[:, ro:ro + w.L] != 0)[:, None, :, None]
    np.testing.assert_allclose(out, np.where(real, dense, 0.0), atol=1e-12, rtol=0)


def test_finite_differences_with_dropout():
    """Analytic backward == central differences of sum(out * dout) with the keep
    decisions fixed by the seed (fp64, h = 1e-6)."""
    doc = synth.doc_layout(("explicit", (5, 7), 4), 1, 16)
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 2, 8, 4))
    k = rng.standard_normal((1, 1, 16, 4))
    v = rng.standard_normal((1, 1, 16, 4))
    do = rng.standard_normal((1, 2, 8, 4))
    g = oracle.geom(1, 2, 1, 4, 16, 8, 8, 0, 16, window=6, dropout_p=0.4, seed=3)
    z = np.stack([oracle.dropout_factors(g, 0, h) for h in range(2)])
    m = oracle.mask(doc, g)[0]
    assert ((z == 0) & m).any() and ((z > 0) & m).any(), "the case must drop and keep allowed pairs"

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


def test_average_over_seeds_is_the_undropped_output():
    """E[Z] = 1: over n seeds the mean output tends to the dropout-free one, within
    a bound from the per-element variance sum_s P^2 v^2 p / (1 - p) (4.5 sigma)."""
    w, doc, q, k, v, _, ro = _case(B=1, Hq=2, Hkv=1, D=4, S=64, cp=2, layout=("explicit", (20, 30), 14))
    p, n = 0.5, 400
    g0 = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S)
    ref, _ = oracle.fwd(q, k, v, doc, g0)
    acc = np.zeros_like(ref)
    for s in range(n):
        out, _ = oracle.fwd(q, k, v, doc, oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S, dropout_p=p,
                                                       seed=1000 + s))
        acc += out
    mean = acc / n
    m = oracle.mask(doc, g0)
    kr = k.double().numpy().repeat(w.G, axis=1)
    vr = v.double().numpy().repeat(w.G, axis=1)
    sc = np.einsum("bhid,bhjd->bhij", q.double().numpy(), kr) * w.D ** -0.5
    sc = np.where(m[:, None], sc, -np.inf)
    pr = np.exp(sc - sc.max(-1, keepdims=True))
    pr /= pr.sum(-1, keepdims=True)
    T = int(np.floor(p * 65536 + 0.5))
    var = np.einsum("bhij,bhjd->bhid", pr ** 2, vr ** 2) * (T / (65536 - T))
    real = (doc[:, ro:ro + w.L] != 0)[:, None, :, None] & np.ones_like(ref, bool)
    sd = np.sqrt(var / n)
    assert (np.abs(mean - ref)[real] <= 4.5 * sd[real] + 1e-12).all()
    # and a missing keep scale would be far outside the bound
    assert not (np.abs(mean * (1 - p) - ref)[real] <= 4.5 * sd[real] + 1e-12).all()


def test_chunked_merge_equals_unchunked_with_dropout():
    w, doc, q, k, v, _, ro = _case(window=0)
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, 0, w.S, dropout_p=0.25, seed=9)
    out, lse = oracle.fwd(q, k, v, doc, g)
    o_acc, l_acc = None, None
    for a, e in ((0, 37), (37, 90), (90, w.S)):
        gc = oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, ro, a, e - a, dropout_p=0.25, seed=9)
        oc, lc = oracle.fwd_chunk(q, k[:, :, a:e], v[:, :, a:e], doc, gc)
        if o_acc is None:
            o_acc, l_acc = oc, lc
        else:
            o_acc, l_acc = oracle.merge(o_acc, l_acc, oc, lc)
    np.testing.assert_allclose(o_acc, out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l_acc, lse, atol=1e-12, rtol=0)
