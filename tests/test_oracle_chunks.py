"""Pins for the oracle's chunked forward and merge (gemma4_moe.cp_local_ring:
forward over one K/V chunk returning (out, lse), and the -inf-safe online
softmax merge of chunk results).

Each pin checks the oracle against something other than itself: a numpy
brute force of the softmax over the allowed keys inside a chunk (the allow
rule retyped from the definition), the identity that merging the results of a
partition of the keys gives the full-range forward, and the algebra of the
merge (identity element, commutativity, both sides empty)."""
import numpy as np
import pytest

import oracle


def _case(seed, B=1, Hq=2, Hkv=1, D=16, S=96, cp=2, r=1, window=0, lengths=(30, 25, 20), pad=21):
    rng = np.random.default_rng(seed)
    doc = np.zeros((B, S), np.int32)
    pos = 0
    for d, n in enumerate(lengths, start=1):
        doc[:, pos:pos + n] = d
        pos += n
    assert pos + pad == S
    L = S // cp
    q = rng.standard_normal((B, Hq, L, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    return dict(doc=doc, q=q, k=k, v=v, B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, L=L, ro=r * L, window=window)


def _geom(c, kv_offset, S_kv):
    return oracle.geom(c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["L"], c["ro"], kv_offset, S_kv, c["window"])


def _brute_chunk(c, a, e):
    """Softmax over the allowed keys in [a, e), written from the definition."""
    B, Hq, L, D, G = c["B"], c["Hq"], c["L"], c["D"], c["Hq"] // c["Hkv"]
    out = np.zeros((B, Hq, L, D))
    lse = np.full((B, Hq, L), -np.inf)
    scale = D ** -0.5
    for b in range(B):
        doc = c["doc"][b]
        for i in range(L):
            p = c["ro"] + i
            if doc[p] == 0:
                continue
            keys = [s for s in range(a, e)
                    if (doc[s] == doc[p] and s <= p and (c["window"] <= 0 or p - s < c["window"])) or s == p]
            if not keys:
                continue
            for h in range(Hq):
                x = np.array([scale * c["q"][b, h, i] @ c["k"][b, h // G, s] for s in keys])
                m = x.max()
                w = np.exp(x - m)
                out[b, h, i] = (w[:, None] * c["v"][b, h // G, keys]).sum(0) / w.sum()
                lse[b, h, i] = m + np.log(w.sum())
    return out, lse


@pytest.mark.parametrize("a,e,window", [(0, 96, 0), (10, 40, 0), (40, 70, 0), (55, 96, 7), (0, 20, 0), (70, 96, 0)])
def test_chunk_forward_matches_brute_force(a, e, window):
    c = _case(1, window=window)
    g = _geom(c, a, e - a)
    out, lse = oracle.fwd_chunk(c["q"], c["k"][:, :, a:e], c["v"][:, :, a:e], c["doc"], g)
    ref_out, ref_lse = _brute_chunk(c, a, e)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bounds", [(0, 48, 96), (0, 17, 50, 51, 96), (0, 30, 55, 75, 96)])
@pytest.mark.parametrize("window", [0, 9])
def test_merging_a_partition_gives_the_full_forward(bounds, window):
    c = _case(2, window=window)
    full_out, full_lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], _geom(c, 0, c["S"]))
    acc_out = np.zeros_like(full_out)
    acc_lse = np.full(full_lse.shape, -np.inf)
    for a, e in zip(bounds[:-1], bounds[1:]):
        g = _geom(c, a, e - a)
        o, l = oracle.fwd_chunk(c["q"], c["k"][:, :, a:e], c["v"][:, :, a:e], c["doc"], g)
        acc_out, acc_lse = oracle.merge(acc_out, acc_lse, o, l)
    assert np.array_equal(np.isneginf(acc_lse), np.isneginf(full_lse))
    fin = np.isfinite(full_lse)
    np.testing.assert_allclose(acc_lse[fin], full_lse[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(acc_out, full_out, rtol=0, atol=1e-12)


def test_rows_without_keys_in_a_chunk_are_empty():
    c = _case(3)
    # keys [80, 96) are the last document's tail and padding: rows of the shard
    # (positions 48..95) in earlier documents see none of them
    g = _geom(c, 80, 16)
    out, lse = oracle.fwd_chunk(c["q"], c["k"][:, :, 80:], c["v"][:, :, 80:], c["doc"], g)
    doc = c["doc"][0]
    for i in range(c["L"]):
        p = c["ro"] + i
        sees = doc[p] != 0 and any(doc[s] == doc[p] and s <= p for s in range(80, 96))
        assert np.isneginf(lse[0, :, i]).all() != sees
        if not sees:
            assert (out[0, :, i] == 0).all()


def test_merge_algebra():
    rng = np.random.default_rng(4)
    o1, o2 = rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    l1, l2 = rng.standard_normal(5) * 3, rng.standard_normal(5) * 3
    empty_l = np.full(5, -np.inf)
    # -inf is the identity, whatever the empty side's out holds
    o, l = oracle.merge(o1, l1, rng.standard_normal((5, 8)), empty_l)
    np.testing.assert_array_equal(l, l1)
    np.testing.assert_allclose(o, o1, rtol=0, atol=1e-15)
    # commutative
    oa, la = oracle.merge(o1, l1, o2, l2)
    ob, lb = oracle.merge(o2, l2, o1, l1)
    np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-14)
    # the weights: out is the exp(lse)-weighted mean, lse the log of the summed weights
    w1, w2 = np.exp(l1), np.exp(l2)
    np.testing.assert_allclose(la, np.log(w1 + w2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(oa, (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None], rtol=0, atol=1e-12)
    # both empty
    o, l = oracle.merge(o1, empty_l, o2, empty_l)
    assert np.isneginf(l).all() and (o == 0).all()
