"""Pins of the exchange-plan oracle (oracle/exchange.py) to things other than
itself: hand-worked plans (tests/golden/exchange_plans.json), the needed K/V
range read off the attention oracle's dense mask by brute force, the page's
claim that the needed-only exchange's backward sums what the all-gather's
reduce-scatter would, the adjoint of the gather, and closed forms."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import exchange as ex
from sliding_window_attention_device_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "exchange_plans.json")


def _doc_from_runs(rows):
    out = []
    for runs in rows:
        out.append(np.concatenate([np.full(n, d, np.int32) for d, n in runs]))
    return np.stack(out)


def _runs(idx):
    return [list(range(a, e)) for a, e in idx]


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"][:24])
def test_hand_worked_plans(case):
    doc = _doc_from_runs(case["doc_runs"])
    p = ex.plan(doc, case["cp_size"])
    for k in ("s_first", "real_end", "back", "use_halo", "halo_size", "counts"):
        assert p[k] == case[k], k
    assert not p["layout_error"]
    for r, want in case["rank_splits"].items():
        i, o, s = ex.a2a_split(p, int(r))
        assert i == want["in_splits"] and o == want["out_splits"]
        assert s == [t for run in _runs(want["send_index_runs"]) for t in run]


def _layouts():
    out = []
    for seed, (layout, B, S, W) in enumerate([
        (("uniform", 5, 40, 9), 2, 96, 4),
        (("uniform", 1, 300, 20), 3, 240, 8),
        (("lognormal", 30.0, 1.0, 1, 200, 15), 2, 192, 6),
        (("single",), 1, 64, 4),
        (("explicit", (100, 90, 50), 16), 1, 256, 4),
        (("uniform", 20, 70, 0), 1, 120, 3),
        (("uniform", 3, 9, 30), 4, 64, 2),
        (("uniform", 100, 400, 0), 2, 200, 1),
    ]):
        out.append((synth.doc_layout(layout, B, S, seed), W))
    return out


@pytest.mark.parametrize("doc,W", _layouts())
def test_needed_ranges_from_the_dense_mask(doc, W):
    """[s_first_r, real_end_r) = the smallest range holding every key a real
    local row of rank r may attend (any batch row), read off og_mask."""
    B, S = doc.shape
    L = S // W
    p = ex.plan(doc, W)
    for r in range(W):
        g = oracle.geom(B, 1, 1, 8, S, L, r * L, 0, S, 0)
        m = oracle.mask(doc, g)  # [B, L, S]
        real = doc[:, r * L:(r + 1) * L] != 0
        keys = np.nonzero((m & real[:, :, None]).any(axis=(0, 1)))[0]
        if keys.size == 0:
            assert (p["s_first"][r], p["real_end"][r], p["back"][r]) == (r * L, r * L, 0)
            continue
        assert (p["s_first"][r], p["real_end"][r]) == (int(keys.min()), int(keys.max()) + 1)
        assert keys.size == keys.max() - keys.min() + 1  # the needed keys are contiguous
        assert p["back"][r] == r * L - int(keys.min())
    # use_halo: every key a rank needs below its own chunk lies in the left neighbour's chunk
    fits = all(p["s_first"][r] >= (r - 1) * L for r in range(W))
    assert p["use_halo"] == fits


@pytest.mark.parametrize("doc,W", _layouts())
def test_a2a_pieces_assemble_each_needed_range(doc, W):
    p = ex.plan(doc, W)
    L = p["L"]
    splits = [ex.a2a_split(p, s) for s in range(W)]
    for s, (ins, outs, idx) in enumerate(splits):
        assert len(idx) == sum(ins)
        assert all(0 <= t < L for t in idx)
        assert outs == [splits[src][0][s] for src in range(W)]
    for r in range(W):
        got = []
        for s, (ins, _, idx) in enumerate(splits):  # pieces arrive in source order
            off = sum(ins[:r])
            got += [s * L + t for t in idx[off:off + ins[r]]]
        assert got == list(range(p["s_first"][r], p["real_end"][r]))


@pytest.mark.parametrize("doc,W", _layouts()[:5])
def test_backward_sums_like_the_all_gather_reduce_scatter(doc, W):
    """Page claim: the needed-only exchange's index_add matches the sum the
    all-gather's reduce_scatter would give for each owned token."""
    rng = np.random.default_rng(7)
    p = ex.plan(doc, W)
    L, S = p["L"], p["S"]
    C, D = 2, 3
    grads = [rng.standard_normal((1, C, p["real_end"][r] - p["s_first"][r], D)) for r in range(W)]
    full = np.zeros((1, C, S, D))
    for r in range(W):
        full[:, :, p["s_first"][r]:p["real_end"][r]] += grads[r]
    for s in range(W):
        ins, _, idx = ex.a2a_split(p, s)
        pieces = []
        for r in range(W):
            a = max(s * L, p["s_first"][r])
            pieces.append(grads[r][:, :, a - p["s_first"][r]:a - p["s_first"][r] + ins[r]])
        local = ex.scatter_add(np.concatenate(pieces, axis=2), idx, L)
        np.testing.assert_allclose(local, full[:, :, s * L:(s + 1) * L], rtol=0, atol=1e-12)


def test_gather_and_scatter_add_are_adjoint():
    rng = np.random.default_rng(3)
    idx = [5, 0, 7, 7, 2, 5, 5, 1]
    x = rng.standard_normal((2, 3, 8, 4))
    y = rng.standard_normal((2, 3, len(idx), 4))
    lhs = float((ex.gather(x, idx) * y).sum())
    rhs = float((x * ex.scatter_add(y, idx, 8)).sum())
    assert abs(lhs - rhs) < 1e-12
    assert np.array_equal(ex.gather(x, idx)[:, :, 2], x[:, :, 7])


@pytest.mark.parametrize("W", [1, 2, 3, 8])
def test_single_document_closed_form(W):
    L = 16
    p = ex.plan(np.ones((1, W * L), np.int32), W)
    assert p["s_first"] == [0] * W
    assert p["real_end"] == [(r + 1) * L for r in range(W)]
    assert p["back"] == [r * L for r in range(W)]
    assert p["use_halo"] == (W <= 2)
    assert p["counts"] == [[L if s <= r else 0 for r in range(W)] for s in range(W)]
    assert p["halo_size"] == (W - 1) * L


def test_all_padding_rank_and_layout_errors():
    doc = np.array([[1, 1, 1, 2, 2, 0, 0, 0, 0, 0, 0, 0]], np.int32)
    p = ex.plan(doc, 3)
    assert (p["s_first"], p["real_end"], p["back"]) == ([0, 3, 8], [4, 5, 8], [0, 1, 0])
    assert not p["layout_error"]
    assert ex.plan(np.array([[1, 1, 0, 2]], np.int32), 2)["layout_error"]
    assert ex.plan(np.array([[1, -1, 2, 2]], np.int32), 2)["layout_error"]
