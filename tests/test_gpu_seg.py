"""K1 segmentation and K2 tile classification on the GPU, bit-exact against the oracle.

Segments: every field of the definition (n_real, n_seg, s_first, real_end,
cu_q, cu_k, max_q, max_k) plus first_q / first_k / max_tail / need_lo and the
LAYOUT / KV_RANGE status bits. Tiles: the classification is compared with a
brute-force classification of the oracle's dense mask, and the work lists
must be permutations ordered by decreasing work.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_attention_device_gb300 import bdattn, synth

pytestmark = pytest.mark.gpu

FIELDS = ("n_real", "n_seg", "s_first", "real_end", "max_q", "max_k", "first_q", "first_k", "max_tail")


def _gpu_seg(doc, g):
    d = torch.from_numpy(np.ascontiguousarray(doc, dtype=np.int32)).cuda()
    seg, status = bdattn.bd_attn_seg_build(d, g)
    torch.cuda.synchronize()
    return bdattn.read_seg(seg, g), int(status.item())


def _check_segments(doc, B, S, L, ro, kvo, skv, window):
    g = bdattn.geom(B, 2, 1, 64, S, L, ro, kvo, skv, window)
    og = oracle.geom(B, 2, 1, 64, S, L, ro, kvo, skv, window)
    tab, status = _gpu_seg(doc, g)
    ref = oracle.segments(doc, og)
    exp_status = 0
    for b in range(B):
        got, exp = tab["rows"][b], ref[b]
        for f in FIELDS:
            assert got[f] == exp[f], (b, f, got[f], exp[f])
        assert got["kv_need_lo"] == exp["kv_need_lo"], (b, got["kv_need_lo"], exp["kv_need_lo"])
        np.testing.assert_array_equal(got["cu_q"], exp["cu_q"])
        np.testing.assert_array_equal(got["cu_k"], exp["cu_k"])
        row_bits = (bdattn.STATUS_LAYOUT if exp["layout_error"] else 0) | \
                   (bdattn.STATUS_KV_RANGE if exp["kv_range_error"] else 0)
        assert got["row_status"] == row_bits, (b, got["row_status"], row_bits)
        exp_status |= row_bits
    assert status == exp_status
    return tab


@pytest.mark.parametrize("key", ["C1", "C2", "C3", "C4", "C5", "C5w4096", "C5w512"])
def test_segments_named_workloads(key):
    w = synth.WORKLOADS[key]
    doc = synth.doc_layout(w.layout, w.B, w.S, 0)
    for r in w.ranks:
        if w.kv == "needed":
            og = oracle.geom(w.B, 1, 1, 64, w.S, w.L, r * w.L, 0, w.S, w.window)
            segs = oracle.segments(doc, og)
            kvo = min(s["s_first"] for s in segs)
            skv = max(s["real_end"] for s in segs) - kvo
        else:
            kvo, skv = w.prefix_kv(r)
        _check_segments(doc, w.B, w.S, w.L, r * w.L, kvo, skv, w.window)


def _layouts():
    out = []
    rng = np.random.default_rng(7)
    for seed in range(8):
        out.append(("uniform", synth.doc_layout(("uniform", 1, 300, 200), 3, 2048, seed)))
    out.append(("single", synth.doc_layout(("single",), 1, 2048)))
    out.append(("ones", np.concatenate([np.arange(1, 2001, dtype=np.int32), np.zeros(47, np.int32)])[None]))
    # distinct but not increasing ids (valid: each id one contiguous run)
    perm = rng.permutation(np.arange(1, 40)).astype(np.int32)
    out.append(("shuffled", np.repeat(perm, 50)[None, :2048] if len(np.repeat(perm, 50)) >= 2048 else
                np.concatenate([np.repeat(perm, 50), np.zeros(2048 - 39 * 50, np.int32)])[None]))
    # invalid: an id reused in two runs
    bad = synth.doc_layout(("uniform", 50, 300, 100), 1, 2048, 3).copy()
    bad[0, 1500:1600] = bad[0, 10]
    out.append(("reuse", bad))
    # invalid: a document after padding
    bad2 = synth.doc_layout(("uniform", 50, 300, 300), 1, 2048, 4).copy()
    bad2[0, -1] = 77
    out.append(("after_pad", bad2))
    # invalid: negative id
    bad3 = synth.doc_layout(("uniform", 50, 300, 0), 1, 2048, 5).copy()
    bad3[0, 0] = -3
    out.append(("negative", bad3))
    return out


@pytest.mark.parametrize("name,doc", _layouts())
def test_segments_random_and_invalid_layouts(name, doc):
    B, S = doc.shape
    for cp in (1, 4, 16):
        L = S // cp
        for r in range(cp):
            _check_segments(doc, B, S, L, r * L, 0, S, 0)
            _check_segments(doc, B, S, L, r * L, 0, S, 37)


def test_kv_range_errors():
    doc = synth.doc_layout(("uniform", 100, 600, 64), 2, 2048, 1)
    L = 512
    for r in range(4):
        ro = r * L
        for kvo, skv, win in ((ro, L, 0), (ro - 100 if ro >= 100 else 0, 300, 0), (0, ro + 1, 0), (ro - 8, L + 8, 9),
                              (ro - 7, L + 7, 9), (max(0, ro - 300), L + min(ro, 300), 0)):
            if kvo < 0 or kvo + skv > 2048 or skv < 1:
                continue
            _check_segments(doc, 2, 2048, L, ro, kvo, skv, win)


def _brute_tiles(doc, B, S, L, ro, kvo, skv, window):
    """Classification of every 128x128 tile from the oracle's dense mask (real rows only)."""
    og = oracle.geom(B, 1, 1, 64, S, L, ro, kvo, skv, window)
    m = oracle.mask(doc, og)
    real = doc[:, ro:ro + L] != 0
    m = m & real[:, :, None]
    nqt, nkt = -(-L // 128), -(-skv // 128)
    cls = np.zeros((B, nqt, nkt), np.int32)  # 0 empty, 1 partial, 2 full
    for b in range(B):
        for qt in range(nqt):
            for kt in range(nkt):
                t = m[b, qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
                if t.any():
                    cls[b, qt, kt] = 2 if (t.shape == (128, 128) and t.all()) else 1
    return cls, m


@pytest.mark.parametrize("seed,window,cp,kvmode", [(0, 0, 4, "full"), (1, 100, 4, "full"), (2, 0, 8, "needed"),
                                                   (3, 300, 2, "prefix"), (4, 0, 1, "full"), (5, 1, 4, "full")])
def test_tile_classification(seed, window, cp, kvmode):
    B, S = 2, 2048
    doc = synth.doc_layout(("uniform", 20, 700, 150), B, S, seed)
    L = S // cp
    for r in range(cp):
        ro = r * L
        if kvmode == "full":
            kvo, skv = 0, S
        elif kvmode == "prefix":
            kvo, skv = 0, ro + L
        else:
            segs = oracle.segments(doc, oracle.geom(B, 1, 1, 64, S, L, ro, 0, S, window))
            kvo = min(s["s_first"] for s in segs)
            skv = max(1, max(s["real_end"] for s in segs) - kvo)
        tab = _check_segments(doc, B, S, L, ro, kvo, skv, window)
        cls, m = _brute_tiles(doc, B, S, L, ro, kvo, skv, window)
        nqt, nkt = cls.shape[1:]
        attended = set()  # K/V tiles (b * nkt + kt) some local row attends
        for b in range(B):
            row = tab["rows"][b]
            for qt in range(nqt):
                nz = np.nonzero(cls[b, qt])[0]
                lo, hi = row["qt_krange"][qt]
                if nz.size == 0:
                    assert hi < lo, (b, qt, lo, hi)
                    continue
                assert (lo, hi) == (nz[0], nz[-1]) and nz.size == hi - lo + 1, (b, qt, lo, hi, nz)
                for kt in range(lo, hi + 1):
                    bit = (int(row["full_bits"][qt][kt >> 5]) >> (kt & 31)) & 1
                    assert bit == (cls[b, qt, kt] == 2), (b, qt, kt, bit, cls[b, qt, kt])
            for kt in range(nkt):
                rows = np.nonzero(m[b, :, kt * 128:(kt + 1) * 128].any(axis=1))[0]
                a, e = row["kt_qrange"][kt]
                if rows.size == 0:
                    assert a == e == 0
                else:
                    attended.add(b * nkt + kt)
                    assert (a, e) == (rows[0], rows[-1] + 1) and rows.size == e - a, (b, kt, a, e, rows)
        n_full, n_part = int((cls == 2).sum()), int((cls == 1).sum())
        assert tuple(tab["counts"][:3]) == (n_full, n_part, cls.size - n_full - n_part)
        # the attended K/V tiles are counted and lead the backward work list
        assert int(tab["counts"][3]) == len(attended)
        assert set(tab["bwd_work"][:len(attended)].tolist()) == attended
        # work lists: permutations ordered by decreasing work
        fw = tab["fwd_work"]
        assert sorted(fw.tolist()) == list(range(B * nqt))
        kr = np.concatenate([tab["rows"][b]["qt_krange"] for b in range(B)])
        fkey = np.where(kr[:, 1] >= kr[:, 0], kr[:, 1] - kr[:, 0] + 1, 0)[fw]
        assert (np.diff(fkey) <= 0).all()
        bw = tab["bwd_work"]
        assert sorted(bw.tolist()) == list(range(B * nkt))
        qr = np.concatenate([tab["rows"][b]["kt_qrange"] for b in range(B)])
        bkey = np.where(qr[:, 1] > qr[:, 0], (qr[:, 1] - 1) // 64 - qr[:, 0] // 64 + 1, 0)[bw]
        assert (np.diff(bkey) <= 0).all()
