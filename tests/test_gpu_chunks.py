"""Chunked K/V (gemma4_moe.cp_local_ring: per-step forward over one K/V chunk
returning (out, lse), the -inf-safe merge of chunk results, and the per-chunk
backward with the globally merged out / lse), on the GPU through the C ABI,
against the fp64 oracle.

Each case splits the shard's K/V range into chunks, some of whose edges fall
inside a 128-row tile, plus one chunk after the shard's rows that no row sees:
  * every chunk's forward matches oracle.fwd_chunk (rows with no key in the
    chunk: out = 0, lse = -inf);
  * merging all chunks on the GPU, from lse = -inf over a NaN-filled out,
    matches the full-range oracle forward, both with the merge kernel and
    with the forward's merging epilogue;
  * prep once with the merged out / lse, then one backward main per chunk
    (dq accumulating, dk / dv per chunk) matches the full-range oracle backward.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import LSE_ABS, assert_close, make_case
from sliding_window_attention_device_gb300 import synth

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = [
    # name, workload, rank, chunk edges inside the case's K/V buffer (None: its end)
    ("d128_ragged", W("ca", "chunked, D 128, ragged shard", B=2, Hq=4, Hkv=2, D=128, S=1280, cp_size=4,
                      layout=("uniform", 20, 300, 40)), 2, (0, 200, 384, 700, None)),
    ("d64_window", W("cb", "chunked, D 64, window 100", B=1, Hq=3, Hkv=3, D=64, S=1024, cp_size=2,
                     layout=("uniform", 50, 400, 70), window=100), 1, (0, 128, 517, None)),
    ("d256_window", W("cc", "chunked, D 256, window 150", B=1, Hq=4, Hkv=2, D=256, S=1280, cp_size=4,
                      layout=("uniform", 100, 600, 30), window=150, kv="prefix"), 3, (0, 830, 1000, None)),
    ("d256_after", W("ce", "chunked, D 256, GQA 2, a chunk after the rows", B=2, Hq=4, Hkv=2, D=256, S=1024,
                     cp_size=4, layout=("uniform", 60, 500, 20), kv="prefix"), 1, (0, 200, None)),
    ("d512_prefix", W("cd", "chunked, D 512, GQA 2", B=1, Hq=4, Hkv=2, D=512, S=1024, cp_size=4,
                      layout=("uniform", 60, 500, 20), kv="prefix"), 2, (0, 300, 700, None)),
]


def _geom(w, c, kv_offset, S_kv):
    from sliding_window_attention_device_gb300 import bdattn
    return bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], kv_offset, S_kv, w.window)


def _ogeom(w, c, kv_offset, S_kv):
    return oracle.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], kv_offset, S_kv, w.window)


def _chunks(c, edges):
    """(kv_offset, S_kv, lo, hi) of each chunk [lo, hi) of the case's K/V buffer."""
    e = [x if x is not None else c["S_kv"] for x in edges]
    return [(c["kv_offset"] + a, b - a, a, b) for a, b in zip(e[:-1], e[1:]) if b > a]


@pytest.mark.parametrize("name,w,r,edges", CASES, ids=[x[0] for x in CASES])
def test_chunked_forward_merge_and_backward(name, w, r, edges):
    from sliding_window_attention_device_gb300 import bdattn
    dev = torch.device("cuda")
    c = make_case(w, r)
    doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
    q, do = c["q"].to(dev), c["do"].to(dev)
    chunks = _chunks(c, edges)
    # a chunk after the shard's last row: keys every local row is causally blind to
    after = c["row_offset"] + w.L
    if after + 128 <= w.S:
        k_after, v_after = synth.kv_rows(w, 0, after, after + 128)
        extra = (after, 128, k_after, v_after)
    else:
        extra = None

    # forward per chunk, merged on the GPU: by the merge kernel (acc_*) and by
    # the forward's own merging epilogue (fus_*), both from lse = -inf over a
    # NaN-filled out
    g_full = _geom(w, c, c["kv_offset"], c["S_kv"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    acc_out = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    acc_lse = torch.full((w.B, w.Hq, w.L), float("-inf"), dtype=torch.float32, device=dev)
    fus_out, fus_lse = acc_out.clone(), acc_lse.clone()
    runs = []
    for kv_off, S_kv, lo, hi in chunks:
        runs.append((kv_off, S_kv, c["k"][:, :, lo:hi].contiguous(), c["v"][:, :, lo:hi].contiguous()))
    if extra is not None:
        runs.append(extra)
    segs = []
    for kv_off, S_kv, k, v in runs:
        g = _geom(w, c, kv_off, S_kv)
        seg, _ = bdattn.bd_attn_seg_build_chunk(doc, g, status=status)
        out = torch.full_like(acc_out, float("nan"))
        lse = torch.full_like(acc_lse, float("nan"))
        kd, vd = k.to(dev), v.to(dev)
        bdattn.bd_attn_fwd(q, kd, vd, seg, g, status, out=out, lse=lse)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref_out, ref_lse = oracle.fwd_chunk(c["q"], k, v, c["doc"], _ogeom(w, c, kv_off, S_kv))
        got_lse = lse.double().cpu().numpy()
        assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), f"{name}: empty rows differ"
        fin = np.isfinite(ref_lse)
        assert np.abs(got_lse[fin] - ref_lse[fin]).max(initial=0.0) <= LSE_ABS
        assert_close(f"{name} chunk [{kv_off},{kv_off + S_kv}) out", out, ref_out)
        bdattn.bd_attn_merge(acc_out, acc_lse, out, lse, g, status)
        bdattn.bd_attn_fwd_merge(q, kd, vd, seg, g, status, fus_out, fus_lse)
        segs.append((g, seg, kd, vd))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    full_out, full_lse = oracle.fwd(c["q"], c["k"], c["v"], c["doc"], _ogeom(w, c, c["kv_offset"], c["S_kv"]))
    got_lse = acc_lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(full_lse))
    fin = np.isfinite(full_lse)
    assert np.abs(got_lse[fin] - full_lse[fin]).max(initial=0.0) <= LSE_ABS
    assert_close(f"{name} merged out", acc_out, full_out)
    got_lse = fus_lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(full_lse))
    assert np.abs(got_lse[fin] - full_lse[fin]).max(initial=0.0) <= LSE_ABS
    assert_close(f"{name} forward-merged out", fus_out, full_out)

    # backward per chunk with the merged out / lse
    ws = torch.empty(bdattn.bwd_workspace_bytes(g_full), dtype=torch.uint8, device=dev)
    dq = torch.full((w.B, w.Hq, w.L, w.D), float("nan"), dtype=torch.float32, device=dev)
    bdattn.bd_attn_bwd_prep(do, acc_out, g_full, status, ws)
    dks, dvs = [], []
    for g, seg, kd, vd in segs:
        dk = torch.full((w.B, w.Hkv, g.S_kv, w.D), float("nan"), dtype=torch.float32, device=dev)
        dv = torch.full_like(dk, float("nan"))
        bdattn.bd_attn_bwd_main(do, q, kd, vd, acc_lse, seg, g, status, ws, dk, dv)
        dks.append(dk)
        dvs.append(dv)
    bdattn.bd_attn_bwd_finalize(g_full, status, ws, dq)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_dq, ref_dk, ref_dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"],
                                        _ogeom(w, c, c["kv_offset"], c["S_kv"]))
    n_main = len(chunks)
    assert_close(f"{name} dq", dq, ref_dq)
    assert_close(f"{name} dk", torch.cat(dks[:n_main], dim=2), ref_dk)
    assert_close(f"{name} dv", torch.cat(dvs[:n_main], dim=2), ref_dv)
    if extra is not None:  # no row sees the chunk after the rows: zero gradients there
        assert (dks[-1] == 0).all() and (dvs[-1] == 0).all()


@pytest.mark.parametrize("D", [64, 512])
def test_merge_edge_cases(D):
    """Both sides empty stays (0, -inf); an empty side is the identity even
    when its out is not finite; merging equal lse gives the average."""
    from sliding_window_attention_device_gb300 import bdattn
    dev = torch.device("cuda")
    g = bdattn.geom(1, 2, 1, D, 256, 128, 0, 0, 256, 0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(5)
    a = torch.randn(1, 2, 128, D, generator=gen).to(torch.bfloat16)
    b = torch.randn(1, 2, 128, D, generator=gen).to(torch.bfloat16)
    la = torch.randn(1, 2, 128, generator=gen) * 3
    lb = torch.randn(1, 2, 128, generator=gen) * 3
    # rows 0..31: a empty; 32..63: b empty; 64..95: both empty; 96..127: equal lse
    la[..., 0:32] = float("-inf")
    lb[..., 32:64] = float("-inf")
    la[..., 64:96] = float("-inf")
    lb[..., 64:96] = float("-inf")
    lb[..., 96:] = la[..., 96:]
    a_in = a.clone()
    a_in[..., 0:32, :] = float("nan")  # an empty side may hold anything
    out, lse = a_in.to(dev), la.to(dev)
    bdattn.bd_attn_merge(out, lse, b.to(dev), lb.to(dev), g, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_out, ref_lse = oracle.merge(a.double().numpy(), la.double().numpy(), b.double().numpy(), lb.double().numpy())
    got_out, got_lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(got_out).all()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=1e-5)
    np.testing.assert_allclose(got_out, ref_out, rtol=0, atol=2e-2)
    assert (got_out[..., 64:96, :] == 0).all()
    np.testing.assert_array_equal(got_out[..., 32:64, :], a.double().numpy()[..., 32:64, :])


@pytest.mark.slow
@pytest.mark.parametrize("key,r,fused", [("C2", 3, True), ("C2", 7, False), ("C3", 7, True), ("C5w512", 5, True),
                                         ("G512", 6, True)])
def test_ring_chunks_full_size_sampled(key, r, fused):
    """Full size, through the chunking and calls the benchmark's ring modes time
    (merges in the forward's epilogue, or by the merge kernel):
    sampled rows (out, lse, dq) and keys (dk, dv) against the oracle over the
    whole K/V range; keys in a skipped block get no gradient from any row; and
    sum over all keys of dV equals the sum of dO over the real rows."""
    import bench
    from test_gpu_full import _oracle_sampled, _pick, _check
    w = synth.WORKLOADS[key]
    dev = torch.device("cuda")
    rep = bench.RingChunkReplica(w, 0, dev, torch.float32, ranks={r}, fused=fused)
    rep.step()
    torch.cuda.synchronize()
    assert int(rep.status.item()) == 0
    s = rep.shards[0]
    c = make_case(w, r, seed=0)
    assert (c["kv_offset"], c["S_kv"]) == (s["g"].kv_offset, s["g"].S_kv)
    rows, keys = _pick(c, np.random.default_rng(321))
    ref_rows, ref_keys = _oracle_sampled(c, rows, keys)
    out, lse, dq = s["out"].float().cpu(), s["lse"].cpu(), s["dq"].cpu()
    for (b, h, i), (o_ref, l_ref, dq_ref) in ref_rows.items():
        _check(f"{key} r{r} out[{b},{h},{i}]", out[b, h, i].numpy(), o_ref)
        _check(f"{key} r{r} dq[{b},{h},{i}]", dq[b, h, i].numpy(), dq_ref)
        if np.isneginf(l_ref):
            assert torch.isneginf(lse[b, h, i])
        else:
            assert abs(float(lse[b, h, i]) - l_ref) <= LSE_ABS
    for (b, hk, j), (dk_ref, dv_ref) in ref_keys.items():
        pos = c["kv_offset"] + j
        ch = [x for x in s["chunks"] if x["g"].kv_offset <= pos < x["g"].kv_offset + x["g"].S_kv]
        if not ch:  # a skipped block: no local row may reach it
            assert not np.any(dk_ref) and not np.any(dv_ref), (key, r, b, hk, j)
            continue
        jj = pos - ch[0]["g"].kv_offset
        _check(f"{key} r{r} dk[{b},{hk},{j}]", ch[0]["dk"][b, hk, jj].cpu().numpy(), dk_ref)
        _check(f"{key} r{r} dv[{b},{hk},{j}]", ch[0]["dv"][b, hk, jj].cpu().numpy(), dv_ref)
    real = torch.from_numpy(c["doc"][:, c["row_offset"]:c["row_offset"] + w.L] != 0).to(dev)
    do = s["do"].double() * real[:, None, :, None]
    lhs = sum(x["dv"].double().sum(2) for x in s["chunks"])
    rhs = do.view(w.B, w.Hkv, w.G, w.L, w.D).sum((2, 3))
    rel = ((lhs - rhs).norm() / rhs.norm().clamp_min(1e-30)).item()
    assert rel < 1e-2, f"{key} r{r}: sum dV identity rel err {rel:.3e}"
