"""Failure handling on the GPU without any fault: bad layouts and K/V ranges set
status bits and later kernels skip their work; a bounded wait that nobody
releases reports a timeout instead of hanging."""
import numpy as np
import pytest
import torch

from sliding_window_attention_device_gb300 import bdattn, synth

pytestmark = pytest.mark.gpu


def _inputs(g, seed=0):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(g.B, g.Hq, g.L, g.D, generator=gen).bfloat16().cuda()
    k = torch.randn(g.B, g.Hkv, g.S_kv, g.D, generator=gen).bfloat16().cuda()
    v = torch.randn(g.B, g.Hkv, g.S_kv, g.D, generator=gen).bfloat16().cuda()
    return q, k, v


def _run(doc, g):
    d = torch.from_numpy(np.ascontiguousarray(doc, dtype=np.int32)).cuda()
    seg, status = bdattn.bd_attn_seg_build(d, g)
    q, k, v = _inputs(g)
    sentinel = torch.full((g.B, g.Hq, g.L, g.D), 7.0, dtype=torch.bfloat16, device="cuda")
    out, lse = bdattn.bd_attn_fwd(q, k, v, seg, g, status, out=sentinel.clone())
    dq, dk, dv = bdattn.bd_attn_bwd(q, q, k, v, out, lse, seg, g, status,
                                    dq=torch.full((g.B, g.Hq, g.L, g.D), 7.0, device="cuda"))
    torch.cuda.synchronize()
    return int(status.item()), out, dq


def test_layout_error_skips_work():
    doc = synth.doc_layout(("uniform", 50, 300, 100), 1, 1024, 2).copy()
    doc[0, 1023] = 5  # a document after the padding tail
    g = bdattn.geom(1, 2, 1, 128, 1024, 256, 512, 0, 1024)
    st, out, dq = _run(doc, g)
    assert st & bdattn.STATUS_LAYOUT
    assert (out.float() == 7.0).all() and (dq == 7.0).all()  # untouched


def test_kv_range_error_skips_work():
    doc = synth.doc_layout(("uniform", 300, 600, 0), 1, 1024, 3)
    g = bdattn.geom(1, 2, 1, 128, 1024, 256, 512, 600, 168)  # K/V misses local rows 512..599
    st, out, dq = _run(doc, g)
    assert st == bdattn.STATUS_KV_RANGE
    assert (out.float() == 7.0).all() and (dq == 7.0).all()


def test_geometry_mismatch_sets_bounds():
    doc = synth.doc_layout(("uniform", 50, 300, 10), 1, 1024, 4)
    g = bdattn.geom(1, 2, 1, 128, 1024, 256, 256, 0, 1024)
    d = torch.from_numpy(doc).cuda()
    seg, status = bdattn.bd_attn_seg_build(d, g)
    g2 = bdattn.geom(1, 2, 1, 128, 1024, 256, 512, 0, 1024)  # table built for another shard
    q, k, v = _inputs(g2)
    bdattn.bd_attn_fwd(q, k, v, seg, g2, status)
    torch.cuda.synchronize()
    assert int(status.item()) & bdattn.STATUS_BOUNDS


def test_bounded_wait_times_out():
    status = bdattn.new_status("cuda")
    bdattn.selftest_wait_timeout(20_000_000, status)  # 20 ms, nobody arrives
    torch.cuda.synchronize()
    assert int(status.item()) == bdattn.STATUS_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda") * 2
    assert x.sum().item() == 8.0


def test_argument_errors_raise():
    g = bdattn.geom(1, 2, 1, 128, 1024, 256, 512, 0, 1024)
    with pytest.raises(ValueError):
        bdattn.bd_attn_seg_build(torch.zeros(1, 1000, dtype=torch.int32, device="cuda"), g)
    with pytest.raises(ValueError):
        bdattn.bd_attn_seg_build(torch.zeros(1, 1024, dtype=torch.int64, device="cuda"), g)
