"""The allocation-free backward, bd_attn_bwd_noalloc, called through the C ABI.

Some callers can give the library their input and output buffers but cannot
allocate device memory while they run (a host that reserved its whole memory
budget at start-up, a plugin whose framework allows only its own allocator).
This entry point keeps the backward's scratch in a static per-GPU array
instead of a caller workspace. Its results must match bd_attn_bwd's and the
fp64 oracle's within the parity tolerance, in both gradient dtypes, on
consecutive calls that reuse the same scratch (the first call on a different
problem, so that anything the second call failed to clear would show), with
and without attention dropout, and a problem larger than the scratch must be
refused with a clear error.

This file is collected last, so that a run stopping at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import MAX_ABS, MEAN_ABS, assert_close, assert_close_bf16, make_case, oracle_geom
from sliding_window_attention_device_gb300 import bdattn, synth

pytestmark = pytest.mark.gpu

SCRATCH_TOO_SMALL = 4
DTYPES = {"f32": (bdattn.BD_DTYPE_F32, torch.float32), "bf16": (bdattn.BD_DTYPE_BF16, torch.bfloat16)}


def _noalloc():
    lib = bdattn.load()
    f = lib.bd_attn_bwd_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(bdattn.Geom), ctypes.c_int, P, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def test_noalloc_setup_call():
    """Every pointer NULL: only the per-device set-up, nothing enqueued."""
    f = _noalloc()
    assert f(*([None] * 7), None, 0, *([None] * 5)) == 0


@pytest.mark.parametrize("drop", [0.0, 0.3])
@pytest.mark.parametrize("dtype", sorted(DTYPES))
def test_noalloc_matches_bwd_and_oracle_on_consecutive_calls(dtype, drop):
    code, tdt = DTYPES[dtype]
    w = synth.Workload("N", "noalloc", B=2, Hq=4, Hkv=2, D=128, S=1280, cp_size=4,
                       layout=("uniform", 20, 300, 40), window=0)
    dev = torch.device("cuda")
    f = _noalloc()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two different problems of the same geometry, one call each, in a row
    for call, seed in enumerate((7, 3)):
        c = make_case(w, 2, seed=seed)
        c["dropout_p"], c["drop_seed"] = drop, 1000 + seed
        g = bdattn.geom(w.B, w.Hq, w.Hkv, w.D, w.S, w.L, c["row_offset"], c["kv_offset"], c["S_kv"], w.window,
                        dropout_p=drop, seed=1000 + seed)
        assert bdattn.bwd_workspace_bytes(g) <= (16 << 20)
        doc = torch.from_numpy(np.ascontiguousarray(c["doc"])).to(dev)
        q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
        seg, status = bdattn.bd_attn_seg_build(doc, g)
        out, lse = bdattn.bd_attn_fwd(q, k, v, seg, g, status)
        ref = bdattn.bd_attn_bwd(do, q, k, v, out, lse, seg, g, status, grad_dtype=tdt)
        dq = torch.full_like(ref[0], float("nan"))
        dk = torch.full_like(ref[1], float("nan"))
        dv = torch.full_like(ref[2], float("nan"))
        rc = f(P(do), P(q), P(k), P(v), P(out), P(lse), P(seg), ctypes.byref(g), code, P(dq), P(dk), P(dv),
               P(status), stream)
        assert rc == 0, bdattn.strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        og = oracle_geom(c)
        o_dq, o_dk, o_dv = oracle.bwd(c["q"], c["k"], c["v"], c["do"], c["doc"], og)
        close = assert_close if dtype == "f32" else assert_close_bf16
        # with dropout the parity bar is scaled by the keep scale 2^16 / (2^16 - T)
        keep = 65536.0 / (65536 - int(np.floor(drop * 65536 + 0.5)))
        bar = (MAX_ABS * keep, MEAN_ABS * keep)
        for name, got, r, o in (("dq", dq, ref[0], o_dq), ("dk", dk, ref[1], o_dk), ("dv", dv, ref[2], o_dv)):
            assert got.dtype == tdt
            close(f"call {call} {name} vs bd_attn_bwd", got, r.double().cpu().numpy(), *bar)
            close(f"call {call} {name} vs oracle", got, o, *bar)
        # the same kernels sum dK / dV inside one CTA in a fixed order
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_noalloc_refuses_problems_larger_than_its_scratch():
    g = bdattn.geom(2, 32, 8, 128, 32768, 4096, 0, 0, 32768)  # needs ~135 MB of scratch
    assert bdattn.bwd_workspace_bytes(g) > (16 << 20)
    f = _noalloc()
    P = ctypes.c_void_p
    rc = f(P(16), P(16), P(16), P(16), P(16), P(16), P(16), ctypes.byref(g), bdattn.BD_DTYPE_F32, P(16), P(16),
           P(16), P(16), None)
    assert rc == SCRATCH_TOO_SMALL
    assert "16 MiB" in bdattn.strerror(rc)
