"""The C ABI on the host: the library loads, exports every symbol include/bdattn.h
declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from sliding_window_attention_device_gb300 import bdattn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bdattn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return bdattn.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_attn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in bdattn.h but not exported"
    assert set(names) == set(bdattn.EXPORTS)


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define\s+(BD_\w+)\s+(0x[0-9a-fA-F]+|\d+)", text))
    val = lambda k: int(consts[k], 0)
    assert val("BD_OK") == bdattn.BD_OK and val("BD_ERR_ARG") == bdattn.BD_ERR_ARG
    assert val("BD_STATUS_LAYOUT") == bdattn.STATUS_LAYOUT
    assert val("BD_STATUS_KV_RANGE") == bdattn.STATUS_KV_RANGE
    assert val("BD_STATUS_BOUNDS") == bdattn.STATUS_BOUNDS
    assert val("BD_STATUS_TIMEOUT") == bdattn.STATUS_TIMEOUT
    assert val("BD_SEG_HDR_WORDS") == bdattn.HDR_WORDS
    assert val("BD_SEG_NOFF") == len(bdattn.REGIONS)
    for i, name in enumerate(("N_REAL", "N_SEG", "S_FIRST", "REAL_END", "MAX_Q", "MAX_K", "FIRST_Q", "FIRST_K",
                              "MAX_TAIL", "KV_NEED_LO", "ROW_STATUS")):
        assert val(f"BD_SEG_{name}") == i and bdattn.HDR_FIELDS[i] == name.lower().replace("row_status", "row_status")


def test_sizes_and_layout(lib):
    g = bdattn.geom(2, 32, 8, 128, 32768, 4096, 0, 0, 32768)
    lay = bdattn.seg_layout(g)
    assert lay["nqt"] == 32 and lay["nkt"] == 256 and lay["nkw"] == 8
    order = [lay[r] for r in bdattn.REGIONS]
    assert order == sorted(order) and all(o % 4 == 0 for o in order)
    assert bdattn.seg_bytes(g) == 4 * lay["total"]
    assert lay["cu_k"] - lay["cu_q"] >= 2 * 4097
    rows = 2 * 32 * 4096
    assert bdattn.bwd_workspace_bytes(g) >= rows * 128 * 4 + rows * 4


@pytest.mark.parametrize("bad", [
    dict(D=96), dict(Hq=6, Hkv=4), dict(L=0), dict(row_offset=32000), dict(kv_offset=-1),
    dict(S_kv=40000), dict(B=0),
])
def test_bad_geometry_rejected(lib, bad):
    base = dict(B=1, Hq=4, Hkv=2, D=128, S_full=32768, L=4096, row_offset=0, kv_offset=0, S_kv=32768)
    base.update(bad)
    g = bdattn.geom(**base)
    assert lib.bd_attn_seg_bytes(ctypes.byref(g)) == 0
    assert lib.bd_attn_bwd_workspace_bytes(ctypes.byref(g)) == 0
    # argument checks run before any CUDA call, so this needs no GPU
    rc = lib.bd_attn_seg_build(ctypes.c_void_p(16), ctypes.byref(g), ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert rc == bdattn.BD_ERR_ARG


@pytest.mark.parametrize("D", [32, 96, 384, 1024])
def test_unsupported_head_dims_rejected(lib, D):
    g = bdattn.geom(1, 2, 1, D, 256, 64, 0, 0, 256)
    assert lib.bd_attn_seg_bytes(ctypes.byref(g)) == 0
    assert lib.bd_attn_bwd_workspace_bytes(ctypes.byref(g)) == 0


@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_every_head_dim_has_sizes(lib, D):
    """Every mode runs at every supported head dim: the table and the backward
    workspace (fp32 dq accumulator + delta) are sized for it."""
    g = bdattn.geom(1, 4, 2, D, 1024, 256, 256, 0, 1024)
    assert lib.bd_attn_seg_bytes(ctypes.byref(g)) > 0
    rows = 4 * 256
    assert lib.bd_attn_bwd_workspace_bytes(ctypes.byref(g)) >= rows * D * 4 + rows * 4


def test_null_pointers_rejected(lib):
    g = bdattn.geom(1, 2, 1, 64, 256, 64, 128, 0, 256)
    P = ctypes.c_void_p
    assert lib.bd_attn_seg_build(None, ctypes.byref(g), P(16), P(16), None) == bdattn.BD_ERR_ARG
    assert lib.bd_attn_fwd(P(16), None, P(16), P(16), ctypes.byref(g), P(16), P(16), P(16), None) == bdattn.BD_ERR_ARG
    assert lib.bd_attn_fwd(P(16), P(16), P(16), P(16), ctypes.byref(g), P(8), P(16), P(16), None) == bdattn.BD_ERR_ARG
    assert lib.bd_attn_bwd(P(16), P(16), P(16), P(16), P(16), P(16), P(16), ctypes.byref(g), 7, P(16), P(16), P(16),
                           P(256), P(16), None) == bdattn.BD_ERR_ARG
    assert lib.bd_attn_selftest_wait_timeout(None, 1000, None) == bdattn.BD_ERR_ARG
    assert bdattn.strerror(bdattn.BD_ERR_ARG).startswith("invalid argument")


def test_plan_constants_and_layout(lib):
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define\s+(BD_PLAN_\w+)\s+(0x[0-9a-fA-F]+|\d+)", text))
    for i, name in enumerate(bdattn.PLAN_HDR_FIELDS):
        assert int(consts[f"BD_PLAN_{name.upper()}"], 0) == i
    assert int(consts["BD_PLAN_HDR_WORDS"]) == bdattn.PLAN_HDR_WORDS
    assert int(consts["BD_PLAN_NOFF"]) == len(bdattn.PLAN_REGIONS)
    for i, name in enumerate(bdattn.PLAN_REGIONS):
        assert int(consts[f"BD_PLAN_OFF_{name.upper()}"]) == i
    B, W, L = 3, 8, 100
    lay = bdattn.plan_layout(B, W, L)
    sizes = dict(hdr=16, s_first=W, real_end=W, back=W, halo_send=W, counts=W * W, in_splits=W, out_splits=W,
                 send_off=W, recv_off=W, send_index=W * L, row_range=2 * B * W)
    names = bdattn.PLAN_REGIONS
    for a, b in zip(names[:-1], names[1:]):
        assert lay[a] % 4 == 0 and lay[b] - lay[a] >= sizes[a] and lay[b] - lay[a] < sizes[a] + 4
    assert bdattn.plan_bytes(B, W, L) == 4 * lay["total"]
    assert lib.bd_attn_plan_bytes(0, 8, 100) == 0 and lib.bd_attn_plan_bytes(1, 1025, 4) == 0
    assert lib.bd_attn_exchange_plan(None, 1, 64, 4, 0, None, None, None) == bdattn.BD_ERR_ARG


def test_kv_layout_constants_and_validation(lib):
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define\s+(BD_KV_\w+)\s+(\d+)", text))
    assert int(consts["BD_KV_BHSD"]) == bdattn.KV_BHSD and int(consts["BD_KV_SBHD"]) == bdattn.KV_SBHD
    fields = re.search(r"typedef struct \{(.*?)\} bd_geom;", text, re.S).group(1)
    names = re.findall(r"\b(?:int|float|uint32_t)\s+(\w+);", fields)
    assert names == [n for n, _ in bdattn.Geom._fields_]
    g = bdattn.geom(1, 2, 1, 64, 256, 64, 0, 0, 256, 0, kv_layout=bdattn.KV_SBHD)
    assert bdattn.kv_shape(g) == (256, 1, 1, 64) and lib.bd_attn_seg_bytes(ctypes.byref(g)) > 0
    g.kv_layout = 2
    assert lib.bd_attn_seg_bytes(ctypes.byref(g)) == 0


def test_deterministic_backward_rejects_null_pointers(lib):
    g = bdattn.geom(1, 2, 1, 512, 256, 64, 0, 0, 256, 0)
    assert lib.bd_attn_bwd_deterministic(None, None, None, None, None, None, None, ctypes.byref(g), 0, None, None,
                                         None, None, None, None) == bdattn.BD_ERR_ARG


def test_dropout_arguments_are_checked_on_the_host():
    """dropout_p outside [0, 1), or rounding to a threshold of 2^16, is refused
    before anything touches a device."""
    lib = bdattn.load()
    P = ctypes.c_void_p
    for p in (1.0, -0.1, float("nan"), 0.99999999):
        g = bdattn.geom(1, 2, 1, 128, 1024, 256, 256, 0, 1024, dropout_p=p, seed=3)
        assert lib.bd_attn_fwd(P(16), P(16), P(16), P(16), ctypes.byref(g), P(16), P(16), P(16), None) == \
            bdattn.BD_ERR_ARG, p
        assert lib.bd_attn_seg_bytes(ctypes.byref(g)) == 0
    for D in (64, 128, 256, 512):  # a valid probability passes the host checks at every head dim
        g = bdattn.geom(1, 2, 1, D, 1024, 256, 256, 0, 1024, dropout_p=0.1, seed=3)
        assert lib.bd_attn_seg_bytes(ctypes.byref(g)) > 0
