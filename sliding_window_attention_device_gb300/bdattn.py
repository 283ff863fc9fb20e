"""ctypes binding of libbdattn.so (declared in include/bdattn.h).

Argument marshalling only: every computation runs in the CUDA kernels behind
the C ABI. Tensors are PyTorch CUDA tensors (PyTorch provides the device
memory and the current stream); outputs the caller does not pass are
allocated here with torch. There is no CPU fallback: without the compiled
library, or without a GPU, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbdattn.so")

# return codes
BD_OK, BD_ERR_ARG, BD_ERR_CUDA, BD_ERR_UNSUPPORTED = 0, 1, 2, 3
# device status bits
STATUS_LAYOUT, STATUS_KV_RANGE, STATUS_BOUNDS, STATUS_TIMEOUT = 0x1, 0x2, 0x4, 0x8
# gradient dtypes
BD_DTYPE_F32, BD_DTYPE_BF16 = 0, 1
# per-row header fields of the segment table
HDR_FIELDS = ("n_real", "n_seg", "s_first", "real_end", "max_q", "max_k", "first_q", "first_k", "max_tail",
              "kv_need_lo", "row_status")
HDR_WORDS = 32
# region indices of the segment table (BD_SEG_OFF_*)
REGIONS = ("hdr", "cu_q", "cu_k", "row_lo", "qt_krange", "kt_qrange", "full_bits", "fwd_work", "bwd_work",
           "counts", "total")

EXPORTS = ("bd_attn_seg_bytes", "bd_attn_seg_layout", "bd_attn_seg_build", "bd_attn_seg_build_chunk",
           "bd_attn_fwd", "bd_attn_fwd_merge", "bd_attn_merge",
           "bd_attn_bwd_workspace_bytes", "bd_attn_bwd", "bd_attn_bwd_deterministic", "bd_attn_bwd_prep",
           "bd_attn_bwd_main",
           "bd_attn_bwd_finalize", "bd_attn_bwd_prep_dq", "bd_attn_bwd_main_dq",
           "bd_attn_bwd_noalloc", "bd_attn_plan_bytes", "bd_attn_plan_layout", "bd_attn_exchange_plan",
           "bd_attn_needed_gather", "bd_attn_needed_scatter_add", "bd_attn_strerror",
           "bd_attn_selftest_wait_timeout")

# exchange plan: header fields (BD_PLAN_*) and regions (BD_PLAN_OFF_*)
PLAN_HDR_FIELDS = ("magic", "cp_size", "L", "rank", "B", "use_halo", "halo_size", "total_send", "total_recv")
PLAN_HDR_WORDS = 16
PLAN_REGIONS = ("hdr", "s_first", "real_end", "back", "halo_send", "counts", "in_splits", "out_splits", "send_off",
                "recv_off", "send_index", "row_range", "total")
PLAN_MAGIC = 0x62647870


class Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("S_full", ctypes.c_int), ("L", ctypes.c_int), ("row_offset", ctypes.c_int),
                ("kv_offset", ctypes.c_int), ("S_kv", ctypes.c_int), ("window", ctypes.c_int),
                ("scale", ctypes.c_float), ("kv_layout", ctypes.c_int), ("dropout_p", ctypes.c_float),
                ("seed_lo", ctypes.c_uint32), ("seed_hi", ctypes.c_uint32)]

    def __repr__(self):
        return "Geom(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


KV_BHSD, KV_SBHD = 0, 1  # K/V layouts: [B, Hkv, S_kv, D] or token-major [S_kv, B, Hkv, D]


def geom(B, Hq, Hkv, D, S_full, L, row_offset, kv_offset, S_kv, window=0, scale=0.0, kv_layout=KV_BHSD,
         dropout_p=0.0, seed=0) -> Geom:
    """Geometry of one query shard: local rows [row_offset, row_offset+L) of a
    padded sequence of S_full positions, K/V buffer rows = positions
    [kv_offset, kv_offset+S_kv). scale <= 0 means D**-0.5; window <= 0: none;
    kv_layout: KV_BHSD or KV_SBHD (token-major k, v, dk, dv); dropout_p > 0:
    attention dropout drawn from the 64-bit `seed` (the same p and seed in the
    forward and the backward of a step)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return Geom(int(B), int(Hq), int(Hkv), int(D), int(S_full), int(L), int(row_offset), int(kv_offset),
                int(S_kv), int(window), float(scale or 0.0), int(kv_layout), float(dropout_p), seed & 0xFFFFFFFF,
                seed >> 32)


def kv_shape(g: Geom) -> tuple:
    """Shape of k, v, dk, dv for the geometry's K/V layout."""
    return (g.S_kv, g.B, g.Hkv, g.D) if g.kv_layout == KV_SBHD else (g.B, g.Hkv, g.S_kv, g.D)


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libbdattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m sliding_window_attention_device_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, G = ctypes.c_void_p, ctypes.POINTER(Geom)
        lib.bd_attn_seg_bytes.argtypes = [G]
        lib.bd_attn_seg_bytes.restype = ctypes.c_size_t
        lib.bd_attn_seg_layout.argtypes = [G, P]
        lib.bd_attn_seg_layout.restype = ctypes.c_int
        lib.bd_attn_bwd_workspace_bytes.argtypes = [G]
        lib.bd_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.bd_attn_seg_build.argtypes = [P, G, P, P, P]
        lib.bd_attn_seg_build.restype = ctypes.c_int
        lib.bd_attn_seg_build_chunk.argtypes = [P, G, P, P, P]
        lib.bd_attn_seg_build_chunk.restype = ctypes.c_int
        lib.bd_attn_merge.argtypes = [P, P, P, P, G, P, P]
        lib.bd_attn_merge.restype = ctypes.c_int
        lib.bd_attn_fwd.argtypes = [P, P, P, P, G, P, P, P, P]
        lib.bd_attn_fwd.restype = ctypes.c_int
        lib.bd_attn_fwd_merge.argtypes = [P, P, P, P, G, P, P, P, P]
        lib.bd_attn_fwd_merge.restype = ctypes.c_int
        lib.bd_attn_bwd.argtypes = [P, P, P, P, P, P, P, G, ctypes.c_int, P, P, P, P, P, P]
        lib.bd_attn_bwd.restype = ctypes.c_int
        lib.bd_attn_bwd_deterministic.argtypes = [P, P, P, P, P, P, P, G, ctypes.c_int, P, P, P, P, P, P]
        lib.bd_attn_bwd_deterministic.restype = ctypes.c_int
        lib.bd_attn_bwd_prep.argtypes = [P, P, G, P, P, P]
        lib.bd_attn_bwd_prep.restype = ctypes.c_int
        lib.bd_attn_bwd_main.argtypes = [P, P, P, P, P, P, G, ctypes.c_int, P, P, P, P, P]
        lib.bd_attn_bwd_main.restype = ctypes.c_int
        lib.bd_attn_bwd_finalize.argtypes = [G, ctypes.c_int, P, P, P, P]
        lib.bd_attn_bwd_finalize.restype = ctypes.c_int
        lib.bd_attn_bwd_prep_dq.argtypes = [P, P, G, P, P, P, P]
        lib.bd_attn_bwd_prep_dq.restype = ctypes.c_int
        lib.bd_attn_bwd_main_dq.argtypes = [P, P, P, P, P, P, G, ctypes.c_int, P, P, P, P, P, P]
        lib.bd_attn_bwd_main_dq.restype = ctypes.c_int
        I = ctypes.c_int
        lib.bd_attn_plan_bytes.argtypes = [I, I, I]
        lib.bd_attn_plan_bytes.restype = ctypes.c_size_t
        lib.bd_attn_plan_layout.argtypes = [I, I, I, P]
        lib.bd_attn_plan_layout.restype = I
        lib.bd_attn_exchange_plan.argtypes = [P, I, I, I, I, P, P, P]
        lib.bd_attn_exchange_plan.restype = I
        lib.bd_attn_needed_gather.argtypes = [P, P, I, I, I, I, I, P, I, P, P]
        lib.bd_attn_needed_gather.restype = I
        lib.bd_attn_needed_scatter_add.argtypes = [P, P, I, I, I, I, I, P, I, P, P]
        lib.bd_attn_needed_scatter_add.restype = I
        lib.bd_attn_strerror.argtypes = [ctypes.c_int]
        lib.bd_attn_strerror.restype = ctypes.c_char_p
        lib.bd_attn_selftest_wait_timeout.argtypes = [P, ctypes.c_uint64, P]
        lib.bd_attn_selftest_wait_timeout.restype = ctypes.c_int
        _lib = lib
        return lib


def strerror(code: int) -> str:
    return load().bd_attn_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != BD_OK:
        raise RuntimeError(f"{what} failed: {strerror(rc)} (code {rc})")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on {device or 'a CUDA device'}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def seg_bytes(g: Geom) -> int:
    n = load().bd_attn_seg_bytes(ctypes.byref(g))
    if n == 0:
        raise ValueError(f"invalid geometry {g}")
    return int(n)


def seg_layout(g: Geom) -> dict:
    arr = (ctypes.c_int32 * (len(REGIONS) + 3))()
    _check(load().bd_attn_seg_layout(ctypes.byref(g), arr), "bd_attn_seg_layout")
    d = {name: int(arr[i]) for i, name in enumerate(REGIONS)}
    d["nqt"], d["nkt"], d["nkw"] = int(arr[len(REGIONS)]), int(arr[len(REGIONS) + 1]), int(arr[len(REGIONS) + 2])
    return d


def bwd_workspace_bytes(g: Geom) -> int:
    n = load().bd_attn_bwd_workspace_bytes(ctypes.byref(g))
    if n == 0:
        raise ValueError(f"invalid geometry {g}")
    return int(n)


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def bd_attn_seg_build(doc_ids: torch.Tensor, g: Geom, seg: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, stream=None):
    """Segment table of the shard (device); returns (seg, status)."""
    dev = doc_ids.device
    _need(doc_ids, "doc_ids", torch.int32, (g.B, g.S_full), None)
    if seg is None:
        seg = torch.empty(seg_bytes(g) // 4, dtype=torch.int32, device=dev)
    if status is None:
        status = new_status(dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_seg_build(_ptr(doc_ids), ctypes.byref(g), _ptr(seg), _ptr(status), _stream(stream)),
           "bd_attn_seg_build")
    return seg, status


def bd_attn_seg_build_chunk(doc_ids: torch.Tensor, g: Geom, seg: torch.Tensor | None = None,
                            status: torch.Tensor | None = None, stream=None):
    """Segment table for one chunk of the K/V range (no K/V range requirement); returns (seg, status)."""
    dev = doc_ids.device
    _need(doc_ids, "doc_ids", torch.int32, (g.B, g.S_full), None)
    if seg is None:
        seg = torch.empty(seg_bytes(g) // 4, dtype=torch.int32, device=dev)
    if status is None:
        status = new_status(dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_seg_build_chunk(_ptr(doc_ids), ctypes.byref(g), _ptr(seg), _ptr(status),
                                          _stream(stream)), "bd_attn_seg_build_chunk")
    return seg, status


def bd_attn_merge(out, lse, out_chunk, lse_chunk, g: Geom, status, stream=None):
    """Merge a K/V chunk's (out, lse) into the running (out, lse), in place."""
    dev = out.device
    for name, t in (("out", out), ("out_chunk", out_chunk)):
        _need(t, name, torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    for name, t in (("lse", lse), ("lse_chunk", lse_chunk)):
        _need(t, name, torch.float32, (g.B, g.Hq, g.L), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_merge(_ptr(out), _ptr(lse), _ptr(out_chunk), _ptr(lse_chunk), ctypes.byref(g),
                                _ptr(status), _stream(stream)), "bd_attn_merge")


def bd_attn_fwd(q, k, v, seg, g: Geom, status, out=None, lse=None, stream=None):
    """out [B,Hq,L,D] bf16 and lse [B,Hq,L] fp32 (natural log; -inf on padding rows)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(k, "k", torch.bfloat16, kv_shape(g), dev)
    _need(v, "v", torch.bfloat16, kv_shape(g), dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    if out is None:
        out = torch.empty(g.B, g.Hq, g.L, g.D, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(g.B, g.Hq, g.L, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(lse, "lse", torch.float32, (g.B, g.Hq, g.L), dev)
    _check(load().bd_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(seg), ctypes.byref(g), _ptr(out), _ptr(lse),
                              _ptr(status), _stream(stream)), "bd_attn_fwd")
    return out, lse


def bd_attn_fwd_merge(q, k, v, seg, g: Geom, status, out, lse, stream=None):
    """Forward over one K/V chunk merged into the running (out, lse), in place."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(k, "k", torch.bfloat16, kv_shape(g), dev)
    _need(v, "v", torch.bfloat16, kv_shape(g), dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _need(out, "out", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(lse, "lse", torch.float32, (g.B, g.Hq, g.L), dev)
    _check(load().bd_attn_fwd_merge(_ptr(q), _ptr(k), _ptr(v), _ptr(seg), ctypes.byref(g), _ptr(out), _ptr(lse),
                                    _ptr(status), _stream(stream)), "bd_attn_fwd_merge")
    return out, lse


def bd_attn_bwd(dout, q, k, v, out, lse, seg, g: Geom, status, grad_dtype=torch.float32, dq=None, dk=None,
                dv=None, workspace=None, stream=None, _fn="bd_attn_bwd"):
    """dq [B,Hq,L,D], dk / dv [B,Hkv,S_kv,D] (summed over each GQA group) in grad_dtype."""
    dev = q.device
    if grad_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("grad_dtype must be torch.float32 or torch.bfloat16")
    for name, t in (("dout", dout), ("q", q), ("out", out)):
        _need(t, name, torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(k, "k", torch.bfloat16, kv_shape(g), dev)
    _need(v, "v", torch.bfloat16, kv_shape(g), dev)
    _need(lse, "lse", torch.float32, (g.B, g.Hq, g.L), dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    if dq is None:
        dq = torch.empty(g.B, g.Hq, g.L, g.D, dtype=grad_dtype, device=dev)
    if dk is None:
        dk = torch.empty(kv_shape(g), dtype=grad_dtype, device=dev)
    if dv is None:
        dv = torch.empty(kv_shape(g), dtype=grad_dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(g), dtype=torch.uint8, device=dev)
    _need(dq, "dq", grad_dtype, (g.B, g.Hq, g.L, g.D), dev)
    _need(dk, "dk", grad_dtype, kv_shape(g), dev)
    _need(dv, "dv", grad_dtype, kv_shape(g), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    code = BD_DTYPE_BF16 if grad_dtype == torch.bfloat16 else BD_DTYPE_F32
    _check(getattr(load(), _fn)(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seg),
                                ctypes.byref(g), code, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), _ptr(status),
                                _stream(stream)), _fn)
    return dq, dk, dv


def bd_attn_bwd_deterministic(dout, q, k, v, out, lse, seg, g: Geom, status, grad_dtype=torch.float32, dq=None,
                              dk=None, dv=None, workspace=None, stream=None):
    """bd_attn_bwd with bitwise reproducible results (dq by a fixed-order pass)."""
    return bd_attn_bwd(dout, q, k, v, out, lse, seg, g, status, grad_dtype, dq, dk, dv, workspace, stream,
                       _fn="bd_attn_bwd_deterministic")


def bd_attn_bwd_prep(dout, out, g: Geom, status, workspace, stream=None):
    """Stage 1 of bd_attn_bwd: delta and a zeroed dq accumulator in `workspace`."""
    dev = out.device
    _need(dout, "dout", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(out, "out", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_bwd_prep(_ptr(dout), _ptr(out), ctypes.byref(g), _ptr(workspace), _ptr(status),
                                   _stream(stream)), "bd_attn_bwd_prep")


def bd_attn_bwd_main(dout, q, k, v, lse, seg, g: Geom, status, workspace, dk, dv, stream=None):
    """Stage 2 of bd_attn_bwd: dk, dv (dtype of dk) and the dq accumulation."""
    dev = q.device
    gd = dk.dtype
    if gd not in (torch.float32, torch.bfloat16):
        raise ValueError("dk / dv must be float32 or bfloat16")
    for name, t in (("dout", dout), ("q", q)):
        _need(t, name, torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(k, "k", torch.bfloat16, kv_shape(g), dev)
    _need(v, "v", torch.bfloat16, kv_shape(g), dev)
    _need(lse, "lse", torch.float32, (g.B, g.Hq, g.L), dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(dk, "dk", gd, kv_shape(g), dev)
    _need(dv, "dv", gd, kv_shape(g), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    _need(status, "status", torch.int32, (1,), dev)
    code = BD_DTYPE_BF16 if gd == torch.bfloat16 else BD_DTYPE_F32
    _check(load().bd_attn_bwd_main(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(seg), ctypes.byref(g),
                                   code, _ptr(dk), _ptr(dv), _ptr(workspace), _ptr(status), _stream(stream)),
           "bd_attn_bwd_main")


def bd_attn_bwd_finalize(g: Geom, status, workspace, dq, stream=None):
    """Stage 3 of bd_attn_bwd: dq = the (already scaled) accumulator, in the dtype of dq."""
    dev = dq.device
    if dq.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dq must be float32 or bfloat16")
    _need(dq, "dq", dq.dtype, (g.B, g.Hq, g.L, g.D), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    _need(status, "status", torch.int32, (1,), dev)
    code = BD_DTYPE_BF16 if dq.dtype == torch.bfloat16 else BD_DTYPE_F32
    _check(load().bd_attn_bwd_finalize(ctypes.byref(g), code, _ptr(dq), _ptr(workspace), _ptr(status),
                                       _stream(stream)), "bd_attn_bwd_finalize")


def bd_attn_bwd_prep_dq(dout, out, g: Geom, status, workspace, dq, stream=None):
    """Stage 1 with the fp32 dq as accumulator: delta in `workspace`, dq zeroed."""
    dev = out.device
    _need(dout, "dout", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(out, "out", torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    _need(dq, "dq", torch.float32, (g.B, g.Hq, g.L, g.D), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_bwd_prep_dq(_ptr(dout), _ptr(out), ctypes.byref(g), _ptr(workspace), _ptr(dq),
                                      _ptr(status), _stream(stream)), "bd_attn_bwd_prep_dq")


def bd_attn_bwd_main_dq(dout, q, k, v, lse, seg, g: Geom, status, workspace, dq, dk, dv, stream=None):
    """Stage 2 with the fp32 dq as accumulator: dk, dv (dtype of dk) and dq += scale * dS K."""
    dev = q.device
    gd = dk.dtype
    if gd not in (torch.float32, torch.bfloat16):
        raise ValueError("dk / dv must be float32 or bfloat16")
    for name, t in (("dout", dout), ("q", q)):
        _need(t, name, torch.bfloat16, (g.B, g.Hq, g.L, g.D), dev)
    _need(k, "k", torch.bfloat16, kv_shape(g), dev)
    _need(v, "v", torch.bfloat16, kv_shape(g), dev)
    _need(lse, "lse", torch.float32, (g.B, g.Hq, g.L), dev)
    _need(seg, "seg", torch.int32, (seg_bytes(g) // 4,), dev)
    _need(dq, "dq", torch.float32, (g.B, g.Hq, g.L, g.D), dev)
    _need(dk, "dk", gd, kv_shape(g), dev)
    _need(dv, "dv", gd, kv_shape(g), dev)
    _need(workspace, "workspace", torch.uint8, (bwd_workspace_bytes(g),), dev)
    _need(status, "status", torch.int32, (1,), dev)
    code = BD_DTYPE_BF16 if gd == torch.bfloat16 else BD_DTYPE_F32
    _check(load().bd_attn_bwd_main_dq(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(seg), ctypes.byref(g),
                                      code, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), _ptr(status),
                                      _stream(stream)), "bd_attn_bwd_main_dq")


def selftest_wait_timeout(limit_ns: int, status: torch.Tensor, stream=None):
    _need(status, "status", torch.int32, (1,), None)
    _check(load().bd_attn_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)),
           "bd_attn_selftest_wait_timeout")


def read_seg(seg: torch.Tensor, g: Geom) -> dict:
    """Copy the segment table to the host and decode it (synchronises; tests and tools only)."""
    lay = seg_layout(g)
    a = seg.cpu().numpy()
    L, B, nqt, nkt, nkw = g.L, g.B, lay["nqt"], lay["nkt"], lay["nkw"]
    rows = []
    for b in range(B):
        h = a[lay["hdr"] + b * HDR_WORDS: lay["hdr"] + (b + 1) * HDR_WORDS]
        d = {name: int(h[i]) for i, name in enumerate(HDR_FIELDS)}
        n = d["n_seg"]
        cq = a[lay["cu_q"] + b * (L + 1): lay["cu_q"] + (b + 1) * (L + 1)]
        ck = a[lay["cu_k"] + b * (L + 1): lay["cu_k"] + (b + 1) * (L + 1)]
        d["cu_q"] = cq[:n + 1].copy()
        d["cu_k"] = ck[:n + 1].copy()
        d["row_lo"] = a[lay["row_lo"] + b * L: lay["row_lo"] + (b + 1) * L].copy()
        d["qt_krange"] = a[lay["qt_krange"] + b * nqt * 2: lay["qt_krange"] + (b + 1) * nqt * 2].reshape(nqt, 2).copy()
        d["kt_qrange"] = a[lay["kt_qrange"] + b * nkt * 2: lay["kt_qrange"] + (b + 1) * nkt * 2].reshape(nkt, 2).copy()
        d["full_bits"] = a[lay["full_bits"] + b * nqt * nkw: lay["full_bits"] + (b + 1) * nqt * nkw].reshape(nqt, nkw).copy()
        rows.append(d)
    return {"rows": rows,
            "fwd_work": a[lay["fwd_work"]: lay["fwd_work"] + B * nqt].copy(),
            "bwd_work": a[lay["bwd_work"]: lay["bwd_work"] + B * nkt].copy(),
            "counts": a[lay["counts"]: lay["counts"] + 4].copy(),
            "layout": lay}


# ------------------------------------------------------------ exchange plans
def plan_bytes(B: int, cp_size: int, L: int) -> int:
    n = load().bd_attn_plan_bytes(int(B), int(cp_size), int(L))
    if n == 0:
        raise ValueError(f"invalid plan size B={B} cp_size={cp_size} L={L}")
    return int(n)


def plan_layout(B: int, cp_size: int, L: int) -> dict:
    arr = (ctypes.c_int32 * len(PLAN_REGIONS))()
    _check(load().bd_attn_plan_layout(int(B), int(cp_size), int(L), arr), "bd_attn_plan_layout")
    return {name: int(arr[i]) for i, name in enumerate(PLAN_REGIONS)}


def bd_attn_exchange_plan(doc_ids: torch.Tensor, cp_size: int, rank: int, plan: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, stream=None):
    """Exchange plan of `rank` from the replicated doc ids [B, S] (device); returns (plan, status)."""
    dev = doc_ids.device
    B, S = doc_ids.shape
    _need(doc_ids, "doc_ids", torch.int32, (B, S), None)
    if S % cp_size:
        raise ValueError("the sequence must split into cp_size equal chunks")
    n = plan_bytes(B, cp_size, S // cp_size) // 4
    if plan is None:
        plan = torch.empty(n, dtype=torch.int32, device=dev)
    if status is None:
        status = new_status(dev)
    _need(plan, "plan", torch.int32, (n,), dev)
    _need(status, "status", torch.int32, (1,), dev)
    _check(load().bd_attn_exchange_plan(_ptr(doc_ids), int(B), int(S), int(cp_size), int(rank), _ptr(plan),
                                        _ptr(status), _stream(stream)), "bd_attn_exchange_plan")
    return plan, status


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BD_DTYPE_BF16
    if t.dtype == torch.float32:
        return BD_DTYPE_F32
    raise ValueError("bfloat16 or float32 expected")


def bd_attn_needed_gather(x_local: torch.Tensor, plan: torch.Tensor, send: torch.Tensor, status, stream=None):
    """send [max_rows, B, C, D] (token-major) from x_local [B, C, L, D] by the plan's send_index."""
    B, C, L, D = x_local.shape
    max_rows = send.shape[0]
    _need(x_local, "x_local", x_local.dtype, (B, C, L, D), None)
    _need(send, "send", x_local.dtype, (max_rows, B, C, D), x_local.device)
    _need(status, "status", torch.int32, (1,), x_local.device)
    _check(load().bd_attn_needed_gather(_ptr(x_local), _ptr(plan), B, C, L, D, _dtype_code(x_local), _ptr(send),
                                        int(max_rows), _ptr(status), _stream(stream)), "bd_attn_needed_gather")
    return send


def bd_attn_needed_scatter_add(grad_send: torch.Tensor, plan: torch.Tensor, grad_local: torch.Tensor, status,
                               stream=None):
    """grad_local [B, C, L, D] = the index-add of grad_send [max_rows, B, C, D] (token-major)."""
    B, C, L, D = grad_local.shape
    max_rows = grad_send.shape[0]
    _need(grad_local, "grad_local", grad_local.dtype, (B, C, L, D), None)
    _need(grad_send, "grad_send", grad_local.dtype, (max_rows, B, C, D), grad_local.device)
    _need(status, "status", torch.int32, (1,), grad_local.device)
    _check(load().bd_attn_needed_scatter_add(_ptr(grad_send), _ptr(plan), B, C, L, D, _dtype_code(grad_local),
                                             _ptr(grad_local), int(max_rows), _ptr(status), _stream(stream)),
           "bd_attn_needed_scatter_add")
    return grad_local


def read_plan(plan: torch.Tensor, B: int, cp_size: int, L: int) -> dict:
    """Copy a plan to the host and decode it (synchronises; tests and tools only)."""
    lay = plan_layout(B, cp_size, L)
    a = plan.cpu().numpy()
    W = cp_size
    h = a[lay["hdr"]: lay["hdr"] + PLAN_HDR_WORDS]
    d = {name: int(h[i]) for i, name in enumerate(PLAN_HDR_FIELDS)}
    for name in ("s_first", "real_end", "back", "halo_send", "in_splits", "out_splits", "send_off", "recv_off"):
        d[name] = [int(x) for x in a[lay[name]: lay[name] + W]]
    d["counts"] = [[int(x) for x in a[lay["counts"] + s * W: lay["counts"] + (s + 1) * W]] for s in range(W)]
    d["send_index"] = [int(x) for x in a[lay["send_index"]: lay["send_index"] + max(0, d["total_send"])]]
    return d
