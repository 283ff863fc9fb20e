"""Per-document causal (block-diagonal) attention for one context-parallel shard, GB300-native.

The compute lives in ``libbdattn.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/bdattn.h``); :mod:`.bdattn` is its thin ctypes
binding and :mod:`.synth` draws seeded synthetic inputs.
"""
from importlib import import_module

__all__ = ["bdattn", "synth", "bd_attn_seg_build", "bd_attn_fwd", "bd_attn_bwd"]


def __getattr__(name):
    if name in ("bdattn", "synth"):
        return import_module(f"{__name__}.{name}")
    if name in ("bd_attn_seg_build", "bd_attn_fwd", "bd_attn_bwd"):
        return getattr(import_module(f"{__name__}.bdattn"), name)
    raise AttributeError(name)
