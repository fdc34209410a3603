"""GB300-native LAMB optimizer step for one ZeRO-2 shard.

The compute path is ``liblamb_gb300.so`` (hand-written CUDA for sm_103a behind
the C ABI of ``include/lamb.h``); this package only binds it to torch tensors.
"""
from ._lib import LambError, library_path, load
from .lamb import Lamb, plan, plan_limits

__all__ = ["Lamb", "LambError", "plan", "plan_limits", "library_path", "load"]
