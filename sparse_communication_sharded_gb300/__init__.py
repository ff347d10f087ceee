"""GB300-native SCAPE sharded sparse optimizer step (sm_103a CUDA behind a C ABI)."""
from . import _scape
from ._scape import ScapeError, load
from .optimizer import Scape

__all__ = ["Scape", "ScapeError", "load", "_scape"]
