"""GB300-native decode-time KV-cache eviction pass.

The pass (attention with probability capture, head pooling, layer-sequential
EMA, LRFU priority, budgeted selection, stable compaction) runs in the CUDA
library built from ``csrc/`` (``libkvev.so``); ``kvev`` is its Python binding.
"""
from . import kvev  # noqa: F401
from .kvev import EvictionPass, KvevError  # noqa: F401
