"""GB300-native decode hot path of ECHO (lossless KV-cache offloading for
sparse-attention LLMs): FP8 indexer scores on tcgen05, exact top-k with an EMA
threshold predictor and early fetch, and the fixed-size GPU cache step with
zero-copy recall from a pinned host pool.  The compute lives in ``libecho.so``
(CUDA for sm_103a, C ABI in ``include/echo.h``); this package binds it.
"""
from . import _lib as lib  # noqa: F401
from .decode import DecodeLayer, DecodeStack  # noqa: F401
