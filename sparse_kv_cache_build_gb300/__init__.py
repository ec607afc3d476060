"""Sparse paged-KV decode attention for GB300: a C-ABI CUDA library and a thin binding."""

from . import inputs  # noqa: F401
