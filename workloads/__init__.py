"""Seeded synthetic inputs shared by the CUDA path's tests and bench and by the
CPU oracle's tests.  Holds no attention, scatter or copy arithmetic."""
from .configs import CONFIGS, DecodeConfig, LONG_CONTEXT_BLOCK_SIZES, get  # noqa: F401
from .gen import (PagedDecodeWorkload, StepInputs, TORCH_DTYPES, fill_cache,  # noqa: F401
                  normal, step_values, TAG_CACHE_K, TAG_CACHE_V)
