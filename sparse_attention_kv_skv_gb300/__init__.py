"""Sparse-attention KV assembly for GB300 (sm_103a).

The compute path lives in ``libskv.so`` (CUDA, built by ``build.py``); this
package only binds it.  See ``include/skv.h`` for the C ABI.
"""
from .skv import (  # noqa: F401
    Config,
    Context,
    SkvError,
    SKV_DEVERR_BAD_INDEX,
    SKV_DEVERR_BAD_REQUEST,
    SKV_DEVERR_CONTEXT_FULL,
    SKV_DEVERR_DUPLICATE,
    LIB_PATH,
)
