"""Sparse-attention KV assembly for GB300 (sm_103a).

The compute path lives in ``libskv.so`` (CUDA, built by ``build.py``); this
package only binds it.  See ``include/skv.h`` for the C ABI.

The binding is loaded on first use of any exported name, so that
``sparse_attention_kv_skv_gb300.build`` can run before the library exists;
using the API without the library raises ImportError (there is no fallback).
"""
_EXPORTS = ("Config", "Context", "SkvError", "SKV_DEVERR_BAD_INDEX", "SKV_DEVERR_BAD_REQUEST",
            "SKV_DEVERR_CONTEXT_FULL", "SKV_DEVERR_DUPLICATE", "LIB_PATH", "skv")

__all__ = list(_EXPORTS)


def __getattr__(name):
    if name in _EXPORTS:
        import importlib
        mod = importlib.import_module(".skv", __name__)
        return mod if name == "skv" else getattr(mod, name)
    raise AttributeError(name)
