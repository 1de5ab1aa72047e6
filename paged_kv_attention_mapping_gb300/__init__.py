"""Paged-KV attention for one packed decode/prefill tick on GB300 (sm_103a).

The compute runs in ``libpagedkv.so`` (hand-written CUDA behind a C ABI,
declared in ``include/pagedkv.h``); ``binding`` marshals torch tensors into
that ABI. ``workloads`` draws the seeded synthetic inputs.
"""
__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
