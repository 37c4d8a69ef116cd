"""GB300-native (sm_103a) forward of a top-K routed MoE SwiGLU FFN layer with
always-on shared experts.

The compute lives in the C-ABI library ``libmoe.so`` built from ``csrc/``
(declared in ``include/moe.h``); ``api`` is a thin ctypes binding over it
that marshals torch CUDA tensors into plain device pointers. The binding is
loaded on first use, so importing this package (for example to reach the
``workloads`` input generator) needs neither a GPU nor the built library.
"""

__all__ = ["api", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
