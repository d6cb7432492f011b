"""GB300 (sm_103a) csgmv multi-adapter LoRA path.

The compute lives in libcsgmv.so (include/csgmv.h); ``binding`` exposes the
same calls on torch tensors.  ``workloads`` draws the seeded synthetic inputs.
The binding is imported lazily so that the input generator works on machines
without a GPU or a built library.
"""

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in ("binding", "workloads", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
