"""GB300 (sm_103a) NVFP4 W4A4 residual-compensation path: libquads and its Python binding.

    from nvfp4_w4a4_quantized_quant_gb300 import quads, inputs
"""
from . import inputs  # noqa: F401

__all__ = ["quads", "inputs", "build"]


def __getattr__(name):
    if name in ("quads", "build", "layer"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
