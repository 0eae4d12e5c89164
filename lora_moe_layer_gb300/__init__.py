"""lora_moe_layer_gb300 -- multi-LoRA fused MoE layer forward for GB300 (sm_103a).

The compute lives in libmoelora.so (CUDA C++, built by ``build.build()``);
``binding`` is its ctypes binding, ``layer`` a small convenience wrapper that
owns device copies of a layer's weights, and ``workloads`` the seeded
synthetic inputs.  Submodules load lazily so that importing the package does
not open the CUDA library.
"""
import importlib

__all__ = ["binding", "build", "layer", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
