"""Gated bidirectional linear attention (SANA-Video 2.0) for B300 (sm_103a).

The forward runs in ``libsla.so`` (hand-written CUDA kernels behind the C ABI
of ``include/sla.h``); ``gated_linear_attention_attn_b300.sla`` is its Python
binding and ``gated_linear_attention_attn_b300.workloads`` names the workload
shapes and draws seeded inputs.  The binding is imported on first use, so the
workload module works without the library.
"""

import importlib

__all__ = ["sla", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
