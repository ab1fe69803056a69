"""Paged split-KV GQA decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libga.so`` (hand-written CUDA);
:mod:`paged_split_kv_gqa_gb300.ga` is its thin ctypes binding and is loaded on
first use.  :mod:`paged_split_kv_gqa_gb300.workloads` draws seeded inputs.
"""
import importlib

__all__ = ["ga", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
