"""paged_kv_split_gb300: paged split-KV decode attention for GB300 (sm_103a).

The compute path is libpd.so (hand-written CUDA behind a C ABI, declared in
include/pd.h). ``paged_kv_split_gb300.binding`` marshals torch tensors into
those calls; importing it fails loudly when libpd.so has not been built.
``paged_kv_split_gb300.inputs`` holds the seeded synthetic workloads.
"""
import importlib

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
