"""Load-balanced paged GQA decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libhpcdecode.so`` (CUDA kernels in
``csrc/``); :mod:`.binding` marshals torch tensors into its calls. Nothing in
this package computes attention on the CPU: if the library is missing the
calls raise.

The binding is imported on first attribute access, so that
:mod:`.workloads` (the seeded input generator) can be used on its own.
"""
import importlib

_BINDING_NAMES = {
    "KV_BF16", "KV_FP8_E4M3", "HpcError", "Plan", "build", "default_num_ctas",
    "hpc_decode_attn", "hpc_decode_combine", "hpc_decode_plan", "hpc_decode_plan_static",
    "hpc_decode_read_error", "hpc_decode_step_host", "lib", "split_buffers", "decode",
    "sm_count", "hpc_rope_norm",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
