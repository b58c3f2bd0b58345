"""QEvict decode-time path on GB300: a C-ABI CUDA library (libqevict.so) and its thin binding.

    from recoverable_quantized_kv_gb300 import binding, synth
    cache = binding.Cache(binding.make_config(synth.workload("llama8b_32k")))

The CUDA library must be built first (recoverable_quantized_kv_gb300.build.build()); without
it the binding raises instead of falling back to anything else.
"""
from . import synth  # noqa: F401

__all__ = ["binding", "build", "synth"]
