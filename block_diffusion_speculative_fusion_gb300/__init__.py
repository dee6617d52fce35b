"""GB300-native DFlash hot path: context-KV materialisation, bidirectional block
attention, greedy and sampled verify and the DLoop gate, as hand-written
sm_103a CUDA behind a small C ABI (``libdflash.so``).

The ctypes binding is imported lazily (``from . import api``) so that the
workload and input-generator modules load without the compiled library.
"""
__all__ = ["workloads", "synth", "api"]
