"""Speculative-decoding verify step on sm_103a (GB300).

The compute lives in libsdverify.so (include/sd_verify.h): split-KV
tree-masked verify attention, argmax + greedy path selection, and the KV
commit.  ``native`` is its ctypes binding (same names as the C ABI),
``step.VerifyStep`` runs a whole step, ``synth`` draws seeded synthetic
workloads, and ``build`` compiles the library in-tree.
"""

__all__ = ["native", "step", "synth", "build"]
