"""Bit-exact float_moment and float_psnr of 8- to 16-bit luma frames on GB300.

The computation runs in libvmx (CUDA, sm_103a), reached through a C ABI
(``include/vmx.h``); ``api`` marshals torch tensors to it. ``synth`` draws the
seeded synthetic workloads; ``build`` compiles the library in-tree.
"""

__all__ = ["api", "build", "synth"]
