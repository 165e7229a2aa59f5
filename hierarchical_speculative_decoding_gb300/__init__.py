"""TriForce decode-step attention on GB300: a C-ABI CUDA library plus a thin binding.

Submodules:
  binding  ctypes marshalling over libtriforce_attn.so (built in-tree)
  synth    seeded synthetic inputs shaped like the decode-step workloads
"""
