"""GB300-native compression pass of Compressed PagedAttention (Zipage).

Submodules:
  zipage  ctypes binding of the C-ABI library libzipage.so (CUDA kernels for sm_103a)
  build   compiles libzipage.so in-tree with nvcc
  synth   seeded synthetic workloads (inputs only)
"""
