"""libtpmlp: the tensor-parallel Transformer MLP block (forward and backward)
as hand-written sm_103a CUDA behind a C ABI (include/tpmlp.h).

Modules:
  build    compiles csrc/*.cu into _build/libtpmlp.so with nvcc
  binding  ctypes binding with the C ABI's names (marshalling only)
  block    device buffers for one block and the calls that run it
  inputs   seeded synthetic workloads (shared with the tests)

Importing the package does not load the library; importing ``binding`` does,
and fails loudly if it has not been built.
"""
