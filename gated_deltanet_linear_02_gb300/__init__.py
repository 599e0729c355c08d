"""Gated-DeltaNet token mixer for GB300 (sm_103a).

The compute lives in ``libgdn.so`` (hand-written CUDA behind a C ABI, see
``include/gdn.h``). This package is its thin ctypes binding: ``ops`` marshals
torch tensors into the C calls, ``inputs`` draws seeded synthetic workloads.
Nothing is imported eagerly, so ``inputs`` works on a machine without the
library or a GPU.
"""

DIMS = dict(Hv=32, Hk=16, dk=128, dv=128, conv_k=4)
C_CONV = 2 * DIMS["Hk"] * DIMS["dk"] + DIMS["Hv"] * DIMS["dv"]   # 8192
D_INNER = DIMS["Hv"] * DIMS["dv"]                                   # 4096
