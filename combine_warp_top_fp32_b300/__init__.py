"""B300-native MoE expert-parallel dispatch and combine.

The product is the C-ABI library ``libep_b300.so`` (hand-written sm_103a CUDA
kernels behind ``include/ep.h``). :mod:`.binding` loads it through ctypes and
exposes the same entry points over torch CUDA tensors; :mod:`.workloads`
holds the seeded synthetic inputs. Importing this package does not load the
library; the first call into :mod:`.binding` does, and fails loudly when the
library has not been built.
"""

__all__ = ["binding", "workloads"]
