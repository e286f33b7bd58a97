"""GB300 (sm_103a) split Shared / Non-Shared beam-search decode attention.

The compute path is the C-ABI library `libxattn.so` (CUDA kernels for sm_103a); this
package holds its ctypes binding (`xattn`), its build step (`build`) and the seeded
workload generator (`workloads`). Importing the package loads nothing; the binding loads
the library on first use and raises if it is missing.
"""

__all__ = ["workloads", "build", "xattn"]
