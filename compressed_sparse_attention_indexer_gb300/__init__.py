"""GB300-native compressed sparse attention (CSA) decode step.

The compute path is the CUDA library ``libcsa`` (sm_103a) behind a C ABI
(``include/csa.h``); ``csa`` below is its thin ctypes binding.  Importing the
package does not load the library: the first call does, and it raises if the
library has not been built.  There is no CPU fallback.
"""
from .workloads import CsaConfig, Dists, Workload, WORKLOADS, make_batch, to_device  # noqa: F401
