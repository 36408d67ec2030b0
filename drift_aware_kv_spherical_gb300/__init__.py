"""libpolestar: the drift-scoring and sparse-refresh path of Polestar-Cache /
Polestar-Commit on one GB300 (sm_103a), behind a C ABI (include/polestar.h).

``polestar`` is the ctypes binding (import it explicitly; it loads the CUDA
library), ``workloads`` the seeded synthetic inputs, ``pipeline`` the step
driver that chains the six calls.
"""
