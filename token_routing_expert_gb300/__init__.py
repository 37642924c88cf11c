"""GB300 (sm_103a) routed / latent Mixture-of-Experts layer forward.

The compute path is the native library ``libmoe_gb300.so`` (hand-written
CUDA: tcgen05 / TMEM / TMA GEMMs, warp-per-token router, permutation and
combine kernels) behind a C ABI; ``native`` is its thin ctypes binding.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "native", "build"]
