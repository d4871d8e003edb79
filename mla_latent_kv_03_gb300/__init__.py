"""libmla: MLA latent-KV paged decode for GB300 (sm_103a).

The compute path is the C-ABI shared library ``libmla.so`` built from
``csrc/``; ``mla_latent_kv_03_gb300.libmla`` is a thin ctypes binding over it.
Importing this package loads nothing; the binding loads the library on first
use and raises if it is missing (there is no fallback path).
"""

__all__ = ["workloads"]
