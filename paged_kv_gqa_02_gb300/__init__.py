"""Paged-KV grouped-query attention for GB300 (sm_103a).

The CUDA library ``libpaged_gqa.so`` (C ABI, ``include/paged_gqa.h``) does
all the work; ``paged_kv_gqa_02_gb300.ops`` is a thin ctypes binding that
marshals torch CUDA tensors into it.  ``inputs`` and ``workloads`` hold the
seeded synthetic inputs and the workload shapes.
"""

__all__ = ["inputs", "workloads", "ops"]
