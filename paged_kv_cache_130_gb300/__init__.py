"""Paged KV-cache decode path for GB300 (sm_103a).

The compute runs in the CUDA library ``libpkv.so`` built from ``csrc/``; this
package holds its thin ctypes binding (``binding``), the host block allocator
(``block_manager``) and the seeded workload generator (``workloads``).
"""
