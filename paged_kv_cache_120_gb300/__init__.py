"""PagedAttention decode for GB300 (sm_103a).

The product is ``libpa.so``: a C-ABI library (declared in ``include/pa.h``)
with the paged KV-cache write (``pa_reshape_and_cache``), the paged decode
(``pa_decode``, split-K included) and copy-on-write block copies
(``pa_copy_blocks``), plus a host C++ block allocator that builds block
tables and slot mappings. ``paged_kv_cache_120_gb300.binding`` is a thin
ctypes layer with the same names; importing this package loads nothing.
"""

__all__ = ["binding", "workloads", "build"]
