"""GB300-native paged KV cache: paged decode attention, KV append and copy-on-write block
copies as CUDA kernels for sm_103a behind a C ABI (``libpkv.so``), plus a host C block manager.

Importing the package loads nothing; ``paged_kv_cache_258_gb300.pkv`` is the ctypes binding
and loads the compiled library on first use.
"""
__all__ = ["pkv", "workloads"]
