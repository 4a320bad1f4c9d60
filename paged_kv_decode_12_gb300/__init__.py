"""paged_kv_decode_12_gb300: paged-KV decode attention for GB300 (sm_103a).

The compute path is ``libpkv.so`` (CUDA kernels behind a C ABI, declared in
``include/pkv.h``); ``paged_kv_decode_12_gb300.pkv`` is its thin ctypes binding.
``workloads`` draws the seeded synthetic inputs.  Importing the package does not
load the native library; the first call into ``pkv`` does, and fails loudly if
the library has not been built.
"""
__all__ = ["pkv", "workloads"]
