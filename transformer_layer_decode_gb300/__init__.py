"""Batch-1 decode of a Llama-style decoder stack as fused sm_103a CUDA kernels.

The compute path lives in the C-ABI library ``libtld_gb300.so`` (declared in
``include/dec.h``); :mod:`.dec` is its thin ctypes binding.  Importing this
package does not load the library: :func:`.dec.load_library` does, and it
raises if the library has not been built.
"""
