"""GB300 (sm_103a) implementation of SPEAR's gated W4 + low-rank error-compensated linear.

The compute path lives in a C-ABI shared library (``csrc/`` -> ``lib/libspear.so``,
declared in ``include/spear.h``); ``spear`` is its thin ctypes binding.  Import
``quantized_gemm_error_gb300.spear`` to load the library; this package root
stays light so that the seeded input generators (``inputs``) load without CUDA.

Modules on top of the binding: ``stack`` (a Llama-7B decoder-block stack of W4
layers stepped as CUDA graphs), ``scheduler`` (latency tables for prefill chunk
selection), ``shard`` (column-parallel split of a layer over ranks), ``build``
(compiles the library).
"""

__all__ = ["build", "inputs", "scheduler", "shard", "spear", "stack"]
