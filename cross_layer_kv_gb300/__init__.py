"""FusedKV attention for GB300: cross-layer KV reconstruction computed inside
hand-written sm_103a CUDA kernels, exposed through a C ABI (include/fusedkv.h)
with a thin ctypes binding (``fusedkv``)."""

from .fusedkv import (FKV_FUSED, FKV_LITE, FKV_SCALED, FKV_VANILLA, Context, FkvError, header_symbols,  # noqa: F401
                      load, status_string)
