"""GB300-native packed ternary-weight decode.

The compute path is the C ABI library ``_lib/libnt.so`` (hand-written sm_103a CUDA, declared
in include/nt.h); :mod:`packed_weight_gemv_gb300.nt` is its thin ctypes binding with the same
call names. Build with :func:`packed_weight_gemv_gb300.build.build`.
"""
from . import nt  # noqa: F401
