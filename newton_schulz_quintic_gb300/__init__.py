"""GB300-native batched quintic Newton-Schulz orthogonalization.

The compute runs in the CUDA library ``libns.so`` (sources under ``csrc/``,
C ABI declared in ``include/ns.h``); this package is a thin ctypes binding
that marshals torch tensors' device pointers and the current CUDA stream.
The library is loaded on first use, and every call fails loudly when it is
missing: there is no CPU fallback.
"""
from .api import (  # noqa: F401
    NS_BF16,
    NS_F32,
    NSError,
    cost,
    get_status,
    library_path,
    load_library,
    orthogonalize_batched,
    orthogonalize_batched_host,
    workspace_bytes,
)
