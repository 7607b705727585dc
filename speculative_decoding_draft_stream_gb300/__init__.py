"""Dynamic-vocabulary draft LM head (NanoSpec / MicroSpec) for GB300 (sm_103a).

The compute path is the C-ABI library ``libnanospec.so`` (include/nanospec.h),
built from ``csrc/`` by ``build.build()``; ``nanospec`` is its ctypes binding.
"""

from .nanospec import (  # noqa: F401
    EXPORTED,
    FLAG_BAD_ID,
    FLAG_OVERFLOW,
    FLAG_TIMEOUT,
    Handle,
    NanoSpecError,
    load_library,
)
