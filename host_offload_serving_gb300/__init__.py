"""HiSparse RESOLVE hot path for GB300 (sm_103a).

``hisparse`` is the ctypes binding of ``include/hisparse.h``; ``runtime``
wraps it with torch-managed device memory and streams.
"""
from . import hisparse  # noqa: F401
