"""GB300-native paged decode attention.

The compute path lives in a C-ABI shared library built from csrc/ for
sm_103a (declared in include/pa.h); this package's Python layer only loads
that library and marshals arguments to it.  Importing the package does not
load the library: `from paged_kv_cache_124_gb300 import api` does, and fails
loudly if it has not been built.
"""

__all__ = ["api", "inputs", "build"]
