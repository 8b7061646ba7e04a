"""Float64 CPU oracle for differential attention: test infrastructure only.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg import this package.
The library's product path never does.
"""
from . import diffattn_ref  # noqa: F401
