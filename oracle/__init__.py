"""Independent CPU oracle (test infrastructure only).

Importable only from ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``. The CUDA library never imports it, and it imports nothing
from the library.
"""
from . import fp4q_oracle  # noqa: F401
