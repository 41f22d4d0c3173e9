"""CPU oracle for indexer-routed sparse attention — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package. The CUDA library and its Python binding never
import it, and it never imports them.
"""
from . import irs_oracle  # noqa: F401
