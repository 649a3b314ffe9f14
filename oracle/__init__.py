"""CPU oracle for physically sparse QSA decode -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does.
"""
from .qsa_oracle import *  # noqa: F401,F403
