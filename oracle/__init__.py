"""fp64 CPU oracle for the Ulysses attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product path.  It shares
no code with the CUDA library.  See ``usp_oracle`` for the definitions and the
passages they follow.
"""
from .usp_oracle import *  # noqa: F401,F403
from .usp_oracle import __all__  # noqa: F401
