"""CPU oracle for MLA latent-space decode attention.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 restatement of
what the pages define; it exists to check the CUDA library against.  Only the
test suite, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg
and its ``--impl reference`` arm) may import it.  The product path never calls
it, and it shares no code with the CUDA library: it reads the same seeded
bf16 inputs (``mla_inputs``) and nothing else.

Parity status per function is stated in ``oracle/mla.py``.
"""
from .mla import *  # noqa: F401,F403
from .mla import __all__  # noqa: F401
