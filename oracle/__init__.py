"""fp64 CPU oracle for the gated bidirectional linear-attention forward.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import it.  The CUDA library never does, and this
package imports nothing from the library.
"""
from .linattn import *  # noqa: F401,F403
from .linattn import __all__  # noqa: F401
