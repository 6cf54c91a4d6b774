"""CPU oracle for the dual-path quantized-base + LoRA overlay library.

TEST INFRASTRUCTURE ONLY.  Nothing on the library's product path imports,
calls or links this package: it is used by ``tests/``, by the smoke check in
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``.  It shares no code with the CUDA library.

Every function is a plain, slow, obviously-correct restatement of a
definition from the pages (fp64 arithmetic, library matmul as the only
primitive).  Parity status of each function is listed in ``ovl_oracle``'s
module docstring.
"""
from .ovl_oracle import *  # noqa: F401,F403
