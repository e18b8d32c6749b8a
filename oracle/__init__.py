"""CPU oracle (test infrastructure only).

Plain, slow numpy restatement of what the Lynx hot path computes, used to check
the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` import it; the library never does, and the two share no
code.  See ``lynx_oracle`` (quantiser and reconstruction) and ``attention``
(float64 decode / verification attention).
"""
from . import lynx_oracle, attention  # noqa: F401
