"""Plain CPU oracle for the dropless-MoE hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product (``grouped_gemm_top_gb300``) never imports it and shares no code
with it.
"""
from .moe_oracle import *  # noqa: F401,F403
