"""Plain CPU oracle for paged KV-cache decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s ``cpu_baseline`` leg (and its ``--impl reference`` arm) may import,
call or execute anything in this package.  The CUDA library and its Python binding
never import it, and it shares no code, tables or helpers with them: it is written
from the pages' prose (cited per function) in plain numpy, fp64 for every
floating-point step except the fp32 quantisation division that the quantisation
reading fixes.

Every function here is pinned by ``tests/test_oracle_*.py`` against values printed on
the pages (``tests/golden/``), closed forms, library routines (torch SDPA, torch's
float8 cast, numpy's round-half-even) and brute force on tiny inputs.
"""

from .paged_kv import *  # noqa: F401,F403
from .prefix_cache import *  # noqa: F401,F403
