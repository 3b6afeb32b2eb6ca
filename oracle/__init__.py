"""Float64 CPU oracle for LRKV (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path
(``rank_kv_attention_gb300``) never imports, links or calls it, and this
package imports nothing from the product path.
"""
from .lrkv_oracle import *  # noqa: F401,F403
from . import fp8  # noqa: F401  (8-bit cache storage)
from . import rope  # noqa: F401  (exact rotary position embedding)
from . import norm  # noqa: F401  (joint RMSNorm of the keys)
from . import grouped  # noqa: F401  (a shared basis per group of heads)
