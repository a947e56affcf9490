"""CPU oracle for the fused weight-gradient + AdamW step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.
"""
from .forge_oracle import *  # noqa: F401,F403
from .regime1 import *  # noqa: F401,F403
from .accum import *  # noqa: F401,F403
from .sr import *  # noqa: F401,F403
from .fp8 import *  # noqa: F401,F403
