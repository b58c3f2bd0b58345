"""CPU oracle for QEvict's decode-time path: test infrastructure only.

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import it.
"""
from .qevict_oracle import *  # noqa: F401,F403
from .qevict_oracle import Config, Budget, Unit, Ledger  # noqa: F401
