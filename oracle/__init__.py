"""fp64 CPU oracle (test infrastructure only; see dora_oracle.py)."""
from .dora_oracle import *  # noqa: F401,F403
from .dora_oracle import __all__  # noqa: F401
