"""fp64 CPU oracle (test infrastructure only; never called by the library)."""
from .bt_oracle import *  # noqa: F401,F403
