"""fp64 CPU oracle (test infrastructure only; see kd_oracle's header)."""
from .kd_oracle import *  # noqa: F401,F403
