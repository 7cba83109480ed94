"""CPU oracle (test infrastructure only; see mx_oracle's header)."""
from .mx_oracle import *  # noqa: F401,F403
