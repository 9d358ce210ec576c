"""fp64 CPU oracle (test infrastructure only; see ulysses_oracle.py)."""
from .ulysses_oracle import *  # noqa: F401,F403
