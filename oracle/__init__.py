"""fp64 CPU oracle (test infrastructure; see tp_oracle.py)."""
from .tp_oracle import *  # noqa: F401,F403
