"""CPU oracle of the sharded Linear (test infrastructure; see tp_oracle)."""
from .tp_oracle import *  # noqa: F401,F403
