"""CPU oracle of the RLT hot path (test infrastructure only; see rlt_oracle)."""
from .rlt_oracle import *  # noqa: F401,F403
from . import rlt_oracle  # noqa: F401
