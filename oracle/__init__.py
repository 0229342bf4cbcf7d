"""CPU oracle (test infrastructure only; see rocketkv_oracle)."""
from .rocketkv_oracle import *  # noqa: F401,F403
