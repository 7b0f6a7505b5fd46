"""CPU oracle (test infrastructure only; see snapkv_oracle.py)."""
from .snapkv_oracle import *  # noqa: F401,F403
