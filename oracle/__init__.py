"""CPU oracle (test infrastructure only): float64 restatement of one Medusa verify step."""
from .medusa_oracle import *  # noqa: F401,F403
from . import medusa_oracle  # noqa: F401
