"""fp64 CPU oracle (test infrastructure; never used by the product path)."""

from .mla_oracle import *  # noqa: F401,F403
from . import mla_oracle  # noqa: F401
