"""CPU oracle (test infrastructure only; never used by the product path)."""
from .peagle_oracle import *  # noqa: F401,F403
