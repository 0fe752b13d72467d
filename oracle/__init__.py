"""CPU oracle of the GIFT gradient codec (test infrastructure; see gift_oracle.py)."""
from .gift_oracle import *  # noqa: F401,F403
