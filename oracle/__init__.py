"""CPU oracle package: test infrastructure only (see coda_oracle.py)."""
from .coda_oracle import *  # noqa: F401,F403
from . import coda_oracle  # noqa: F401
