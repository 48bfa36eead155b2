"""CPU fp64 oracle (test infrastructure only; see oracle/reference.py)."""
from .reference import *  # noqa: F401,F403
from . import reference  # noqa: F401
