"""CPU oracle for QUOKA (test infrastructure only; see quoka_oracle.py)."""
from . import quoka_oracle  # noqa: F401
