"""fp64 CPU oracle for exact attention (test infrastructure; see attention.py)."""
from .attention import *  # noqa: F401,F403
