"""CPU oracle for the Quasar W8A8 verification path (test infrastructure only)."""
from .quasar_oracle import *  # noqa: F401,F403
