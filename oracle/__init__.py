"""CPU oracle for Compressed Sparse Attention (test infrastructure; see csa_oracle)."""
from .csa_oracle import *  # noqa: F401,F403
from . import csa_oracle  # noqa: F401
