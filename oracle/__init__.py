"""CPU oracle for the W4A16 GEMM (test infrastructure only; see ``wq4_oracle``)."""
from .wq4_oracle import *  # noqa: F401,F403
from . import wq4_oracle  # noqa: F401
