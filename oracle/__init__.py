"""Float64 CPU oracle for the POET-X layer (test infrastructure only; see
poetx_oracle's header)."""
from .poetx_oracle import *  # noqa: F401,F403
