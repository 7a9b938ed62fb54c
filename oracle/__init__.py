"""Float64 CPU oracle (test infrastructure only; see vg_oracle)."""
from .vg_oracle import *  # noqa: F401,F403
