"""Float64 CPU oracle (test infrastructure only; see diffattn_oracle)."""

from .diffattn_oracle import *  # noqa: F401,F403
