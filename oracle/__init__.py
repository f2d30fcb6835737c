"""Float64 CPU oracle (test infrastructure only; the library never imports it)."""
from .palu_oracle import *  # noqa: F401,F403
