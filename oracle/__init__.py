"""CPU oracle (test infrastructure; see lin_state_oracle's header)."""
from . import lin_state_oracle  # noqa: F401
