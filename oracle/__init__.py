"""fp64 CPU oracle (test infrastructure only; see ``lin_oracle``)."""

from .lin_oracle import *  # noqa: F401,F403
from .lin_oracle import __all__  # noqa: F401
