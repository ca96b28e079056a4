"""Oracle package: test infrastructure only (see latentmoe_oracle's docstring)."""
from .latentmoe_oracle import *  # noqa: F401,F403
