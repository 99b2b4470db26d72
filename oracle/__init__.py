"""CPU oracle of the DDTree verify step (test infrastructure only).

Import only from tests, the smoke check and the bench's CPU-baseline leg.
"""
from .ddt_oracle import *  # noqa: F401,F403
