"""CPU oracle of the two-tier sparse-attention step: test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the library. See dsa_oracle.py.
"""
from .dsa_oracle import *  # noqa: F401,F403
from .dsa_oracle import StepConfig  # noqa: F401
