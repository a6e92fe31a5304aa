"""CPU oracle of the DSpark proposal head and greedy verify step.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's CPU
baseline.  The library never imports it.
"""
from .dspark_oracle import *  # noqa: F401,F403
from . import dspark_oracle, check  # noqa: F401
