"""CPU oracle of the attention hot path (test infrastructure only).

Imported by tests, the smoke check and the benchmark's CPU-baseline leg; the
product library never imports it.
"""
from .reference import *  # noqa: F401,F403
