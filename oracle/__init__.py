"""CPU oracle of the GPT2 tile-task training step.

TEST INFRASTRUCTURE: imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg. The library never imports it and shares no code
with it.
"""
from .gpt2 import *  # noqa: F401,F403
