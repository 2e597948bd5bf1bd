"""Float64 CPU oracle for MLA absorbed decode (test infrastructure only).

Imported only by tests, the smoke check and the benchmark's CPU baseline.
The CUDA path never imports it.
"""
from .mla_oracle import *  # noqa: F401,F403
