"""CPU oracle for the LoPA branch-verification step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use it; the CUDA
library never imports it and it never imports the library."""
from .lopa_oracle import *  # noqa: F401,F403
from . import lopa_oracle  # noqa: F401
