"""fp64 CPU oracle for MLA latent-cache decode: test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import it; the product path never does.
"""
from .mla_oracle import *  # noqa: F401,F403
