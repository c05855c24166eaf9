"""QSA oracle -- test infrastructure only.

A plain fp64 CPU statement of the Qwen Sparse Attention layer (see
``qsa_oracle.c`` for the sources and the readings it takes).  Only the tests,
the package smoke check and the benchmark's CPU-baseline leg may import this
package; the CUDA product path never does.
"""
from .oracle import *  # noqa: F401,F403
