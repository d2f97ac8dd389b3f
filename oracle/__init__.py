"""fp64 CPU oracle for the DSV sparse-attention hot path (test infrastructure only).

Only tests, the smoke check and bench.py's CPU-baseline leg may import this
package; the CUDA path never does.
"""
from .dsv_oracle import *  # noqa: F401,F403
