"""CPU oracle of the quantized linear projection.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with
the CUDA path.
"""
from . import vqlin_oracle  # noqa: F401
