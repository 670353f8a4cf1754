"""Seeded synthetic inputs for the quantized-linear path.

This package is shared by the oracle, the tests and the benchmark.  It only
draws random numbers and rounds them to bf16 storage; none of the
quantization arithmetic lives here.
"""
from .generators import (  # noqa: F401
    sub_rng,
    f32_to_bf16_bits,
    bf16_bits_to_f32,
    activations,
    weights,
    random_codes,
    outlier_channels,
)
from .workloads import WORKLOADS, Projection, layer_projections  # noqa: F401
