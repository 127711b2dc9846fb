"""Seeded synthetic inputs for the paged KV-cache decode path.

Both the CUDA path (its tests and ``bench.py``) and the CPU oracle's tests take
their inputs from here.  The module only draws random numbers and lays out the
structure of a workload (sequence lengths, which physical block a logical block
sits in, which sequences fork); it computes none of the method's arithmetic.
"""

from .gen import (  # noqa: F401
    DTYPES,
    BeamPlan,
    DecodeBatch,
    MixedServingPlan,
    SamplingPlan,
    beam_search,
    decode_13b,
    lognormal_lengths,
    long_context,
    mixed_serving,
    parallel_sampling,
    random_decode_batch,
    tiny_decode,
)
