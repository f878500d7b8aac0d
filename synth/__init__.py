"""Seeded synthetic inputs shared by the tests, the benchmark and smoke().

This package only draws inputs (lengths, block permutations, values).  It
holds none of the attention or addressing arithmetic: slot mappings, cache
writes and attention are computed separately by the oracle and by the CUDA
library.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    DecodeCase,
    MlaCase,
    PrefillCase,
    decode_case,
    mla_case,
    prefill_case,
    make_config,
)
