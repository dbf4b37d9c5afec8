"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests.

This package only draws random numbers and lays them out (sequence lengths,
physical block ids, Q/K/V values, fp8 scales).  It holds none of the paged
attention arithmetic: no softmax, no slot arithmetic, no block-manager logic.
Both the oracle (``oracle/``) and the CUDA library receive exactly the same
tensors from here.
"""
from .configs import (  # noqa: F401
    DecodeCase,
    PrefillChunk,
    make_decode_case,
    tiny_config,
    qwen7b_gqa_config,
    mha13b_config,
    long_splitkv_config,
    mixed_config,
    CONFIG_BUILDERS,
)
