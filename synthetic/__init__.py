"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the benchmark.

This package only *describes and draws inputs*: model shapes, weights drawn from N(0, std)
and rounded to bf16, the NVFP4 and MXFP4 / FP8 encodings of expert weights, token streams. It holds none of the
decode-step arithmetic; the oracle (``oracle/``) and the CUDA path (``decode_megakernel_04_gb300``)
each implement that on their own and share nothing but what this package hands them.
"""
from .workloads import (  # noqa: F401
    ModelConfig,
    CONFIGS,
    config,
    make_weights,
    make_tokens,
    weight_names,
)
from .nvfp4 import quantize_nvfp4, quantize_nvfp4_experts, E2M1_GRID  # noqa: F401
from .mxfp4 import quantize_mxfp4, reencode_fp8_rows  # noqa: F401
