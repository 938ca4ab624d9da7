"""CPU oracle for the whole-stack small-batch decode step.

TEST INFRASTRUCTURE ONLY. It exists to check the CUDA megakernel, and only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may
import it. The product package never imports it and it never imports the product package; the two
share only the seeded inputs drawn by ``synthetic``.

Everything is numpy in float64: activations, accumulations, the recurrent state. Weights are the
bf16-rounded draws (exact in float64); NVFP4 weights are decoded exactly as e2m1 * e4m3 * fp32, and
the pages' own expert format (FP8-E4M3 gate / up with a bf16 scale per 256 rows, MXFP4 down) exactly as
e4m3 * bf16 and e2m1 * 2^(E8M0 - 127).
The KV cache and the MLA latent cache hold the exact (float64) keys, values and latents: the pages fix
no cache precision, so a narrower storage type is the implementation's choice and its rounding is
absorbed by the comparison tolerance, not built into the definition.

Parity status of each function is recorded in its docstring; the pins live in tests/test_oracle_*.py.
"""
from .model import Oracle  # noqa: F401
from . import ops  # noqa: F401
