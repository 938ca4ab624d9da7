"""GPU parity at the context lengths the benchmark runs (4096 and 8192 cached positions), with the real
attention shapes of the workloads and narrow everything else, so the oracle's prefill stays affordable.

At these lengths an attention instruction covers hundreds of positions: its online softmax folds many
weight-ring chunks (each 32 KB of K and V, or of MLA latents) and many 32-key blocks per chunk, carrying
the running (max, sum, output) across them; each test asserts from the compiled program that every
attention instruction streams at least four ring chunks. Contexts are prefilled once per model (the
oracle in blocks of rows, the GPU in 8-row launches) and forked to the other sequences, which then decode
their own tokens."""
import dataclasses

import pytest

from synthetic import config

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_megakernel_04_gb300 import _build
    _build.build()


def _check(rep):
    assert not rep.errors, "\n".join(rep.errors[:10])
    assert rep.token_mismatch == 0
    assert rep.compared >= 2


def _gdn_gqa():
    """One gated-delta-net layer and one GQA layer with the hybrid workload's attention (24 q / 4 kv heads
    of 256) and delta-rule shapes (16 heads of 128), d_model 512."""
    return dataclasses.replace(config("hybrid_gdn_gqa"), n_layers=2, mixers=("gdn", "gqa"), d_model=512,
                               ffn_dim=1024, vocab=4096)


def _gqa_48():
    """One GQA layer with the NVFP4 MoE workload's attention shape (48 q / 8 kv heads of 128), dense FFN."""
    return dataclasses.replace(config("hybrid_gdn_gqa"), n_layers=1, mixers=("gqa",), n_q_heads=48,
                               n_kv_heads=8, head_dim=128, d_model=512, ffn_dim=1024, vocab=4096)


def _mla(heads):
    """One MLA layer with the KDA/MLA workload's latent (512 + 64), q_lora 1536, nope 128, v_head 128."""
    return dataclasses.replace(config("moe_kda_mla"), n_layers=1, mixers=("mla",), ffn="dense", ffn_dim=1024,
                               d_model=1024, vocab=4096, mla_heads=heads)


@pytest.mark.parametrize("B", [1, 8])
def test_gqa_24x256_ctx4096(B):
    from gpu_harness import run_case
    rep = run_case(_gdn_gqa(), B=B, T=4096, decode_steps=2, verify_accepts=(3, 6) if B == 1 else (5,),
                   tol=TOL, max_ctx=4200, fork=True, oracle_block=128, min_ring_chunks=4)
    _check(rep)


@pytest.mark.parametrize("B", [1, 8])
def test_gqa_48x128_ctx8192(B):
    from gpu_harness import run_case
    rep = run_case(_gqa_48(), B=B, T=8192, decode_steps=2, verify_accepts=(3, 6) if B == 1 else (),
                   tol=TOL, max_ctx=8300, fork=True, oracle_block=256, min_ring_chunks=4)
    _check(rep)


def test_mla_64_heads_ctx2048():
    from gpu_harness import run_case
    rep = run_case(_mla(64), B=1, T=2048, decode_steps=2, verify_accepts=(3, 6), tol=TOL, max_ctx=2150,
                   fork=True, oracle_block=256, min_ring_chunks=4)
    _check(rep)


def test_mla_8_heads_ctx8192_batch8():
    from gpu_harness import run_case
    rep = run_case(_mla(8), B=8, T=8192, decode_steps=2, verify_accepts=(4,), tol=TOL, max_ctx=8300,
                   fork=True, oracle_block=256, min_ring_chunks=4)
    _check(rep)
