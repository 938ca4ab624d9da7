"""mk_decode_step_static: the decode step for callers that cannot allocate device memory at decode time
(for instance a serving process whose own pool already holds all free HBM). It runs the same kernel as
mk_decode_step with its working memory in a fixed device array inside the library, and the caller's
own buffers for the caches and the per-sequence bookkeeping.

This file is collected last on purpose: the test reuses the library's one static array, and a failure
here should come after every other test has run."""
import ctypes as C

import numpy as np
import pytest
import torch

from synthetic import config, make_tokens, make_weights

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16-path tolerance of the parity tests


def _state_buffers(cfg, desc, dev):
    """Zero-filled persistent buffers sized as include/mk.h describes (GQA-only model)."""
    n_gqa = sum(1 for m in cfg.mixers if m == "gqa")
    kv = n_gqa * desc.max_batch * cfg.n_kv_heads * desc.max_ctx * cfg.head_dim
    kc = torch.zeros(kv, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros(kv, dtype=torch.bfloat16, device=dev)
    seq = torch.zeros(desc.max_batch * 4, dtype=torch.int32, device=dev)
    return (kc, vc, seq)


def test_static_entry_point_matches_handle_entry_point():
    from decode_megakernel_04_gb300 import Megakernel, _build, binding
    _build.build()
    lib = binding.load()
    cfg = config("tiny_dense")
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=4, device=dev)
    B, R, max_ctx = 2, 8, 64
    mk = Megakernel(cfg, w, max_batch=B, max_rows=R, max_ctx=max_ctx)
    kc, vc, seq = _state_buffers(cfg, mk.desc, dev)
    sb = binding.StateBuffers(kcache=kc.data_ptr(), vcache=vc.data_ptr(), state=None, pending=None,
                              seq=seq.data_ptr(), epoch=0)
    # two calls in a row: an 8-row block from an empty context, then one row after committing all 8
    calls = [(make_tokens(4, "a", (B, R), cfg.vocab, device=dev), [0, 0]),
             (make_tokens(4, "b", (B, 1), cfg.vocab, device=dev), [R, R])]
    for toks, pos in calls:
        toks = toks.contiguous()
        pos_t = torch.tensor(pos, dtype=torch.int32, device=dev)
        n = toks.numel()
        la = torch.empty((n, cfg.vocab), device=dev)
        aa = torch.empty((n,), dtype=torch.int32, device=dev)
        mk.step(toks, pos_t, la, aa)
        assert mk.status() == 0
        lb = torch.full((n, cfg.vocab), float("nan"), device=dev)
        ab = torch.full((n,), -1, dtype=torch.int32, device=dev)
        rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(mk.wtab), C.byref(sb), toks.data_ptr(),
                                       pos_t.data_ptr(), B, toks.shape[1], lb.data_ptr(), ab.data_ptr(), None)
        assert rc == 0, binding.STATUS.get(rc, rc)
        err = float((la - lb).abs().max())
        assert err <= TOL, err
        np.testing.assert_array_equal(aa.cpu().numpy(), ab.cpu().numpy())
    assert sb.epoch == 2
    mk.close()


def test_static_entry_point_rejects_oversized_step():
    """A step whose working memory exceeds the static array is refused before anything runs."""
    from decode_megakernel_04_gb300 import Megakernel, _build, binding
    _build.build()
    lib = binding.load()
    # one small layer, but 8 q heads of width 256 per kv head and 8 rows: the attention partials alone
    # need more than the static array holds
    cfg = config("tiny_dense", n_layers=1, d_model=64, vocab=97, n_q_heads=8, n_kv_heads=1, head_dim=256,
                 ffn_dim=64)
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=0, device=dev)
    mk = Megakernel(cfg, w, max_batch=1, max_rows=8, max_ctx=32)
    kc, vc, seq = _state_buffers(cfg, mk.desc, dev)
    sb = binding.StateBuffers(kcache=kc.data_ptr(), vcache=vc.data_ptr(), state=None, pending=None,
                              seq=seq.data_ptr(), epoch=0)
    toks = torch.zeros((1, 8), dtype=torch.int32, device=dev)
    pos = torch.zeros((1,), dtype=torch.int32, device=dev)
    lg = torch.empty((8, cfg.vocab), device=dev)
    rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(mk.wtab), C.byref(sb), toks.data_ptr(),
                                   pos.data_ptr(), 1, 8, lg.data_ptr(), None, None)
    assert rc == 2  # MK_ERR_UNSUPPORTED
    assert sb.epoch == 0
    # a single row fits and runs
    lg1 = torch.empty((1, cfg.vocab), device=dev)
    rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(mk.wtab), C.byref(sb), toks.data_ptr(),
                                   pos.data_ptr(), 1, 1, lg1.data_ptr(), None, None)
    assert rc == 0
    assert torch.isfinite(lg1).all()
    mk.close()
