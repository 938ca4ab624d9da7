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
    """Zero-filled persistent buffers sized as include/mk.h describes: the KV cache of the GQA layers, the
    recurrent state and the two halves of the pending-row store of the delta-rule layers, and the
    per-sequence counts. Returns the tensors (kept alive by the caller) and the StateBuffers record."""
    from decode_megakernel_04_gb300 import binding
    n_gqa = sum(1 for m in cfg.mixers if m == "gqa")
    n_lin = sum(1 for m in cfg.mixers if m in ("gdn", "kda"))
    keep = []

    def zeros(n, dtype):
        if n == 0:
            return None
        t = torch.zeros(n, dtype=dtype, device=dev)
        keep.append(t)
        return t.data_ptr()

    kv = n_gqa * desc.max_batch * cfg.n_kv_heads * desc.max_ctx * cfg.head_dim
    rec = (2 * cfg.lin_dk + cfg.lin_dv + 1 + 3) // 4 * 4
    state = n_lin * desc.max_batch * cfg.lin_heads * cfg.lin_dv * cfg.lin_dk
    pending = n_lin * 2 * desc.max_batch * desc.max_rows * cfg.lin_heads * rec
    sb = binding.StateBuffers(kcache=zeros(kv, torch.bfloat16), vcache=zeros(kv, torch.bfloat16),
                              state=zeros(state, torch.float32), pending=zeros(pending, torch.float32),
                              seq=zeros(desc.max_batch * 4, torch.int32), epoch=0)
    return keep, sb


def _packed_weights(mk, dev):
    """The caller's tiled copy of the projection matrices (mk_pack_weights into a 1024-byte aligned buffer
    the caller owns) and a weight table that points to it, as mk_decode_step_static requires."""
    from decode_megakernel_04_gb300 import binding
    n = binding.packed_weight_bytes(mk.desc, mk.wtab, dev.index or 0)
    buf = torch.empty(n + 1024, dtype=torch.uint8, device=dev)
    ptr = (buf.data_ptr() + 1023) // 1024 * 1024
    binding.pack_weights(mk.desc, mk.wtab, ptr, dev.index or 0)
    torch.cuda.synchronize()
    wt = binding.Weights()
    C.memmove(C.byref(wt), C.byref(mk.wtab), C.sizeof(wt))
    wt.packed = ptr
    return buf, wt


def _compare_calls(lib, mk, sb, cfg, calls, dev):
    """Runs each (tokens, positions) call through mk_decode_step on the handle and through
    mk_decode_step_static on the caller's buffers; logits within TOL, greedy tokens equal, and the
    caller's call counter advanced by one per call."""
    from decode_megakernel_04_gb300 import binding
    packed_buf, wt = _packed_weights(mk, dev)
    for i, (toks, pos) in enumerate(calls):
        toks = toks.contiguous()
        B, R = toks.shape
        pos_t = torch.tensor(pos, dtype=torch.int32, device=dev)
        n = toks.numel()
        la = torch.empty((n, cfg.vocab), device=dev)
        aa = torch.empty((n,), dtype=torch.int32, device=dev)
        mk.step(toks, pos_t, la, aa)
        assert mk.status() == 0
        lb = torch.full((n, cfg.vocab), float("nan"), device=dev)
        ab = torch.full((n,), -1, dtype=torch.int32, device=dev)
        rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(wt), C.byref(sb), toks.data_ptr(),
                                       pos_t.data_ptr(), B, R, lb.data_ptr(), ab.data_ptr(), None)
        assert rc == 0, binding.STATUS.get(rc, rc)
        err = float((la - lb).abs().max())
        assert err <= TOL, (i, err)
        np.testing.assert_array_equal(aa.cpu().numpy(), ab.cpu().numpy())
        assert sb.epoch == i + 1


def test_static_entry_point_matches_handle_entry_point():
    from decode_megakernel_04_gb300 import Megakernel, _build, binding
    _build.build()
    lib = binding.load()
    cfg = config("tiny_dense")
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=4, device=dev)
    B, R, max_ctx = 2, 8, 64
    mk = Megakernel(cfg, w, max_batch=B, max_rows=R, max_ctx=max_ctx)
    keep, sb = _state_buffers(cfg, mk.desc, dev)
    # two calls in a row: an 8-row block from an empty context, then one row after committing all 8
    calls = [(make_tokens(4, "a", (B, R), cfg.vocab, device=dev), [0, 0]),
             (make_tokens(4, "b", (B, 1), cfg.vocab, device=dev), [R, R])]
    _compare_calls(lib, mk, sb, cfg, calls, dev)
    mk.close()


def test_handle_on_caller_packed_weights():
    """mk_create with weights->packed set reads the caller's tiled copy (mk_pack_weights) instead of making its
    own: the same step gives the same logits, bit for bit, and the handle owns less device memory."""
    from decode_megakernel_04_gb300 import Megakernel, binding
    cfg = config("hybrid_gdn_gqa", n_layers=2, d_model=256, ffn_dim=512, vocab=2048, n_q_heads=4, n_kv_heads=2,
                 head_dim=64, lin_heads=4, lin_dk=64, lin_dv=32)
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=7, device=dev)
    a = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64)
    buf, wt = _packed_weights(a, dev)
    b = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64, packed=wt.packed)
    ia, ib = binding.Info(), binding.Info()
    assert a.lib.mk_get_info(a.h, C.byref(ia)) == 0 and b.lib.mk_get_info(b.h, C.byref(ib)) == 0
    n = binding.packed_weight_bytes(a.desc, a.wtab, dev.index or 0)
    assert ia.device_bytes - ib.device_bytes == n
    toks = make_tokens(7, "p", (2, 8), cfg.vocab, device=dev).contiguous()
    pos = torch.zeros(2, dtype=torch.int32, device=dev)
    la, lb = torch.empty((16, cfg.vocab), device=dev), torch.empty((16, cfg.vocab), device=dev)
    a.step(toks, pos, la)
    b.step(toks, pos, lb)
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(la, lb)
    a.close()
    b.close()


def test_static_entry_point_hybrid_state_and_pending_rows():
    """A gated-delta-net + GQA stack, where the step also depends on the caller's recurrent state and on
    its pending-row store (which half a call reads and writes follows the caller's call counter): 8-row
    verify blocks with partial acceptance and single rows in between, every call equal to the handle's."""
    from decode_megakernel_04_gb300 import Megakernel, _build, binding
    _build.build()
    lib = binding.load()
    cfg = config("hybrid_gdn_gqa", n_layers=4, d_model=256, ffn_dim=512, vocab=2048, n_q_heads=4, n_kv_heads=2,
                 head_dim=64, lin_heads=4, lin_dk=64, lin_dv=32)
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=6, device=dev)
    B, R, max_ctx = 2, 8, 64
    mk = Megakernel(cfg, w, max_batch=B, max_rows=R, max_ctx=max_ctx)
    keep, sb = _state_buffers(cfg, mk.desc, dev)
    calls = [(make_tokens(6, "a", (B, R), cfg.vocab, device=dev), [0, 0]),      # verify block from empty
             (make_tokens(6, "b", (B, 1), cfg.vocab, device=dev), [3, 5]),      # accept 3 and 5 of its rows
             (make_tokens(6, "c", (B, R), cfg.vocab, device=dev), [4, 6]),      # another block
             (make_tokens(6, "d", (B, 1), cfg.vocab, device=dev), [12, 8])]     # accept 8 and 2
    _compare_calls(lib, mk, sb, cfg, calls, dev)
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
    keep, sb = _state_buffers(cfg, mk.desc, dev)
    toks = torch.zeros((1, 8), dtype=torch.int32, device=dev)
    pos = torch.zeros((1,), dtype=torch.int32, device=dev)
    lg = torch.empty((8, cfg.vocab), device=dev)
    # without the caller's packed weights the call is refused
    rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(mk.wtab), C.byref(sb), toks.data_ptr(),
                                   pos.data_ptr(), 1, 1, lg.data_ptr(), None, None)
    assert rc == 1  # MK_ERR_INVALID_ARG
    packed_buf, wt = _packed_weights(mk, dev)
    rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(wt), C.byref(sb), toks.data_ptr(),
                                   pos.data_ptr(), 1, 8, lg.data_ptr(), None, None)
    assert rc == 2  # MK_ERR_UNSUPPORTED
    assert sb.epoch == 0
    # a single row fits and runs
    lg1 = torch.empty((1, cfg.vocab), device=dev)
    rc = lib.mk_decode_step_static(C.byref(mk.desc), C.byref(wt), C.byref(sb), toks.data_ptr(),
                                   pos.data_ptr(), 1, 1, lg1.data_ptr(), None, None)
    assert rc == 0
    assert torch.isfinite(lg1).all()
    mk.close()
