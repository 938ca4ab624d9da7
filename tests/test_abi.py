"""The C-ABI library builds, loads without a GPU and exports every entry point include/mk.h declares;
the ctypes structures match the C layout; host-side argument checks need no GPU."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

from decode_megakernel_04_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mk.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def _c_layout():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "mk.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("mk_model_desc %zu\n", sizeof(mk_model_desc));
  printf("mk_layer_weights %zu\n", sizeof(mk_layer_weights));
  printf("mk_weights %zu\n", sizeof(mk_weights));
  printf("mk_info %zu\n", sizeof(mk_info));
  printf("mk_state_buffers %zu\n", sizeof(mk_state_buffers));
  F(mk_model_desc, mixer) F(mk_model_desc, n_q_heads) F(mk_model_desc, route_scale) F(mk_model_desc, max_ctx)
  F(mk_layer_weights, w_dq) F(mk_layer_weights, w_router) F(mk_layer_weights, e_gate_scales)
  F(mk_layer_weights, s_down_gscale) F(mk_weights, layers) F(mk_info, device_bytes)
  F(mk_state_buffers, seq) F(mk_state_buffers, epoch)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I" + os.path.dirname(HEADER), c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return dict((k, int(v)) for k, v in (line.split() for line in out.strip().splitlines()))


def test_struct_layout_matches_header():
    c = _c_layout()
    assert C.sizeof(binding.ModelDesc) == c["mk_model_desc"]
    assert C.sizeof(binding.LayerWeights) == c["mk_layer_weights"]
    assert C.sizeof(binding.Weights) == c["mk_weights"]
    assert C.sizeof(binding.Info) == c["mk_info"]
    assert C.sizeof(binding.StateBuffers) == c["mk_state_buffers"]
    for key, off in c.items():
        if "." not in key:
            continue
        struct, field = key.split(".")
        cls = {"mk_model_desc": binding.ModelDesc, "mk_layer_weights": binding.LayerWeights,
               "mk_weights": binding.Weights, "mk_info": binding.Info,
               "mk_state_buffers": binding.StateBuffers}[struct]
        assert getattr(cls, field).offset == off, key


def test_host_argument_checks_need_no_gpu(lib):
    h = C.c_void_p()
    # NULL arguments are rejected before any CUDA call
    assert lib.mk_create(None, None, 0, C.byref(h)) == 1
    assert lib.mk_decode_step(None, None, None, 1, 1, None, None, None) == 1
    assert lib.mk_prefill_kv(None, None, 1, 1, None) == 1
    assert lib.mk_get_status(None, None) == 1
    assert lib.mk_set_wait_limit(None, 1) == 1
    # an inconsistent description is rejected by the host checks (no device touched)
    d = binding.ModelDesc()
    d.n_layers = 0
    w = binding.Weights()
    assert lib.mk_create(C.byref(d), C.byref(w), 0, C.byref(h)) == 1
    assert lib.mk_last_error(None) == b""
