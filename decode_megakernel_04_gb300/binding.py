"""Thin ctypes binding of libmk (include/mk.h). Argument marshalling only: every step of the decode
path runs in the library's CUDA kernels. Loading fails loudly when the library is missing; nothing
here computes on the CPU."""
from __future__ import annotations

import ctypes as C
import os

MK_MAX_LAYERS = 128
MIXERS = {"gqa": 0, "gdn": 1, "kda": 2, "mla": 3}
STATUS = {0: "MK_OK", 1: "MK_ERR_INVALID_ARG", 2: "MK_ERR_UNSUPPORTED", 3: "MK_ERR_NOMEM", 4: "MK_ERR_CUDA",
          5: "MK_ERR_TIMEOUT", 6: "MK_ERR_DEVICE"}
MK_OK, MK_ERR_TIMEOUT, MK_ERR_DEVICE = 0, 5, 6

_I = C.c_int32
_F = C.c_float
_P = C.c_void_p


class ModelDesc(C.Structure):
    _fields_ = [
        ("n_layers", _I), ("d_model", _I), ("vocab", _I), ("tied_embedding", _I),
        ("norm_eps", _F), ("rope_theta", _F), ("mixer", _I * MK_MAX_LAYERS),
        ("n_q_heads", _I), ("n_kv_heads", _I), ("head_dim", _I),
        ("lin_heads", _I), ("lin_dk", _I), ("lin_dv", _I),
        ("mla_heads", _I), ("q_lora", _I), ("kv_lora", _I), ("qk_nope", _I), ("qk_rope", _I), ("v_head", _I),
        ("ffn_kind", _I), ("ffn_dim", _I), ("n_experts", _I), ("top_k", _I), ("n_shared", _I),
        ("expert_dim", _I), ("expert_format", _I), ("route_scale", _F),
        ("max_batch", _I), ("max_rows", _I), ("max_ctx", _I),
    ]


LAYER_FIELDS = [
    "attn_norm", "ffn_norm", "wq", "wk", "wv", "wo", "wa", "wb",
    "w_dq", "q_norm", "w_uq", "w_dkv", "kv_norm", "w_uk", "w_uv",
    "w_gate", "w_up", "w_down", "w_router", "router_bias",
    "e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down",
    "e_gate_scales", "e_up_scales", "e_down_scales", "s_gate_scales", "s_up_scales", "s_down_scales",
    "e_gate_gscale", "e_up_gscale", "e_down_gscale", "s_gate_gscale", "s_up_gscale", "s_down_gscale",
]


class LayerWeights(C.Structure):
    _fields_ = [(f, _P) for f in LAYER_FIELDS]


class Weights(C.Structure):
    _fields_ = [("embed", _P), ("final_norm", _P), ("lm_head", _P), ("layers", LayerWeights * MK_MAX_LAYERS),
                ("packed", _P)]


class Info(C.Structure):
    _fields_ = [("n_sm", _I), ("threads_per_cta", _I), ("smem_bytes", _I), ("ring_slots", _I),
                ("ring_slot_bytes", _I), ("n_ops_last", _I), ("device_bytes", C.c_int64)]


PLAN_OP_FIELDS = ["type", "n_instr", "layer", "rows", "K", "k_begin", "ldw", "mma", "staged", "kc", "rg", "passes",
                  "out_kind", "nchunk", "groups", "head_dim", "n_heads", "n_kv_heads", "col_group"]


PLAN_OP_FIELDS += ["ncols", "pa0", "patoms", "pk_offset"]


class PlanOp(C.Structure):
    _fields_ = [(f, _I) for f in PLAN_OP_FIELDS[:-1]] + [("pk_offset", C.c_int64)]


class PlanInstr(C.Structure):
    _fields_ = [("op", _I), ("sm", _I), ("a", _I), ("b", _I), ("c", _I)]


class StateBuffers(C.Structure):
    """Caller-owned persistent buffers of mk_decode_step_static (see include/mk.h)."""
    _fields_ = [("kcache", _P), ("vcache", _P), ("state", _P), ("pending", _P), ("seq", _P), ("epoch", C.c_uint32)]


EXPORTS = ["mk_create", "mk_prefill_kv", "mk_decode_step", "mk_decode_step_host", "mk_get_status",
           "mk_last_error", "mk_get_info", "mk_destroy", "mk_decode_step_static", "mk_set_routing_log",
           "mk_fork_sequence", "mk_plan", "mk_set_wait_limit",
           "mk_set_routing_override", "mk_decode_steps", "mk_decode_steps_host", "mk_verify_step",
           "mk_packed_weight_bytes", "mk_pack_weights"]

_lib = None


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmk.so")


def load(path: str | None = None) -> C.CDLL:
    """Load libmk.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libmk.so not found at {p}: build it with decode_megakernel_04_gb300._build.build()")
    lib = C.CDLL(p)
    lib.mk_create.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.c_int, C.POINTER(_P)]
    lib.mk_prefill_kv.argtypes = [_P, _P, C.c_int, C.c_int, _P]
    lib.mk_decode_step.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, _P, _P]
    lib.mk_decode_step_host.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, _P, _P]
    lib.mk_get_status.argtypes = [_P, _P]
    lib.mk_last_error.argtypes = [_P]
    lib.mk_last_error.restype = C.c_char_p
    lib.mk_get_info.argtypes = [_P, C.POINTER(Info)]
    lib.mk_destroy.argtypes = [_P]
    lib.mk_destroy.restype = None
    lib.mk_set_routing_log.argtypes = [_P, _P]
    lib.mk_fork_sequence.argtypes = [_P, C.c_int, C.c_int, _P]
    lib.mk_set_wait_limit.argtypes = [_P, C.c_uint64]
    lib.mk_set_routing_override.argtypes = [_P, _P]
    lib.mk_decode_steps.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, _P, _P]
    lib.mk_decode_steps_host.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, _P]
    lib.mk_verify_step.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, _P, _P, _P]
    lib.mk_plan.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.c_int, C.c_int, C.c_int, C.c_int,
                            C.POINTER(PlanOp), C.c_int, C.POINTER(C.c_int), C.POINTER(PlanInstr), C.c_int,
                            C.POINTER(C.c_int)]
    lib.mk_decode_step_static.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.POINTER(StateBuffers),
                                          _P, _P, C.c_int, C.c_int, _P, _P, _P]
    lib.mk_packed_weight_bytes.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.c_int, C.POINTER(C.c_uint64)]
    lib.mk_pack_weights.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.c_int, _P, _P]
    for f in ("mk_packed_weight_bytes", "mk_pack_weights", "mk_create", "mk_prefill_kv", "mk_decode_step", "mk_decode_step_host", "mk_get_status", "mk_get_info",
              "mk_decode_step_static", "mk_set_routing_log", "mk_fork_sequence", "mk_plan", "mk_set_wait_limit",
              "mk_set_routing_override", "mk_decode_steps", "mk_decode_steps_host", "mk_verify_step"):
        getattr(lib, f).restype = C.c_int
    if path is None:
        _lib = lib
    return lib


def plan(desc: ModelDesc, weights: Weights, n_sm: int, batch: int, rows: int, head: bool = True):
    """mk_plan: the program of one step shape for an n_sm-SM device, compiled on the host. Returns
    (ops, instrs) as lists of dicts (fields of mk_plan_op / mk_plan_instr)."""
    lib = load()
    n_ops, n_instr = C.c_int(0), C.c_int(0)
    rc = lib.mk_plan(C.byref(desc), C.byref(weights), n_sm, batch, rows, int(head), None, 0, C.byref(n_ops), None, 0,
                     C.byref(n_instr))
    if rc != MK_OK:
        raise MKError(rc, "mk_plan")
    ops = (PlanOp * max(1, n_ops.value))()
    ins = (PlanInstr * max(1, n_instr.value))()
    rc = lib.mk_plan(C.byref(desc), C.byref(weights), n_sm, batch, rows, int(head), ops, n_ops.value, C.byref(n_ops),
                     ins, n_instr.value, C.byref(n_instr))
    if rc != MK_OK:
        raise MKError(rc, "mk_plan")
    as_dict = lambda r, names: {f: getattr(r, f) for f in names}
    return ([as_dict(ops[i], PLAN_OP_FIELDS) for i in range(n_ops.value)],
            [as_dict(ins[i], ("op", "sm", "a", "b", "c")) for i in range(n_instr.value)])


def packed_weight_bytes(desc: ModelDesc, weights: Weights, device: int = 0) -> int:
    """mk_packed_weight_bytes: size of the tiled copy of the projection matrices on `device`."""
    n = C.c_uint64(0)
    rc = load().mk_packed_weight_bytes(C.byref(desc), C.byref(weights), device, C.byref(n))
    if rc != MK_OK:
        raise MKError(rc, "mk_packed_weight_bytes")
    return n.value


def pack_weights(desc: ModelDesc, weights: Weights, packed_ptr: int, device: int = 0, stream: int = 0) -> None:
    """mk_pack_weights: fill the caller's device buffer (packed_weight_bytes long, 1024-byte aligned)."""
    rc = load().mk_pack_weights(C.byref(desc), C.byref(weights), device, packed_ptr, stream or None)
    if rc != MK_OK:
        raise MKError(rc, "mk_pack_weights")


class MKError(RuntimeError):
    def __init__(self, code, msg=""):
        self.code = code
        super().__init__(f"{STATUS.get(code, code)}: {msg}")


def model_desc(cfg, max_batch: int, max_rows: int, max_ctx: int) -> ModelDesc:
    """Fill the C model description from a config object with the attribute names of mk_model_desc."""
    d = ModelDesc()
    d.n_layers = cfg.n_layers
    d.d_model = cfg.d_model
    d.vocab = cfg.vocab
    d.tied_embedding = int(cfg.tied)
    d.norm_eps = cfg.norm_eps
    d.rope_theta = cfg.rope_theta
    for i, m in enumerate(cfg.mixers):
        d.mixer[i] = MIXERS[m]
    for f in ("n_q_heads", "n_kv_heads", "head_dim", "lin_heads", "lin_dk", "lin_dv", "mla_heads", "q_lora",
              "kv_lora", "qk_nope", "qk_rope", "v_head", "ffn_dim", "n_experts", "top_k", "n_shared", "expert_dim"):
        setattr(d, f, int(getattr(cfg, f)))
    d.ffn_kind = 0 if cfg.ffn == "dense" else 1
    if cfg.expert_fmt not in ("bf16", "nvfp4"):
        raise ValueError(f"expert format {cfg.expert_fmt!r} has no kernel path (bf16 and nvfp4 do)")
    d.expert_format = 0 if cfg.expert_fmt == "bf16" else 1
    d.route_scale = cfg.route_scale
    d.max_batch, d.max_rows, d.max_ctx = max_batch, max_rows, max_ctx
    return d


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def weight_table(cfg, w: dict) -> Weights:
    """Device pointers of the named weight tensors (names as drawn by the synthetic workloads)."""
    W = Weights()
    W.embed = _ptr(w["embed"])
    W.final_norm = _ptr(w["final_norm"])
    W.lm_head = _ptr(w.get("lm_head"))
    nvfp4 = cfg.expert_fmt == "nvfp4"
    for i in range(cfg.n_layers):
        L = W.layers[i]
        p = f"layers.{i}."
        for f in LAYER_FIELDS:
            if f.endswith("_scales") or f.endswith("_gscale"):
                continue
            key = p + f
            if f in ("e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down") and nvfp4:
                if key + ".q" in w:
                    setattr(L, f, _ptr(w[key + ".q"]))
                    setattr(L, f + "_scales", _ptr(w[key + ".s"]))
                    setattr(L, f + "_gscale", _ptr(w[key + ".g"]))
            elif key in w:
                setattr(L, f, _ptr(w[key]))
    return W


class Megakernel:
    """One handle of the C library: a model on one GPU plus its caches and states."""

    def __init__(self, cfg, weights: dict, max_batch: int, max_rows: int, max_ctx: int, device: int = 0,
                 packed: int = 0):
        """packed: device address of a tiled copy of the projection matrices written by pack_weights for this
        model (kept alive by the caller), or 0 to let the handle make its own."""
        self.lib = load()
        self.cfg = cfg
        self._weights = weights  # keep the tensors alive for the handle's lifetime
        self.desc = model_desc(cfg, max_batch, max_rows, max_ctx)
        self.wtab = weight_table(cfg, weights)
        self.wtab.packed = packed or None
        h = _P()
        rc = self.lib.mk_create(C.byref(self.desc), C.byref(self.wtab), device, C.byref(h))
        if rc != MK_OK:
            raise MKError(rc, "mk_create failed (details on stderr)")
        self.h = h

    def _check(self, rc):
        if rc != MK_OK:
            raise MKError(rc, self.lib.mk_last_error(self.h).decode())

    def prefill(self, tokens, stream=None):
        """tokens: device int32 [B, T] (contiguous)."""
        B, T = tokens.shape
        self._check(self.lib.mk_prefill_kv(self.h, tokens.data_ptr(), B, T, stream))

    def step(self, tokens, positions, logits=None, argmax=None, stream=None):
        """tokens: device int32 [B, R]; positions: device int32 [B]; outputs preallocated device tensors."""
        B, R = tokens.shape
        self._check(self.lib.mk_decode_step(self.h, tokens.data_ptr(), positions.data_ptr(), B, R,
                                             _ptr(logits), _ptr(argmax), stream))

    def step_host(self, tokens_np, positions_np, argmax_np, logits_np=None, stream=None):
        """Host (numpy int32 / float32, C-contiguous) variant: copies in, runs, copies out, waits."""
        B, R = tokens_np.shape
        rc = self.lib.mk_decode_step_host(
            self.h, tokens_np.ctypes.data, positions_np.ctypes.data, B, R,
            None if logits_np is None else logits_np.ctypes.data, argmax_np.ctypes.data, stream)
        self._check(rc)

    def verify(self, tokens, positions, accept_out, logits=None, argmax=None, stream=None):
        """Verify step with on-device greedy acceptance. tokens: device int32 [B, R] (anchor + drafts);
        accept_out: device int32 [3, B] (accepted length, bonus token, next position)."""
        B, R = tokens.shape
        self._check(self.lib.mk_verify_step(self.h, tokens.data_ptr(), positions.data_ptr(), B, R, _ptr(logits),
                                             _ptr(argmax), accept_out.data_ptr(), stream))

    def steps(self, tokens, positions, n_steps: int, tokens_out, logits=None, stream=None):
        """n_steps greedy steps in one launch. tokens, positions: device int32 [B]; tokens_out: device int32
        [n_steps, B]; logits: device fp32 [B, V] or None (the last step's)."""
        B = tokens.shape[0]
        self._check(self.lib.mk_decode_steps(self.h, tokens.data_ptr(), positions.data_ptr(), B, n_steps,
                                              tokens_out.data_ptr(), _ptr(logits), stream))

    def steps_host(self, tokens_np, positions_np, n_steps: int, tokens_out_np, stream=None):
        """Host (numpy int32) variant of steps: copies in, runs, copies the tokens [n_steps, B] out, waits."""
        B = tokens_np.shape[0]
        self._check(self.lib.mk_decode_steps_host(self.h, tokens_np.ctypes.data, positions_np.ctypes.data, B,
                                                   n_steps, tokens_out_np.ctypes.data, stream))

    def fork(self, src: int, dst: int, stream=None):
        """Make sequence ``dst`` a copy of sequence ``src`` (caches, states, pending rows, counts)."""
        self._check(self.lib.mk_fork_sequence(self.h, src, dst, stream))

    def set_routing_log(self, log=None):
        """Route the expert ids of every MoE row into ``log`` (device int32 [n_layers, max_batch, max_ctx,
        top_k], kept alive by this object while set); None turns the log off."""
        self._route_log = log
        self._check(self.lib.mk_set_routing_log(self.h, None if log is None else log.data_ptr()))

    def set_routing_override(self, ids=None):
        """Make MoE rows use the expert ids in ``ids`` (device int32, the routing log's layout; rows whose
        first id is < 0 use their own picks), kept alive by this object while set; None turns it off."""
        self._route_force = ids
        self._check(self.lib.mk_set_routing_override(self.h, None if ids is None else ids.data_ptr()))

    def set_wait_limit(self, limit_ns: int):
        """Time limit of every wait inside the kernel (default 2 s); see mk_set_wait_limit."""
        self._check(self.lib.mk_set_wait_limit(self.h, int(limit_ns)))

    def status(self, stream=None) -> int:
        return self.lib.mk_get_status(self.h, stream)

    def info(self) -> Info:
        i = Info()
        self._check(self.lib.mk_get_info(self.h, C.byref(i)))
        return i

    def close(self):
        if getattr(self, "h", None):
            self.lib.mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
