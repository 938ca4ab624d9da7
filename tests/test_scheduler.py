"""The host scheduler, checked on the CPU through mk_plan (include/mk.h): the program of a step shape is
compiled exactly as mk_decode_step compiles it, for a device with a given number of SMs, and its ops and
per-SM instruction queues are checked for coverage and ordering. No GPU is used: the weight pointers are
fake (present and 16-byte aligned, never dereferenced)."""
import collections
import dataclasses

import pytest

from decode_megakernel_04_gb300 import _build, binding
from synthetic import config
from synthetic.workloads import weight_names

EMBED, GEMV, ROPE, ATTN, DELTA, MLA_PREP, MLA_ATTN, ROUTE, MOE_UP, MOE_DOWN, FINAL, COMBINE, QABS, UV = range(14)
RESID, SWIGLU, LOGITS = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return binding.load()


def fake_weights(cfg) -> binding.Weights:
    W = binding.Weights()
    addr = [0x100000]

    def nxt():
        addr[0] += 0x1000
        return addr[0]

    W.embed = nxt()
    W.final_norm = nxt()
    W.lm_head = None if cfg.tied else nxt()
    for name in weight_names(cfg):
        if not name.startswith("layers."):
            continue
        _, i, field = name.split(".", 2)
        L = W.layers[int(i)]
        setattr(L, field, nxt())
        if cfg.expert_fmt == "nvfp4" and field in ("e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down"):
            setattr(L, field + "_scales", nxt())
            setattr(L, field + "_gscale", nxt())
    return W


def make_plan(cfg, n_sm, B, R, head=True, max_batch=8, max_rows=8, max_ctx=4096):
    desc = binding.model_desc(cfg, max_batch, max_rows, max_ctx)
    return binding.plan(desc, fake_weights(cfg), n_sm, B, R, head)


def pk_split(rows, n_sm, s):
    """first logical row of SM s's share of a GEMV: whole 8-row units, balanced"""
    units = -(-rows // 8)
    return min(rows, 8 * (units * s // n_sm))


def walk_chunks(o, instrs, packed_groups):
    """The ring chunks of a GEMV op, in the producer's (= the consumers') order: per instruction, row groups
    (one packed block on mma.sync; as many blocks as fit 512 TMEM columns on tcgen05), K parts (the whole K on
    mma.sync; 256 / ncols atoms on tcgen05), blocks of at most 128 physical rows (64 logical rows for SwiGLU),
    runs of at most 32 KB of atoms. Each chunk is one contiguous range of the group's packed copy; the ranges
    are recorded per group so that the op (or its K parts together) can be checked to read every byte once."""
    sw = 1 if o["out_kind"] == SWIGLU else 0
    br = 128
    A, nat = o["patoms"], -(-o["K"] // 64)
    tc = o["mma"] == 2
    KP = 256 // o["ncols"] if tc else nat
    per_group = packed_groups.setdefault(o["pk_offset"], {"bytes": (-(-o["rows"] // 8) * 8) * A * 128 * (1 + sw),
                                                          "ranges": []})
    def group_end(g0, b):
        # as many blocks as fit 512 TMEM columns: ncols per tile, times the block's K-stacking factor (up to 4
        # atoms per MMA for non-SwiGLU blocks of at most 64 rows with 16 activation columns)
        cols, r = 0, g0
        while r < b:
            e = min(b, r + br)
            P = (-(-(e - r) // 8) * 8) << sw
            st = 1 if (sw or o["ncols"] != 16) else max(1, min(4, 128 // P, nat))
            c = (1 + sw) * o["ncols"] * st
            if r > g0 and cols + c > 512:
                break
            cols, r = cols + c, e
        return r

    for x in instrs:
        a, b = x["a"], x["b"]
        if b <= a:
            continue
        g0 = a
        while g0 < b:
            g1 = group_end(g0, b) if tc else min(b, g0 + br)
            for a0 in range(0, nat, KP):
                r = g0
                while r < g1:
                    e = min(g1, r + br)
                    rows8 = -(-(e - r) // 8) * 8
                    P = rows8 << sw
                    bat = max(1, 256 // P)
                    base = r * A * 128 * (1 + sw) + (o["pa0"]) * P * 128
                    cc = a0
                    while cc < min(nat, a0 + KP):
                        na = min(bat, min(nat, a0 + KP) - cc)
                        off, nb = base + cc * P * 128, na * P * 128
                        assert 0 < nb <= 32768 and off % 1024 == 0 and off + nb <= per_group["bytes"]
                        per_group["ranges"].append((off, nb))
                        cc += na
                    r = e
            g0 = g1


def check_program(cfg, n_sm, B, R, head=True):
    ops, ins = make_plan(cfg, n_sm, B, R, head)
    N = B * R
    by_op = collections.defaultdict(list)
    for x in ins:
        by_op[x["op"]].append(x)
    # every op's instruction count is its counter target; each SM runs its queue in op order
    for k, o in enumerate(ops):
        assert o["n_instr"] == len(by_op[k]), (k, o)
    last = collections.defaultdict(lambda: -1)
    for x in ins:
        assert x["op"] >= last[x["sm"]], "an SM's queue must follow the op order"
        last[x["sm"]] = x["op"]
    assert ops[-1]["type"] == FINAL and ops[-1]["n_instr"] == 1 and by_op[len(ops) - 1][0]["sm"] == 0
    assert ops[0]["type"] == EMBED
    assert len(ops) <= 32 * cfg.n_layers + 16

    def partition(k, total):
        """instructions of op k: one per SM, [a, b) ranges tiling [0, total) in SM order"""
        xs = sorted(by_op[k], key=lambda x: x["sm"])
        assert [x["sm"] for x in xs] == list(range(n_sm)), "one instruction per SM"
        pos = 0
        for x in xs:
            assert x["a"] == pos and x["b"] >= x["a"]
            pos = x["b"]
        assert pos == total

    d = cfg.d_model
    k = 0
    splits = []
    packed_groups = {}
    for k, o in enumerate(ops):
        t = o["type"]
        if t == EMBED:
            partition(k, d)
        elif t == GEMV:
            partition(k, o["rows"])
            assert 0 <= o["k_begin"] and o["k_begin"] + o["K"] <= o["ldw"]
            for x in by_op[k]:
                assert x["a"] == pk_split(o["rows"], n_sm, x["sm"]), "shares of whole 8-row units"
            if o["mma"] == 1:
                # mma.sync: up to 4 rows, hi / lo columns of whole atoms (and the residual slice) staged
                assert N <= 4 and o["k_begin"] == 64 * o["pa0"]
                xrows = max(x["b"] - x["a"] for x in by_op[k]) if o["out_kind"] == RESID else 0
                assert N * (64 * -(-o["K"] // 64) + 8 + xrows) * 4 <= 82176 - 32
            else:
                assert o["mma"] == 2 and o["ncols"] == -(-2 * N // 16) * 16
                assert o["k_begin"] == 0 and o["K"] == o["ldw"] and o["pa0"] == 0, "no K split on the tcgen05 path"
            assert o["patoms"] == -(-o["ldw"] // 64)
            walk_chunks(o, by_op[k], packed_groups)
            if o["k_begin"] > 0 or o["K"] < o["ldw"]:
                splits.append(k)
        elif t == ROPE:
            assert sorted(x["sm"] for x in by_op[k]) == list(range(n_sm))
        elif t == ATTN:
            seen = collections.Counter()
            for x in by_op[k]:
                lo, hi = x["c"] & 0xFF, x["c"] >> 8
                assert 0 <= lo < hi <= R and 0 <= x["b"] < o["nchunk"]
                for r in range(lo, hi):
                    seen[(x["a"], x["b"], r)] += 1
            assert set(seen.values()) == {1}
            assert len(seen) == B * o["n_kv_heads"] * o["nchunk"] * R
        elif t == MLA_ATTN:
            seen = collections.Counter()
            for x in by_op[k]:
                lo, hi = x["c"] & 0xFF, x["c"] >> 8
                assert 0 <= lo < hi <= R and hi - lo <= 2, "at most 2 rows per warp"
                for r in range(lo, hi):
                    seen[(x["a"], x["b"], r)] += 1
            assert set(seen.values()) == {1}
            assert len(seen) == B * (cfg.mla_heads // 8) * o["nchunk"] * R
            assert o["groups"] == 8 and o["n_kv_heads"] == cfg.mla_heads // 8
        elif t == COMBINE:
            heads = cfg.mla_heads if o["head_dim"] == 512 else cfg.n_q_heads
            got = sorted((x["a"], x["b"], x["c"]) for x in by_op[k])
            assert got == sorted((b, r, h) for b in range(B) for r in range(R) for h in range(heads))
        elif t == DELTA:
            ng = -(-cfg.lin_dv // o["col_group"])
            got = sorted((x["a"], x["b"], x["c"]) for x in by_op[k])
            assert got == sorted((b, h, j) for b in range(B) for h in range(cfg.lin_heads) for j in range(ng))
            assert o["col_group"] in (8, 16, 32, 64, 128)
        elif t == MLA_PREP:
            sms = sorted(x["sm"] for x in by_op[k])
            assert sms == list(range(len(sms))) and 8 * len(sms) >= 2 * N
        elif t == QABS:
            got = sorted((x["a"], x["b"]) for x in by_op[k])
            assert got == sorted((h, cb) for h in range(cfg.mla_heads) for cb in range(cfg.kv_lora // 128))
        elif t == UV:
            got = sorted((x["a"], x["b"]) for x in by_op[k])
            assert got == sorted((h, j) for h in range(cfg.mla_heads) for j in range(-(-cfg.v_head // 64)))
        elif t == ROUTE:
            assert len(by_op[k]) == 1
        elif t == MOE_UP:
            partition(k, cfg.expert_dim)
            assert o["rg"] == (16 if N <= 4 else 8)
        elif t == MOE_DOWN:
            partition(k, d)
            assert ops[k - 1]["type"] == MOE_UP and ops[k - 2]["type"] == ROUTE
    # a K-split residual GEMV: consecutive parts tile the input width
    groups = []
    for k in splits:
        if groups and groups[-1][-1] == k - 1 and ops[k]["ldw"] == ops[k - 1]["ldw"]:
            groups[-1].append(k)
        else:
            groups.append([k])
    for g in groups:
        assert all(ops[k]["out_kind"] == RESID for k in g)
        assert ops[g[0]]["k_begin"] == 0
        for a, b in zip(g, g[1:]):
            assert ops[b]["k_begin"] == ops[a]["k_begin"] + ops[a]["K"]
        assert ops[g[-1]]["k_begin"] + ops[g[-1]]["K"] == ops[g[-1]]["ldw"]
    # every GEMV weight group is read exactly once per step: its ops' chunks tile its packed copy
    assert packed_groups
    for g in packed_groups.values():
        pos = 0
        for off, nb in sorted(g["ranges"]):
            assert off == pos, "chunks of a packed group must not overlap or leave gaps"
            pos = off + nb
        assert pos == g["bytes"]
    # one LM head when asked for, none otherwise
    assert sum(o["type"] == GEMV and o["out_kind"] == LOGITS for o in ops) == (1 if head else 0)
    return ops, ins


@pytest.mark.parametrize("name,layers", [("tiny_dense", None), ("hybrid_gdn_gqa", 4), ("moe_kda_mla", 4),
                                         ("moe_nvfp4_gqa", 2)])
@pytest.mark.parametrize("B,R", [(1, 1), (2, 1), (4, 1), (8, 1), (1, 8), (2, 8), (8, 8)])
def test_program_coverage(name, layers, B, R):
    cfg = config(name, n_layers=layers)
    check_program(cfg, 152, B, R)


@pytest.mark.parametrize("n_sm", [7, 37, 148])
def test_program_coverage_other_sm_counts(n_sm):
    check_program(config("hybrid_gdn_gqa", n_layers=4), n_sm, 2, 8)
    check_program(config("moe_kda_mla", n_layers=4), n_sm, 3, 1)


def test_prefill_program_has_no_head():
    check_program(config("hybrid_gdn_gqa", n_layers=4), 152, 1, 8, head=False)


def test_layer_op_sequences():
    """The op kinds of one layer, in program order, for each mixer / FFN kind (batch 1, decode)."""
    cfg = dataclasses.replace(config("moe_kda_mla"), n_layers=2, mixers=("kda", "mla"))
    ops, _ = make_plan(cfg, 152, 1, 1)
    kinds = [o["type"] for o in ops]
    kda = [GEMV, DELTA, GEMV]
    mla = [GEMV, MLA_PREP, GEMV, QABS, MLA_ATTN, COMBINE, UV, GEMV]
    moe = [GEMV, ROUTE, MOE_UP, MOE_DOWN]
    assert kinds == [EMBED] + kda + moe + mla + moe + [GEMV, FINAL]
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    ops, _ = make_plan(cfg, 152, 1, 1)
    kinds = [o["type"] for o in ops]
    gdn = [GEMV, DELTA, GEMV, GEMV, GEMV]
    gqa = [GEMV, ROPE, ATTN, COMBINE, GEMV, GEMV, GEMV]
    assert kinds == [EMBED] + gdn * 3 + gqa + [GEMV, FINAL]


def test_staging_decisions():
    """Batch 1 to 4 of the d = 5120 stack take the mma.sync GEMV for every projection (4 rows of width 5120
    fit the staging area as hi/lo pairs); 8 rows (and 8-row verify) take the tcgen05 / TMEM GEMV."""
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    ops, _ = make_plan(cfg, 152, 1, 8)
    assert all(o["mma"] == 2 for o in ops if o["type"] == GEMV)
    for B, want in ((1, 1), (2, 1), (4, 1), (8, 2)):
        ops, _ = make_plan(cfg, 152, B, 1)
        gemvs = [o for o in ops if o["type"] == GEMV and o["K"] == cfg.d_model]
        assert gemvs and all(o["mma"] == want for o in gemvs), B
    # MoE up to 2 rows stages its inputs; 4 rows of width 7168 do not fit
    cfg = config("moe_kda_mla", n_layers=4)
    for B, want in ((1, 1), (2, 1), (4, 0)):
        ops, _ = make_plan(cfg, 152, B, 1)
        assert all(o["staged"] == want for o in ops if o["type"] in (MOE_UP, MOE_DOWN)), B


def test_plan_rejects_bad_shapes():
    cfg = config("moe_kda_mla", n_layers=4)
    with pytest.raises(binding.MKError):
        make_plan(cfg, 152, 9, 1)                       # batch above max_batch
    with pytest.raises(binding.MKError):
        make_plan(cfg, 152, 1, 9)                       # rows above max_rows
    with pytest.raises(binding.MKError):
        make_plan(dataclasses.replace(cfg, kv_lora=256), 152, 1, 1)   # latent width the kernel does not take
    with pytest.raises(binding.MKError):
        make_plan(dataclasses.replace(cfg, n_experts=300), 152, 1, 1)
    with pytest.raises(binding.MKError):
        make_plan(dataclasses.replace(cfg, top_k=17), 152, 1, 1)
    nv = config("moe_nvfp4_gqa", n_layers=2)
    with pytest.raises(binding.MKError):
        make_plan(dataclasses.replace(nv, expert_dim=2000), 152, 1, 1)  # NVFP4 rows need multiples of 256


def test_one_sm_residual_gemv_takes_tcgen05():
    """With one SM a residual GEMV's share is all 5120 rows: for 4 activation rows their slice of x no longer
    fits beside any K part of the staged inputs, so those GEMVs take the tcgen05 path (whose epilogue reads x
    from HBM), and the program still covers every row and reads every packed byte once."""
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    ops, _ = check_program(cfg, 1, 4, 1)
    resid = [o for o in ops if o["type"] == GEMV and o["out_kind"] == RESID]
    assert resid and all(o["mma"] == 2 for o in resid)
    check_program(cfg, 1, 2, 8)


def test_batch_above_eight_rows_per_call():
    """Concurrency above batch 8: a handle may hold up to 64 sequences; one call takes at most 64 rows, so 64
    single-row sequences run (every GEMV on the tcgen05 path, 128 TMEM columns per tile) and 16 sequences of
    8-row verify blocks are refused."""
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    ops, ins = make_plan(cfg, 152, 64, 1, max_batch=64)
    gemvs = [o for o in ops if o["type"] == GEMV]
    assert gemvs and all(o["mma"] == 2 and o["ncols"] == 128 for o in gemvs)
    ops, _ = make_plan(cfg, 152, 8, 8, max_batch=64)
    assert all(o["mma"] == 2 for o in ops if o["type"] == GEMV)
    with pytest.raises(binding.MKError):
        make_plan(cfg, 152, 16, 8, max_batch=64)
