"""CPU checks of the C-ABI library: it loads, exports every declared symbol, and
its host-only logic (capacity bound, block choice, argument validation) is
right. No compute call is made here (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import weight_quantized_moe_align_gb300 as w

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wna16_moe.h")


@pytest.fixture(scope="module")
def lib():
    w.build()
    return w.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wna16_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(w.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_capacity_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for _ in range(500):
        P = int(rng.integers(0, 20000))
        E = int(rng.integers(1, 257))
        B = int(rng.choice([16, 32, 64, 128, 256]))
        assert w.align_capacity(P, E, B) == oracle.align_capacity(P, E, B)
    assert lib.wna16_align_capacity(-1, 8, 16) == -1


def test_block_choice(lib):
    for M, k, E in [(1, 8, 256), (4, 2, 8), (1024, 8, 256), (1024, 2, 8), (8192, 2, 8), (512, 8, 64)]:
        b = w.choose_block(M, k, E)
        assert b in (16, 32, 64, 128, 256)
    assert w.choose_block(1, 8, 256) == 16  # decode: one pair per expert
    assert w.choose_block(8192, 2, 8) == 128


def test_status_strings(lib):
    for code in range(8):
        assert lib.wna16_status_string(code)


def _call_fused(lib, **over):
    args = dict(hidden=16, act=0, M=4, H=256, I=512, E=8, topk=2, w13_q=16, w13_s=16, w13_z=None,
                w2_q=16, w2_s=16, w2_z=None, sdt=0, bits=4, G=128, ids=16, tw=16, out=16, ws=16,
                ws_bytes=1 << 30, block=0, split=0, stream=None)
    args.update(over)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.wna16_fused_moe(v(args["hidden"]), args["act"], args["M"], args["H"], args["I"], args["E"],
                               args["topk"], v(args["w13_q"]), v(args["w13_s"]), v(args["w13_z"]),
                               v(args["w2_q"]), v(args["w2_s"]), v(args["w2_z"]), args["sdt"], args["bits"],
                               args["G"], v(args["ids"]), v(args["tw"]), v(args["out"]), v(args["ws"]),
                               args["ws_bytes"], args["block"], args["split"], args["stream"])


def test_fused_argument_errors_are_host_side(lib):
    # each of these returns before anything would touch a device
    assert _call_fused(lib, M=0) == 0  # empty batch: OK, nothing launched
    assert _call_fused(lib, hidden=None) == 1
    assert _call_fused(lib, hidden=8) == 1  # misaligned
    assert _call_fused(lib, bits=3) == 2
    assert _call_fused(lib, H=200) == 2
    assert _call_fused(lib, I=96) == 2
    assert _call_fused(lib, G=96) == 2
    assert _call_fused(lib, G=0) == 1
    assert _call_fused(lib, E=300) == 2
    assert _call_fused(lib, topk=9) == 2
    assert _call_fused(lib, block=48) == 1
    assert _call_fused(lib, block=512) == 1
    assert _call_fused(lib, split=9) == 1
    assert _call_fused(lib, split=-1) == 1
    assert _call_fused(lib, act=2) == 1  # fp32 is for router logits only
    assert _call_fused(lib, w13_z=16) == 1  # zeros for one projection only
    assert _call_fused(lib, act=5) == 1
    assert _call_fused(lib, ws_bytes=16) == 3


def test_workspace_bytes_cover_the_layout(lib):
    n = w.workspace_bytes(1024, 7168, 2048, 256, 8, 4, 128)
    P = 1024 * 8
    B = w.choose_block(1024, 8, 256)
    cap = oracle.align_capacity(P, 256, B)
    assert n >= cap * 4 + cap * 2048 * 2 + P * 7168 * 4
    assert lib.wna16_fused_moe_workspace_bytes(4, 256, 512, 8, 2, 3, 128, 0, 0) == 0


def _call_routing(lib, **over):
    a = dict(logits=16, dt=2, M=4, E=256, k=8, scoring=1, renorm=1, ng=8, tg=4, ids=16, w=16)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.wna16_topk_routing(vp(a["logits"]) if a["logits"] else None, a["dt"], a["M"], a["E"], a["k"],
                                  a["scoring"], a["renorm"], a["ng"], a["tg"],
                                  vp(a["ids"]) if a["ids"] else None, vp(a["w"]) if a["w"] else None, None)


def test_routing_argument_errors_are_host_side(lib):
    assert _call_routing(lib, M=0) == 0  # nothing launched
    assert _call_routing(lib, logits=None) == 1
    assert _call_routing(lib, logits=18) == 1  # fp32 logits need 4-byte alignment
    assert _call_routing(lib, ids=None) == 1
    assert _call_routing(lib, E=257) == 1
    assert _call_routing(lib, k=33) == 1
    assert _call_routing(lib, E=4, k=5, ng=1) == 1  # topk > E
    assert _call_routing(lib, ng=7) == 1  # groups must divide E
    assert _call_routing(lib, ng=64, E=256) == 1  # at most 32 groups
    assert _call_routing(lib, ng=4, E=4, k=1, tg=1) == 1  # groups of one expert
    assert _call_routing(lib, tg=9) == 1
    assert _call_routing(lib, tg=0) == 1
    assert _call_routing(lib, k=9, E=32, ng=8, tg=2) == 1  # only 8 experts kept
    assert _call_routing(lib, scoring=2) == 1
    assert _call_routing(lib, dt=3) == 1



class _Opt(ctypes.Structure):
    _fields_ = [("w13_bias", ctypes.c_void_p), ("w2_bias", ctypes.c_void_p), ("activation", ctypes.c_int),
                ("swiglu_alpha", ctypes.c_float), ("swiglu_beta", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("w13_perm", ctypes.c_void_p), ("w2_inv_perm", ctypes.c_void_p),
                ("router_logits", ctypes.c_void_p), ("logits_dtype", ctypes.c_int), ("scoring", ctypes.c_int),
                ("renormalize", ctypes.c_int), ("n_groups", ctypes.c_int), ("topk_groups", ctypes.c_int),
                ("routed_ids", ctypes.c_void_p), ("routed_weights", ctypes.c_void_p)]


def _call_fused_ex(lib, opt):
    v = ctypes.c_void_p
    return lib.wna16_fused_moe_ex(v(16), 0, 4, 256, 512, 8, 2, v(16), v(16), None, v(16), v(16), None, 0, 4, 128,
                                  v(16), v(16), v(16), v(16), 1 << 30, 0, 0, None, None, ctypes.byref(opt))


def test_options_errors_are_host_side(lib):
    nan = float("nan")
    assert _call_fused_ex(lib, _Opt(None, None, 2, 1.0, 0.0, 0.0)) == 1  # unknown activation
    assert _call_fused_ex(lib, _Opt(17, None, 0, 1.0, 0.0, 0.0)) == 1  # misaligned bias
    assert _call_fused_ex(lib, _Opt(None, 33, 0, 1.0, 0.0, 0.0)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 1, nan, 1.0, 7.0)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 1, 1.7, float("inf"), 7.0)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 1, 1.7, 1.0, nan)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 0, 1.0, 0.0, 0.0, 18, None)) == 1  # misaligned permutation
    assert _call_fused_ex(lib, _Opt(None, None, 0, 1.0, 0.0, 0.0, None, 34)) == 1
    # routing from logits: output buffers required; bad routing arguments before any launch
    assert _call_fused_ex(lib, _Opt(None, None, 0, 1.0, 0.0, 0.0, None, None, 16, 2, 0, 1, 1, 1, None, 16)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 0, 1.0, 0.0, 0.0, None, None, 16, 2, 5, 1, 1, 1, 16, 16)) == 1
    assert _call_fused_ex(lib, _Opt(None, None, 0, 1.0, 0.0, 0.0, None, None, 16, 2, 0, 1, 3, 1, 16, 16)) == 1
    v = ctypes.c_void_p
    # M = 0 with valid options: OK, nothing launched
    assert lib.wna16_fused_moe_ex(v(16), 0, 0, 256, 512, 8, 2, v(16), v(16), None, v(16), v(16), None, 0, 4, 128,
                                  v(16), v(16), v(16), v(16), 1 << 30, 0, 0, None, None,
                                  ctypes.byref(_Opt(16, 16, 1, 1.7, 1.0, 7.0))) == 0


def test_act_order_prepare_errors_are_host_side(lib):
    v = ctypes.c_void_p
    defaults = (("q", v(16)), ("g", v(16)), ("E", 4), ("N", 256), ("K", 512), ("bits", 4), ("G", 128),
                ("qo", v(16)), ("perm", v(16)), ("inv", None), ("st", v(16)))
    call = lambda **o: lib.wna16_act_order_prepare(*[o.get(k, d) for k, d in defaults], None)
    assert call(G=0) == 1
    assert call(G=-1) == 1  # one group per channel has no order to restore
    assert call(G=96) == 2  # K % G != 0
    assert call(bits=3) == 1
    assert call(q=None) == 1  # q and q_out go together
    assert call(q=None, qo=None, perm=None) == 1
    assert call(st=None) == 1
    assert call(perm=v(18)) == 1


def test_convert_checkpoint_errors_are_host_side(lib):
    v = ctypes.c_void_p
    defaults = (("fmt", 0), ("q", v(16)), ("z", v(16)), ("E", 4), ("N", 256), ("K", 512), ("bits", 4), ("G", 128),
                ("qo", v(16)), ("zo", v(16)))
    call = lambda **o: lib.wna16_convert_checkpoint(*[o.get(k, d) for k, d in defaults], None)
    assert call(fmt=3) == 1
    assert call(fmt=2, bits=8) == 2  # AWQ is 4-bit
    assert call(G=0) == 1
    assert call(G=96) == 2
    assert call(N=4) == 2  # N must hold whole zero-point words
    assert call(q=None) == 1
    assert call(zo=None) == 1  # zeros in, no zeros out
    assert call(z=None, zo=None, E=0) == 1
    assert call(qo=v(18)) == 1


def test_large_tiles_refused_for_many_experts(lib):
    # more than 16 experts: 128/256-token tiles are refused (workspace size 0,
    # the fused call answers unsupported); 64 is accepted, and so are large
    # tiles for 16 experts or fewer
    assert lib.wna16_fused_moe_workspace_bytes(256, 7168, 2048, 256, 8, 4, 128, 128, 0) == 0
    assert lib.wna16_fused_moe_workspace_bytes(128, 3584, 2560, 64, 8, 4, 128, 256, 0) == 0
    assert lib.wna16_fused_moe_workspace_bytes(256, 7168, 2048, 256, 8, 4, 128, 64, 0) > 0
    assert lib.wna16_fused_moe_workspace_bytes(256, 4096, 14336, 16, 2, 4, 128, 128, 0) > 0
    p = ctypes.c_void_p(256)
    st = lib.wna16_fused_moe(p, 0, 256, 7168, 2048, 256, 8, p, p, p, p, p, p, 0, 4, 128, p, p, p, p,
                             1 << 40, 128, 0, None)
    assert st == 2  # WNA16_ERR_UNSUPPORTED, before any launch
