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
    for code in range(7):
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
