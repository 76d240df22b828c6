"""GPU checks of the prepacked weight form (wna16_prepack, wna16_fused_moe_prepacked).

A stage image is byte-identical to the shared-memory stage the GEMM kernels
build from the plain layout. The only differences are bytes outside the
matrices, which only ever meet zero token values. So the layer on prepacked
weights must equal the layer on the plain weights bit for bit, in every
configuration, and through them the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, Workload, make_expert_weights, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def small(**kw):
    base = dict(name="pp", H=384, I=320, E=6, topk=2, bits=4, has_zeros=True, group_size=128,
                act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")
    base.update(kw)
    return Workload(**base)


def packed(li):
    wl = li.wl
    w13 = w.prepack(li.w13_q, li.w13_s, li.w13_z, wl.bits, wl.group_size, gate_up=True)
    w2 = w.prepack(li.w2_q, li.w2_s, li.w2_z, wl.bits, wl.group_size, gate_up=False)
    return w13, w2


def both(li, block, split_k=0):
    w13, w2 = packed(li)
    a = w.fused_moe_prepacked(li.hidden, w13, w2, li.topk_ids, li.topk_w, block=block, split_k=split_k)
    b = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    li.wl.bits, li.wl.group_size, block=block, split_k=split_k)
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("bits,zeros,G,act,sdt", [
    (4, True, 128, "f16", "f16"), (4, False, 128, "bf16", "bf16"), (4, True, 64, "f16", "f16"),
    (4, True, 256, "bf16", "f16"), (4, True, -1, "f16", "f16"), (8, False, -1, "bf16", "f16"),
    (8, True, 64, "f16", "bf16"), (8, False, 128, "f16", "f16")])
@pytest.mark.parametrize("block", [16, 32, 64, 128])
def test_prepacked_equals_plain(bits, zeros, G, act, sdt, block):
    # H = 384 and I = 320: ragged down-GEMM row tile (384 = 3 x 128 exact, but
    # the gate/up tiles of I = 320 end mid-stage) and a half-width last K stage
    # of the down GEMM when G permits
    H, I = (384, 320) if G in (64, -1) else (512, 256 * (2 if G == 256 else 1) + (0 if G == 256 else 128))
    wl = small(bits=bits, has_zeros=zeros, group_size=G, act_dtype=act, scale_dtype=sdt, H=H, I=I)
    li = make_layer_inputs(wl, 29).to(DEV)
    for split in ((0, 2) if block <= 32 else (0,)):
        a, b = both(li, block, split)
        assert torch.equal(a, b), (bits, zeros, G, act, block, split)


def test_prepacked_matches_oracle():
    wl = small(H=512, I=384, group_size=128)
    li = make_layer_inputs(wl, 21).to(DEV)
    w13, w2 = packed(li)
    y = w.fused_moe_prepacked(li.hidden, w13, w2, li.topk_ids, li.topk_w, block=16)
    torch.cuda.synchronize()
    ref = bits_to_f64(oracle.fused_moe_grouped(oracle_layer_dict(li)), "f16")
    assert max_rel_err(bits_to_f64(halfbits(y), "f16"), ref) <= 1e-2


def test_prepack_size_and_mixtral_decode_bit_exact():
    wl = WORKLOADS["mixtral8x7b"]
    weights = make_expert_weights(wl, DEV)
    li = make_layer_inputs(wl, 16, DEV, weights=weights)
    # G = 128 divides every stage: the packed form is exactly as large as the plain one
    plain13 = li.w13_q.numel() * 4 + li.w13_s.numel() * 2 + li.w13_z.numel() * 4
    assert w.load().wna16_prepack_bytes(wl.E, 2 * wl.I, wl.H, 4, 128, 1, 1) == plain13
    a, b = both(li, 0)
    assert torch.equal(a, b)
    del weights


def test_prepack_rejects_bad_shapes():
    L = w.load()
    assert L.wna16_prepack_bytes(8, 100, 4096, 4, 128, 1, 0) == 0   # N not a multiple of 64
    assert L.wna16_prepack_bytes(8, 4096, 4096, 4, 96, 1, 0) == 0   # G neither 64 nor a multiple of 128
    assert L.wna16_prepack_bytes(8, 4096, 4096, 3, 128, 1, 0) == 0  # bits
