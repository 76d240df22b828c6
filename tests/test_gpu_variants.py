"""GPU parity of the model-variant options (wna16_fused_moe_ex): per-expert
biases of both projections and the clamped SwiGLU, on both GEMM kernels, with
K splits and on prepacked weights, against the float64 oracle (max relative
error 1e-2)."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import Workload, make_biases, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def small(**kw):
    base = dict(name="variants", H=384, I=256, E=6, topk=2, bits=4, has_zeros=True, group_size=128,
                act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")
    base.update(kw)
    return Workload(**base)


def check(li, b13=None, b2=None, glu=None, block=0, split_k=0, packed=False):
    kw = dict(w13_bias=b13, w2_bias=b2)
    if glu is not None:
        kw.update(activation="swiglu_clamp", swiglu=glu)
    wl = li.wl
    if packed:
        p13 = w.prepack(li.w13_q, li.w13_s, li.w13_z, wl.bits, wl.group_size, gate_up=True)
        p2 = w.prepack(li.w2_q, li.w2_s, li.w2_z, wl.bits, wl.group_size, gate_up=False)
        y = w.fused_moe_prepacked(li.hidden, p13, p2, li.topk_ids, li.topk_w, block=block, split_k=split_k, **kw)
    else:
        y = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids,
                        li.topk_w, wl.bits, wl.group_size, block=block, split_k=split_k, **kw)
    torch.cuda.synchronize()
    L = oracle_layer_dict(li)
    if b13 is not None:
        L["w13_b"] = halfbits(b13)
    if b2 is not None:
        L["w2_b"] = halfbits(b2)
    L["glu"] = glu
    ref = oracle.fused_moe_grouped(L)
    r, g = bits_to_f64(ref, wl.act_dtype), bits_to_f64(halfbits(y), wl.act_dtype)
    assert np.all(np.isfinite(g))
    err = max_rel_err(g, r)
    assert err <= TOL, (err, block, split_k, glu)
    return y


# deferred-scale kernel (16/32-token tiles, G = 128 / per-channel) and the
# general kernel (G = 64, 64+ token tiles, int8 with bf16)
FORMATS = [
    (dict(), 16),
    (dict(act_dtype="bf16", scale_dtype="bf16", has_zeros=False), 16),
    (dict(), 32),
    (dict(group_size=64), 16),
    (dict(), 64),
    (dict(bits=8, has_zeros=False, group_size=-1, act_dtype="bf16", scale_dtype="f16"), 32),
    (dict(bits=8, has_zeros=False, group_size=-1), 16),
]
VARIANTS = [
    dict(bias=True, glu=None),
    dict(bias=False, glu=(1.702, 1.0, 7.0)),
    # a limit inside the range of the gate/up values: the clamp is active
    dict(bias=True, glu=(1.702, 1.0, 0.04)),
    dict(bias=True, glu=(1.0, 0.0, 0.0)),  # no clamp, reduces to silu(g) * u
]


@pytest.mark.parametrize("variant", VARIANTS, ids=["bias", "swiglu", "bias+clamped", "bias+plain"])
@pytest.mark.parametrize("fmt,block", FORMATS, ids=[f"{i}" for i in range(len(FORMATS))])
def test_variants(fmt, block, variant):
    wl = small(**fmt)
    li = make_layer_inputs(wl, 37).to(DEV)
    b13 = b2 = None
    if variant["bias"]:
        b13, b2 = make_biases(wl, 5, DEV)
    check(li, b13, b2, variant["glu"], block=block)


@pytest.mark.parametrize("block", [16, 64])
def test_down_bias_added_once_across_k_splits(block):
    wl = small(I=640)
    li = make_layer_inputs(wl, 20).to(DEV)
    b13, b2 = make_biases(wl, 6, DEV, std=0.2)
    for split in (2, 3):
        check(li, b13, b2, (1.702, 1.0, 0.05), block=block, split_k=split)


def test_bias_only_down_projection_and_gate_up_only():
    wl = small()
    li = make_layer_inputs(wl, 9).to(DEV)
    b13, b2 = make_biases(wl, 7, DEV)
    check(li, b13, None, block=16)
    check(li, None, b2, block=16)


@pytest.mark.parametrize("block", [16, 64])
def test_variants_on_prepacked_weights(block):
    wl = small()
    li = make_layer_inputs(wl, 29).to(DEV)
    b13, b2 = make_biases(wl, 8, DEV)
    y_plain = check(li, b13, b2, (1.702, 1.0, 0.04), block=block)
    y_pack = check(li, b13, b2, (1.702, 1.0, 0.04), block=block, packed=True)
    assert torch.equal(y_plain, y_pack)


def test_default_options_match_the_plain_call():
    wl = small()
    li = make_layer_inputs(wl, 11).to(DEV)
    zero13 = torch.zeros(wl.E, 2 * wl.I, dtype=li.hidden.dtype, device=DEV)
    zero2 = torch.zeros(wl.E, wl.H, dtype=li.hidden.dtype, device=DEV)
    base = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                       wl.bits, wl.group_size, block=16).clone()
    # zero biases through the options entry point: same bits
    y = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    wl.bits, wl.group_size, block=16, w13_bias=zero13, w2_bias=zero2)
    torch.cuda.synchronize()
    assert torch.equal(base, y)


def test_bad_bias_shape_is_rejected():
    wl = small()
    li = make_layer_inputs(wl, 3).to(DEV)
    with pytest.raises(ValueError):
        w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    wl.bits, wl.group_size, w13_bias=torch.zeros(wl.E, wl.I, dtype=li.hidden.dtype, device=DEV))
    with pytest.raises(ValueError):
        w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    wl.bits, wl.group_size, activation="gelu")
