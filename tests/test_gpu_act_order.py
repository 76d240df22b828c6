"""GPU parity of act-order (GPTQ desc_act) weights: wna16_act_order_prepare's
permutations and repacked codes bit-exact against the oracle, and the layer on
repacked weights with the permutations against the oracle's direct g_idx
dequantization (max relative error 1e-2)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import Workload, make_g_idx, make_layer_inputs, pack_along_last, quantize_expert_act_order
from tests.helpers import bits_to_f64, halfbits, max_rel_err, np_i32, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def small(**kw):
    base = dict(name="actorder", H=512, I=384, E=5, topk=2, bits=4, has_zeros=True, group_size=128,
                act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")
    base.update(kw)
    return Workload(**base)


def act_order_inputs(wl, M, seed, order13=True, order2=True):
    """Layer inputs whose experts are quantized with act-order groups; returns
    (inputs, g_idx13 [E, H], g_idx2 [E, I]) (plain k // G where not ordered)."""
    li = make_layer_inputs(wl, M, seed=seed)
    gen = torch.Generator().manual_seed(seed)
    out, gidx = {}, {}
    for name, (N, K), on in (("w13", (2 * wl.I, wl.H), order13), ("w2", (wl.H, wl.I), order2)):
        qs, ss, zs, gs = [], [], [], []
        for e in range(wl.E):
            wt = torch.randn(N, K, generator=gen) * 0.02
            g = make_g_idx(K, wl.group_size, 1000 * seed + 10 * e + len(name)) if on else \
                torch.arange(K) // wl.group_size
            codes, s, z = quantize_expert_act_order(wt, wl.bits, wl.has_zeros, wl.group_size, wl.scale_dtype, g)
            qs.append(pack_along_last(codes, wl.bits))
            ss.append(s)
            zs.append(None if z is None else pack_along_last(z, wl.bits))
            gs.append(g.to(torch.int32))
        out[name] = (torch.stack(qs), torch.stack(ss), None if zs[0] is None else torch.stack(zs))
        gidx[name] = torch.stack(gs)
    li = dataclasses.replace(li, w13_q=out["w13"][0], w13_s=out["w13"][1], w13_z=out["w13"][2],
                             w2_q=out["w2"][0], w2_s=out["w2"][1], w2_z=out["w2"][2])
    return li.to(DEV), gidx["w13"], gidx["w2"]


@pytest.mark.parametrize("bits", [4, 8])
def test_prepare_is_the_oracle_permutation(bits):
    E, N, K, G = 3, 64, 1024, 128
    g = torch.stack([make_g_idx(K, G, 40 + e) for e in range(E)]).to(torch.int32)
    q = torch.randint(-2 ** 31, 2 ** 31 - 1, (E, N, K * bits // 32), dtype=torch.int64).to(torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_out, perm, inv = w.act_order_prepare(q.to(DEV), g.to(DEV), bits, G, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for e in range(E):
        p, i = oracle.act_order_permutation(g[e].numpy())
        assert np.array_equal(perm[e].cpu().numpy(), p)
        assert np.array_equal(inv[e].cpu().numpy(), i)
        u = oracle.unpack_codes(np_i32(q[e]), bits)
        u_out = oracle.unpack_codes(np_i32(q_out[e]), bits)
        assert np.array_equal(u_out, u[:, p])


def test_bad_groups_are_flagged_and_outputs_stay_in_range():
    E, N, K, G = 2, 16, 512, 128
    g = torch.stack([make_g_idx(K, G, 7), make_g_idx(K, G, 8)]).to(torch.int32)
    g[1, :10] = 0  # group 0 of expert 1 now holds more than G columns
    q = torch.zeros(E, N, K // 8, dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_out, perm, inv = w.act_order_prepare(q.to(DEV), g.to(DEV), 4, G, status=status)
    assert w.read_device_status(status) & w.DEV_BAD_GROUPS
    for t in (perm, inv):
        v = t.cpu().numpy()
        assert v.min() >= 0 and v.max() < K
    # expert 0 is valid and unaffected
    p, _ = oracle.act_order_permutation(g[0].numpy())
    assert np.array_equal(perm[0].cpu().numpy(), p)


def run(li, g13, g2, block=0, order13=True, order2=True, packed=False, **kw):
    wl = li.wl
    q13, perm13, _ = w.act_order_prepare(li.w13_q, g13.to(DEV), wl.bits, wl.group_size)
    q2, _, inv2 = w.act_order_prepare(li.w2_q, g2.to(DEV), wl.bits, wl.group_size)
    opts = dict(w13_perm=perm13 if order13 else None, w2_inv_perm=inv2 if order2 else None)
    if not order13:
        q13 = li.w13_q
    if not order2:
        q2 = li.w2_q
    if packed:
        p13 = w.prepack(q13, li.w13_s, li.w13_z, wl.bits, wl.group_size, gate_up=True)
        p2 = w.prepack(q2, li.w2_s, li.w2_z, wl.bits, wl.group_size, gate_up=False)
        y = w.fused_moe_prepacked(li.hidden, p13, p2, li.topk_ids, li.topk_w, block=block, **opts, **kw)
    else:
        y = w.fused_moe(li.hidden, q13, li.w13_s, li.w13_z, q2, li.w2_s, li.w2_z, li.topk_ids, li.topk_w, wl.bits,
                        wl.group_size, block=block, **opts, **kw)
    torch.cuda.synchronize()
    L = oracle_layer_dict(li)
    L["w13_g_idx"] = g13.numpy()
    L["w2_g_idx"] = g2.numpy()
    return y, L


def check(y, L, dt):
    ref = oracle.fused_moe_grouped(L)
    r, g = bits_to_f64(ref, dt), bits_to_f64(halfbits(y), dt)
    assert np.all(np.isfinite(g))
    err = max_rel_err(g, r)
    assert err <= TOL, err
    return err


FORMATS = [
    dict(),
    dict(act_dtype="bf16", scale_dtype="bf16", has_zeros=False),
    dict(bits=8, has_zeros=False),
    dict(group_size=64),
]


@pytest.mark.parametrize("block", [16, 64])
@pytest.mark.parametrize("fmt", FORMATS, ids=["int4-f16", "int4sym-bf16", "int8", "g64"])
def test_layer(fmt, block):
    wl = small(**fmt)
    li, g13, g2 = act_order_inputs(wl, 37, 3)
    y, L = run(li, g13, g2, block=block)
    check(y, L, wl.act_dtype)


@pytest.mark.parametrize("order13,order2", [(True, False), (False, True)])
def test_one_projection_in_act_order(order13, order2):
    wl = small()
    li, g13, g2 = act_order_inputs(wl, 20, 4, order13, order2)
    y, L = run(li, g13, g2, block=16, order13=order13, order2=order2)
    check(y, L, wl.act_dtype)


def test_act_order_with_biases_swiglu_and_prepacked_weights():
    wl = small()
    li, g13, g2 = act_order_inputs(wl, 29, 5)
    b13 = (torch.randn(wl.E, 2 * wl.I, generator=torch.Generator().manual_seed(1)) * 0.05).half().to(DEV)
    b2 = (torch.randn(wl.E, wl.H, generator=torch.Generator().manual_seed(2)) * 0.05).half().to(DEV)
    kw = dict(w13_bias=b13, w2_bias=b2, activation="swiglu_clamp", swiglu=(1.702, 1.0, 0.05))
    y1, L = run(li, g13, g2, block=32, **kw)
    y2, _ = run(li, g13, g2, block=32, packed=True, **kw)
    L.update(w13_b=halfbits(b13), w2_b=halfbits(b2), glu=(1.702, 1.0, 0.05))
    check(y1, L, wl.act_dtype)
    assert torch.equal(y1, y2)


def test_identity_groups_match_the_plain_layer():
    # g_idx = k // G: prepare is the identity and the act-order path (general
    # kernel, permuted gather and epilogue) gives the plain result
    wl = small()
    li, g13, g2 = act_order_inputs(wl, 16, 6, False, False)
    y_ord, L = run(li, g13, g2, block=64)
    y_plain = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids,
                          li.topk_w, wl.bits, wl.group_size, block=64)
    torch.cuda.synchronize()
    assert torch.equal(y_ord, y_plain)
