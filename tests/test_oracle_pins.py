"""Pins of the float64 oracle against facts that do not come from the oracle.

The pages print no tensors and no worked example, so the oracle is pinned by
closed forms of its own definitions, by the quantizer's round-trip bound
(|dequant - w| <= scale/2, the bound the weight-only quantization recipe gives),
by brute force on tiny inputs and by invariants of the layer. Each group of
checks below is chosen so that a plausible slip (a wrong shift, a transposed
scale, a dropped zero point, a swapped gate/up half, a wrong slot order) fails.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import Workload, pack_along_last, quantize_expert
from tests.helpers import halfbits

# ----------------------------------------------------------------------------
# T1: packed-code layout (LSB first along the packed axis)
# ----------------------------------------------------------------------------


def test_unpack_literal_words_int4():
    # Layout rule: code of element i sits in bits [4*(i%8), 4*(i%8)+4).
    words = np.array([[0x76543210, np.int32(np.uint32(0xFEDCBA98).view(np.int32))]],
                     dtype=np.int32)
    assert oracle.unpack_codes(words, 4).tolist() == [list(range(16))]


def test_unpack_literal_words_int8():
    words = np.array([0x03020100, np.uint32(0xFFFEFDFC).view(np.int32)], dtype=np.int32)
    assert oracle.unpack_codes(words, 8).tolist() == [0, 1, 2, 3, 252, 253, 254, 255]


@pytest.mark.parametrize("bits", [4, 8])
def test_unpack_every_code_at_every_position(bits):
    pf = 32 // bits
    for pos, code in itertools.product(range(pf), range(1 << bits)):
        word = np.uint32(code << (bits * pos)).view(np.int32)
        out = oracle.unpack_codes(np.array([word], dtype=np.int32), bits)
        expect = [0] * pf
        expect[pos] = code
        assert out.tolist() == expect


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_round_trip(bits):
    g = torch.Generator().manual_seed(7)
    codes = torch.randint(0, 1 << bits, (5, 3, 64), generator=g)
    words = pack_along_last(codes, bits).numpy()
    assert words.shape == (5, 3, 64 * bits // 32)
    assert np.array_equal(oracle.unpack_codes(words, bits), codes.numpy())


# ----------------------------------------------------------------------------
# T2: quantize -> dequantize round trip is within half a quantization step
# ----------------------------------------------------------------------------

CASES = [  # (bits, has_zeros, G, scale dtype)
    (4, True, 128, "f16"), (4, True, 64, "f16"), (4, True, 256, "bf16"),
    (4, False, 128, "bf16"), (4, False, 128, "f16"), (4, True, -1, "f16"),
    (8, False, -1, "f16"), (8, False, 128, "bf16"), (8, True, 64, "f16"),
]


@pytest.mark.parametrize("bits,has_zeros,G,sdt", CASES)
def test_round_trip_within_half_step(bits, has_zeros, G, sdt):
    N, K = 48, 512
    g = torch.Generator().manual_seed(bits * 100 + G)
    w = torch.randn(N, K, generator=g) * 0.02
    Gk = K if G == -1 else G
    codes, scales, zeros = quantize_expert(w, bits, has_zeros, Gk, sdt)
    q = pack_along_last(codes, bits).numpy()
    zw = None if zeros is None else pack_along_last(zeros, bits).numpy()
    W = oracle.dequantize_expert(q, halfbits(scales), zw, bits, G, sdt)
    s = oracle.halfbits_to_f64(halfbits(scales), sdt)  # [K/G, N]
    step = s.T[:, np.arange(K) // Gk]  # scale of each element's own group
    err = np.abs(W - w.double().numpy())
    assert np.all(err <= step / 2 * (1 + 1e-6)), float(np.max(err / step))
    # and the error is not trivially small: the codes really are coarse
    assert np.max(err / step) > 0.3


def test_dequant_codes_equal_zero_points_is_zero():
    N, K, G, bits = 16, 256, 128, 4
    z = torch.randint(0, 16, (K // G, N), generator=torch.Generator().manual_seed(3))
    codes = z.t()[:, torch.arange(K) // G]  # every code equals its zero point
    s = torch.rand(K // G, N, generator=torch.Generator().manual_seed(4)).half() + 0.5
    W = oracle.dequantize_expert(pack_along_last(codes, bits).numpy(), halfbits(s),
                                 pack_along_last(z, bits).numpy(), bits, G, "f16")
    assert np.all(W == 0.0)


def test_dequant_symmetric_zero_point_is_half_range():
    # no zeros tensor: int4 zero point 8, int8 zero point 128
    for bits, zp in ((4, 8), (8, 128)):
        codes = torch.full((8, 64), zp + 3)
        s = torch.full((1, 8), 0.25, dtype=torch.float16)
        W = oracle.dequantize_expert(pack_along_last(codes, bits).numpy(), halfbits(s),
                                     None, bits, -1, "f16")
        assert np.all(W == 0.75)


def test_dequant_group_index_boundaries():
    # scale of group g applies exactly to k in [g*G, (g+1)*G)
    N, K, G, bits = 8, 256, 64, 4
    codes = torch.full((N, K), 9)  # 9 - 8 = 1 with the symmetric zero point
    s = torch.tensor([[1.0], [2.0], [4.0], [8.0]]).repeat(1, N).half()  # [K/G, N]
    W = oracle.dequantize_expert(pack_along_last(codes, bits).numpy(), halfbits(s),
                                 None, bits, G, "f16")
    expect = np.repeat([1.0, 2.0, 4.0, 8.0], G)
    assert np.array_equal(W, np.tile(expect, (N, 1)))


# ----------------------------------------------------------------------------
# rounding to the output dtype (round-to-nearest-even, single rounding)
# ----------------------------------------------------------------------------


def _bf16_value(b):
    return oracle.halfbits_to_f64(np.array([b], dtype=np.uint16), "bf16")[0]


def test_bf16_rounding_closed_forms():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    r = lambda v: _bf16_value(oracle.round_to_halfbits(np.array([v]), "bf16")[0])
    assert r(one + ulp / 2) == one  # tie -> even (1.0)
    assert r(one + 3 * ulp / 2) == one + 2 * ulp  # tie -> even
    assert r(one + ulp / 2 + 2.0 ** -40) == one + ulp  # above the tie
    assert r(-(one + ulp / 2 + 2.0 ** -40)) == -(one + ulp)
    assert r(3.0e-41) == 2.0 ** -133 * round(3.0e-41 / 2.0 ** -133)  # subnormal
    assert np.isinf(r(3.5e38))
    assert r(0.0) == 0.0


def test_f16_rounding_closed_forms():
    r = lambda v: float(oracle.round_to_halfbits(np.array([v]), "f16").view(np.float16)[0])
    ulp = 2.0 ** -10
    assert r(1 + ulp / 2) == 1.0
    assert r(1 + 3 * ulp / 2) == 1 + 2 * ulp
    assert r(1 + ulp / 2 + 2.0 ** -30) == 1 + ulp


# ----------------------------------------------------------------------------
# T3: moe_align_block_size against brute force and its invariants
# ----------------------------------------------------------------------------


def brute_align(ids, E, B):
    """Sort valid pairs by (expert, pair index); pad each expert to a multiple of B."""
    P = len(ids)
    order = sorted((p for p in range(P) if 0 <= ids[p] < E), key=lambda p: (ids[p], p))
    slots, blocks = [], []
    for e in range(E):
        mine = [p for p in order if ids[p] == e]
        if not mine:
            continue
        n = -(-len(mine) // B) * B
        slots += mine + [P] * (n - len(mine))
        blocks += [e] * (n // B)
    return slots, blocks


def check_align(ids, E, B):
    ids = np.asarray(ids, dtype=np.int32)
    sorted_ids, expert_ids, npp, counts = oracle.moe_align_block_size(ids, E, B)
    ids = ids.reshape(-1)
    P = ids.size
    slots, blocks = brute_align(ids.tolist(), E, B)
    cap = sorted_ids.size
    assert cap % B == 0 and expert_ids.size == cap // B
    assert cap >= len(slots)
    assert npp == len(slots)
    assert sorted_ids[:npp].tolist() == slots
    assert np.all(sorted_ids[npp:] == P)
    assert expert_ids[: npp // B].tolist() == blocks
    assert np.all(expert_ids[npp // B:] == -1)
    # invariants: a permutation of the valid pairs plus sentinel padding only
    valid = sorted(p for p in range(P) if 0 <= ids[p] < E)
    assert sorted(int(v) for v in sorted_ids if v != P) == valid
    for e in range(E):
        assert counts[e] == int(np.sum(ids == e))
    assert npp == sum(-(-int(c) // B) * B for c in counts)


@pytest.mark.parametrize("seed", range(20))
def test_align_random_vs_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.choice([1, 2, 7, 8, 64, 256]))
    M = int(rng.integers(0, 70))
    k = int(rng.integers(1, min(E, 8) + 1))
    B = int(rng.choice([16, 32, 64, 128]))
    ids = rng.integers(0, E, size=(M, k))
    check_align(ids, E, B)


def test_align_special_cases():
    check_align([[3]], 256, 16)  # one pair, 256 experts
    check_align(np.zeros((40, 1)), 8, 16)  # every pair on one expert
    check_align(np.full((5, 2), 7), 8, 64)  # only the last expert used
    check_align(np.zeros((0, 2)), 8, 16)  # no tokens
    check_align([[0, 0], [0, 0]], 4, 16)  # duplicate ids inside a token
    check_align([[1, 9], [-1, 2], [3, 1]], 8, 16)  # out-of-range ids are dropped


def test_align_capacity_closed_form():
    # decode: one token, top-8 of 256 experts, block 16 -> 8 blocks at most
    assert oracle.align_capacity(8, 256, 16) == 128
    assert oracle.align_capacity(2, 8, 16) == 32
    assert oracle.align_capacity(8192, 256, 16) == 8192 + 256 * 15 + 0 - (8192 + 256 * 15) % 16 + (
        16 if (8192 + 256 * 15) % 16 else 0)
    # the bound is tight: every expert one pair over a block multiple
    E, B = 5, 16
    ids = np.repeat(np.arange(E), B + 1)
    _, _, npp, _ = oracle.moe_align_block_size(ids, E, B)
    assert npp == E * 2 * B <= oracle.align_capacity(ids.size, E, B)


# ----------------------------------------------------------------------------
# T4: the layer
# ----------------------------------------------------------------------------


def _small_layer(M=3, H=64, I=32, E=4, k=2, bits=4, has_zeros=True, G=32,
                 act="f16", sdt="f16", seed=0):
    g = torch.Generator().manual_seed(seed)
    L = dict(act_dtype=act, scale_dtype=sdt, bits=bits, group_size=G)
    x = (torch.randn(M, H, generator=g) * 0.5).to(torch.float16 if act == "f16" else torch.bfloat16)
    L["x"] = halfbits(x)
    for name, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
        qs, ss, zs = [], [], []
        for e in range(E):
            w = torch.randn(N, K, generator=g) * 0.1
            c, s, z = quantize_expert(w, bits, has_zeros, K if G == -1 else G, sdt)
            qs.append(pack_along_last(c, bits))
            ss.append(halfbits(s))
            zs.append(None if z is None else pack_along_last(z, bits).numpy())
        L[name + "_q"] = torch.stack(qs).numpy()
        L[name + "_s"] = np.stack(ss)
        L[name + "_z"] = None if zs[0] is None else np.stack(zs)
    ids = np.stack([np.random.default_rng(seed + t).choice(E, k, replace=False) for t in range(M)])
    L["topk_ids"] = ids.astype(np.int32)
    L["topk_w"] = np.random.default_rng(seed).random((M, k)).astype(np.float32)
    return L


def _scalar_layer(L):
    """Brute force with scalar Python loops over every index."""
    bits = L["bits"]
    pf = 32 // bits
    mask = (1 << bits) - 1
    x = oracle.halfbits_to_f64(L["x"], L["act_dtype"])
    M, H = x.shape
    E, twoI, _ = L["w13_q"].shape
    I = twoI // 2

    def weight(name, e, n, kk, K):
        G = K if L["group_size"] == -1 else L["group_size"]
        word = int(L[name + "_q"][e, n, kk // pf]) & 0xFFFFFFFF
        u = (word >> (bits * (kk % pf))) & mask
        s = float(oracle.halfbits_to_f64(L[name + "_s"][e, kk // G, n], L["scale_dtype"]))
        if L[name + "_z"] is None:
            z = 1 << (bits - 1)
        else:
            zw = int(L[name + "_z"][e, kk // G, n // pf]) & 0xFFFFFFFF
            z = (zw >> (bits * (n % pf))) & mask
        return (u - z) * s

    out = np.zeros((M, H))
    for t in range(M):
        for j in range(L["topk_ids"].shape[1]):
            e = int(L["topk_ids"][t, j])
            a = []
            for i in range(I):
                gsum = sum(weight("w13", e, i, kk, H) * x[t, kk] for kk in range(H))
                usum = sum(weight("w13", e, I + i, kk, H) * x[t, kk] for kk in range(H))
                a.append(gsum / (1.0 + math.exp(-gsum)) * usum)
            for h in range(H):
                y = sum(weight("w2", e, h, i, I) * a[i] for i in range(I))
                out[t, h] += float(L["topk_w"][t, j]) * y
    return out


@pytest.mark.parametrize("kw", [dict(), dict(bits=8, has_zeros=False, G=-1, act="bf16"),
                                dict(has_zeros=False, act="bf16", sdt="bf16", G=16)])
def test_layer_vs_scalar_brute_force(kw):
    L = _small_layer(M=2, H=32, I=16, E=3, k=2, **kw) if "G" in kw else _small_layer(
        M=2, H=32, I=16, E=3, k=2, G=16, **kw)
    ref = _scalar_layer(L)
    got = oracle.fused_moe_per_token(L, round_output=False)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-15)
    grouped = oracle.fused_moe_grouped(L, round_output=False)
    assert np.allclose(grouped, ref, rtol=1e-12, atol=1e-15)


def test_layer_top1_single_expert_is_dense_mlp():
    L = _small_layer(M=5, H=64, I=32, E=1, k=1)
    L["topk_w"] = np.ones((5, 1), dtype=np.float32)
    W13 = oracle.dequantize_expert(L["w13_q"][0], L["w13_s"][0], L["w13_z"][0], 4, 32, "f16")
    W2 = oracle.dequantize_expert(L["w2_q"][0], L["w2_s"][0], L["w2_z"][0], 4, 32, "f16")
    X = oracle.halfbits_to_f64(L["x"], "f16")
    G1, U = np.matmul(X, W13[:32].T), np.matmul(X, W13[32:].T)
    dense = np.matmul(G1 * (1.0 / (1.0 + np.exp(-G1))) * U, W2.T)
    got = oracle.fused_moe_per_token(L, round_output=False)
    assert np.allclose(got, dense, rtol=1e-12, atol=1e-14)


def test_layer_closed_form_constant_weights():
    """Every gate weight a, every up weight 2a, every down weight b, x_t = c:
    g = H a c, u = 2 H a c, out_t = sum_j w_tj * I * b * silu(g) * u."""
    H, I, E, k, M, bits, G = 64, 32, 2, 2, 2, 4, 32
    a, b, c = 2.0 ** -6, 2.0 ** -5, 2.0 ** -3
    L = dict(act_dtype="f16", scale_dtype="f16", bits=bits, group_size=G)
    L["x"] = halfbits(torch.full((M, H), c, dtype=torch.float16))
    gate = torch.full((I, H), 9)
    up = torch.full((I, H), 10)  # (10 - 8) * a = 2a
    L["w13_q"] = pack_along_last(torch.cat([gate, up])[None].repeat(E, 1, 1), bits).numpy()
    L["w13_s"] = halfbits(torch.full((E, H // G, 2 * I), a, dtype=torch.float16))
    L["w13_z"] = None
    L["w2_q"] = pack_along_last(torch.full((E, H, I), 9), bits).numpy()
    L["w2_s"] = halfbits(torch.full((E, I // G, H), b, dtype=torch.float16))
    L["w2_z"] = None
    L["topk_ids"] = np.array([[0, 1], [1, 0]], dtype=np.int32)
    L["topk_w"] = np.array([[0.75, 0.25], [0.5, 0.125]], dtype=np.float32)
    g = H * a * c
    u = 2 * H * a * c
    y = I * b * (g / (1 + math.exp(-g))) * u
    got = oracle.fused_moe_per_token(L, round_output=False)
    assert np.allclose(got[0], y * 1.0)
    assert np.allclose(got[1], y * 0.625)


def test_layer_linear_in_topk_weights():
    L = _small_layer()
    base = oracle.fused_moe_per_token(L, round_output=False)
    L2 = dict(L, topk_w=(L["topk_w"] * 2.0).astype(np.float32))
    assert np.allclose(oracle.fused_moe_per_token(L2, round_output=False), 2 * base)
    # one slot at a time sums to the whole
    parts = 0
    for j in range(L["topk_ids"].shape[1]):
        w = np.zeros_like(L["topk_w"])
        w[:, j] = L["topk_w"][:, j]
        parts = parts + oracle.fused_moe_per_token(dict(L, topk_w=w), round_output=False)
    assert np.allclose(parts, base, rtol=1e-12, atol=1e-15)


def test_layer_zero_when_codes_equal_zero_points():
    L = _small_layer(has_zeros=False)
    L["w2_q"] = pack_along_last(torch.full((4, 64, 32), 8), 4).numpy()  # u - 8 = 0
    assert np.all(oracle.fused_moe_per_token(L, round_output=False) == 0.0)


def test_layer_expert_relabeling_invariance():
    L = _small_layer(E=4)
    perm = np.array([2, 0, 3, 1])  # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    L2 = dict(L)
    for key in ("w13_q", "w13_s", "w13_z", "w2_q", "w2_s", "w2_z"):
        L2[key] = L[key][inv]
    L2["topk_ids"] = perm[L["topk_ids"]].astype(np.int32)
    a = oracle.fused_moe_per_token(L, round_output=False)
    b = oracle.fused_moe_per_token(L2, round_output=False)
    assert np.array_equal(a, b)


def test_layer_drops_out_of_range_ids():
    L = _small_layer(E=4)
    L2 = dict(L, topk_ids=np.where(np.arange(2)[None, :] == 1, 99, L["topk_ids"]).astype(np.int32))
    L3 = dict(L, topk_w=np.where(np.arange(2)[None, :] == 1, 0, L["topk_w"]).astype(np.float32))
    assert np.array_equal(oracle.fused_moe_per_token(L2, round_output=False),
                          oracle.fused_moe_per_token(L3, round_output=False))


def test_tiny_workload_oracle_forms_agree():
    from synthetic import WORKLOADS, make_layer_inputs
    from tests.helpers import oracle_layer_dict
    li = make_layer_inputs(WORKLOADS["tiny"], 4)
    L = oracle_layer_dict(li)
    a = oracle.fused_moe_per_token(L)
    b = oracle.fused_moe_grouped(L)
    # both round the same float64 sum (up to summation order) once
    fa = oracle.halfbits_to_f64(a, "f16")
    fb = oracle.halfbits_to_f64(b, "f16")
    assert np.max(np.abs(fa - fb)) <= np.max(np.abs(fa)) * 2.0 ** -10


# ----------------------------------------------------------------------------
# biases and the clamped SwiGLU (vLLM int8 MoE config: w1_bias / w2_bias,
# swiglu_alpha / swiglu_beta / swiglu_limit; readings in the oracle)
# ----------------------------------------------------------------------------

def test_gated_activation_closed_forms():
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))
    act = lambda g, u, glu=None: float(oracle.gated_activation(np.array([g]), np.array([u]), glu)[0])
    assert act(1.0, 2.0) == pytest.approx(2.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    # gate clamped from above only, up from both sides, beta added after the clamp:
    # (9, -8) -> (7, -7): 7 * sigmoid(2 * 7) * (-7 + 1)
    assert act(9.0, -8.0, (2.0, 1.0, 7.0)) == pytest.approx(-42.0 * sig(14.0), rel=1e-15)
    # (-9, 9) -> (-9, 7): -9 * sigmoid(-18) * 8
    assert act(-9.0, 9.0, (2.0, 1.0, 7.0)) == pytest.approx(-72.0 * sig(-18.0), rel=1e-15)
    # inside the limit nothing is clamped
    assert act(3.0, 0.5, (2.0, 1.0, 7.0)) == pytest.approx(3.0 * sig(6.0) * 1.5, rel=1e-15)
    # limit <= 0: no clamp
    assert act(9.0, -8.0, (2.0, 1.0, 0.0)) == pytest.approx(9.0 * sig(18.0) * -7.0, rel=1e-15)
    # alpha = 1, beta = 0, no limit is silu(g) * u
    rng = np.random.default_rng(3)
    g, u = rng.standard_normal(50) * 4, rng.standard_normal(50) * 4
    np.testing.assert_allclose(oracle.gated_activation(g, u, (1.0, 0.0, 0.0)), oracle.gated_activation(g, u),
                               rtol=1e-15)


def _half(v, dt="f16"):
    return halfbits(torch.as_tensor(np.asarray(v, dtype=np.float32)).to(
        torch.float16 if dt == "f16" else torch.bfloat16))


def test_layer_biases_closed_form_zero_weights():
    # all codes at the zero point: W13 = W2 = 0, so y = b2[e] for every slot and
    # out_t = sum_j w_tj b2[e_tj], whatever b13 and the activation are
    L = _small_layer(has_zeros=False)
    E, H, I = 4, 64, 32
    L["w13_q"] = pack_along_last(torch.full((E, 2 * I, H), 8), 4).numpy()
    L["w2_q"] = pack_along_last(torch.full((E, H, I), 8), 4).numpy()
    rng = np.random.default_rng(1)
    b2 = rng.standard_normal((E, H))
    L["w13_b"] = _half(rng.standard_normal((E, 2 * I)) * 4)
    L["w2_b"] = _half(b2)
    b2 = oracle.halfbits_to_f64(L["w2_b"], "f16")
    tw = L["topk_w"].astype(np.float64)
    want = sum(tw[:, j, None] * b2[L["topk_ids"][:, j]] for j in range(2))
    for glu in (None, (1.702, 1.0, 7.0)):
        got = oracle.fused_moe_per_token(dict(L, glu=glu), round_output=False)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)


def test_layer_biases_closed_form_constant_down():
    # W13 = 0 and every down weight b: g_i = b13[e, i], u_i = b13[e, I + i],
    # y_h = b * sum_i act(g_i, u_i) + b2[e, h]; clamped SwiGLU with values past the limit
    L = _small_layer(has_zeros=False, E=2)
    E, H, I, b = 2, 64, 32, 2.0 ** -5
    L["w13_q"] = pack_along_last(torch.full((E, 2 * I, H), 8), 4).numpy()
    L["w2_q"] = pack_along_last(torch.full((E, H, I), 9), 4).numpy()  # (9 - 8) * s
    L["w2_s"] = halfbits(torch.full((E, I // 32, H), b, dtype=torch.float16))
    rng = np.random.default_rng(2)
    L["w13_b"] = _half(rng.standard_normal((E, 2 * I)) * 8)
    L["w2_b"] = _half(rng.standard_normal((E, H)))
    L["topk_ids"] = np.array([[0, 1], [1, 0], [0, 1]], dtype=np.int32)
    b13 = oracle.halfbits_to_f64(L["w13_b"], "f16")
    b2 = oracle.halfbits_to_f64(L["w2_b"], "f16")
    alpha, beta, lim = 1.702, 1.0, 7.0
    y = np.zeros((E, H))
    for e in range(E):
        s = 0.0
        for i in range(I):
            g, u = b13[e, i], b13[e, I + i]
            g, u = min(g, lim), min(max(u, -lim), lim)
            s += g / (1.0 + math.exp(-alpha * g)) * (u + beta)
        y[e] = b * s + b2[e]
    tw = L["topk_w"].astype(np.float64)
    want = np.stack([sum(tw[t, j] * y[L["topk_ids"][t, j]] for j in range(2)) for t in range(3)])
    got = oracle.fused_moe_per_token(dict(L, glu=(alpha, beta, lim)), round_output=False)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
    assert np.any(np.abs(b13) > lim)  # the clamp is exercised


def test_layer_biases_grouped_matches_per_token():
    L = _small_layer(E=4)
    rng = np.random.default_rng(4)
    L["w13_b"] = _half(rng.standard_normal((4, 64)))
    L["w2_b"] = _half(rng.standard_normal((4, 64)))
    for glu in (None, (1.702, 1.0, 0.5)):
        a = oracle.fused_moe_per_token(dict(L, glu=glu), round_output=False)
        b = oracle.fused_moe_grouped(dict(L, glu=glu), round_output=False)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------
# act-order (GPTQ desc_act: group of column k = g_idx[k])
# ----------------------------------------------------------------------------

def test_act_order_permutation_closed_form():
    perm, inv = oracle.act_order_permutation(np.array([1, 0, 1, 0, 2, 2]))
    assert perm.tolist() == [1, 3, 0, 2, 4, 5]  # group 0: k 1, 3; group 1: k 0, 2; group 2: k 4, 5
    assert inv.tolist() == [2, 0, 3, 1, 4, 5]


def test_act_order_default_groups_are_the_plain_layout():
    L = _small_layer(E=2)
    g = np.arange(64) // 32
    a = oracle.dequantize_expert(L["w13_q"][0], L["w13_s"][0], L["w13_z"][0], 4, 32, "f16")
    b = oracle.dequantize_expert(L["w13_q"][0], L["w13_s"][0], L["w13_z"][0], 4, 32, "f16", g_idx=g)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("bits,has_zeros,G", [(4, True, 32), (4, False, 64), (8, False, 32)])
def test_act_order_round_trip_within_half_step(bits, has_zeros, G):
    # the error bound holds only if every column is dequantized with its own group
    from synthetic import make_g_idx, quantize_expert_act_order
    K, N = 256, 48
    w = torch.randn(N, K, generator=torch.Generator().manual_seed(bits + G)) * 0.1
    g = make_g_idx(K, G, 11)
    codes, s, z = quantize_expert_act_order(w, bits, has_zeros, G, "f16", g)
    q = pack_along_last(codes, bits).numpy()
    zw = None if z is None else pack_along_last(z, bits).numpy()
    W = oracle.dequantize_expert(q, halfbits(s), zw, bits, G, "f16", g_idx=g.numpy())
    step = oracle.halfbits_to_f64(halfbits(s), "f16").T[:, g.numpy()]  # [N, K] scale of each weight
    assert np.all(np.abs(W - w.double().numpy()) <= step / 2 + 1e-12)
    # grouping by k // G instead breaks the bound
    W_wrong = oracle.dequantize_expert(q, halfbits(s), zw, bits, G, "f16")
    assert not np.all(np.abs(W_wrong - w.double().numpy()) <= step / 2 + 1e-12)


def test_act_order_repacked_columns_are_the_plain_layout():
    # sorting the columns by group gives a plain grouped matrix:
    # W_actorder[:, perm[i]] = W_plain(codes[:, perm])[:, i]
    from synthetic import make_g_idx, quantize_expert_act_order
    K, N, G = 128, 32, 32
    w = torch.randn(N, K, generator=torch.Generator().manual_seed(5)) * 0.1
    g = make_g_idx(K, G, 3)
    codes, s, z = quantize_expert_act_order(w, 4, True, G, "f16", g)
    perm, _ = oracle.act_order_permutation(g.numpy())
    W = oracle.dequantize_expert(pack_along_last(codes, 4).numpy(), halfbits(s), pack_along_last(z, 4).numpy(), 4, G,
                                 "f16", g_idx=g.numpy())
    Wp = oracle.dequantize_expert(pack_along_last(codes[:, perm], 4).numpy(), halfbits(s),
                                  pack_along_last(z, 4).numpy(), 4, G, "f16")
    assert np.array_equal(W[:, perm], Wp)


def test_act_order_layer_vs_scalar_brute_force():
    from synthetic import make_g_idx
    L = _small_layer(M=2, H=32, I=16, E=2, k=2, G=16)
    L["w13_g_idx"] = np.stack([make_g_idx(32, 16, 20 + e).numpy() for e in range(2)])
    L["w2_g_idx"] = np.stack([make_g_idx(16, 16, 30 + e).numpy() for e in range(2)])
    bits, pf, mask = 4, 8, 15
    x = oracle.halfbits_to_f64(L["x"], "f16")

    def weight(name, e, n, kk):
        word = int(L[name + "_q"][e, n, kk // pf]) & 0xFFFFFFFF
        u = (word >> (bits * (kk % pf))) & mask
        g = int(L[name + "_g_idx"][e, kk])
        s = float(oracle.halfbits_to_f64(L[name + "_s"][e, g, n], "f16"))
        zw = int(L[name + "_z"][e, g, n // pf]) & 0xFFFFFFFF
        return (u - ((zw >> (bits * (n % pf))) & mask)) * s

    out = np.zeros((2, 32))
    for t in range(2):
        for j in range(2):
            e = int(L["topk_ids"][t, j])
            a = []
            for i in range(16):
                gs = sum(weight("w13", e, i, kk) * x[t, kk] for kk in range(32))
                us = sum(weight("w13", e, 16 + i, kk) * x[t, kk] for kk in range(32))
                a.append(gs / (1.0 + math.exp(-gs)) * us)
            for h in range(32):
                out[t, h] += float(L["topk_w"][t, j]) * sum(weight("w2", e, h, i) * a[i] for i in range(16))
    got = oracle.fused_moe_per_token(L, round_output=False)
    np.testing.assert_allclose(got, out, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.fused_moe_grouped(L, round_output=False), out, rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------
# GPTQ / AWQ checkpoint formats
# ----------------------------------------------------------------------------

def test_awq_field_order_literal_word():
    # field i holds column AWQ_PACK_ORDER[i]: 0x76543210 puts 0..7 in columns 0 2 4 6 1 3 5 7
    assert oracle.unpack_awq(np.array([[0x76543210]])).tolist() == [[0, 4, 1, 5, 2, 6, 3, 7]]
    assert oracle.unpack_awq(np.array([[0x0000000F, 0xF0000000]])).tolist() == [[15] + [0] * 7 + [0] * 7 + [15]]


def test_gptq_literal_words():
    # column n of word row r holds k = 8 r + j in field j
    q = np.array([[0x76543210, 0x00000010], [0x00000000, 0xF0000000]])
    codes = oracle.unpack_gptq_qweight(q, 4)
    assert codes.shape == (2, 16)
    assert codes[0].tolist() == list(range(8)) + [0] * 8
    assert codes[1].tolist() == [0, 1] + [0] * 13 + [15]
    q8 = np.array([[0x04030201]])
    assert oracle.unpack_gptq_qweight(q8, 8).tolist() == [[1, 2, 3, 4]]
    # v1 zero points: stored z - 1, so 0xF is zero point 0
    assert oracle.unpack_gptq_qzeros(np.array([[0x7654321F]]), 4).tolist() == [[0, 2, 3, 4, 5, 6, 7, 8]]
    assert oracle.unpack_gptq_qzeros(np.array([[0x7654321F]]), 4, False).tolist() == [[15, 1, 2, 3, 4, 5, 6, 7]]


def _gptq_pack(codes, bits):
    """[N, K] codes -> GPTQ qweight [K/pf, N], with explicit loops."""
    N, K = codes.shape
    pf = 32 // bits
    out = np.zeros((K // pf, N), dtype=np.int64)
    for n in range(N):
        for k in range(K):
            out[k // pf, n] |= int(codes[n, k]) << (bits * (k % pf))
    return out


def _awq_pack(vals):
    """[R, N] 4-bit values -> AWQ words [R, N/8], with explicit loops."""
    R, N = vals.shape
    out = np.zeros((R, N // 8), dtype=np.int64)
    for r in range(R):
        for c in range(N // 8):
            for i in range(8):
                out[r, c] |= int(vals[r, 8 * c + oracle.AWQ_PACK_ORDER[i]]) << (4 * i)
    return out


@pytest.mark.parametrize("fmt,bits", [("gptq", 4), ("gptq", 8), ("awq", 4)])
def test_checkpoint_formats_dequantize_like_the_plain_layout(fmt, bits):
    # the same codes, zero points and scales in a checkpoint layout and in the
    # plain layout give the same float64 weights
    rng = np.random.default_rng(bits)
    N, K, G = 32, 64, 32
    codes = rng.integers(0, 1 << bits, size=(N, K))
    zeros = rng.integers(0, 1 << bits, size=(K // G, N))
    s = halfbits((torch.rand(K // G, N) * 0.01 + 0.001).half())
    plain = oracle.dequantize_expert(pack_along_last(torch.as_tensor(codes), bits).numpy(), s,
                                     pack_along_last(torch.as_tensor(zeros), bits).numpy(), bits, G, "f16")
    if fmt == "gptq":
        u = oracle.unpack_gptq_qweight(_gptq_pack(codes, bits), bits)
        zw = np.zeros((K // G, N * bits // 32), dtype=np.int64)
        for g in range(K // G):
            for n in range(N):
                zw[g, n * bits // 32] |= ((int(zeros[g, n]) - 1) % (1 << bits)) << (bits * (n % (32 // bits)))
        z = oracle.unpack_gptq_qzeros(zw, bits)
    else:
        u = oracle.unpack_awq(_awq_pack(codes.T)).T  # AWQ packs [K, N] along N
        z = oracle.unpack_awq(_awq_pack(zeros))
    sf = oracle.halfbits_to_f64(s, "f16")
    g_of_k = np.arange(K) // G
    W = (u - z.T[:, g_of_k]) * sf.T[:, g_of_k]
    assert np.array_equal(u, codes) and np.array_equal(z, zeros)
    assert np.array_equal(W, plain)



def test_round_intermediate_diagnosis_mode():
    # rounding the activation to the act dtype moves the output by about that
    # rounding; with codes equal to zero points it changes nothing (a = 0)
    from tests.helpers import max_rel_err, norm_rel_err
    L = _small_layer()
    a = oracle.fused_moe_per_token(L, round_output=False)
    b = oracle.fused_moe_per_token(L, round_output=False, round_intermediate=True)
    c = oracle.fused_moe_grouped(L, round_output=False, round_intermediate=True)
    np.testing.assert_allclose(b, c, rtol=1e-12, atol=1e-15)
    assert 0 < max_rel_err(b, a) < 2.0 ** -9 and 0 < norm_rel_err(b, a) < 2.0 ** -9
    Z = dict(L, w13_q=pack_along_last(torch.full((4, 64, 64), 8), 4).numpy(), w13_z=None)
    assert np.array_equal(oracle.fused_moe_per_token(Z, round_output=False),
                          oracle.fused_moe_per_token(Z, round_output=False, round_intermediate=True))
