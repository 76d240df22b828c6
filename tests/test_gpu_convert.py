"""GPU parity of wna16_convert_checkpoint: GPTQ / AWQ checkpoint tensors to the
layer's layout, bit-exact against the oracle's unpacking of each layout, and a
layer run on converted weights against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, Workload, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, np_i32, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _rand_words(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-2 ** 31, 2 ** 31 - 1, shape, generator=g, dtype=torch.int64).to(torch.int32)


@pytest.mark.parametrize("fmt,bits", [("gptq", 4), ("gptq", 8), ("gptq_v2", 4), ("awq", 4)])
@pytest.mark.parametrize("N,K,G", [(96, 512, 128), (40, 256, -1), (1056, 4160, 64)])
def test_random_words_bit_exact(fmt, bits, N, K, G):
    pf = 32 // bits
    if N % pf:
        pytest.skip("N must hold whole zero-point words")
    E = 3
    Gk = K if G == -1 else G
    qw = _rand_words((E, K, N // 8) if fmt == "awq" else (E, K // pf, N), N + K + bits)
    qz = _rand_words((E, K // Gk, N // pf), N * K + bits)
    q_out, z_out = w.convert_checkpoint(fmt, qw.to(DEV), qz.to(DEV), bits, G)
    torch.cuda.synchronize()
    for e in range(E):
        if fmt == "awq":
            codes = oracle.unpack_awq(np_i32(qw[e])).T  # [K, N] -> [N, K]
            zeros = oracle.unpack_awq(np_i32(qz[e]))
        else:
            codes = oracle.unpack_gptq_qweight(np_i32(qw[e]), bits)
            zeros = oracle.unpack_gptq_qzeros(np_i32(qz[e]), bits, stored_minus_one=fmt == "gptq")
        assert np.array_equal(oracle.unpack_codes(np_i32(q_out[e]), bits), codes)
        assert np.array_equal(oracle.unpack_zeros(np_i32(z_out[e]), bits), zeros)


def test_symmetric_weights_without_zeros():
    qw = _rand_words((2, 64, 128), 9)
    q_out, z_out = w.convert_checkpoint("gptq", qw.to(DEV), None, 4, 128)
    torch.cuda.synchronize()
    assert z_out is None
    assert np.array_equal(oracle.unpack_codes(np_i32(q_out[1]), 4), oracle.unpack_gptq_qweight(np_i32(qw[1]), 4))


def _pack_fields(vals, bits, order=None):
    """[..., W*pf] field values -> [..., W] int32 words (LSB first, or in `order`)."""
    pf = 32 // bits
    v = vals.reshape(*vals.shape[:-1], vals.shape[-1] // pf, pf).astype(np.int64)
    if order is not None:
        v = v[..., list(order)]
    words = np.zeros(v.shape[:-1], dtype=np.int64)
    for i in range(pf):
        words |= v[..., i] << (bits * i)
    return torch.from_numpy(words.astype(np.uint32).view(np.int32))


@pytest.mark.parametrize("fmt", ["gptq", "awq"])
def test_layer_from_checkpoint_layout(fmt):
    # a layer's weights written out in the checkpoint layout convert back to the
    # very same words, and the layer on them matches the oracle
    wl = Workload(name="ckpt", H=512, I=384, E=4, topk=2, bits=4, has_zeros=True, group_size=128,
                  act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")
    li = make_layer_inputs(wl, 24).to(DEV)
    conv = {}
    for name in ("w13", "w2"):
        q = getattr(li, name + "_q").cpu()
        z = getattr(li, name + "_z").cpu()
        if fmt == "gptq":
            qw = q.transpose(1, 2).contiguous()  # the same words, [K/pf, N]
            zv = np.stack([oracle.unpack_zeros(np_i32(z[e]), 4) for e in range(wl.E)])
            qz = _pack_fields((zv - 1) % 16, 4)
        else:
            codes = np.stack([oracle.unpack_codes(np_i32(q[e]), 4).T for e in range(wl.E)])  # [E, K, N]
            qw = _pack_fields(codes, 4, oracle.AWQ_PACK_ORDER)
            zv = np.stack([oracle.unpack_zeros(np_i32(z[e]), 4) for e in range(wl.E)])
            qz = _pack_fields(zv, 4, oracle.AWQ_PACK_ORDER)
        q_out, z_out = w.convert_checkpoint(fmt, qw.to(DEV), qz.to(DEV), 4, wl.group_size)
        torch.cuda.synchronize()
        assert torch.equal(q_out, getattr(li, name + "_q"))
        assert torch.equal(z_out, getattr(li, name + "_z"))
        conv[name] = (q_out, z_out)
    y = w.fused_moe(li.hidden, conv["w13"][0], li.w13_s, conv["w13"][1], conv["w2"][0], li.w2_s, conv["w2"][1],
                    li.topk_ids, li.topk_w, wl.bits, wl.group_size)
    torch.cuda.synchronize()
    ref = oracle.fused_moe_grouped(oracle_layer_dict(li))
    assert max_rel_err(bits_to_f64(halfbits(y), "f16"), bits_to_f64(ref, "f16")) <= 1e-2


def test_mixtral_sized_gate_up_conversion_is_bit_exact():
    # one Mixtral-8x7B-shaped expert: w13 [2I = 28672, H = 4096] in GPTQ layout
    wl = WORKLOADS["mixtral8x7b"]
    N, K = 2 * wl.I, wl.H
    qw = _rand_words((1, K // 8, N), 77).to(DEV)
    q_out, _ = w.convert_checkpoint("gptq", qw, None, 4, 128)
    torch.cuda.synchronize()
    assert torch.equal(q_out[0], qw[0].t())
