"""GPU parity of the fused layer against the float64 oracle.

Bar: max |y - r| / max |r| <= 1e-2 on the layer output (fp32 accumulation,
fp16/bf16 output), element by element on every output of every case here.
The shapes span several weight-row tiles of both GEMMs, several K stages and
quantization groups, ragged token blocks (block sizes that do not divide the
per-expert counts), every block size and K split, both weight widths, both
activation dtypes and both scale dtypes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, Workload, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, norm_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def run_layer(li, block=0, split_k=0, out=None, workspace=None, ids=None):
    return w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z,
                       li.topk_ids if ids is None else ids, li.topk_w, li.wl.bits, li.wl.group_size,
                       out=out, workspace=workspace, block=block, split_k=split_k)


def check(li, block=0, split_k=0, tokens=None):
    y = run_layer(li, block, split_k)
    torch.cuda.synchronize()
    L = oracle_layer_dict(li)
    if tokens is None:
        ref = oracle.fused_moe_grouped(L)
        got = halfbits(y)
    else:
        ref = oracle.fused_moe_per_token(L, tokens=tokens)
        got = halfbits(y)[tokens]
    dt = li.wl.act_dtype
    r, g = bits_to_f64(ref, dt), bits_to_f64(got, dt)
    assert np.all(np.isfinite(g))
    err = max_rel_err(g, r)
    assert err <= TOL, (err, norm_rel_err(g, r), block, split_k)
    return err


def small(name="small", **kw):
    base = dict(name=name, H=384, I=192, E=6, topk=2, bits=4, has_zeros=True, group_size=64,
                act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")
    base.update(kw)
    return Workload(**base)


def test_tiny_workload():
    wl = WORKLOADS["tiny"]
    li = make_layer_inputs(wl, 4).to(DEV)
    check(li, block=wl.block)


@pytest.mark.parametrize("block", [16, 32, 64, 128, 256])
def test_blocks_ragged_tails(block):
    li = make_layer_inputs(small(), 37).to(DEV)
    check(li, block=block)


@pytest.mark.parametrize("split_k", [1, 2, 3])
def test_split_k(split_k):
    li = make_layer_inputs(small(I=640), 5).to(DEV)
    check(li, block=16, split_k=split_k)


@pytest.mark.parametrize("act,sdt", [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f16"), ("f16", "bf16")])
@pytest.mark.parametrize("bits,zeros,G", [(4, True, 64), (4, False, 128), (8, False, -1), (8, True, 64)])
def test_formats(act, sdt, bits, zeros, G):
    wl = small(bits=bits, has_zeros=zeros, group_size=G, act_dtype=act, scale_dtype=sdt, H=256, I=256)
    li = make_layer_inputs(wl, 19).to(DEV)
    check(li, block=16)
    check(li, block=64)


@pytest.mark.parametrize("act,sdt,bits,zeros", [("f16", "f16", 4, True), ("f16", "bf16", 4, False),
                                                ("bf16", "bf16", 4, True), ("bf16", "f16", 4, False),
                                                ("f16", "f16", 8, True), ("f16", "bf16", 8, False)])
@pytest.mark.parametrize("G", [128, 256, -1])
@pytest.mark.parametrize("block", [16, 32])
def test_deferred_scale_tiles(act, sdt, bits, zeros, G, block):
    # 16- and 32-token tiles whose K stages lie inside one group run the
    # deferred-scale kernel: magic-number codes, offsets and zero point removed
    # by a correction MMA, scale applied to each stage's fp32 partial sum
    wl = small(bits=bits, has_zeros=zeros, group_size=G, act_dtype=act, scale_dtype=sdt, H=512, I=768)
    li = make_layer_inputs(wl, 37 if block == 16 else 75).to(DEV)
    for split in (1, 2, 3):
        check(li, block=block, split_k=split)


@pytest.mark.parametrize("bits,act", [(4, "f16"), (4, "bf16"), (8, "f16")])
def test_deferred_scale_half_stage(bits, act):
    # per-channel scales, H and I = 64 (mod 128): the last K stage of both GEMMs
    # holds a single 64-wide half, whose token sums stay zero
    wl = small(H=320, I=192, group_size=-1, bits=bits, has_zeros=True, act_dtype=act, scale_dtype=act)
    li = make_layer_inputs(wl, 23).to(DEV)
    check(li, block=16)
    check(li, block=16, split_k=2)
    check(li, block=32, split_k=2)


@pytest.mark.parametrize("M,block", [(1, 16), (3, 16), (2, 32)])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_gate_up_k_split(M, block, act):
    # few work units and K = 2048 (16 stages): the gate/up GEMM splits K in two;
    # split units publish fp32 partial sums and the last one of each lane quarter
    # adds them up before silu(gate) * up. Called twice: the arrival counters
    # must start from zero again.
    wl = small(H=2048, I=256, E=4, topk=1, group_size=128, act_dtype=act, scale_dtype=act)
    li = make_layer_inputs(wl, M).to(DEV)
    check(li, block=block)
    check(li, block=block)


def test_deferred_scale_large_activations():
    # hidden values 50x larger: the fp16 token sums of the correction operand
    # (stored at 1/32) and the magic-number offsets must not lose the result
    wl = small(H=512, I=256, group_size=128)
    li = make_layer_inputs(wl, 16).to(DEV)
    li.hidden.mul_(50.0)
    check(li, block=16)
    check(li, block=32)


@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_int8_256_token_tiles_single_a_slot(act):
    # 8-bit codes with 256-token tiles leave room for two ring stages and so a
    # single TMEM A slot: the two dequant warpgroups must take turns on it
    wl = small(bits=8, has_zeros=False, group_size=-1, act_dtype=act, scale_dtype="f16", H=384, I=256, E=2, topk=1)
    li = make_layer_inputs(wl, 300).to(DEV)
    check(li, block=256)


def test_hidden_not_multiple_of_row_tile():
    # H = 320: the down GEMM's last 128-row tile is half outside the matrix
    li = make_layer_inputs(small(H=320, I=128, group_size=64), 11).to(DEV)
    check(li, block=32)


def test_many_experts_top8():
    wl = small(E=64, topk=8, H=256, I=128, routing="softmax", zipf_s=1.1, act_dtype="bf16", scale_dtype="bf16",
               has_zeros=False, group_size=128)
    li = make_layer_inputs(wl, 33).to(DEV)
    check(li)  # automatic block and split


def test_256_experts_grouped_routing():
    wl = small(E=256, topk=8, H=256, I=128, routing="sigmoid_grouped", n_groups=8, topk_groups=4, group_size=128)
    for M in (1, 16):
        li = make_layer_inputs(wl, M).to(DEV)
        check(li)


def test_duplicate_ids_in_a_token():
    li = make_layer_inputs(small(), 6).to(DEV)
    li.topk_ids[:, 1] = li.topk_ids[:, 0]
    check(li, block=16)


def test_empty_batch():
    li = make_layer_inputs(small(), 0).to(DEV)
    y = run_layer(li)
    assert y.shape == (0, 384)


def test_bad_expert_id_is_dropped_and_reported():
    li = make_layer_inputs(small(), 9).to(DEV)
    ids = li.topk_ids.clone()
    ids[3, 1] = 99
    ids[5, 0] = -1
    need = w.workspace_bytes(9, 384, 192, 6, 2, 4, 64, 16, 0)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    y = run_layer(li, block=16, workspace=ws, ids=ids)
    bits = w.read_device_status(ws[:4].view(torch.int32))
    assert bits == w.DEV_BAD_EXPERT_ID
    L = oracle_layer_dict(li)
    L["topk_ids"] = ids.cpu().numpy()
    ref = bits_to_f64(oracle.fused_moe_grouped(L), "f16")
    assert max_rel_err(bits_to_f64(halfbits(y), "f16"), ref) <= TOL
    # a clean call resets the status word
    run_layer(li, block=16, workspace=ws)
    assert w.read_device_status(ws[:4].view(torch.int32)) == 0


def test_output_canaries_and_no_stray_writes():
    li = make_layer_inputs(small(), 13).to(DEV)
    canary = torch.tensor(-7.25, dtype=torch.float16)
    buf = torch.full((13 + 2, 384), float(canary), dtype=torch.float16, device=DEV)
    out = buf[1:14]
    run_layer(li, block=32, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[0] == canary) and torch.all(buf[14] == canary)


def test_cuda_graph_replay_is_bit_identical():
    li = make_layer_inputs(small(E=8, topk=2), 21).to(DEV)
    need = w.workspace_bytes(21, 384, 192, 8, 2, 4, 64, 0, 0)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = torch.empty(21, 384, dtype=torch.float16, device=DEV)
    eager = run_layer(li, workspace=ws).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        run_layer(li, out=out, workspace=ws)  # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            run_layer(li, out=out, workspace=ws)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    # new routing written into the captured input buffers is picked up on replay
    li.topk_ids.copy_(torch.flip(li.topk_ids, dims=[0]))
    li.topk_w.copy_(torch.flip(li.topk_w, dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    L = oracle_layer_dict(li)
    ref = bits_to_f64(oracle.fused_moe_grouped(L), "f16")
    assert max_rel_err(bits_to_f64(halfbits(out), "f16"), ref) <= TOL


def test_deterministic_across_calls():
    li = make_layer_inputs(small(), 40).to(DEV)
    a = run_layer(li, block=16).clone()
    b = run_layer(li, block=16)
    assert torch.equal(a, b)


@pytest.mark.parametrize("block", [16, 32, 64])
@pytest.mark.parametrize("split_k", [1, 2, 3])
def test_atomic_down_reduction(block, split_k):
    # the fp32-atomic variant of the down GEMM's reduction (slots and K splits
    # added into one [M, H] row per token): within the tolerance of the oracle
    # and of the ordered reduction, though not bit-reproducible
    wl = small(H=512, I=768, group_size=128, E=6, topk=3)
    li = make_layer_inputs(wl, 37).to(DEV)
    ordered = run_layer(li, block=block, split_k=split_k).clone()
    y = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    wl.bits, wl.group_size, block=block, split_k=split_k, atomic_reduce=True)
    torch.cuda.synchronize()
    ref = bits_to_f64(oracle.fused_moe_grouped(oracle_layer_dict(li)), wl.act_dtype)
    g = bits_to_f64(halfbits(y), wl.act_dtype)
    assert max_rel_err(g, ref) <= TOL
    assert max_rel_err(g, bits_to_f64(halfbits(ordered), wl.act_dtype)) <= TOL
