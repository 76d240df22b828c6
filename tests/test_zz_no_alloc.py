"""GPU check of wna16_fused_moe_noalloc, the entry point for callers that have
no allocator to give the library a workspace (a plain C host program, or a
plugin inside a process whose memory manager owns the device memory and would
be bypassed by an extra cudaMalloc). It must produce what the ordinary entry
point produces, call after call, although every call reuses one library-owned
scratch area that still holds the previous call's data, and it must not
allocate device memory.

Both entry points run the same deterministic kernels on the same inputs, so the
outputs are compared bit for bit (which is within the parity tolerance). The
layers cover the scratch contents that must be rewritten or cleared by each
call: the token sums of a K stage half with no elements (H and I not multiples
of 128) and the arrival counters of the gate/up GEMM's K split, after a larger
call has filled the area with other data.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before this one.
"""
import ctypes

import pytest
import torch

import weight_quantized_moe_align_gb300 as w
from synthetic import Workload, make_expert_weights, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2  # the layer-output tolerance of the parity tests
NOALLOC_BYTES = 64 << 20  # WNA16_NOALLOC_SCRATCH_BYTES
WORKSPACE_TOO_SMALL = 3

LAYERS = {
    # groups of 128, stages fully inside H and I
    "g128": Workload("noalloc_g128", H=384, I=640, E=8, topk=2, bits=4, has_zeros=True, group_size=128,
                     act_dtype="f16", scale_dtype="f16", routing="softmax_renorm"),
    # one group per channel, H % 128 == I % 128 == 64: the last stage of each
    # GEMM has an empty 64-wide half whose token sums the call must zero
    "half_stage": Workload("noalloc_half", H=448, I=576, E=8, topk=2, bits=4, has_zeros=False,
                           group_size=-1, act_dtype="bf16", scale_dtype="bf16", routing="softmax_renorm"),
    # decode batch over a long K and few row tiles: the gate/up GEMM is split
    # over K and uses per-unit arrival counters in the scratch area
    "k_split": Workload("noalloc_ksplit", H=4096, I=512, E=8, topk=2, bits=4, has_zeros=True, group_size=128,
                        act_dtype="f16", scale_dtype="f16", routing="softmax_renorm"),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _with_workspace(li):
    return w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids,
                       li.topk_w, li.wl.bits, li.wl.group_size)


def _without_workspace(li, out):
    return w.fused_moe_noalloc(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z,
                               li.topk_ids, li.topk_w, li.wl.bits, li.wl.group_size, out)


def _same(got, ref, dt):
    g = bits_to_f64(halfbits(got), dt)
    r = bits_to_f64(halfbits(ref), dt)
    assert max_rel_err(g, r) <= TOL
    assert torch.equal(got, ref)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    weights = {k: make_expert_weights(wl, DEV) for k, wl in LAYERS.items()}
    # fill the scratch area with another call's data first
    big = make_layer_inputs(LAYERS["g128"], 200, DEV, weights=weights["g128"], seed=3)
    _without_workspace(big, torch.empty_like(big.hidden))
    torch.cuda.synchronize()
    for key, wl in LAYERS.items():
        # two calls in a row with different batches: the second finds the
        # first call's data in the shared scratch area
        for M, seed in ((37, 11), (3, 12)):
            li = make_layer_inputs(wl, M, DEV, weights=weights[key], seed=seed)
            need = w.workspace_bytes(M, wl.H, wl.I, wl.E, wl.topk, wl.bits, wl.group_size)
            assert need <= NOALLOC_BYTES
            out = torch.empty_like(li.hidden)
            got = _without_workspace(li, out)
            ref = _with_workspace(li)
            torch.cuda.synchronize()
            assert w.noalloc_read_status() == 0, (key, M)
            _same(got, ref, wl.act_dtype)


def test_noalloc_allocates_nothing():
    wl = LAYERS["k_split"]
    weights = make_expert_weights(wl, DEV)
    li = make_layer_inputs(wl, 5, DEV, weights=weights, seed=21)
    out = torch.empty_like(li.hidden)
    _without_workspace(li, out)  # kernels loaded, address looked up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated(DEV)
    free_before, _ = torch.cuda.mem_get_info(DEV)
    for _ in range(2):
        _without_workspace(li, out)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info(DEV)
    assert torch.cuda.memory_allocated(DEV) == torch_before
    assert free_after == free_before
    _same(out, _with_workspace(li), wl.act_dtype)


def test_noalloc_status_word_reports_dropped_pairs():
    wl = LAYERS["g128"]
    weights = make_expert_weights(wl, DEV)
    li = make_layer_inputs(wl, 9, DEV, weights=weights, seed=31)
    li.topk_ids[4, 1] = wl.E + 3  # a host-made id outside [0, E): that pair is dropped
    out = torch.empty_like(li.hidden)
    _without_workspace(li, out)
    assert w.noalloc_read_status() & w.DEV_BAD_EXPERT_ID
    _same(out, _with_workspace(li), wl.act_dtype)
    # the next call resets the word
    li.topk_ids[4, 1] = 0
    _without_workspace(li, out)
    assert w.noalloc_read_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = w.load()
    # Mixtral-8x7B shapes at M = 1024 need far more than 64 MiB of workspace;
    # the call must refuse before touching any pointer (dummy aligned ones here).
    M, H, I, E, topk = 1024, 4096, 14336, 8, 2
    assert w.workspace_bytes(M, H, I, E, topk, 4, 128) > NOALLOC_BYTES
    p = ctypes.c_void_p(256)
    st = lib.wna16_fused_moe_noalloc(p, 0, M, H, I, E, topk, p, p, p, p, p, p, 0, 4, 128, p, p, p, 0, 0, None)
    assert st == WORKSPACE_TOO_SMALL
