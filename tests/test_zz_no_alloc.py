"""GPU check of wna16_fused_moe_noalloc, the entry point for callers that have
no allocator to give the library a workspace (a plain C host program, or a
plugin inside a process whose memory manager owns the device memory and would
be bypassed by an extra cudaMalloc). It must produce what the ordinary entry
point produces, call after call, although every call reuses one library-owned
scratch area that still holds the previous call's data.

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


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _layer():
    return Workload("noalloc", H=384, I=640, E=8, topk=2, bits=4, has_zeros=True, group_size=128,
                    act_dtype="f16", scale_dtype="f16", routing="softmax_renorm")


def _with_workspace(li):
    return w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids,
                       li.topk_w, li.wl.bits, li.wl.group_size)


def _without_workspace(li):
    out = torch.empty_like(li.hidden)
    return w.fused_moe_noalloc(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z,
                               li.topk_ids, li.topk_w, li.wl.bits, li.wl.group_size, out)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    wl = _layer()
    weights = make_expert_weights(wl, DEV)
    # two calls in a row with different batches: the second finds the first
    # call's data in the shared scratch area
    for M, seed in ((37, 11), (5, 12)):
        li = make_layer_inputs(wl, M, DEV, weights=weights, seed=seed)
        need = w.workspace_bytes(M, wl.H, wl.I, wl.E, wl.topk, wl.bits, wl.group_size)
        assert need <= NOALLOC_BYTES
        got = _without_workspace(li)
        ref = _with_workspace(li)
        torch.cuda.synchronize()
        g = bits_to_f64(halfbits(got), "f16")
        r = bits_to_f64(halfbits(ref), "f16")
        assert max_rel_err(g, r) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = w.load()
    # Mixtral-8x7B shapes at M = 1024 need far more than 64 MiB of workspace;
    # the call must refuse before touching any pointer (dummy aligned ones here).
    M, H, I, E, topk = 1024, 4096, 14336, 8, 2
    assert w.workspace_bytes(M, H, I, E, topk, 4, 128) > NOALLOC_BYTES
    p = ctypes.c_void_p(256)
    st = lib.wna16_fused_moe_noalloc(p, 0, M, H, I, E, topk, p, p, p, p, p, p, 0, 4, 128, p, p, p, 0, 0, None)
    assert st == WORKSPACE_TOO_SMALL
