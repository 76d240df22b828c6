"""The failure path on the GPU, without a fault: a bounded pipeline wait that
nothing completes gives up, reports WNA16_DEV_TIMEOUT in the status word, the
CTA's other waiting role leaves through the abort flag, and the context stays
usable for the next layer call."""
import time

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def test_bounded_wait_gives_up_reports_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    roles = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    w.check_wait_timeout(status, roles)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert w.read_device_status(status) & w.DEV_TIMEOUT
    assert int(roles.item()) == 2  # both waiting warps left
    assert 1.0 < dt < 30.0  # about one wait bound (2 s), no longer
    # the next layer call runs normally and its own status word is clean
    wl = WORKLOADS["tiny"]
    li = make_layer_inputs(wl, 4).to(DEV)
    ws = torch.empty(w.workspace_bytes(4, wl.H, wl.I, wl.E, wl.topk, wl.bits, wl.group_size), dtype=torch.uint8,
                     device=DEV)
    y = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids, li.topk_w,
                    wl.bits, wl.group_size, workspace=ws)
    torch.cuda.synchronize()
    assert w.read_device_status(ws[:4].view(torch.int32)) == 0
    ref = oracle.fused_moe_per_token(oracle_layer_dict(li))
    assert max_rel_err(bits_to_f64(halfbits(y), wl.act_dtype), bits_to_f64(ref, wl.act_dtype)) <= 1e-2


def test_bad_status_pointer_is_rejected_on_the_host():
    with pytest.raises(ValueError):
        w.check_wait_timeout(torch.zeros(2, dtype=torch.int32, device=DEV))
