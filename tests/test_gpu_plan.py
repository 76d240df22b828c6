"""GPU checks of the plan entry points (wna16_plan_create / wna16_fused_moe_plan):
a plan built once for a set of weights must give, call after call and for
batches of different sizes, exactly the output of wna16_fused_moe on the same
inputs (same kernels, same launch plan, so bit for bit), and the float64 oracle
within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, Workload, make_expert_weights, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2

LAYERS = [
    WORKLOADS["tiny"],
    Workload("plan_sym_bf16", H=512, I=768, E=16, topk=4, bits=4, has_zeros=False, group_size=128,
             act_dtype="bf16", scale_dtype="bf16", routing="softmax"),
    Workload("plan_w8", H=384, I=512, E=8, topk=2, bits=8, has_zeros=False, group_size=-1,
             act_dtype="bf16", scale_dtype="f16", routing="softmax_renorm"),
]
DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


@pytest.mark.parametrize("wl", LAYERS, ids=lambda x: x.name)
def test_plan_matches_fused_call_and_oracle(wl):
    weights = make_expert_weights(wl, DEV)
    (q13, s13, z13), (q2, s2, z2) = weights["w13"], weights["w2"]
    plan = w.Plan(q13, s13, z13, q2, s2, z2, wl.bits, wl.group_size, wl.topk, act_dtype=DT[wl.act_dtype])
    for M, seed in ((1, 5), (37, 6), (200, 7), (37, 8)):
        li = make_layer_inputs(wl, M, DEV, weights=weights, seed=seed)
        ws = torch.empty(plan.workspace_bytes(M), dtype=torch.uint8, device=DEV)
        out = torch.empty_like(li.hidden)
        plan(li.hidden, li.topk_ids, li.topk_w, out, ws)
        ref = w.fused_moe(li.hidden, q13, s13, z13, q2, s2, z2, li.topk_ids, li.topk_w, wl.bits, wl.group_size)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (wl.name, M)
        if M <= 37:
            r = bits_to_f64(oracle.fused_moe_per_token(oracle_layer_dict(li)), wl.act_dtype)
            assert max_rel_err(bits_to_f64(halfbits(out), wl.act_dtype), r) <= TOL


def test_plan_rejects_bad_weights():
    wl = WORKLOADS["tiny"]
    weights = make_expert_weights(wl, DEV)
    (q13, s13, z13), (q2, s2, z2) = weights["w13"], weights["w2"]
    with pytest.raises((w.WNA16Error, ValueError)):
        w.Plan(q13, s13, z13, q2, s2, z2, wl.bits, 96, wl.topk)  # group size 96: unsupported
    with pytest.raises(ValueError):
        w.Plan(q13, s13, None, q2, s2, z2, wl.bits, wl.group_size, wl.topk)  # zeros for one projection only
