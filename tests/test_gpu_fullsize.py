"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic block size and K split).

The float64 oracle cannot run whole full-size batches in test time, so:
* sampled outputs: two tokens of the largest batch of each workload (the last
  token, which sits in the ragged tail of its expert blocks, and the first)
  are computed one by one by the oracle and compared element by element
  (max |y - r| / max |r| <= 1e-2 over their rows);
* a property that holds at any size: a token's output does not depend on the
  batch it is in. Every M of the workload's sweep is run and each token's row
  is compared with the same token computed alone (M = 1) or in the largest
  batch, within the same tolerance.
The alignment outputs at these sizes are checked bit-exactly against the
oracle in test_gpu_align.py.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, make_expert_weights, make_layer_inputs
from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2
FULL = ["mixtral8x7b", "qwen2_57b", "deepseek_v3", "mixtral8x22b_w8"]


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _run(li):
    return w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, li.topk_ids,
                       li.topk_w, li.wl.bits, li.wl.group_size)


def _oracle_rows(li, tokens):
    """Oracle rows for `tokens`, moving only the experts they route to."""
    ids = li.topk_ids[tokens].cpu()
    experts = sorted(set(int(e) for e in ids.flatten().tolist()))
    ex = torch.tensor(experts, dtype=torch.long, device=li.w13_q.device)
    remap = {e: i for i, e in enumerate(experts)}
    pick = lambda t: None if t is None else t.index_select(0, ex)
    sub = li.__class__(li.wl, len(tokens), li.hidden[tokens], pick(li.w13_q), pick(li.w13_s), pick(li.w13_z),
                       pick(li.w2_q), pick(li.w2_s), pick(li.w2_z),
                       torch.tensor([[remap[int(e)] for e in row] for row in ids.tolist()], dtype=torch.int32),
                       li.topk_w[tokens].cpu())
    L = oracle_layer_dict(sub)
    return bits_to_f64(oracle.fused_moe_per_token(L), li.wl.act_dtype)


@pytest.mark.parametrize("name", FULL)
def test_full_size(name):
    wl = WORKLOADS[name]
    weights = make_expert_weights(wl, DEV)
    dt = wl.act_dtype
    M_big = max(wl.m_sweep)
    big = make_layer_inputs(wl, M_big, DEV, weights=weights)
    y_big = bits_to_f64(halfbits(_run(big)), dt)
    assert np.all(np.isfinite(y_big))
    # sampled outputs against the oracle
    tokens = [M_big - 1, 0] if M_big > 1 else [0]
    ref = _oracle_rows(big, tokens)
    assert max_rel_err(y_big[tokens], ref) <= TOL, name
    # batch invariance over the sweep: every token of every smaller batch equals
    # the same token (same hidden row, same routing) inside the largest batch
    for M in wl.m_sweep:
        if M == M_big:
            continue
        li = make_layer_inputs(wl, M, DEV, weights=weights)
        y = bits_to_f64(halfbits(_run(li)), dt)
        alone = []
        for t in range(min(M, 4)):
            one = li.__class__(wl, 1, li.hidden[t:t + 1].contiguous(), li.w13_q, li.w13_s, li.w13_z, li.w2_q,
                               li.w2_s, li.w2_z, li.topk_ids[t:t + 1].contiguous(), li.topk_w[t:t + 1].contiguous())
            alone.append(bits_to_f64(halfbits(_run(one)), dt)[0])
        assert max_rel_err(y[: len(alone)], np.stack(alone)) <= TOL, (name, M)
    del weights, big
    torch.cuda.empty_cache()
