"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic block size and K split).

The float64 oracle cannot run whole full-size batches in test time, so:
* sampled outputs: two tokens of the largest batch of each workload (the last
  token, which sits in the ragged tail of its expert blocks, and the first)
  are computed one by one by the oracle and compared element by element
  (max |y - r| / max |r| <= 1e-2 over their rows);
* the same at the decode-sized batches the benchmark reports, which run the
  16- and 32-token deferred-scale kernels over the whole K of every workload
  (their per-stage partial sums and correction MMAs at full length): first,
  middle and last token against the oracle;
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
    """Oracle rows for `tokens`, moving only the experts they route to (one
    token at a time, so at most top-k dequantized experts are held)."""
    if len(tokens) > 1:
        return np.concatenate([_oracle_rows(li, [t]) for t in tokens])
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


# (workload, M): the decode points of the benchmark's sweep, in the launch
# configuration it times. Mixtral-8x7B M=1 runs the 16-token deferred kernel
# with the down GEMM split over K (ordered fp32 slab); M=16 and Qwen2-57B M=8 /
# DeepSeek-V3 M=16 the 16-token deferred kernel over K = 4096, 3584 and 7168
# (32, 28 and 56 stages of per-stage partial sums), DeepSeek-V3 M=1 / 64 too;
# Mixtral-8x7B M=64 and Qwen2-57B M=128 the 32-token deferred tile.
DECODE_POINTS = [("mixtral8x7b", 1), ("mixtral8x7b", 16), ("mixtral8x7b", 64), ("qwen2_57b", 8),
                 ("qwen2_57b", 128), ("deepseek_v3", 1), ("deepseek_v3", 16), ("deepseek_v3", 64)]


@pytest.fixture(scope="module")
def weight_cache():
    cache = {}
    yield cache
    cache.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,M", DECODE_POINTS)
def test_decode_points_vs_oracle(name, M, weight_cache):
    wl = WORKLOADS[name]
    if name not in weight_cache:
        weight_cache.clear()
        torch.cuda.empty_cache()
        weight_cache[name] = make_expert_weights(wl, DEV)
    li = make_layer_inputs(wl, M, DEV, weights=weight_cache[name])
    block = w.choose_block(M, wl.topk, wl.E)
    assert block in (16, 32), (name, M, block)  # the deferred-scale kernel's tiles
    y = bits_to_f64(halfbits(_run(li)), wl.act_dtype)
    assert np.all(np.isfinite(y))
    tokens = sorted({0, M // 2, M - 1})
    ref = _oracle_rows(li, tokens)
    err = max_rel_err(y[tokens], ref)
    assert err <= TOL, (name, M, block, err)
