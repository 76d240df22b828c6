"""Workload shapes and seeded input makers for the fused W4A16 / W8A16 MoE layer.

The layer shapes follow the models the pages on weight-quantized fused MoE
kernels run (vLLM PR #12185 "add triton fused moe kernel for gptq/awq":
DeepSeek-V3-AWQ decode and Qwen1.5-MoE-GPTQ; vLLM PR #6502 "Add Support for
GPTQ Fused MOE": Qwen2-57B-A14B-GPTQ-Int4; vLLM PR #14967 "Integrate Fused MoE
Kernels from AITER": Mixtral-8x7B). Inputs are synthetic: activations are
N(0, 0.1^2) like the benchmark script of vLLM PR #14138 ("randn / 10"), expert
weights are N(0, 0.02^2) and are quantized here before they reach the layer.

Nothing in this module dequantizes or multiplies: it draws numbers, rounds them
to codes/scales the way a GPTQ/AWQ-style quantizer would, and packs codes into
int32 words. The packed layout is the library's documented input format:

* ``q[e, n, w]`` int32 holds codes for ``k = w*pf .. w*pf+pf-1`` of output row
  ``n``, code of ``k`` in bits ``[bits*(k%pf), bits*(k%pf)+bits)`` (LSB first),
  ``pf = 32 // bits``;
* ``scales[e, g, n]`` (fp16 or bf16) is the scale of group ``g`` (K range
  ``[g*G, (g+1)*G)``) of row ``n``;
* ``zeros[e, g, w]`` int32 packs the integer zero points of rows
  ``w*pf .. w*pf+pf-1`` of group ``g`` with the same LSB-first rule; when there
  is no zeros tensor the zero point is ``2**(bits-1)``.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Optional

import torch

_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and recipe of one synthetic MoE layer."""

    name: str
    H: int  # hidden size (K of the gate/up GEMM, N of the down GEMM)
    I: int  # intermediate size per expert
    E: int  # number of experts
    topk: int
    bits: int  # 4 or 8
    has_zeros: bool  # asymmetric (integer zero points) or symmetric
    group_size: int  # -1 = one group per output channel (G = K)
    act_dtype: str  # "f16" | "bf16"
    scale_dtype: str  # "f16" | "bf16"
    routing: str  # "softmax_renorm" | "softmax" | "sigmoid_grouped"
    m_sweep: tuple = (4,)
    zipf_s: Optional[float] = None
    n_groups: int = 1  # expert groups for grouped sigmoid routing
    topk_groups: int = 1
    block: int = 0  # align block size pinned by the workload (0 = library choice)
    weight_std: float = 0.02
    act_std: float = 0.1

    def G(self, K: int) -> int:
        return K if self.group_size == -1 else self.group_size

    @property
    def pf(self) -> int:
        return 32 // self.bits

    def weight_bytes_per_expert(self) -> int:
        """Packed bytes of one expert: codes + scales + zeros of w13 and w2."""
        total = 0
        for N, K in ((2 * self.I, self.H), (self.H, self.I)):
            G = self.G(K)
            total += N * K * self.bits // 8
            total += (K // G) * N * 2
            if self.has_zeros:
                total += (K // G) * N * self.bits // 8
        return total


WORKLOADS = {
    "tiny": Workload(
        "tiny", H=256, I=512, E=8, topk=2, bits=4, has_zeros=True, group_size=128,
        act_dtype="f16", scale_dtype="f16", routing="softmax_renorm",
        m_sweep=(4,), block=16),
    "mixtral8x7b": Workload(
        "mixtral8x7b", H=4096, I=14336, E=8, topk=2, bits=4, has_zeros=True,
        group_size=128, act_dtype="f16", scale_dtype="f16", routing="softmax_renorm",
        m_sweep=(1, 16, 64, 256, 1024)),
    # GPTQ checkpoints store fp16 scales; a bf16 model loads them in its own dtype,
    # so the scales of this bf16 layer are bf16.
    "qwen2_57b": Workload(
        "qwen2_57b", H=3584, I=2560, E=64, topk=8, bits=4, has_zeros=False,
        group_size=128, act_dtype="bf16", scale_dtype="bf16", routing="softmax",
        m_sweep=(1, 8, 32, 128, 512), zipf_s=1.1),
    "deepseek_v3": Workload(
        "deepseek_v3", H=7168, I=2048, E=256, topk=8, bits=4, has_zeros=True,
        group_size=128, act_dtype="f16", scale_dtype="f16", routing="sigmoid_grouped",
        m_sweep=(1, 4, 16, 64, 256, 1024), n_groups=8, topk_groups=4),
    "mixtral8x22b_w8": Workload(
        "mixtral8x22b_w8", H=6144, I=16384, E=8, topk=2, bits=8, has_zeros=False,
        group_size=-1, act_dtype="bf16", scale_dtype="f16", routing="softmax_renorm",
        m_sweep=(8192,)),
}


def _seed(*parts) -> int:
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# ----------------------------------------------------------------------------
# routing (inputs of the layer: top-k expert ids and weights)
# ----------------------------------------------------------------------------

def make_router_logits(wl: Workload, M: int, seed: int) -> torch.Tensor:
    """Router logits [M, E] float32 on CPU: N(0, 1), plus log p_rank(e) for the
    Zipf-skewed workloads (p_r ~ r^-s over a seeded rank permutation)."""
    g = _gen(seed, "cpu")
    logits = torch.randn(M, wl.E, generator=g, dtype=torch.float64)
    if wl.zipf_s is not None:
        rank = torch.randperm(wl.E, generator=_gen(_seed(wl.name, "zipf"), "cpu")) + 1
        p = rank.double() ** (-wl.zipf_s)
        logits = logits + torch.log(p / p.sum())[None, :]
    return logits.float().contiguous()


def routing_params(wl: Workload) -> dict:
    """The workload's routing as keyword arguments of the routing call."""
    if wl.routing == "softmax_renorm":
        return dict(scoring="softmax", renormalize=True, n_groups=1, topk_groups=1)
    if wl.routing == "softmax":
        return dict(scoring="softmax", renormalize=False, n_groups=1, topk_groups=1)
    if wl.routing == "sigmoid_grouped":
        return dict(scoring="sigmoid", renormalize=True, n_groups=wl.n_groups, topk_groups=wl.topk_groups)
    raise ValueError(wl.routing)


def make_routing(wl: Workload, M: int, seed: int):
    """Router logits -> (topk_ids [M,k] int32, topk_weights [M,k] fp32), on CPU.

    softmax_renorm: softmax over the top-k logits (Mixtral style);
    softmax: softmax over all experts, keep the top-k probabilities as they are;
    sigmoid_grouped: sigmoid scores, group score = sum of the two best scores of
    each group, keep the best ``topk_groups`` groups, take the top-k experts in
    them, weights = score / sum of the selected scores (DeepSeek-V3 style).
    Zipf skew (Qwen2 workload): logits += log p_rank(e), p_r ~ r^-s with a seeded
    rank permutation, so a few experts get most tokens.
    """
    logits = make_router_logits(wl, M, seed).double()
    if wl.routing == "softmax_renorm":
        top, ids = torch.topk(logits, wl.topk, dim=-1)
        w = torch.softmax(top, dim=-1)
    elif wl.routing == "softmax":
        probs = torch.softmax(logits, dim=-1)
        w, ids = torch.topk(probs, wl.topk, dim=-1)
    elif wl.routing == "sigmoid_grouped":
        scores = torch.sigmoid(logits)
        gs = wl.E // wl.n_groups
        grp = scores.view(M, wl.n_groups, gs).topk(2, dim=-1).values.sum(-1)
        keep = grp.topk(wl.topk_groups, dim=-1).indices
        mask = torch.zeros(M, wl.n_groups, dtype=torch.bool)
        mask.scatter_(1, keep, True)
        masked = scores.masked_fill(~mask.repeat_interleave(gs, dim=1), -1.0)
        top, ids = torch.topk(masked, wl.topk, dim=-1)
        w = top / top.sum(-1, keepdim=True)
    else:
        raise ValueError(wl.routing)
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def make_biases(wl: Workload, seed: int, device="cpu", std: float = 0.05):
    """Per-expert biases in the activation dtype: w13 [E, 2I] (gate rows, then up
    rows) and w2 [E, H], N(0, std^2)."""
    g = _gen(seed, "cpu")
    dt = _TORCH_DTYPE[wl.act_dtype]
    b13 = (torch.randn(wl.E, 2 * wl.I, generator=g) * std).to(dt).to(device)
    b2 = (torch.randn(wl.E, wl.H, generator=g) * std).to(dt).to(device)
    return b13.contiguous(), b2.contiguous()


def make_hidden(wl: Workload, M: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(M, wl.H, generator=g, device=device, dtype=torch.float32) * wl.act_std
    return x.to(_TORCH_DTYPE[wl.act_dtype]).contiguous()


# ----------------------------------------------------------------------------
# quantization of one expert matrix into codes / scales / zero points
# ----------------------------------------------------------------------------

def _round_up_to(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Smallest representable value of ``dtype`` that is >= x (x > 0, fp32)."""
    y = x.to(dtype)
    low = y.to(torch.float32) < x
    bits = y.view(torch.int16)
    bits = torch.where(low, bits + 1, bits)  # positive values: next ulp up
    return bits.view(dtype)


def pack_along_last(codes: torch.Tensor, bits: int) -> torch.Tensor:
    """Pack unsigned codes (< 2**bits) along the last dim, LSB first, into int32."""
    pf = 32 // bits
    L = codes.shape[-1]
    assert L % pf == 0, (L, pf)
    c = codes.to(torch.int64).reshape(*codes.shape[:-1], L // pf, pf)
    shifts = torch.arange(pf, device=codes.device, dtype=torch.int64) * bits
    words = (c << shifts).sum(-1)
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words)
    return words.to(torch.int32).contiguous()


def quantize_expert(w: torch.Tensor, bits: int, has_zeros: bool, G: int,
                    scale_dtype: str):
    """Quantize one fp32 matrix ``w[N, K]`` group-wise along K.

    Returns (codes [N,K] int64, scales [K/G, N], zeros [K/G, N] int64 or None).
    asym: lo=min(min,0), hi=max(max,0), s=up((hi-lo)/(2^b-1)), z=rne(-lo/s),
          u=clamp(rne(w/s)+z, 0, 2^b-1).
    sym int4 (zero 8): s=up(2*absmax/15), u=clamp(rne(w/s)+8, 0, 15).
    sym int8: s=up(absmax/127), u=clamp(rne(w/s), -127, 127)+128.
    ``up`` rounds the scale up to the scale dtype so the clamp never cuts a value
    further than half a step.
    """
    N, K = w.shape
    assert K % G == 0
    qmax = (1 << bits) - 1
    wg = w.to(torch.float32).reshape(N, K // G, G)
    sdt = _TORCH_DTYPE[scale_dtype]
    if has_zeros:
        lo = wg.amin(-1).clamp(max=0.0)
        hi = wg.amax(-1).clamp(min=0.0)
        assert bool((hi > lo).all()), "degenerate quantization group"
        s = _round_up_to((hi - lo) / qmax, sdt)
        sf = s.to(torch.float32)
        z = torch.round(-lo / sf).clamp(0, qmax)
        u = (torch.round(wg / sf[..., None]) + z[..., None]).clamp(0, qmax)
        zeros = z.to(torch.int64).t().contiguous()
    else:
        amax = wg.abs().amax(-1)
        assert bool((amax > 0).all()), "degenerate quantization group"
        if bits == 4:
            s = _round_up_to(2.0 * amax / 15.0, sdt)
            sf = s.to(torch.float32)
            u = (torch.round(wg / sf[..., None]) + 8).clamp(0, 15)
        elif bits == 8:
            s = _round_up_to(amax / 127.0, sdt)
            sf = s.to(torch.float32)
            u = torch.round(wg / sf[..., None]).clamp(-127, 127) + 128
        else:
            raise ValueError(bits)
        zeros = None
    codes = u.to(torch.int64).reshape(N, K)
    return codes, s.t().contiguous(), zeros


def make_g_idx(K: int, G: int, seed: int) -> torch.Tensor:
    """Act-order groups (GPTQ desc_act): a seeded order of the K columns is cut
    into groups of G, so every group holds G columns spread over K."""
    order = torch.randperm(K, generator=_gen(seed, "cpu"))
    g = torch.empty(K, dtype=torch.int64)
    g[order] = torch.arange(K) // G
    return g


def quantize_expert_act_order(w: torch.Tensor, bits: int, has_zeros: bool, G: int, scale_dtype: str,
                              g_idx: torch.Tensor):
    """``quantize_expert`` with the groups of ``g_idx`` (columns k with
    g_idx[k] = g form group g): the columns are gathered group by group,
    quantized as contiguous groups, and the codes put back in the original
    column order. Scales / zeros stay [K/G, N] per group."""
    order = torch.argsort(g_idx, stable=True)
    codes, s, z = quantize_expert(w[:, order], bits, has_zeros, G, scale_dtype)
    back = torch.empty_like(codes)
    back[:, order] = codes
    return back, s, z


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class LayerInputs:
    wl: Workload
    M: int
    hidden: torch.Tensor  # [M, H] act dtype
    w13_q: torch.Tensor  # [E, 2I, H/pf] int32
    w13_s: torch.Tensor  # [E, H/G, 2I] scale dtype
    w13_z: Optional[torch.Tensor]  # [E, H/G, 2I/pf] int32
    w2_q: torch.Tensor  # [E, H, I/pf] int32
    w2_s: torch.Tensor  # [E, I/G, H]
    w2_z: Optional[torch.Tensor]  # [E, I/G, H/pf]
    topk_ids: torch.Tensor  # [M, k] int32
    topk_w: torch.Tensor  # [M, k] fp32

    @property
    def group_size(self) -> int:
        return self.wl.group_size

    def to(self, device) -> "LayerInputs":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, hidden=f(self.hidden), w13_q=f(self.w13_q), w13_s=f(self.w13_s),
            w13_z=f(self.w13_z), w2_q=f(self.w2_q), w2_s=f(self.w2_s), w2_z=f(self.w2_z),
            topk_ids=f(self.topk_ids), topk_w=f(self.topk_w))


def make_expert_weights(wl: Workload, device="cpu", experts=None):
    """Quantized, packed w13 and w2 of all experts (seeded per expert/matrix)."""
    H, I, E, bits, pf = wl.H, wl.I, wl.E, wl.bits, wl.pf
    out = {}
    for mat, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
        G = wl.G(K)
        q = torch.empty(E, N, K // pf, dtype=torch.int32, device=device)
        s = torch.empty(E, K // G, N, dtype=_TORCH_DTYPE[wl.scale_dtype], device=device)
        z = (torch.empty(E, K // G, N // pf, dtype=torch.int32, device=device)
             if wl.has_zeros else None)
        for e in range(E) if experts is None else experts:
            g = _gen(_seed(wl.name, wl.H, wl.I, e, mat), device)
            w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * wl.weight_std
            codes, sc, zc = quantize_expert(w, bits, wl.has_zeros, G, wl.scale_dtype)
            del w
            q[e] = pack_along_last(codes, bits)
            s[e] = sc
            if z is not None:
                z[e] = pack_along_last(zc, bits)
            del codes
        out[mat] = (q, s, z)
    return out


def make_layer_inputs(wl: Workload, M: int, device="cpu", weights=None,
                      seed: Optional[int] = None) -> LayerInputs:
    """Hidden states, routing and (unless given) quantized weights for M tokens."""
    seed = 1000 + M if seed is None else seed
    if weights is None:
        weights = make_expert_weights(wl, device)
    ids, tw = make_routing(wl, M, _seed(wl.name, "route", seed))
    x = make_hidden(wl, M, _seed(wl.name, "hidden", seed), device)
    (q13, s13, z13), (q2, s2, z2) = weights["w13"], weights["w2"]
    return LayerInputs(wl, M, x, q13, s13, z13, q2, s2, z2, ids.to(device), tw.to(device))

