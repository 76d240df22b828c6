"""Float64 oracle of the fused W4A16 / W8A16 Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library, and it imports nothing of
the library. It is deliberately plain: explicit shifts and masks, one float64
matrix-vector product per (token, slot), no blocking or fusion.

What it follows (the pages give prose, no formulas):

* vLLM PR #12185 "[Kernel] add triton fused moe kernel for gptq/awq": one fused
  MoE over GPTQ/AWQ int4 weights with per-group scales and zero points; its note
  1 on ``moe_align_block_size`` (per-expert grouping of (token, slot) pairs,
  padded to the GEMM block size, graph-safe);
* vLLM PR #6502 "[Model] Add Support for GPTQ Fused MOE", the bug report on
  ``BLOCK_SIZE_K`` versus the quantization group size: every K index uses the
  scale of its own group ``k // G``;
* vLLM ``fused_moe/oracle/int8.py`` (``int8_w8a16_moe_quant_config`` and the
  channel-strategy schema): int8 weights, symmetric, one scale per output
  channel;
* vLLM PR #14138 "optimize performance of gptq marlin kernel when n is small",
  benchmark script: ``quantize_weights(weight, uint4, group_size=128, zero
  points)`` and ``is_zp_float=False`` -> unsigned codes with integer zero points.

Stated readings where the pages are silent (each also listed in the design
notes): codes are packed LSB first along K in int32 words; scales are stored
group-major ``[E, K/G, N]``; zero points are the true integer zero, packed LSB
first along N ``[E, K/G, N/pf]``; without a zeros tensor the zero point is
``2**(bits-1)``; rows ``[0, I)`` of w13 are the gate projection and ``[I, 2I)``
the up projection; the activation is ``silu(gate) * up``; the output is the
top-k weighted sum in slot order, rounded once (round-to-nearest-even) to the
activation dtype. Pair ids outside ``[0, E)`` are dropped.

Half-precision inputs (fp16 or bf16 activations and scales) are passed as their
raw 16-bit patterns (``uint16`` arrays) with a dtype tag, so that bf16 needs no
library support and every conversion to float64 is exact.
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------


def halfbits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of raw fp16 or bf16 bit patterns."""
    b = np.asarray(bits).astype(np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def _round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (8 significant bits), nearest-even, once."""
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    m, e = np.frexp(np.where(finite, x, 0.0))  # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 keeps 8 significant bits for normals (exponent e-1 >= -126); below
    # that the spacing is fixed at 2**-133 (subnormals).
    normal = e - 1 >= -126
    with np.errstate(over="ignore", invalid="ignore"):
        r_norm = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
        r_sub = np.ldexp(np.rint(np.ldexp(np.where(normal, 0.0, x), 133)), -133)
    out = np.where(normal, r_norm, r_sub)
    out = np.where(finite, out, x)
    with np.errstate(over="ignore"):
        f32 = out.astype(np.float32)  # exact (8 significant bits) or +-inf
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def round_to_halfbits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 to fp16/bf16 (nearest-even, single rounding); raw bits."""
    if dtype == "f16":
        # numpy converts float64 -> float16 with one correctly rounded step.
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return _round_to_bf16_bits(x)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# unpack and dequantize
# ----------------------------------------------------------------------------


def unpack_codes(words: np.ndarray, bits: int) -> np.ndarray:
    """Codes from int32 words packed along the last axis, LSB first.

    code of element ``i`` = ``(word[i // pf] >> (bits * (i % pf))) & (2**bits - 1)``
    with ``pf = 32 // bits``.
    """
    pf = 32 // bits
    mask = (1 << bits) - 1
    w = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    out = np.empty(w.shape[:-1] + (w.shape[-1] * pf,), dtype=np.int64)
    for i in range(pf):
        out[..., i::pf] = (w >> (bits * i)) & mask
    return out


def unpack_zeros(zero_words: np.ndarray, bits: int) -> np.ndarray:
    """Integer zero points ``[..., K/G, N]`` from words packed along N."""
    return unpack_codes(zero_words, bits)


def dequantize_expert(q: np.ndarray, scales_bits: np.ndarray, zero_words, bits: int,
                      group_size: int, scale_dtype: str, g_idx=None) -> np.ndarray:
    """Float64 weights ``W[n, k] = (u[n, k] - z[g(k), n]) * s[g(k), n]``.

    ``q`` [N, K/pf] int32, ``scales_bits`` [K/G, N] raw half bits, ``zero_words``
    [K/G, N/pf] int32 or None (zero point ``2**(bits-1)``). ``group_size`` -1
    means one group per output channel (G = K). The group of k is ``k // G``,
    or with act-order (GPTQ ``desc_act``; vLLM PR #14138 passes the ``g_idx``
    tensor, empty there) ``g(k) = g_idx[k]``.
    """
    u = unpack_codes(q, bits)  # [N, K]
    N, K = u.shape
    G = K if group_size == -1 else group_size
    assert K % G == 0
    s = halfbits_to_f64(scales_bits, scale_dtype)  # [K/G, N]
    assert s.shape == (K // G, N), (s.shape, K, G, N)
    if zero_words is None:
        z = np.full((K // G, N), float(1 << (bits - 1)))
    else:
        z = unpack_zeros(zero_words, bits).astype(np.float64)  # [K/G, N]
        assert z.shape == (K // G, N)
    g_of_k = np.arange(K) // G if g_idx is None else np.asarray(g_idx, dtype=np.int64)
    assert g_of_k.shape == (K,) and g_of_k.min() >= 0 and g_of_k.max() < K // G
    return (u.astype(np.float64) - z.T[:, g_of_k]) * s.T[:, g_of_k]


def act_order_permutation(g_idx: np.ndarray):
    """K order that makes act-order groups contiguous: ``perm`` lists k by
    ascending group, ascending k within a group (a stable sort of ``g_idx``);
    ``inv[perm[i]] = i``. Returns (perm, inv) int32."""
    g = np.asarray(g_idx, dtype=np.int64)
    perm = np.array(sorted(range(g.size), key=lambda k: (g[k], k)), dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return perm.astype(np.int32), inv.astype(np.int32)


# ----------------------------------------------------------------------------
# checkpoint formats (vLLM PR #12185: the fused kernel's weight format "is
# just compatible with gptq/awq"; the formats themselves are those of the
# public GPTQ and AWQ packers, restated here)
# ----------------------------------------------------------------------------
#
# GPTQ: qweight [K/pf, N] int32, the codes of column n packed along K (word r
#   holds k = r*pf + j in bits [bits*j, +bits)); qzeros [K/G, N/pf] packed along
#   N the same way, storing z - 1 in the original format ("v1") and z itself in
#   the later one ("v2"); scales [K/G, N].
# AWQ (4-bit): qweight [K, N/8] int32 packed along N with the field order
#   AWQ_PACK_ORDER (field i of word c holds column 8c + AWQ_PACK_ORDER[i]);
#   qzeros [K/G, N/8] packed the same way; scales [K/G, N]; zero points stored
#   as they are.

AWQ_PACK_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


def _fields(words: np.ndarray, bits: int) -> np.ndarray:
    """[..., W] int32 words -> [..., W, 32/bits] fields, LSB first."""
    w = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    pf = 32 // bits
    shifts = bits * np.arange(pf)
    return (w[..., None] >> shifts) & ((1 << bits) - 1)


def unpack_gptq_qweight(qweight: np.ndarray, bits: int) -> np.ndarray:
    """GPTQ qweight [K/pf, N] -> codes [N, K]."""
    f = _fields(qweight, bits)  # [K/pf, N, pf]: field j of word (r, n) is k = r*pf + j
    Kw, N, pf = f.shape
    return np.transpose(f, (1, 0, 2)).reshape(N, Kw * pf)


def unpack_gptq_qzeros(qzeros: np.ndarray, bits: int, stored_minus_one: bool = True) -> np.ndarray:
    """GPTQ qzeros [K/G, N/pf] -> zero points [K/G, N] (v1 adds the 1 back, mod 2^bits)."""
    z = _fields(qzeros, bits).reshape(qzeros.shape[0], -1)
    return (z + 1) % (1 << bits) if stored_minus_one else z


def unpack_awq(words: np.ndarray) -> np.ndarray:
    """AWQ words [R, N/8] (4-bit, interleaved) -> values [R, N] in column order."""
    f = _fields(words, 4)  # [R, N/8, 8]: field i holds column 8c + AWQ_PACK_ORDER[i]
    out = np.empty_like(f)
    out[..., list(AWQ_PACK_ORDER)] = f
    return out.reshape(f.shape[0], -1)


# ----------------------------------------------------------------------------
# moe_align_block_size
# ----------------------------------------------------------------------------


def align_capacity(P: int, E: int, block: int) -> int:
    """Padded-slot capacity: at most min(P, E) experts are non-empty and each
    pads fewer than ``block`` slots; rounded up to a whole block."""
    raw = P + min(P, E) * (block - 1)
    return int(math.ceil(raw / block)) * block


def moe_align_block_size(topk_ids: np.ndarray, E: int, block: int):
    """Group (token, slot) pairs by expert, padded to the GEMM block size.

    Pair ``p = t * topk + j`` (row-major over ``topk_ids[M, topk]``).
    Returns ``(sorted_ids [cap], expert_ids [cap/block], num_post_pad, counts [E])``:
    ``cnt[e] = #{p : id_p = e}`` (ids outside [0, E) are dropped);
    ``padded[e] = ceil(cnt[e]/block) * block``; ``off[e] = sum_{e'<e} padded[e']``;
    ``sorted_ids[off[e] + r]`` is the r-th smallest pair with id e for r < cnt[e]
    and the sentinel ``P`` for the padding; ``expert_ids[b] = e`` for the blocks of
    expert e; slots at or past ``num_post_pad = sum padded`` hold ``P`` and
    their blocks ``-1``.
    """
    ids = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    P = ids.size
    cap = align_capacity(P, E, block)
    counts = np.zeros(E, dtype=np.int64)
    for p in range(P):
        if 0 <= ids[p] < E:
            counts[ids[p]] += 1
    padded = [((int(c) + block - 1) // block) * block for c in counts]
    offsets = [0] * E
    run = 0
    for e in range(E):
        offsets[e] = run
        run += padded[e]
    num_post_pad = run
    sorted_ids = np.full(cap, P, dtype=np.int32)
    fill = list(offsets)
    for p in range(P):  # ascending p: stable within each expert
        e = ids[p]
        if 0 <= e < E:
            sorted_ids[fill[e]] = p
            fill[e] += 1
    expert_ids = np.full(cap // block, -1, dtype=np.int32)
    for e in range(E):
        for b in range(offsets[e] // block, (offsets[e] + padded[e]) // block):
            expert_ids[b] = e
    return sorted_ids, expert_ids, int(num_post_pad), counts.astype(np.int32)


# ----------------------------------------------------------------------------
# routing: router logits -> top-k expert ids and weights
# ----------------------------------------------------------------------------
#
# The pages name top-k routing ids and weights as the first stage of the layer
# (the Mixtral, Qwen2-MoE and DeepSeek-V3 models of vLLM PR #12185 and PR #6502)
# but give no formulas. Stated readings:
# * softmax scores p_e = exp(l_e) / sum_e' exp(l_e'); sigmoid scores
#   s_e = 1 / (1 + exp(-l_e));
# * experts are ranked by logit, larger first, ties to the lower index, NaN
#   ranked as -inf (both score functions are increasing in the logit, so
#   this is the ranking by score, decided on the exact inputs);
# * grouped selection (DeepSeek-V3 style): experts split into n_groups equal
#   groups of consecutive ids; a group's score is the sum of the scores of its
#   two best-ranked experts; the topk_groups best groups are kept (larger score
#   first, ties to the lower group, NaN as -inf); the top-k experts are ranked
#   among the kept groups only;
# * weights: the selected scores, or with ``renormalize`` the selected scores
#   divided by their sum (for softmax, the softmax over the selected logits);
# * output slot j holds the j-th best selected expert.


def _rank_order(logits_row, allowed=None):
    """Expert indices, best first: larger logit, then lower index; NaN as -inf."""
    idx = range(len(logits_row)) if allowed is None else allowed

    def key(e):
        v = float(logits_row[e])
        return (math.inf if math.isnan(v) else -v, e)

    return sorted(idx, key=key)


def routing_scores(logits: np.ndarray, scoring: str) -> np.ndarray:
    """Softmax (over all experts of a row) or sigmoid scores, float64."""
    l = np.asarray(logits, dtype=np.float64)
    if scoring == "softmax":
        m = np.max(l, axis=-1, keepdims=True)
        ex = np.exp(l - m)
        return ex / np.sum(ex, axis=-1, keepdims=True)
    if scoring == "sigmoid":
        return 1.0 / (1.0 + np.exp(-l))
    raise ValueError(scoring)


def routing_group_scores(logits: np.ndarray, scoring: str, n_groups: int) -> np.ndarray:
    """[M, n_groups]: sum of the scores of the two best-ranked experts of each group."""
    l = np.asarray(logits, dtype=np.float64)
    M, E = l.shape
    gs = E // n_groups
    sc = routing_scores(l, scoring)
    out = np.zeros((M, n_groups), dtype=np.float64)
    for t in range(M):
        for g in range(n_groups):
            members = list(range(g * gs, (g + 1) * gs))
            best2 = _rank_order(l[t], members)[:2]
            out[t, g] = sc[t, best2[0]] + sc[t, best2[1]]
    return out


def topk_routing(logits: np.ndarray, topk: int, scoring: str = "softmax", renormalize: bool = True,
                 n_groups: int = 1, topk_groups: int = 1):
    """Router logits [M, E] -> (topk_ids [M, topk] int32, topk_weights [M, topk] float64).

    See the readings above. ``n_groups == 1`` is plain top-k; with
    ``n_groups > 1`` the group size E / n_groups must be at least 2.
    """
    l = np.asarray(logits, dtype=np.float64)
    M, E = l.shape
    if not (1 <= topk <= E) or E % n_groups:
        raise ValueError("bad routing shape")
    sc = routing_scores(l, scoring)
    gsc = routing_group_scores(l, scoring, n_groups) if n_groups > 1 else None
    gs = E // n_groups
    ids = np.zeros((M, topk), dtype=np.int32)
    w = np.zeros((M, topk), dtype=np.float64)
    for t in range(M):
        allowed = None
        if n_groups > 1:
            kept = sorted(range(n_groups),
                          key=lambda g: (math.inf if math.isnan(gsc[t, g]) else -gsc[t, g], g))[:topk_groups]
            allowed = [e for g in sorted(kept) for e in range(g * gs, (g + 1) * gs)]
        sel = _rank_order(l[t], allowed)[:topk]
        ids[t] = sel
        if renormalize and scoring == "softmax":
            ex = np.exp(l[t, sel] - l[t, sel[0]])
            w[t] = ex / ex.sum()
        elif renormalize:
            w[t] = sc[t, sel] / sc[t, sel].sum()
        else:
            w[t] = sc[t, sel]
    return ids, w


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def gated_activation(g: np.ndarray, u: np.ndarray, glu=None) -> np.ndarray:
    """The gate/up activation.

    ``glu`` None: silu(g) * u. ``glu = (alpha, beta, limit)`` (the clamped SwiGLU
    that vLLM's int8 MoE config passes as swiglu_alpha / swiglu_beta /
    swiglu_limit, with no formula on the pages; the reading taken): with
    limit > 0, g' = min(g, limit) and u' = clamp(u, -limit, limit), else g' = g,
    u' = u; result g' * sigmoid(alpha * g') * (u' + beta). alpha = 1, beta = 0
    and no limit give silu(g) * u.
    """
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    if glu is None:
        return silu(g) * u
    alpha, beta, limit = (float(v) for v in glu)
    if limit > 0:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return g / (1.0 + np.exp(-alpha * g)) * (u + beta)


def _bias(L, key, e, dtype):
    b = L.get(key)
    return None if b is None else halfbits_to_f64(b[e], dtype)


def _expert_matrices(L, e, cache):
    if e not in cache:
        g13 = L.get("w13_g_idx")
        g2 = L.get("w2_g_idx")
        w13 = dequantize_expert(L["w13_q"][e], L["w13_s"][e],
                                None if L["w13_z"] is None else L["w13_z"][e],
                                L["bits"], L["group_size"], L["scale_dtype"], None if g13 is None else g13[e])
        w2 = dequantize_expert(L["w2_q"][e], L["w2_s"][e],
                               None if L["w2_z"] is None else L["w2_z"][e],
                               L["bits"], L["group_size"], L["scale_dtype"], None if g2 is None else g2[e])
        cache[e] = (w13, w2)
    return cache[e]


def _round_intermediate(a: np.ndarray, dtype: str) -> np.ndarray:
    """The activation rounded once to the activation dtype (nearest-even), as a
    kernel that stores it in that dtype between the GEMMs would see it."""
    return halfbits_to_f64(round_to_halfbits(a, dtype), dtype)


def fused_moe_per_token(L: dict, tokens=None, round_output=True, round_intermediate=False):
    """The layer, one (token, slot) at a time, in float64.

    ``L`` holds: ``x`` [M, H] raw half bits, ``act_dtype``, ``w13_q`` [E, 2I, H/pf],
    ``w13_s`` [E, H/G, 2I] raw bits, ``w13_z`` [E, H/G, 2I/pf] or None, ``w2_q``
    [E, H, I/pf], ``w2_s`` [E, I/G, H], ``w2_z`` [E, I/G, H/pf] or None,
    ``scale_dtype``, ``bits``, ``group_size``, ``topk_ids`` [M, k], ``topk_w`` [M, k]
    float32; optional ``w13_b`` [E, 2I] / ``w2_b`` [E, H] raw half bits of the
    activation dtype (biases), ``glu`` (see :func:`gated_activation`) and
    ``w13_g_idx`` [E, H] / ``w2_g_idx`` [E, I] (act-order groups, original K
    order; see :func:`dequantize_expert`). For each
    token t and slot j with expert e = ids[t, j] in [0, E):
    g = W13[e, :I] x_t + b13[e, :I], u = W13[e, I:] x_t + b13[e, I:],
    a = act(g, u), y = W2[e] a + b2[e]; out_t = sum_j w[t, j] y_{t,j} in slot
    order. Returns float64 [T, H], or the raw half bits of its single rounding
    when ``round_output``. ``round_intermediate`` (diagnosis only, off for
    parity) rounds ``a`` to the activation dtype before the down projection.
    """
    x = halfbits_to_f64(L["x"], L["act_dtype"])
    ids = np.asarray(L["topk_ids"])
    tw = np.asarray(L["topk_w"], dtype=np.float32).astype(np.float64)
    M, k = ids.shape
    E = L["w13_q"].shape[0]
    I = L["w13_q"].shape[1] // 2
    H = x.shape[1]
    tokens = range(M) if tokens is None else tokens
    cache = {}
    rows = []
    for t in tokens:
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            e = int(ids[t, j])
            if not (0 <= e < E):
                continue
            w13, w2 = _expert_matrices(L, e, cache)
            gu = w13 @ x[t]
            b13 = _bias(L, "w13_b", e, L["act_dtype"])
            if b13 is not None:
                gu = gu + b13
            a = gated_activation(gu[:I], gu[I:], L.get("glu"))
            if round_intermediate:
                a = _round_intermediate(a, L["act_dtype"])
            y = w2 @ a
            b2 = _bias(L, "w2_b", e, L["act_dtype"])
            if b2 is not None:
                y = y + b2
            acc = acc + tw[t, j] * y
        rows.append(acc)
    out = np.stack(rows) if rows else np.zeros((0, H))
    return round_to_halfbits(out, L["act_dtype"]) if round_output else out


def fused_moe_grouped(L: dict, round_output=True, round_intermediate=False):
    """Same layer, grouped per expert: dequantize one expert at a time and run
    one float64 matrix product over all of its routed (token, slot) pairs.
    Identical mathematics to :func:`fused_moe_per_token`; only the loop order
    differs (the per-slot terms are still added in slot order)."""
    x = halfbits_to_f64(L["x"], L["act_dtype"])
    ids = np.asarray(L["topk_ids"])
    tw = np.asarray(L["topk_w"], dtype=np.float32).astype(np.float64)
    M, k = ids.shape
    E = L["w13_q"].shape[0]
    I = L["w13_q"].shape[1] // 2
    H = x.shape[1]
    y = np.zeros((M, k, H), dtype=np.float64)
    for e in range(E):
        tt, jj = np.nonzero(ids == e)
        if tt.size == 0:
            continue
        w13, w2 = _expert_matrices(L, e, {})
        gu = x[tt] @ w13.T
        b13 = _bias(L, "w13_b", e, L["act_dtype"])
        if b13 is not None:
            gu = gu + b13[None, :]
        a = gated_activation(gu[:, :I], gu[:, I:], L.get("glu"))
        if round_intermediate:
            a = _round_intermediate(a, L["act_dtype"])
        ye = a @ w2.T
        b2 = _bias(L, "w2_b", e, L["act_dtype"])
        if b2 is not None:
            ye = ye + b2[None, :]
        y[tt, jj] = ye * tw[tt, jj][:, None]
    out = np.zeros((M, H), dtype=np.float64)
    for j in range(k):
        out = out + y[:, j]
    return round_to_halfbits(out, L["act_dtype"]) if round_output else out
