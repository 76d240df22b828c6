"""Thin ctypes binding of ``include/wna16_moe.h``.

Argument marshalling only: each function checks the torch tensors it is given
(device, dtype, shape, contiguity), passes their device pointers and the
current CUDA stream to the C ABI, and raises on a non-OK status. Every step of
the layer runs in the library's CUDA kernels; there is no other code path. If
the library has not been built this module raises instead of computing
anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB

WNA16_OK = 0
STATUS_NAMES = {
    0: "WNA16_OK", 1: "WNA16_ERR_INVALID_ARG", 2: "WNA16_ERR_UNSUPPORTED",
    3: "WNA16_ERR_WORKSPACE_TOO_SMALL", 4: "WNA16_ERR_CUDA",
    5: "WNA16_ERR_DEVICE_BAD_EXPERT_ID", 6: "WNA16_ERR_DEVICE_TIMEOUT", 7: "WNA16_ERR_DEVICE_BAD_GROUPS",
}
DEV_BAD_EXPERT_ID = 0x1
DEV_TIMEOUT = 0x2
DEV_BAD_GROUPS = 0x4

# Every symbol include/wna16_moe.h declares.
EXPORTED = (
    "wna16_align_capacity", "wna16_moe_align_block_size", "wna16_choose_block",
    "wna16_fused_moe_workspace_bytes", "wna16_fused_moe", "wna16_fused_moe_timed",
    "wna16_fused_moe_noalloc", "wna16_prepack_bytes", "wna16_prepack", "wna16_fused_moe_prepacked",
    "wna16_read_device_status", "wna16_status_string", "wna16_topk_routing", "wna16_fused_moe_ex",
    "wna16_fused_moe_prepacked_ex", "wna16_act_order_prepare", "wna16_convert_checkpoint",
    "wna16_check_wait_timeout", "wna16_noalloc_read_status", "wna16_check_launch_plan",
    "wna16_plan_create", "wna16_plan_destroy", "wna16_fused_moe_plan",
)

_DTYPE = {torch.float16: 0, torch.bfloat16: 1}
_LOGIT_DTYPE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
_SCORING = {"softmax": 0, "sigmoid": 1}


class MoeOptions(ctypes.Structure):
    """``wna16_moe_options``: biases and the gate/up activation."""
    _fields_ = [("w13_bias", ctypes.c_void_p), ("w2_bias", ctypes.c_void_p), ("activation", ctypes.c_int),
                ("swiglu_alpha", ctypes.c_float), ("swiglu_beta", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("w13_perm", ctypes.c_void_p), ("w2_inv_perm", ctypes.c_void_p),
                ("router_logits", ctypes.c_void_p), ("logits_dtype", ctypes.c_int), ("scoring", ctypes.c_int),
                ("renormalize", ctypes.c_int), ("n_groups", ctypes.c_int), ("topk_groups", ctypes.c_int),
                ("routed_ids", ctypes.c_void_p), ("routed_weights", ctypes.c_void_p),
                ("atomic_reduce", ctypes.c_int)]


_ACTIVATION = {"silu": 0, "swiglu_clamp": 1}


def _options(hidden, E, I, H, w13_bias, w2_bias, activation, swiglu, w13_perm=None, w2_inv_perm=None,
             atomic_reduce=False):
    """A MoeOptions for the given variant, or None for the default layer."""
    if (w13_bias is None and w2_bias is None and activation == "silu" and w13_perm is None and w2_inv_perm is None
            and not atomic_reduce):
        return None
    if activation not in _ACTIVATION:
        raise ValueError(f"activation must be one of {tuple(_ACTIVATION)}")
    dev = hidden.device
    if w13_bias is not None:
        _check(w13_bias, "w13_bias", hidden.dtype, (E, 2 * I), dev)
    if w2_bias is not None:
        _check(w2_bias, "w2_bias", hidden.dtype, (E, H), dev)
    if w13_perm is not None:
        _check(w13_perm, "w13_perm", torch.int32, (E, H), dev)
    if w2_inv_perm is not None:
        _check(w2_inv_perm, "w2_inv_perm", torch.int32, (E, I), dev)
    alpha, beta, limit = swiglu
    opt = MoeOptions(None if w13_bias is None else w13_bias.data_ptr(),
                     None if w2_bias is None else w2_bias.data_ptr(), _ACTIVATION[activation],
                     float(alpha), float(beta), float(limit),
                     None if w13_perm is None else w13_perm.data_ptr(),
                     None if w2_inv_perm is None else w2_inv_perm.data_ptr())
    opt.atomic_reduce = 1 if atomic_reduce else 0
    return opt


class WNA16Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Loads the built library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(
            f"CUDA library not built ({LIB}); run `python -m weight_quantized_moe_align_gb300.build`")
    L = ctypes.CDLL(LIB)
    c = ctypes
    vp, i64, i32, sz = c.c_void_p, c.c_int64, c.c_int, c.c_size_t
    L.wna16_align_capacity.argtypes = [i64, i32, i32]
    L.wna16_align_capacity.restype = i64
    L.wna16_choose_block.argtypes = [i64, i32, i32]
    L.wna16_choose_block.restype = i32
    L.wna16_moe_align_block_size.argtypes = [vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.wna16_moe_align_block_size.restype = i32
    L.wna16_fused_moe_workspace_bytes.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32]
    L.wna16_fused_moe_workspace_bytes.restype = sz
    L.wna16_fused_moe.argtypes = [vp, i32, i64, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, i32, i32,
                                  i32, vp, vp, vp, vp, sz, i32, i32, vp]
    L.wna16_fused_moe.restype = i32
    L.wna16_fused_moe_timed.argtypes = L.wna16_fused_moe.argtypes + [vp]
    L.wna16_fused_moe_timed.restype = i32
    L.wna16_fused_moe_noalloc.argtypes = L.wna16_fused_moe.argtypes[:19] + [i32, i32, vp]
    L.wna16_fused_moe_noalloc.restype = i32
    L.wna16_noalloc_read_status.argtypes = [c.POINTER(c.c_int32), vp]
    L.wna16_noalloc_read_status.restype = i32
    L.wna16_prepack_bytes.argtypes = [i32, i64, i64, i32, i32, i32, i32]
    L.wna16_prepack_bytes.restype = sz
    L.wna16_prepack.argtypes = [vp, vp, vp, i32, i64, i64, i32, i32, i32, vp, vp]
    L.wna16_prepack.restype = i32
    L.wna16_fused_moe_prepacked.argtypes = [vp, i32, i64, i64, i64, i32, i32, vp, vp, i32, i32, i32, i32, vp, vp,
                                            vp, vp, sz, i32, i32, vp, vp]
    L.wna16_fused_moe_prepacked.restype = i32
    L.wna16_read_device_status.argtypes = [vp, c.POINTER(c.c_int32), vp]
    L.wna16_read_device_status.restype = i32
    L.wna16_fused_moe_ex.argtypes = L.wna16_fused_moe_timed.argtypes + [vp]
    L.wna16_fused_moe_ex.restype = i32
    L.wna16_fused_moe_prepacked_ex.argtypes = L.wna16_fused_moe_prepacked.argtypes + [vp]
    L.wna16_fused_moe_prepacked_ex.restype = i32
    L.wna16_check_wait_timeout.argtypes = [vp, vp, vp]
    L.wna16_check_wait_timeout.restype = i32
    L.wna16_convert_checkpoint.argtypes = [i32, vp, vp, i32, i64, i64, i32, i32, vp, vp, vp]
    L.wna16_convert_checkpoint.restype = i32
    L.wna16_act_order_prepare.argtypes = [vp, vp, i32, i64, i64, i32, i32, vp, vp, vp, vp, vp]
    L.wna16_act_order_prepare.restype = i32
    L.wna16_topk_routing.argtypes = [vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.wna16_topk_routing.restype = i32
    L.wna16_check_launch_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp,
                                          vp, c.c_int32, c.c_char_p, sz]
    L.wna16_check_launch_plan.restype = i64
    L.wna16_plan_create.argtypes = [i32, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                    c.POINTER(vp)]
    L.wna16_plan_create.restype = i32
    L.wna16_plan_destroy.argtypes = [vp]
    L.wna16_plan_destroy.restype = None
    L.wna16_fused_moe_plan.argtypes = [vp, vp, i64, vp, vp, vp, vp, sz, i32, i32, vp]
    L.wna16_fused_moe_plan.restype = i32
    L.wna16_status_string.argtypes = [i32]
    L.wna16_status_string.restype = c.c_char_p
    _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _raise(st: int, what: str):
    if st != WNA16_OK:
        raise WNA16Error(st, what)


def align_capacity(num_pairs: int, E: int, block: int) -> int:
    return int(load().wna16_align_capacity(num_pairs, E, block))


def choose_block(M: int, topk: int, E: int) -> int:
    return int(load().wna16_choose_block(M, topk, E))


def workspace_bytes(M, H, I, E, topk, bits, group_size, block=0, split_k=0) -> int:
    n = int(load().wna16_fused_moe_workspace_bytes(M, H, I, E, topk, bits, group_size, block, split_k))
    if n == 0 and M > 0:
        raise WNA16Error(1, "wna16_fused_moe_workspace_bytes")
    return n


def topk_routing(logits: torch.Tensor, topk: int, scoring: str = "softmax", renormalize: bool = True,
                 n_groups: int = 1, topk_groups: int = 1, topk_ids: Optional[torch.Tensor] = None,
                 topk_weights: Optional[torch.Tensor] = None, stream=None):
    """Router logits [M, E] (fp32/fp16/bf16) -> (topk_ids [M, topk] int32,
    topk_weights [M, topk] fp32) by ``wna16_topk_routing``."""
    _check(logits, "logits", tuple(_LOGIT_DTYPE))
    if logits.dim() != 2:
        raise ValueError("logits must be [M, E]")
    if scoring not in _SCORING:
        raise ValueError(f"scoring must be one of {tuple(_SCORING)}")
    M, E = logits.shape
    dev = logits.device
    if topk_ids is None:
        topk_ids = torch.empty(M, topk, dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty(M, topk, dtype=torch.float32, device=dev)
    _check(topk_ids, "topk_ids", torch.int32, (M, topk), dev)
    _check(topk_weights, "topk_weights", torch.float32, (M, topk), dev)
    st = load().wna16_topk_routing(_ptr(logits), _LOGIT_DTYPE[logits.dtype], M, E, topk, _SCORING[scoring],
                                   int(bool(renormalize)), n_groups, topk_groups, _ptr(topk_ids),
                                   _ptr(topk_weights), _stream(stream))
    _raise(st, "wna16_topk_routing")
    return topk_ids, topk_weights


def moe_align_block_size(topk_ids: torch.Tensor, E: int, block: int, with_counts=True,
                         status: Optional[torch.Tensor] = None, out=None, stream=None):
    """Returns (sorted_ids [cap], expert_ids [cap/block], num_tokens_post_padded [1],
    expert_counts [E] or None) as int32 CUDA tensors."""
    _check(topk_ids, "topk_ids", torch.int32)
    if topk_ids.dim() != 2:
        raise ValueError("topk_ids must be [M, topk]")
    M, topk = topk_ids.shape
    dev = topk_ids.device
    cap = align_capacity(M * topk, E, block)
    if cap < 0:
        raise WNA16Error(1, "wna16_align_capacity")
    if out is None:
        sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        expert_ids = torch.empty(max(cap // block, 1), dtype=torch.int32, device=dev)
        npp = torch.empty(1, dtype=torch.int32, device=dev)
        counts = torch.empty(E, dtype=torch.int32, device=dev) if with_counts else None
    else:
        sorted_ids, expert_ids, npp, counts = out
    if status is not None:
        _check(status, "status", torch.int32, device=dev)
    st = load().wna16_moe_align_block_size(_ptr(topk_ids), M, topk, E, block, _ptr(sorted_ids),
                                           _ptr(expert_ids), _ptr(npp), _ptr(counts), _ptr(status),
                                           _stream(stream))
    _raise(st, "wna16_moe_align_block_size")
    return sorted_ids[:cap], expert_ids[: cap // block], npp, counts


def fused_moe(hidden: torch.Tensor, w13_q: torch.Tensor, w13_scales: torch.Tensor,
              w13_zeros: Optional[torch.Tensor], w2_q: torch.Tensor, w2_scales: torch.Tensor,
              w2_zeros: Optional[torch.Tensor], topk_ids: torch.Tensor, topk_weights: torch.Tensor,
              bits: int, group_size: int, out: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, block: int = 0, split_k: int = 0,
              stream=None, events=None, w13_bias: Optional[torch.Tensor] = None,
              w2_bias: Optional[torch.Tensor] = None, activation: str = "silu",
              swiglu=(1.702, 1.0, 7.0), w13_perm: Optional[torch.Tensor] = None,
              w2_inv_perm: Optional[torch.Tensor] = None, atomic_reduce: bool = False) -> torch.Tensor:
    """The fused layer (see include/wna16_moe.h). Returns ``out`` [M, H].

    ``events``: optional list of 6 ``torch.cuda.Event`` (or None; each must
    already exist on the device, i.e. have been recorded once) recorded before
    the align, gather, gate/up GEMM, down GEMM and combine launches and after
    the last. ``w13_bias`` [E, 2I], ``w2_bias`` [E, H] (activation dtype),
    ``activation`` "silu" or "swiglu_clamp" with ``swiglu`` = (alpha, beta,
    limit), and for act-order weights repacked by :func:`act_order_prepare`
    ``w13_perm`` [E, H] / ``w2_inv_perm`` [E, I]: the model-variant options of
    ``wna16_fused_moe_ex``.
    """
    _check(hidden, "hidden", (torch.float16, torch.bfloat16))
    dev = hidden.device
    M, H = hidden.shape
    E, twoI, kw = w13_q.shape
    I = twoI // 2
    pf = 32 // bits
    G1 = H if group_size == -1 else group_size
    G2 = I if group_size == -1 else group_size
    _check(w13_q, "w13_q", torch.int32, (E, 2 * I, H // pf), dev)
    _check(w2_q, "w2_q", torch.int32, (E, H, I // pf), dev)
    _check(w13_scales, "w13_scales", (torch.float16, torch.bfloat16), (E, H // G1, 2 * I), dev)
    _check(w2_scales, "w2_scales", w13_scales.dtype, (E, I // G2, H), dev)
    if (w13_zeros is None) != (w2_zeros is None):
        raise ValueError("w13_zeros and w2_zeros must both be given or both be None")
    if w13_zeros is not None:
        _check(w13_zeros, "w13_zeros", torch.int32, (E, H // G1, 2 * I // pf), dev)
        _check(w2_zeros, "w2_zeros", torch.int32, (E, I // G2, H // pf), dev)
    _check(topk_ids, "topk_ids", torch.int32, device=dev)
    topk = topk_ids.shape[1] if topk_ids.dim() == 2 else -1
    _check(topk_ids, "topk_ids", torch.int32, (M, topk), dev)
    _check(topk_weights, "topk_weights", torch.float32, (M, topk), dev)
    if out is None:
        out = torch.empty_like(hidden)
    _check(out, "out", hidden.dtype, (M, H), dev)
    need = workspace_bytes(M, H, I, E, topk, bits, group_size, block, split_k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, device=dev)
    args = (_ptr(hidden), _DTYPE[hidden.dtype], M, H, I, E, topk, _ptr(w13_q), _ptr(w13_scales),
            _ptr(w13_zeros), _ptr(w2_q), _ptr(w2_scales), _ptr(w2_zeros), _DTYPE[w13_scales.dtype], bits,
            group_size, _ptr(topk_ids), _ptr(topk_weights), _ptr(out), _ptr(workspace),
            workspace.numel(), block, split_k, _stream(stream))
    opt = _options(hidden, E, I, H, w13_bias, w2_bias, activation, swiglu, w13_perm, w2_inv_perm, atomic_reduce)
    if opt is not None:
        arr = None
        if events is not None:
            if len(events) != 6:
                raise ValueError("events must hold 6 entries")
            arr = (ctypes.c_void_p * 6)(*[None if e is None else e.cuda_event for e in events])
        st = load().wna16_fused_moe_ex(*args, arr, ctypes.byref(opt))
    elif events is None:
        st = load().wna16_fused_moe(*args)
    else:
        if len(events) != 6:
            raise ValueError("events must hold 6 entries")
        arr = (ctypes.c_void_p * 6)(*[None if e is None else e.cuda_event for e in events])
        st = load().wna16_fused_moe_timed(*args, arr)
    _raise(st, "wna16_fused_moe")
    return out


def fused_moe_routed(hidden: torch.Tensor, w13_q: torch.Tensor, w13_scales: torch.Tensor,
                     w13_zeros: Optional[torch.Tensor], w2_q: torch.Tensor, w2_scales: torch.Tensor,
                     w2_zeros: Optional[torch.Tensor], router_logits: torch.Tensor, topk: int, bits: int,
                     group_size: int, scoring: str = "softmax", renormalize: bool = True, n_groups: int = 1,
                     topk_groups: int = 1, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, block: int = 0, split_k: int = 0, stream=None,
                     topk_ids: Optional[torch.Tensor] = None, topk_weights: Optional[torch.Tensor] = None,
                     **variants):
    """The layer from router logits in one library call (``wna16_fused_moe_ex``
    with ``router_logits``): top-k routing on the device, then the layer.
    Returns (out [M, H], topk_ids [M, topk], topk_weights [M, topk]); the last two
    are written by the call. ``variants``: the keyword options of
    :func:`fused_moe` (biases, SwiGLU, act-order permutations)."""
    _check(hidden, "hidden", (torch.float16, torch.bfloat16))
    _check(router_logits, "router_logits", tuple(_LOGIT_DTYPE))
    if scoring not in _SCORING:
        raise ValueError(f"scoring must be one of {tuple(_SCORING)}")
    dev = hidden.device
    M, H = hidden.shape
    E, twoI, _ = w13_q.shape
    I = twoI // 2
    _check(router_logits, "router_logits", device=dev, shape=(M, E))
    if topk_ids is None:
        topk_ids = torch.empty(M, topk, dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty(M, topk, dtype=torch.float32, device=dev)
    _check(topk_ids, "topk_ids", torch.int32, (M, topk), dev)
    _check(topk_weights, "topk_weights", torch.float32, (M, topk), dev)
    if out is None:
        out = torch.empty_like(hidden)
    _check(out, "out", hidden.dtype, (M, H), dev)
    pf = 32 // bits
    G1 = H if group_size == -1 else group_size
    G2 = I if group_size == -1 else group_size
    _check(w13_q, "w13_q", torch.int32, (E, 2 * I, H // pf), dev)
    _check(w2_q, "w2_q", torch.int32, (E, H, I // pf), dev)
    _check(w13_scales, "w13_scales", (torch.float16, torch.bfloat16), (E, H // G1, 2 * I), dev)
    _check(w2_scales, "w2_scales", w13_scales.dtype, (E, I // G2, H), dev)
    need = workspace_bytes(M, H, I, E, topk, bits, group_size, block, split_k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, device=dev)
    opt = _options(hidden, E, I, H, variants.pop("w13_bias", None), variants.pop("w2_bias", None),
                   variants.pop("activation", "silu"), variants.pop("swiglu", (1.702, 1.0, 7.0)),
                   variants.pop("w13_perm", None), variants.pop("w2_inv_perm", None))
    if variants:
        raise TypeError(f"unexpected options {sorted(variants)}")
    if opt is None:
        opt = MoeOptions(None, None, 0, 1.0, 0.0, 0.0, None, None)
    opt.router_logits = router_logits.data_ptr()
    opt.logits_dtype = _LOGIT_DTYPE[router_logits.dtype]
    opt.scoring = _SCORING[scoring]
    opt.renormalize = int(bool(renormalize))
    opt.n_groups = n_groups
    opt.topk_groups = topk_groups
    opt.routed_ids = topk_ids.data_ptr()
    opt.routed_weights = topk_weights.data_ptr()
    st = load().wna16_fused_moe_ex(
        _ptr(hidden), _DTYPE[hidden.dtype], M, H, I, E, topk, _ptr(w13_q), _ptr(w13_scales), _ptr(w13_zeros),
        _ptr(w2_q), _ptr(w2_scales), _ptr(w2_zeros), _DTYPE[w13_scales.dtype], bits, group_size, None, None,
        _ptr(out), _ptr(workspace), workspace.numel(), block, split_k, _stream(stream), None, ctypes.byref(opt))
    _raise(st, "wna16_fused_moe_ex")
    return out, topk_ids, topk_weights


def fused_moe_noalloc(hidden: torch.Tensor, w13_q: torch.Tensor, w13_scales: torch.Tensor,
                      w13_zeros: Optional[torch.Tensor], w2_q: torch.Tensor, w2_scales: torch.Tensor,
                      w2_zeros: Optional[torch.Tensor], topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                      bits: int, group_size: int, out: torch.Tensor, block: int = 0, split_k: int = 0,
                      stream=None) -> torch.Tensor:
    """The fused layer through ``wna16_fused_moe_noalloc``: no workspace is passed
    and none is allocated (the library's fixed scratch area is used; see the
    header). ``out`` [M, H] must be given, so this call allocates nothing either."""
    _check(hidden, "hidden", (torch.float16, torch.bfloat16))
    dev = hidden.device
    M, H = hidden.shape
    E, twoI, _ = w13_q.shape
    I = twoI // 2
    for t, n in ((w13_q, "w13_q"), (w2_q, "w2_q"), (topk_ids, "topk_ids")):
        _check(t, n, torch.int32, device=dev)
    _check(w13_scales, "w13_scales", (torch.float16, torch.bfloat16), device=dev)
    _check(w2_scales, "w2_scales", w13_scales.dtype, device=dev)
    _check(topk_weights, "topk_weights", torch.float32, device=dev)
    _check(out, "out", hidden.dtype, (M, H), dev)
    topk = topk_ids.shape[1]
    st = load().wna16_fused_moe_noalloc(
        _ptr(hidden), _DTYPE[hidden.dtype], M, H, I, E, topk, _ptr(w13_q), _ptr(w13_scales),
        _ptr(w13_zeros), _ptr(w2_q), _ptr(w2_scales), _ptr(w2_zeros), _DTYPE[w13_scales.dtype], bits,
        group_size, _ptr(topk_ids), _ptr(topk_weights), _ptr(out), block, split_k, _stream(stream))
    _raise(st, "wna16_fused_moe_noalloc")
    return out


def noalloc_read_status(stream=None) -> int:
    """Synchronizes the stream and returns the raw device status bits of the
    last ``fused_moe_noalloc`` call on the current device."""
    bits = ctypes.c_int32(0)
    st = load().wna16_noalloc_read_status(ctypes.byref(bits), _stream(stream))
    if st not in (0, 5, 6, 7):
        _raise(st, "wna16_noalloc_read_status")
    return int(bits.value)


class Plan:
    """A ``wna16_plan_t``: the layer for one set of weights, its argument checks
    and weight descriptors done once (see the header). ``plan(hidden, topk_ids,
    topk_weights, out, workspace)`` runs the layer with only the batch's work
    left on the host; the tensors must be contiguous CUDA tensors of the
    documented shapes (checked once per distinct shape), and the weights must
    stay alive and unchanged while the plan is used."""

    def __init__(self, w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros, bits, group_size, topk,
                 act_dtype=torch.float16):
        E, twoI, _ = w13_q.shape
        H = w2_q.shape[1]
        self.E, self.I, self.H, self.topk, self.bits, self.group_size = E, twoI // 2, H, topk, bits, group_size
        self.act_dtype = act_dtype
        dev = w13_q.device
        G1 = H if group_size == -1 else group_size
        G2 = self.I if group_size == -1 else group_size
        pf = 32 // bits
        _check(w13_q, "w13_q", torch.int32, (E, 2 * self.I, H // pf), dev)
        _check(w2_q, "w2_q", torch.int32, (E, H, self.I // pf), dev)
        _check(w13_scales, "w13_scales", (torch.float16, torch.bfloat16), (E, H // G1, 2 * self.I), dev)
        _check(w2_scales, "w2_scales", w13_scales.dtype, (E, self.I // G2, H), dev)
        if (w13_zeros is None) != (w2_zeros is None):
            raise ValueError("w13_zeros and w2_zeros must both be given or both be None")
        if w13_zeros is not None:
            _check(w13_zeros, "w13_zeros", torch.int32, (E, H // G1, 2 * self.I // pf), dev)
            _check(w2_zeros, "w2_zeros", torch.int32, (E, self.I // G2, H // pf), dev)
        self._keep = (w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros)
        self._lib = load()
        h = ctypes.c_void_p()
        st = self._lib.wna16_plan_create(_DTYPE[act_dtype], H, self.I, E, topk, _ptr(w13_q), _ptr(w13_scales),
                                         _ptr(w13_zeros), _ptr(w2_q), _ptr(w2_scales), _ptr(w2_zeros),
                                         _DTYPE[w13_scales.dtype], bits, group_size, ctypes.byref(h))
        _raise(st, "wna16_plan_create")
        self._h = h
        self._seen = set()
        self._run = self._lib.wna16_fused_moe_plan

    def workspace_bytes(self, M, block=0, split_k=0):
        return workspace_bytes(M, self.H, self.I, self.E, self.topk, self.bits, self.group_size, block, split_k)

    def __call__(self, hidden, topk_ids, topk_weights, out, workspace, block=0, split_k=0, stream=None):
        M = hidden.shape[0]
        key = (M, hidden.device, hidden.dtype, out.dtype, workspace.numel())
        if key not in self._seen:
            dev = hidden.device
            _check(hidden, "hidden", self.act_dtype, (M, self.H), dev)
            _check(topk_ids, "topk_ids", torch.int32, (M, self.topk), dev)
            _check(topk_weights, "topk_weights", torch.float32, (M, self.topk), dev)
            _check(out, "out", self.act_dtype, (M, self.H), dev)
            _check(workspace, "workspace", torch.uint8, device=dev)
            self._seen.add(key)
        st = self._run(self._h, hidden.data_ptr(), M, topk_ids.data_ptr(), topk_weights.data_ptr(), out.data_ptr(),
                       workspace.data_ptr(), workspace.numel(), block, split_k,
                       (stream or torch.cuda.current_stream()).cuda_stream)
        if st:
            _raise(st, "wna16_fused_moe_plan")
        return out

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.wna16_plan_destroy(h)
            self._h = None


class PackedWeights:
    """One projection's weights in the prepacked stage-image form (see the
    header): ``data`` (uint8, device) plus the shape information the fused call
    needs."""

    def __init__(self, data: torch.Tensor, E: int, N: int, K: int, bits: int, group_size: int,
                 has_zeros: bool, scale_dtype: torch.dtype, gate_up: bool):
        self.data, self.E, self.N, self.K = data, E, N, K
        self.bits, self.group_size, self.has_zeros = bits, group_size, has_zeros
        self.scale_dtype, self.gate_up = scale_dtype, gate_up


def prepack(q: torch.Tensor, scales: torch.Tensor, zeros: Optional[torch.Tensor], bits: int, group_size: int,
            gate_up: bool, stream=None) -> PackedWeights:
    """``wna16_prepack`` of one projection: w13 (``gate_up=True``, q [E, 2I, H/pf])
    or w2 (q [E, H, I/pf]) with its scales and zero points (or None)."""
    _check(q, "q", torch.int32)
    dev = q.device
    E, N, kw = q.shape
    K = kw * (32 // bits)
    _check(scales, "scales", (torch.float16, torch.bfloat16), device=dev)
    if zeros is not None:
        _check(zeros, "zeros", torch.int32, device=dev)
    n = int(load().wna16_prepack_bytes(E, N, K, bits, group_size, int(zeros is not None), int(gate_up)))
    if n == 0:
        raise WNA16Error(2, "wna16_prepack_bytes")
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    st = load().wna16_prepack(_ptr(q), _ptr(scales), _ptr(zeros), E, N, K, bits, group_size, int(gate_up),
                              _ptr(dst), _stream(stream))
    _raise(st, "wna16_prepack")
    return PackedWeights(dst, E, N, K, bits, group_size, zeros is not None, scales.dtype, gate_up)


def fused_moe_prepacked(hidden: torch.Tensor, w13: PackedWeights, w2: PackedWeights, topk_ids: torch.Tensor,
                        topk_weights: torch.Tensor, out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, block: int = 0, split_k: int = 0,
                        stream=None, events=None, w13_bias: Optional[torch.Tensor] = None,
                        w2_bias: Optional[torch.Tensor] = None, activation: str = "silu",
                        swiglu=(1.702, 1.0, 7.0), w13_perm: Optional[torch.Tensor] = None,
                        w2_inv_perm: Optional[torch.Tensor] = None, atomic_reduce: bool = False) -> torch.Tensor:
    """The fused layer on prepacked weights (``wna16_fused_moe_prepacked``; with
    model-variant options, ``wna16_fused_moe_prepacked_ex``)."""
    _check(hidden, "hidden", (torch.float16, torch.bfloat16))
    dev = hidden.device
    M, H = hidden.shape
    if not (w13.gate_up and not w2.gate_up):
        raise ValueError("w13 must be the gate/up projection and w2 the down projection")
    E, I = w13.E, w13.N // 2
    if (w13.K, w2.N, w2.K, w2.E) != (H, H, I, E) or (w13.bits, w13.group_size, w13.has_zeros) != (
            w2.bits, w2.group_size, w2.has_zeros) or w13.scale_dtype != w2.scale_dtype:
        raise ValueError("w13 and w2 packed with inconsistent shapes or formats")
    _check(w13.data, "w13.data", torch.uint8, device=dev)
    _check(w2.data, "w2.data", torch.uint8, device=dev)
    topk = topk_ids.shape[1] if topk_ids.dim() == 2 else -1
    _check(topk_ids, "topk_ids", torch.int32, (M, topk), dev)
    _check(topk_weights, "topk_weights", torch.float32, (M, topk), dev)
    if out is None:
        out = torch.empty_like(hidden)
    _check(out, "out", hidden.dtype, (M, H), dev)
    need = workspace_bytes(M, H, I, E, topk, w13.bits, w13.group_size, block, split_k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, device=dev)
    arr = None
    if events is not None:
        if len(events) != 6:
            raise ValueError("events must hold 6 entries")
        arr = (ctypes.c_void_p * 6)(*[None if e is None else e.cuda_event for e in events])
    args = (_ptr(hidden), _DTYPE[hidden.dtype], M, H, I, E, topk, _ptr(w13.data), _ptr(w2.data),
            int(w13.has_zeros), _DTYPE[w13.scale_dtype], w13.bits, w13.group_size, _ptr(topk_ids),
            _ptr(topk_weights), _ptr(out), _ptr(workspace), workspace.numel(), block, split_k, _stream(stream), arr)
    opt = _options(hidden, E, I, H, w13_bias, w2_bias, activation, swiglu, w13_perm, w2_inv_perm, atomic_reduce)
    if opt is not None:
        st = load().wna16_fused_moe_prepacked_ex(*args, ctypes.byref(opt))
    else:
        st = load().wna16_fused_moe_prepacked(*args)
    _raise(st, "wna16_fused_moe_prepacked")
    return out


def act_order_prepare(q: torch.Tensor, g_idx: torch.Tensor, bits: int, group_size: int,
                      status: Optional[torch.Tensor] = None, stream=None):
    """Act-order weights -> (q_out, perm, inv_perm) by ``wna16_act_order_prepare``:
    codes [E, N, K/pf] with the columns sorted by group, and the permutations
    [E, K]. ``status`` (int32 [1], zeroed here if not given) receives
    DEV_BAD_GROUPS if ``g_idx`` [E, K] is not a split into groups of G."""
    _check(q, "q", torch.int32)
    dev = q.device
    E, N, kw = q.shape
    K = kw * (32 // bits)
    _check(g_idx, "g_idx", torch.int32, (E, K), dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(status, "status", torch.int32, (1,), dev)
    q_out = torch.empty_like(q)
    perm = torch.empty(E, K, dtype=torch.int32, device=dev)
    inv = torch.empty(E, K, dtype=torch.int32, device=dev)
    st = load().wna16_act_order_prepare(_ptr(q), _ptr(g_idx), E, N, K, bits, group_size, _ptr(q_out), _ptr(perm),
                                        _ptr(inv), _ptr(status), _stream(stream))
    _raise(st, "wna16_act_order_prepare")
    return q_out, perm, inv


_CKPT = {"gptq": 0, "gptq_v2": 1, "awq": 2}


def convert_checkpoint(fmt: str, qweight: torch.Tensor, qzeros: Optional[torch.Tensor], bits: int,
                       group_size: int, stream=None):
    """GPTQ ("gptq": zeros stored minus one; "gptq_v2") or AWQ ("awq") expert
    tensors -> (codes [E, N, K/pf], zeros [E, K/G, N/pf] or None) in the layer's
    layout, by ``wna16_convert_checkpoint``. ``qweight``: GPTQ [E, K/pf, N], AWQ
    [E, K, N/8]; ``qzeros`` [E, K/G, N/pf] or None. Scales need no conversion."""
    if fmt not in _CKPT:
        raise ValueError(f"fmt must be one of {tuple(_CKPT)}")
    _check(qweight, "qweight", torch.int32)
    dev = qweight.device
    pf = 32 // bits
    if fmt == "awq":
        E, K, n8 = qweight.shape
        N = n8 * 8
    else:
        E, kw, N = qweight.shape
        K = kw * pf
    G = K if group_size == -1 else group_size
    if qzeros is not None:
        _check(qzeros, "qzeros", torch.int32, (E, K // G, N // pf), dev)
    q_out = torch.empty(E, N, K // pf, dtype=torch.int32, device=dev)
    z_out = None if qzeros is None else torch.empty(E, K // G, N // pf, dtype=torch.int32, device=dev)
    st = load().wna16_convert_checkpoint(_CKPT[fmt], _ptr(qweight), _ptr(qzeros), E, N, K, bits, group_size,
                                         _ptr(q_out), _ptr(z_out), _stream(stream))
    _raise(st, "wna16_convert_checkpoint")
    return q_out, z_out


def check_wait_timeout(status: torch.Tensor, roles_left: Optional[torch.Tensor] = None, stream=None) -> None:
    """Runs the bounded-wait failure path on purpose (``wna16_check_wait_timeout``):
    about 2 s later ``status`` (int32 [1]) holds DEV_TIMEOUT and ``roles_left``
    (int32 [1], optional) the number of waiting warps that left (2)."""
    _check(status, "status", torch.int32, (1,))
    if roles_left is not None:
        _check(roles_left, "roles_left", torch.int32, (1,), status.device)
    _raise(load().wna16_check_wait_timeout(_ptr(status), _ptr(roles_left), _stream(stream)),
           "wna16_check_wait_timeout")


def check_launch_plan(M, H, I, E, topk, bits, group_size, has_zeros, act_dtype, scale_dtype, topk_ids, sorted_ids,
                      expert_ids, num_tokens_post_padded, block=0, split_k=0, sms=152):
    """Host-only replay of a fused call's launch plan on a given align output
    (``wna16_check_launch_plan``; numpy int32 arrays). Returns (violations,
    report text)."""
    import numpy as np

    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    srt = np.ascontiguousarray(sorted_ids, dtype=np.int32)
    exp = np.ascontiguousarray(expert_ids, dtype=np.int32)
    buf = ctypes.create_string_buffer(4096)
    dt = {"f16": 0, "bf16": 1}
    n = load().wna16_check_launch_plan(M, H, I, E, topk, bits, group_size, int(bool(has_zeros)), dt[act_dtype],
                                       dt[scale_dtype], block, split_k, sms, ids.ctypes.data, srt.ctypes.data,
                                       exp.ctypes.data, int(num_tokens_post_padded), buf, len(buf))
    return int(n), buf.value.decode()


def read_device_status(status_word: torch.Tensor, stream=None) -> int:
    """Synchronizes the stream and returns the raw device status bits."""
    bits = ctypes.c_int32(0)
    st = load().wna16_read_device_status(_ptr(status_word), ctypes.byref(bits), _stream(stream))
    if st not in (0, 5, 6, 7):
        _raise(st, "wna16_read_device_status")
    return int(bits.value)
