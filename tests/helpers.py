"""Glue between the torch-made synthetic inputs and the numpy oracle.

Only converts containers (torch tensors -> numpy arrays, half-precision values
-> raw 16-bit patterns); no arithmetic of the layer lives here.
"""
from __future__ import annotations

import numpy as np
import torch


def halfbits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 tensor as a uint16 numpy array."""
    assert t.dtype in (torch.float16, torch.bfloat16)
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def np_i32(t):
    return None if t is None else t.detach().contiguous().cpu().numpy()


def oracle_layer_dict(li) -> dict:
    """The oracle's input dict for a ``synthetic.LayerInputs``."""
    wl = li.wl
    return dict(
        x=halfbits(li.hidden), act_dtype=wl.act_dtype,
        w13_q=np_i32(li.w13_q), w13_s=halfbits(li.w13_s), w13_z=np_i32(li.w13_z),
        w2_q=np_i32(li.w2_q), w2_s=halfbits(li.w2_s), w2_z=np_i32(li.w2_z),
        scale_dtype=wl.scale_dtype, bits=wl.bits, group_size=wl.group_size,
        topk_ids=np_i32(li.topk_ids), topk_w=li.topk_w.detach().cpu().numpy(),
    )


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def max_rel_err(y: np.ndarray, r: np.ndarray) -> float:
    """max_i |y_i - r_i| / max_i |r_i| (the layer-output parity measure)."""
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.max(np.abs(r)) if r.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(y))) if y.size else 0.0
    return float(np.max(np.abs(y - r)) / den)


def norm_rel_err(y: np.ndarray, r: np.ndarray) -> float:
    """||y - r||_2 / ||r||_2 (reported beside the parity measure)."""
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = float(np.linalg.norm(r))
    return float(np.linalg.norm(y - r)) / den if den else float(np.linalg.norm(y))
