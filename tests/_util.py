"""Shared test helpers: storage conversion, running the CUDA path, ulp metrics."""
from __future__ import annotations

import numpy as np

from persistent_step_megakernel_gb300 import synthetic as S

ULP_BITS = {"bfloat16": 8, "float16": 11, "float32": 24}
EMIN = {"bfloat16": -126, "float16": -14, "float32": -126}


def values(arrays, program):
    """Program-input storage arrays -> exact float64 values."""
    return [S.storage_to_float64(a, s.dtype) for a, s in zip(arrays, program.inputs)]


def to_torch(arr, dtype, device):
    import torch
    if dtype == "bfloat16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def ordered_bits(v, dtype) -> np.ndarray:
    """Values (exactly representable in dtype) -> integers ordered like the values."""
    v = np.asarray(v, dtype=np.float64)
    if dtype == "float16":
        b = v.astype(np.float16).view(np.uint16).astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    b32 = v.astype(np.float32).view(np.uint32).astype(np.int64)
    if dtype == "bfloat16":
        b = b32 >> 16
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.where(b32 & 0x80000000, -(b32 & 0x7FFFFFFF), b32)


def ulp_distance(a, b, dtype) -> np.ndarray:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    d = np.abs(ordered_bits(np.nan_to_num(a), dtype) - ordered_bits(np.nan_to_num(b), dtype))
    nan = np.isnan(a) | np.isnan(b)
    return np.where(nan, np.where(np.isnan(a) & np.isnan(b), 0, 1 << 40), d)


def ulp_of(v, dtype) -> np.ndarray:
    """Spacing of dtype at |v| (the subnormal spacing below the normal range)."""
    a = np.abs(np.asarray(v, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, EMIN[dtype])
    return np.ldexp(1.0, (e - (ULP_BITS[dtype] - 1)).astype(np.int64))
