"""Value tolerances used by every parity test.

T-valued outputs (qNormed, kbar; bf16 or fp16): an element passes when
    |x - ref| <= 1 ulp_T(ref)                                   (2^-7 rel. bf16, 2^-10 fp16)
or, where rope or the norm cancels so that |ref| is tiny next to its head,
    |x - ref| <= 2^-16 * max|ref| over that 128-element head    (the "floor").
The floor covers binary32 reordering error (sum-of-squares tree, rsqrtf, FMA
contraction) that the final cast magnifies only when the output itself is tiny;
tests report how many elements needed it.

FP32 logits: an element passes when
    |x - ref| <= 2^-p * |ref| + 2^-16 * (1/sqrt(128)) * sum_h sum_d |q_hd * k_d|
with p = 7 for bf16 inputs and 10 for fp16 (one ulp of T, relative), plus a
conditioning-aware floor: reordering a 128-term binary32 dot product moves it by
at most ~128 * 2^-24 times that absolute sum.
"""
from __future__ import annotations

import numpy as np

MANT_BITS = {"bf16": 7, "fp16": 10}
MIN_NORMAL_EXP = {"bf16": -126, "fp16": -14}
FLOOR_BITS = 16


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of T bit patterns (independent of the oracle's own converter)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """ulp of T at each |ref| (subnormal spacing below the normal range)."""
    p = MANT_BITS[dtype]
    emin = MIN_NORMAL_EXP[dtype]
    a = np.abs(np.asarray(ref, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.exp2(e - p)


def check_t(x_bits, ref, dtype: str, head_axis_len: int = 128):
    """Compare T outputs (bits) against a reference (T bits or float64 values).

    Returns (ok, stats).  ``ref`` may be uint16 T bits or float64 values.
    """
    x = to_f64(x_bits, dtype)
    r = to_f64(ref, dtype) if np.asarray(ref).dtype == np.uint16 else np.asarray(ref, np.float64)
    assert x.shape == r.shape, (x.shape, r.shape)
    if x.size == 0:
        return True, {"n": 0, "max_ulp": 0.0, "floor_used": 0, "bad": 0}
    finite = np.isfinite(x) & np.isfinite(r)
    diff = np.abs(x - r)
    u = ulp(r, dtype)
    heads = r.reshape(-1, head_axis_len)
    hmax = np.abs(heads).max(axis=1, keepdims=True)
    floor = np.broadcast_to(hmax * 2.0 ** -FLOOR_BITS, heads.shape).reshape(r.shape)
    within_ulp = diff <= u
    within_floor = diff <= floor
    ok_elem = finite & (within_ulp | within_floor)
    stats = {
        "n": int(x.size),
        "max_ulp": float(np.max(np.where(finite, diff / u, np.inf))),
        "floor_used": int(np.sum(finite & ~within_ulp & within_floor)),
        "bad": int(np.sum(~ok_elem)),
    }
    return bool(ok_elem.all()), stats


def logits_floor(q_bits, kbar_bits, dtype: str) -> np.ndarray:
    """Per (row, block) conditioning floor 2^-16/sqrt(128) * sum_h sum_d |q_hd k_gd|.

    q_bits [R, 4, 128] (the rows' heads), kbar_bits [R, NB, 128] or [NB, 128].
    """
    q = np.abs(to_f64(q_bits, dtype))               # [R, 4, 128]
    k = np.abs(to_f64(kbar_bits, dtype))
    qs = q.sum(axis=1)                               # [R, 128]
    if k.ndim == 2:
        s = qs @ k.T                                 # [R, NB]
    else:
        s = np.einsum("rd,rgd->rg", qs, k)
    return s * (2.0 ** -FLOOR_BITS) / np.sqrt(128.0)


def check_logits(x, ref, dtype: str, floor: np.ndarray):
    """FP32 logits: identical masks (bit-exact -FLT_MAX cells), values within tolerance."""
    x = np.asarray(x, np.float32)
    ref = np.asarray(ref, np.float32)
    assert x.shape == ref.shape
    neg = np.float32(-np.finfo(np.float32).max)
    mx = x == neg
    mr = ref == neg
    mask_ok = bool(np.array_equal(mx, mr))
    vis = ~mr
    xd = x.astype(np.float64)
    rd = ref.astype(np.float64)
    diff = np.abs(xd - rd)
    tol = 2.0 ** -MANT_BITS[dtype] * np.abs(rd) + floor
    ok_vals = bool(np.all(np.isfinite(xd[vis])) and np.all(diff[vis] <= tol[vis]))
    rel = np.where(np.abs(rd) > 0, diff / np.maximum(np.abs(rd), 1e-300), 0.0)
    stats = {
        "n": int(x.size),
        "visible": int(vis.sum()),
        "mask_ok": mask_ok,
        "max_rel_err": float(rel[vis].max()) if vis.any() else 0.0,
        "max_err_over_tol": float((diff[vis] / np.maximum(tol[vis], 1e-300)).max()) if vis.any() else 0.0,
        "bad": int(np.sum(vis & ~(diff <= tol))),
    }
    return mask_ok and ok_vals, stats


def check_logits_torch(x, ref, dtype: str, floor):
    """check_logits on torch tensors (any device), for outputs too large for numpy
    float64 arrays: the same mask rule and the same value bound, evaluated in float64."""
    import torch
    neg = float(np.float32(-np.finfo(np.float32).max))
    mx = x == neg
    mr = ref == neg
    mask_ok = bool(torch.equal(mx, mr))
    vis = ~mr
    xd = x.double()
    rd = ref.double()
    diff = (xd - rd).abs()
    tol = (2.0 ** -MANT_BITS[dtype]) * rd.abs() + floor.double()
    ok_elem = torch.isfinite(xd) & (diff <= tol)
    bad = int((vis & ~ok_elem).sum())
    nvis = int(vis.sum())
    worst = float((diff[vis] / tol[vis].clamp(min=1e-300)).max()) if nvis else 0.0
    stats = {"n": int(x.numel()), "visible": nvis, "mask_ok": mask_ok,
             "max_err_over_tol": worst, "bad": bad}
    return mask_ok and bad == 0, stats
