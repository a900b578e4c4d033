"""Shared test utilities: tensor conversion and the parity tolerances.

Tolerances (from the accuracy target of the method's deployment):
  * compressed fp32 values (pooled x, c128 kv and sum):
        |gpu - ref| <= 2e-3 * max(1, |ref|)
  * c128 running max: |gpu - ref| <= 2e-3 (absolute)
  * FP8 codes and scales: bit-exact where the pooled bf16 row agrees with the
    oracle's; stage by stage (rotation, quantisation) everywhere
  * bf16 rounding of the fp32 row: a channel may round to the other bf16
    neighbour than the oracle's exact value only when a rounding boundary lies
    between the two values; the number of such channels is bounded by what
    the measured fp32 error makes likely (bf16_flip_check)
  * scales, ring contents, state-slot selection, cache addresses, plans: exact
"""
import json
import math
import os

import numpy as np
import torch

REL_TOL = 2e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def assert_close_rel(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= REL_TOL, f"{what}: max rel err {worst:.3e} > {REL_TOL}"
    return worst


def assert_close_abs(gpu, ref, tol=REL_TOL, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max abs err {worst:.3e} > {tol}"
    return worst


def cache_rows(cache: np.ndarray, page_size: int, D: int, locs):
    """(codes [n, D], scales [n]) at cache locations (linear in-page layout)."""
    flat = cache.reshape(-1)
    stride = page_size * (D + 4)
    codes, scales = [], []
    for loc in locs:
        page, tok = divmod(int(loc), page_size)
        base = page * stride
        codes.append(flat[base + tok * D: base + tok * D + D])
        scales.append(flat[base + page_size * D + 4 * tok: base + page_size * D + 4 * tok + 4].view(np.float32)[0])
    return np.array(codes).reshape(-1, D), np.array(scales, np.float32)


def report(test, **fields):
    """Append one JSON line of measured figures (flip counts) to the file named
    by CKV_TEST_REPORT, when set; always print it (shown with pytest -rP)."""
    rec = {"test": test, **fields}
    print(json.dumps(rec))
    path = os.environ.get("CKV_TEST_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_spacing(x):
    """Distance between consecutive bf16 values at |x| (8 significant bits;
    subnormal spacing 2^-133 below 2^-126)."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def bf16_flip_check(gpu_x, gpu_xb, ref_x, ref_xb, what, test=None):
    """bf16 rounding of an fp32 row against the oracle's exact row.

    Both sides round to nearest even, so a channel can land on a different
    bf16 value only if a rounding boundary lies between the GPU's fp32 value
    and the oracle's exact one; for a boundary at a uniformly random place
    within the spacing h around x, that happens with probability
    min(1, |x_gpu - x_ref| / h).  The sum E of these probabilities over all
    channels is the expected number of such flips given the measured fp32
    error; the observed count F must satisfy F <= E + 6 sqrt(E) + 6 (a Poisson
    upper tail far below 1e-6), and every flipped channel must have the
    midpoint of its two bf16 values between x_gpu and x_ref.  A wrong rounding
    mode or a rounding stage on the wrong value fails one of the two.
    Returns (rows with a flip, flipped channels, expected flips)."""
    gx = np.asarray(gpu_x, np.float64)
    rx = np.asarray(ref_x, np.float64)
    diff = np.asarray(gpu_xb) != np.asarray(ref_xb)
    F = int(diff.sum())
    err = np.abs(gx - rx)
    E = float(np.minimum(1.0, err / bf16_spacing(rx)).sum())
    bound = E + 6.0 * math.sqrt(E) + 6.0
    rows = int(np.any(diff.reshape(diff.shape[0], -1), axis=1).sum()) if diff.ndim > 1 else int(diff.any())
    report(test or what, rows=int(diff.shape[0]) if diff.ndim > 1 else 1, flipped_rows=rows, flipped_channels=F,
           expected_channels=round(E, 2), bound=round(bound, 2), max_rel_err=float((err / np.maximum(1.0, np.abs(rx))).max())
           if err.size else 0.0)
    assert F <= bound, f"{what}: {F} bf16 flips, more than {bound:.1f} (expected {E:.1f} from the fp32 error)"
    if F:
        g = bf16_values(np.asarray(gpu_xb)[diff])
        r = bf16_values(np.asarray(ref_xb)[diff])
        mid = (g + r) / 2
        lo = np.minimum(gx[diff], rx[diff])
        hi = np.maximum(gx[diff], rx[diff])
        assert np.all((lo <= mid) & (mid <= hi)), f"{what}: a bf16 flip with no rounding boundary between the values"
    return rows, F, E
