"""Shared test utilities: tensor conversion and the parity tolerances.

Tolerances (from the accuracy target of the method's deployment):
  * compressed fp32 values (pooled x, c128 kv and sum):
        |gpu - ref| <= 2e-3 * max(1, |ref|)
  * c128 running max: |gpu - ref| <= 2e-3 (absolute)
  * FP8 codes and scales: bit-exact where the pooled bf16 row agrees with the
    oracle's; stage by stage (rotation, quantisation) everywhere
  * scales, ring contents, state-slot selection, cache addresses, plans: exact
"""
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
