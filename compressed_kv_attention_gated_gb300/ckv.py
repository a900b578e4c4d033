"""Thin Python binding of ``libckv.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls (include/ckv.h)
and takes torch tensors; it checks dtypes/devices, passes raw pointers, sizes
and the current CUDA stream, and raises ``CkvError`` on a nonzero status.  All
arithmetic happens in the CUDA kernels; there is no fallback: if the library
is missing or the tensors are not on a CUDA device, the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

CKV_F32 = 0
CKV_BF16 = 1
PLAN_ENTRY_BYTES = 16
SENTINEL = 0xFFFFFFFF

_STATUS_FUNCS = {
    "ckv_kpool_decode_update": 25,
    "ckv_kpool_compress": 20,
    "ckv_kpool_seed_tail": 10,
    "ckv_c128_online_decode": 13,
    "ckv_c128_online_prefill": 18,
    "ckv_c128_online_decode_fp8": 18,
    "ckv_c128_online_prefill_fp8": 23,
    "ckv_plan_online_prefill": 9,
    "ckv_plan_online_prefill_device": 11,
    "ckv_c128_online_prefill_counted": 17,
    "ckv_c128_online_prefill_counted_fp8": 22,
    "ckv_expand_pools_and_append_tail": 9,
    "ckv_wait_timeout_selftest": 3,
    "ckv_check_distinct": 8,
    "ckv_check_distinct_noalloc": 6,
    "ckv_latency_probe": 9,
}
EXPORTED = tuple(_STATUS_FUNCS) + ("ckv_status_string", "ckv_last_cuda_error", "ckv_abi_version",
                                    "ckv_c128_prefill_set_variant", "ckv_kpool_compress_set_variant")


class CkvError(RuntimeError):
    def __init__(self, func, status, lib):
        msg = lib.ckv_status_string(status).decode()
        if status == 6:
            msg += f" (cudaError {lib.ckv_last_cuda_error()})"
        super().__init__(f"{func}: status {status}: {msg}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libckv.so; raise if it has not been built (no fallback path exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"{_build.LIB} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(_build.LIB)
            for name, nargs in _STATUS_FUNCS.items():
                fn = getattr(L, name)
                fn.restype = ctypes.c_int32
            L.ckv_kpool_decode_update.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p]
            L.ckv_kpool_compress.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p]
            L.ckv_kpool_seed_tail.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_c128_online_decode.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_c128_online_prefill.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_c128_online_decode_fp8.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_c128_online_prefill_fp8.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_plan_online_prefill.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32),
                ctypes.POINTER(ctypes.c_uint32)]
            L.ckv_plan_online_prefill_device.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p]
            L.ckv_c128_online_prefill_counted.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_c128_online_prefill_counted_fp8.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_expand_pools_and_append_tail.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
            L.ckv_wait_timeout_selftest.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
            L.ckv_check_distinct.argtypes = [
                ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_check_distinct_noalloc.argtypes = [
                ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.ckv_latency_probe.argtypes = [
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            L.ckv_status_string.restype = ctypes.c_char_p
            L.ckv_status_string.argtypes = [ctypes.c_int32]
            L.ckv_last_cuda_error.restype = ctypes.c_int32
            L.ckv_last_cuda_error.argtypes = []
            L.ckv_abi_version.restype = ctypes.c_int32
            L.ckv_abi_version.argtypes = []
            for fn in (L.ckv_c128_prefill_set_variant, L.ckv_kpool_compress_set_variant):
                fn.restype = ctypes.c_int32
                fn.argtypes = [ctypes.c_int32]
            _lib = L
    return _lib


# ------------------------------------------------------------------ helpers
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, ref):
    if stream is not None:
        return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    return ctypes.c_void_p(torch.cuda.current_stream(ref.device).cuda_stream)


def _cuda(name, *ts):
    """Every tensor on one CUDA device, the current one: the kernels run on the
    current device, and a pointer into another device's memory would fault."""
    devs = set()
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name}: every tensor must be on a CUDA device")
        devs.add(t.device.index)
    if len(devs) > 1:
        raise ValueError(f"{name}: tensors on several CUDA devices {sorted(devs)}")
    if devs and devs.pop() != torch.cuda.current_device():
        raise ValueError(f"{name}: the tensors are not on the current CUDA device "
                         f"(torch.cuda.set_device or torch.cuda.device(...) first)")


def _check(func, status):
    if status != 0:
        raise CkvError(func, status, load())


def _dtype(t):
    if t.dtype == torch.float32:
        return CKV_F32
    if t.dtype == torch.bfloat16:
        return CKV_BF16
    raise ValueError("input must be float32 or bfloat16")


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def ckv_wait_timeout_selftest(err_word, limit_us=20000, stream=None):
    """Run the bounded-wait self-test (see include/ckv.h); err_word: CUDA int32 [1]."""
    L = load()
    _cuda("ckv_wait_timeout_selftest", err_word)
    _check("ckv_wait_timeout_selftest", L.ckv_wait_timeout_selftest(_ptr(err_word), int(limit_us),
                                                                    _stream(stream, err_word)))


# ------------------------------------------------------------ pooled path
def ckv_kpool_decode_update(kv_cache, tail_ring, tail_slot_mapping, slot_mapping, positions, key,
                            score, ape, round_scale=True, tap_x=None, tap_xb=None, tap_yb=None,
                            use_pdl=False, err_word=None, stream=None):
    """Pooled decode/verify update; see ckv_kpool_decode_update in include/ckv.h.

    kv_cache uint8 [pages, page_size, D+4]; tail_ring bf16 [blocks, 2, P, D];
    index tensors int32 [B, N] (contiguous); key/score bf16 [B, N, D] (last dim
    contiguous); ape float32 [P, D].
    """
    L = load()
    _cuda("ckv_kpool_decode_update", kv_cache, tail_ring, tail_slot_mapping, slot_mapping, positions,
          key, score, ape, tap_x, tap_xb, tap_yb, err_word)
    B, N, D = key.shape
    P = tail_ring.shape[2]
    _need(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 3 and kv_cache.is_contiguous(),
          "kv_cache must be contiguous uint8 [pages, page_size, D+4]")
    _need(tail_ring.dtype == torch.bfloat16 and tail_ring.is_contiguous() and tail_ring.dim() == 4
          and tail_ring.shape[1] == 2 and tail_ring.shape[3] == D, "tail_ring must be bf16 [blocks, 2, P, D]")
    _need(key.dtype == torch.bfloat16 and score.dtype == torch.bfloat16 and score.shape == key.shape
          and key.stride(2) == 1 and score.stride(2) == 1, "key/score must be bf16 [B, N, D], last dim contiguous")
    for t in (tail_slot_mapping, slot_mapping, positions):
        _need(t.dtype == torch.int32 and t.is_contiguous() and tuple(t.shape) == (B, N),
              "index tensors must be contiguous int32 [B, N]")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (P, D),
          "ape must be contiguous float32 [P, D]")
    _check("ckv_kpool_decode_update", L.ckv_kpool_decode_update(
        _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(tail_ring), tail_ring.shape[0],
        _ptr(tail_slot_mapping), _ptr(slot_mapping), _ptr(positions), _ptr(key), key.stride(0),
        key.stride(1), _ptr(score), score.stride(0), score.stride(1), _ptr(ape), B, N, P, D,
        int(bool(round_scale)), _ptr(tap_x), _ptr(tap_xb), _ptr(tap_yb), int(bool(use_pdl)), _ptr(err_word),
        _stream(stream, key)))


def ckv_kpool_compress(slot_k, slot_score, ape, kv_cache=None, loc=None, write_mask=None,
                       write_cache=True, out_fp8=None, out_scale=None, round_scale=True, tap_x=None,
                       tap_xb=None, tap_yb=None, use_pdl=False, err_word=None, stream=None):
    """One-shot pooled compression; see ckv_kpool_compress in include/ckv.h.

    slot_k/slot_score bf16 [n, P, D] contiguous; ape float32 [P, D]; loc int64 [n];
    write_mask bool/uint8 [n]; out_fp8 uint8 (or float8_e4m3fn) [n, D]; out_scale float32 [n].
    """
    L = load()
    _cuda("ckv_kpool_compress", slot_k, slot_score, ape, kv_cache, loc, write_mask, out_fp8, out_scale,
          tap_x, tap_xb, tap_yb, err_word)
    n, P, D = slot_k.shape
    _need(slot_k.dtype == torch.bfloat16 and slot_score.dtype == torch.bfloat16
          and slot_k.is_contiguous() and slot_score.is_contiguous() and slot_score.shape == slot_k.shape,
          "slot_k/slot_score must be contiguous bf16 [n, P, D]")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (P, D),
          "ape must be contiguous float32 [P, D]")
    pages = ps = 0
    if write_cache:
        _need(kv_cache is not None and loc is not None, "write_cache needs kv_cache and loc")
        _need(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 3 and kv_cache.is_contiguous(),
              "kv_cache must be contiguous uint8 [pages, page_size, D+4]")
        _need(loc.dtype == torch.int64 and loc.is_contiguous() and loc.numel() == n, "loc must be int64 [n]")
        pages, ps = kv_cache.shape[0], kv_cache.shape[1]
    if write_mask is not None:
        _need(write_mask.dtype in (torch.bool, torch.uint8) and write_mask.is_contiguous()
              and write_mask.numel() == n, "write_mask must be bool [n]")
    if out_fp8 is not None:
        _need(out_fp8.element_size() == 1 and out_fp8.is_contiguous() and out_fp8.numel() == n * D,
              "out_fp8 must be a contiguous 1-byte tensor [n, D]")
        _need(out_scale is not None and out_scale.dtype == torch.float32 and out_scale.numel() == n,
              "out_scale must be float32 [n]")
    _check("ckv_kpool_compress", L.ckv_kpool_compress(
        _ptr(kv_cache) if write_cache else None, pages, ps, _ptr(slot_k), _ptr(slot_score), _ptr(ape),
        _ptr(loc) if write_cache else None, _ptr(write_mask), int(bool(write_cache)), _ptr(out_fp8),
        _ptr(out_scale), n, P, D, int(bool(round_scale)), _ptr(tap_x), _ptr(tap_xb), _ptr(tap_yb),
        int(bool(use_pdl)), _ptr(err_word), _stream(stream, slot_k)))


def ckv_kpool_seed_tail(tail_ring, key, score, tslot, err_word=None, stream=None):
    """Seed the tail ring from a prefill batch; see ckv_kpool_seed_tail in include/ckv.h."""
    L = load()
    _cuda("ckv_kpool_seed_tail", tail_ring, key, score, tslot, err_word)
    n, D = key.shape
    P = tail_ring.shape[2]
    _need(tail_ring.dtype == torch.bfloat16 and tail_ring.is_contiguous(), "tail_ring must be bf16")
    _need(key.dtype == torch.bfloat16 and score.dtype == torch.bfloat16 and key.is_contiguous()
          and score.is_contiguous() and score.shape == key.shape, "key/score must be contiguous bf16 [n, D]")
    _need(tslot.dtype == torch.int32 and tslot.is_contiguous() and tslot.numel() == n, "tslot must be int32 [n]")
    _check("ckv_kpool_seed_tail", L.ckv_kpool_seed_tail(
        _ptr(tail_ring), tail_ring.shape[0], _ptr(key), _ptr(score), _ptr(tslot), n, P, D,
        _ptr(err_word), _stream(stream, key)))


def ckv_expand_pools_and_append_tail(pool_ids, seq_lens, pool_size, out=None, use_pdl=False, stream=None):
    """Pool -> token index expansion with the tail appended; see include/ckv.h.

    pool_ids: CUDA int32 [rows, n_groups] (last dim contiguous); seq_lens: CUDA
    int64 [rows].  Returns int32 [rows, n_groups * pool_size + pool_size - 1].
    """
    L = load()
    _cuda("ckv_expand_pools_and_append_tail", pool_ids, seq_lens, out)
    _need(pool_ids.dtype == torch.int32 and pool_ids.dim() == 2 and pool_ids.stride(1) == 1,
          "pool_ids must be int32 [rows, n_groups], last dim contiguous")
    _need(seq_lens.dtype == torch.int64 and seq_lens.is_contiguous(), "seq_lens must be int64 [rows]")
    rows, groups = pool_ids.shape
    cols = groups * pool_size + pool_size - 1
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.int32, device=pool_ids.device)
    _need(out.dtype == torch.int32 and out.is_contiguous() and tuple(out.shape) == (rows, cols),
          "out must be contiguous int32 [rows, n_groups * P + P - 1]")
    _check("ckv_expand_pools_and_append_tail", L.ckv_expand_pools_and_append_tail(
        _ptr(pool_ids), pool_ids.stride(0), _ptr(seq_lens), rows, groups, int(pool_size), _ptr(out),
        int(bool(use_pdl)), _stream(stream, pool_ids)))
    return out


# ------------------------------------------------------------ online c128
def ckv_c128_online_decode(state, input, out, ape, indices, seq_lens, use_pdl=False, err_word=None,
                           stream=None):
    """Online c128 decode; see ckv_c128_online_decode in include/ckv.h.

    state float32 [slots, 3, D] (or [slots, 1, 3D]); input float32/bf16 [B, 2D];
    out float32 [B, D]; ape float32 [128, D]; indices/seq_lens int32 [B].
    """
    L = load()
    _cuda("ckv_c128_online_decode", state, input, out, ape, indices, seq_lens, err_word)
    B = input.shape[0]
    D = input.shape[1] // 2
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [B, 2D]")
    _need(out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, D), "out must be float32 [B, D]")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    for t in (indices, seq_lens):
        _need(t.dtype == torch.int32 and t.is_contiguous() and t.numel() == B, "indices/seq_lens must be int32 [B]")
    _check("ckv_c128_online_decode", L.ckv_c128_online_decode(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), _ptr(out), _ptr(ape),
        _ptr(indices), _ptr(seq_lens), B, D, int(bool(use_pdl)), _ptr(err_word), _stream(stream, input)))


def ckv_c128_online_prefill(state, input, out, ape, indices, compress_plan, num_compress, write_plan,
                            num_write, load_indices=None, use_pdl=False, err_word=None, stream=None):
    """Online c128 prefill (compress pass, then write pass); see include/ckv.h.

    state float32 [slots, 3, D]; input float32/bf16 [T, 2D]; out float32 [T, D];
    ape float32 [128, D]; indices (and load_indices) int32 [B]; plans are device
    tensors of 16-byte entries (uint8 [M, 16] or int32 [M, 4]).
    """
    L = load()
    _cuda("ckv_c128_online_prefill", state, input, out, ape, indices, load_indices, compress_plan,
          write_plan, err_word)
    T = input.shape[0]
    D = input.shape[1] // 2
    B = indices.numel()
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [T, 2D]")
    _need(out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (T, D), "out must be float32 [T, D]")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    _need(indices.dtype == torch.int32 and indices.is_contiguous(), "indices must be int32 [B]")
    if load_indices is not None:
        _need(load_indices.dtype == torch.int32 and load_indices.is_contiguous() and load_indices.numel() == B,
              "load_indices must be int32 [B]")
    for pl, cnt in ((compress_plan, num_compress), (write_plan, num_write)):
        _need(pl.is_contiguous() and pl.numel() * pl.element_size() >= cnt * PLAN_ENTRY_BYTES,
              "plan tensors must hold num_* 16-byte entries")
    _check("ckv_c128_online_prefill", L.ckv_c128_online_prefill(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), T, _ptr(out), _ptr(ape),
        _ptr(indices), _ptr(load_indices), B, _ptr(compress_plan), int(num_compress), _ptr(write_plan),
        int(num_write), D, int(bool(use_pdl)), _ptr(err_word), _stream(stream, input)))


def _fp8_cache(kv_cache, cache_loc, D, n_loc):
    blocks = D // 128
    _need(kv_cache.dtype == torch.uint8 and kv_cache.is_contiguous() and kv_cache.dim() == 3
          and kv_cache.shape[2] == D + 4 * blocks, "kv_cache must be contiguous uint8 [pages, page_size, D + 4*D/128]")
    _need(cache_loc.dtype == torch.int64 and cache_loc.is_contiguous() and cache_loc.numel() == n_loc,
          "cache_loc must be contiguous int64")
    return kv_cache.shape[0], kv_cache.shape[1]


def ckv_c128_online_decode_fp8(state, input, out, ape, indices, seq_lens, kv_cache, cache_loc, round_scale=True,
                               use_pdl=False, err_word=None, stream=None):
    """Online c128 decode with the FP8 output stage; see ckv_c128_online_decode_fp8
    in include/ckv.h.  kv_cache uint8 [pages, page_size, D + 4*D/128];
    cache_loc int64 [B]; out float32 [B, D] or None."""
    L = load()
    _cuda("ckv_c128_online_decode_fp8", state, input, out, ape, indices, seq_lens, kv_cache, cache_loc, err_word)
    B = input.shape[0]
    D = input.shape[1] // 2
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [B, 2D]")
    _need(out is None or (out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, D)),
          "out must be float32 [B, D] or None")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    for t in (indices, seq_lens):
        _need(t.dtype == torch.int32 and t.is_contiguous() and t.numel() == B, "indices/seq_lens must be int32 [B]")
    pages, ps = _fp8_cache(kv_cache, cache_loc, D, B)
    _check("ckv_c128_online_decode_fp8", L.ckv_c128_online_decode_fp8(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), _ptr(out), _ptr(ape),
        _ptr(indices), _ptr(seq_lens), B, D, _ptr(kv_cache), pages, ps, _ptr(cache_loc), int(bool(round_scale)),
        int(bool(use_pdl)), _ptr(err_word), _stream(stream, input)))


def ckv_c128_online_prefill_fp8(state, input, out, ape, indices, compress_plan, num_compress, write_plan,
                                num_write, kv_cache, cache_loc, round_scale=True, load_indices=None, use_pdl=False,
                                err_word=None, stream=None):
    """Online c128 prefill with the FP8 output stage; see ckv_c128_online_prefill_fp8
    in include/ckv.h.  kv_cache uint8 [pages, page_size, D + 4*D/128];
    cache_loc int64 [T] (read at compress rows); out float32 [T, D] or None."""
    L = load()
    _cuda("ckv_c128_online_prefill_fp8", state, input, out, ape, indices, load_indices, compress_plan,
          write_plan, kv_cache, cache_loc, err_word)
    T = input.shape[0]
    D = input.shape[1] // 2
    B = indices.numel()
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [T, 2D]")
    _need(out is None or (out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (T, D)),
          "out must be float32 [T, D] or None")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    _need(indices.dtype == torch.int32 and indices.is_contiguous(), "indices must be int32 [B]")
    if load_indices is not None:
        _need(load_indices.dtype == torch.int32 and load_indices.is_contiguous() and load_indices.numel() == B,
              "load_indices must be int32 [B]")
    for pl, cnt in ((compress_plan, num_compress), (write_plan, num_write)):
        _need(pl.is_contiguous() and pl.numel() * pl.element_size() >= cnt * PLAN_ENTRY_BYTES,
              "plan tensors must hold num_* 16-byte entries")
    pages, ps = _fp8_cache(kv_cache, cache_loc, D, T)
    _check("ckv_c128_online_prefill_fp8", L.ckv_c128_online_prefill_fp8(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), T, _ptr(out), _ptr(ape),
        _ptr(indices), _ptr(load_indices), B, _ptr(compress_plan), int(num_compress), _ptr(write_plan),
        int(num_write), D, _ptr(kv_cache), pages, ps, _ptr(cache_loc), int(bool(round_scale)), int(bool(use_pdl)),
        _ptr(err_word), _stream(stream, input)))


def ckv_c128_prefill_set_variant(variant: int) -> int:
    """Select the compress-pass kernel (0 auto, 1 one CTA per segment, 2 TMA pipeline).

    Returns the previous setting; raises on an unknown value."""
    prev = load().ckv_c128_prefill_set_variant(int(variant))
    if prev < 0:
        raise ValueError(f"unknown prefill variant {variant}")
    return prev


def ckv_kpool_compress_set_variant(variant: int) -> int:
    """Select the pooled one-shot kernel (0 auto, 1 one warp per pool, 2 bulk-copy pipeline).

    Returns the previous setting; raises on an unknown value."""
    prev = load().ckv_kpool_compress_set_variant(int(variant))
    if prev < 0:
        raise ValueError(f"unknown kpool compress variant {variant}")
    return prev


def ckv_plan_online_prefill_device(seq_lens, extend_lens, num_tokens, compress_plan=None, write_plan=None,
                                   counts=None, pad_for_graph=False, use_pdl=False, err_word=None, stream=None):
    """Device-side planner; see ckv_plan_online_prefill_device in include/ckv.h.

    seq_lens/extend_lens: CUDA int64 tensors [B].  Returns (compress_plan,
    write_plan, counts) as CUDA tensors (uint8 [num_tokens, 16] x2, int32 [2]);
    nothing is copied to the host.
    """
    L = load()
    _cuda("ckv_plan_online_prefill_device", seq_lens, extend_lens, compress_plan, write_plan, counts, err_word)
    _need(seq_lens.dtype == torch.int64 and extend_lens.dtype == torch.int64 and seq_lens.is_contiguous()
          and extend_lens.is_contiguous() and seq_lens.numel() == extend_lens.numel(),
          "seq_lens/extend_lens must be contiguous int64 [B]")
    dev = seq_lens.device
    if compress_plan is None:
        compress_plan = torch.empty((num_tokens, PLAN_ENTRY_BYTES), dtype=torch.uint8, device=dev)
    if write_plan is None:
        write_plan = torch.empty((num_tokens, PLAN_ENTRY_BYTES), dtype=torch.uint8, device=dev)
    if counts is None:
        counts = torch.zeros((2,), dtype=torch.int32, device=dev)
    for pl in (compress_plan, write_plan):
        _need(pl.is_contiguous() and pl.numel() * pl.element_size() >= num_tokens * PLAN_ENTRY_BYTES,
              "plan buffers must hold num_tokens 16-byte rows")
    _need(counts.numel() >= 2 and counts.element_size() == 4, "counts must be a 4-byte tensor of 2 elements")
    _check("ckv_plan_online_prefill_device", L.ckv_plan_online_prefill_device(
        _ptr(seq_lens), _ptr(extend_lens), seq_lens.numel(), int(num_tokens), _ptr(compress_plan),
        _ptr(write_plan), int(bool(pad_for_graph)), _ptr(counts), int(bool(use_pdl)), _ptr(err_word),
        _stream(stream, seq_lens)))
    return compress_plan, write_plan, counts


def ckv_c128_online_prefill_counted(state, input, out, ape, indices, compress_plan, write_plan, counts,
                                    load_indices=None, use_pdl=False, err_word=None, stream=None):
    """Online c128 prefill with device-resident segment counts; see include/ckv.h."""
    L = load()
    _cuda("ckv_c128_online_prefill_counted", state, input, out, ape, indices, load_indices, compress_plan,
          write_plan, counts, err_word)
    T = input.shape[0]
    D = input.shape[1] // 2
    B = indices.numel()
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [T, 2D]")
    _need(out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (T, D), "out must be float32 [T, D]")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    _need(indices.dtype == torch.int32 and indices.is_contiguous(), "indices must be int32 [B]")
    for pl in (compress_plan, write_plan):
        _need(pl.is_contiguous() and pl.numel() * pl.element_size() >= min(T, T // 128 + B) * PLAN_ENTRY_BYTES,
              "plan tensors too small")
    _check("ckv_c128_online_prefill_counted", L.ckv_c128_online_prefill_counted(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), T, _ptr(out), _ptr(ape), _ptr(indices),
        _ptr(load_indices), B, _ptr(compress_plan), _ptr(write_plan), _ptr(counts), D, int(bool(use_pdl)),
        _ptr(err_word), _stream(stream, input)))


def ckv_c128_online_prefill_counted_fp8(state, input, out, ape, indices, compress_plan, write_plan, counts,
                                        kv_cache, cache_loc, round_scale=True, load_indices=None, use_pdl=False,
                                        err_word=None, stream=None):
    """The device-counted prefill with the FP8 output stage; see include/ckv.h.
    kv_cache uint8 [pages, page_size, D + 4*D/128]; cache_loc int64 [T]; out
    float32 [T, D] or None."""
    L = load()
    _cuda("ckv_c128_online_prefill_counted_fp8", state, input, out, ape, indices, load_indices, compress_plan,
          write_plan, counts, kv_cache, cache_loc, err_word)
    T = input.shape[0]
    D = input.shape[1] // 2
    B = indices.numel()
    _need(state.dtype == torch.float32 and state.is_contiguous() and state.numel() % (3 * D) == 0,
          "state must be contiguous float32 [slots, 3, D]")
    _need(input.is_contiguous() and input.dim() == 2, "input must be contiguous [T, 2D]")
    _need(out is None or (out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (T, D)),
          "out must be float32 [T, D] or None")
    _need(ape.dtype == torch.float32 and ape.is_contiguous() and tuple(ape.shape) == (128, D), "ape must be float32 [128, D]")
    _need(indices.dtype == torch.int32 and indices.is_contiguous(), "indices must be int32 [B]")
    for pl in (compress_plan, write_plan):
        _need(pl.is_contiguous() and pl.numel() * pl.element_size() >= min(T, T // 128 + B) * PLAN_ENTRY_BYTES,
              "plan tensors too small")
    pages, ps = _fp8_cache(kv_cache, cache_loc, D, T)
    _check("ckv_c128_online_prefill_counted_fp8", L.ckv_c128_online_prefill_counted_fp8(
        _ptr(state), state.numel() // (3 * D), _ptr(input), _dtype(input), T, _ptr(out), _ptr(ape), _ptr(indices),
        _ptr(load_indices), B, _ptr(compress_plan), _ptr(write_plan), _ptr(counts), D, _ptr(kv_cache), pages, ps,
        _ptr(cache_loc), int(bool(round_scale)), int(bool(use_pdl)), _ptr(err_word), _stream(stream, input)))


def ckv_plan_online_prefill(seq_lens, extend_lens, num_tokens=None, pad_for_graph=False,
                            compress_plan=None, write_plan=None):
    """Host planner; see ckv_plan_online_prefill in include/ckv.h.

    seq_lens/extend_lens: CPU int64 tensors [B].  Returns (compress_plan,
    write_plan, num_compress, num_write) with the plans as CPU uint8 tensors
    [num_tokens, 16] (pass pinned tensors to fill them in place).
    """
    L = load()
    _need(not seq_lens.is_cuda and not extend_lens.is_cuda, "planner inputs must be host tensors")
    seq_lens = seq_lens.to(torch.int64).contiguous()
    extend_lens = extend_lens.to(torch.int64).contiguous()
    B = seq_lens.numel()
    if num_tokens is None:
        num_tokens = int(extend_lens.sum())
    if compress_plan is None:
        compress_plan = torch.empty((num_tokens, PLAN_ENTRY_BYTES), dtype=torch.uint8)
    if write_plan is None:
        write_plan = torch.empty((num_tokens, PLAN_ENTRY_BYTES), dtype=torch.uint8)
    for pl in (compress_plan, write_plan):
        _need(not pl.is_cuda and pl.is_contiguous() and pl.numel() * pl.element_size() >= num_tokens * 16,
              "plan buffers must be host tensors of num_tokens 16-byte rows")
    nc = ctypes.c_uint32()
    nw = ctypes.c_uint32()
    _check("ckv_plan_online_prefill", L.ckv_plan_online_prefill(
        _ptr(seq_lens), _ptr(extend_lens), B, num_tokens, _ptr(compress_plan), _ptr(write_plan),
        int(bool(pad_for_graph)), ctypes.byref(nc), ctypes.byref(nw)))
    return compress_plan, write_plan, nc.value, nw.value


# ------------------------------------------------------------ contract check
def ckv_check_distinct(ids, id_range, scratch, err_word, stream=None):
    """Flag repeated or out-of-range ids; see ckv_check_distinct in include/ckv.h.

    ids: CUDA int32 or int64 tensor (flattened; negative entries ignored);
    scratch: CUDA int32 tensor of at least ceil(id_range / 32) elements
    (overwritten); err_word: CUDA int32 [1], CKV_DEVERR_DISTINCT (0x40) is
    OR-ed into it on a violation.
    """
    L = load()
    _cuda("ckv_check_distinct", ids, scratch, err_word)
    _need(ids.dtype in (torch.int32, torch.int64) and ids.is_contiguous(), "ids must be contiguous int32/int64")
    _need(scratch.dtype == torch.int32 and scratch.is_contiguous(), "scratch must be contiguous int32")
    _need(err_word.dtype == torch.int32, "err_word must be int32")
    _check("ckv_check_distinct", L.ckv_check_distinct(
        _ptr(ids), ids.element_size(), ids.numel(), int(id_range), _ptr(scratch), scratch.numel(),
        _ptr(err_word), _stream(stream, ids)))


NOALLOC_MAX_RANGE = 1 << 21


def ckv_check_distinct_noalloc(ids, id_range, err_word, stream=None):
    """ckv_check_distinct with the library's own static bitmap (no scratch
    argument, nothing allocated); for callers that cannot allocate device
    memory.  id_range must be at most NOALLOC_MAX_RANGE (2^21).  The first call
    on a device looks up the bitmap's address: make it before any stream
    capture.  Calls that overlap on the GPU share the bitmap and race."""
    L = load()
    _cuda("ckv_check_distinct_noalloc", ids, err_word)
    _need(ids.dtype in (torch.int32, torch.int64) and ids.is_contiguous(), "ids must be contiguous int32/int64")
    _need(err_word.dtype == torch.int32, "err_word must be int32")
    _check("ckv_check_distinct_noalloc", L.ckv_check_distinct_noalloc(
        _ptr(ids), ids.element_size(), ids.numel(), int(id_range), _ptr(err_word), _stream(stream, ids)))


def ckv_latency_probe(hops, n_warps, idx=None, rows=None, out=None, warps_per_cta=4, use_pdl=False, stream=None):
    """Latency floor of a decode-sized launch (see include/ckv.h): hops 0, 1 or
    2 dependent global round trips per warp, 3 for one round trip with the
    pooled decode's first-hop loads, 4 for the pooled decode's memory pattern
    without its arithmetic.  idx int32 [n_warps]; rows and out uint8 [*, 256]
    (out: n_warps rows, 4 * n_warps for hops 4); stream defaults to the current
    stream."""
    L = load()
    _cuda("ckv_latency_probe", idx, rows, out)
    if idx is not None:
        _need(idx.dtype == torch.int32 and idx.is_contiguous() and idx.numel() >= n_warps, "idx must be int32 [n_warps]")
    for t in (rows, out):
        if t is not None:
            _need(t.dtype == torch.uint8 and t.is_contiguous() and t.dim() == 2 and t.shape[1] == 256,
                  "rows/out must be contiguous uint8 [n, 256]")
    if out is not None:
        _need(out.shape[0] >= (4 if hops == 4 else 1) * n_warps, "out must have n_warps rows (4 n_warps for hops 4)")
    num_rows = rows.shape[0] if rows is not None else 0
    if stream is None:
        stream = torch.cuda.current_stream()
    strm = ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    _check("ckv_latency_probe", L.ckv_latency_probe(int(hops), _ptr(idx), _ptr(rows), num_rows, _ptr(out),
                                                    int(n_warps), int(warps_per_cta), int(bool(use_pdl)), strm))
