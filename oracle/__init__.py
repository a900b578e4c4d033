"""CPU oracle for gated-softmax KV compression (TEST INFRASTRUCTURE).

This package is the independent reference the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product path never does.  It shares no
code with the CUDA sources: the arithmetic lives in ``ckv_oracle.cpp`` (plain
loops, double precision except where the pages fix a narrower format), and
this module only compiles that file and marshals numpy arrays into it.

Sources, cited by page title and routine:
  [KPOOL] "vllm.models.glm5next.amd.ops.kpool_compress" (vLLM docs page)
  [C128]  "sgl-project--sglang/.../deepseek_v4/c128_online.cuh" (sglang page)

Every oracle function is pinned by ``tests/test_oracle_pins.py`` against
closed forms, invariants, library routines and brute force.  Functions with
no such pin say so in their docstring ("parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ckv_oracle.cpp")
_LIB = os.path.join(_HERE, "libckv_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-pthread"]


def build(force: bool = False) -> str:
    """Compile ``ckv_oracle.cpp`` into ``libckv_oracle.so`` (g++, host ISA neutral)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", *CFLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _p(a, ct):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ct))


def lib():
    """The oracle library: ``libckv_oracle.so`` built from ``ckv_oracle.cpp``,
    or the build named by CKV_ORACLE_SO (the mutation tests point it at a copy
    with a planted mistake, to show that the pins catch it)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("CKV_ORACLE_SO") or build()
            L = ctypes.CDLL(path)
            P = ctypes.POINTER
            f32, f64, u8, u16, i32, i64, u32 = (ctypes.c_float, ctypes.c_double, ctypes.c_uint8,
                                                ctypes.c_uint16, ctypes.c_int32, ctypes.c_int64,
                                                ctypes.c_uint32)
            ci = ctypes.c_int
            sig = {
                "ora_bf16_from_double": (u16, [f64]),
                "ora_bf16_to_float": (f32, [u16]),
                "ora_e4m3_encode": (u8, [f32]),
                "ora_e4m3_decode": (f32, [u8]),
                "ora_pow2_ceil": (f32, [f32]),
                "ora_hadamard128_exact": (None, [P(f64), P(f64)]),
                "ora_hadamard128_fp32": (None, [P(f32), P(f32)]),
                "ora_quantize_row": (None, [P(u16), ci, ci, P(u8), P(f32)]),
                "ora_rotate_bf16": (None, [P(u16), P(u16)]),
                "ora_pool_compress": (None, [P(f32), P(f32), P(f32), ci, ci, ci, P(f64), P(u16),
                                             P(u16), P(u8), P(f32)]),
                "ora_kpool_compress": (None, [P(u8), i64, i64, P(u16), P(u16), P(f32), P(i64), P(u8),
                                              ci, P(u8), P(f32), i64, ci, ci, ci, P(f64), P(u16),
                                              P(u16), ci]),
                "ora_kpool_decode_update": (None, [P(u8), i64, i64, P(u16), i64, P(i32), P(i32),
                                                   P(i32), P(u16), P(u16), P(f32), ci, ci, ci, ci,
                                                   ci, P(f64), P(u16), P(u16), ci]),
                "ora_kpool_seed_tail": (None, [P(u16), i64, P(u16), P(u16), P(i32), i64, ci, ci]),
                "ora_c128_decode": (None, [P(f32), ctypes.c_void_p, ci, P(f32), P(i32), P(i32), ci,
                                           ci, P(f64), P(f64), P(i32), ci]),
                "ora_c128_prefill": (None, [P(f32), ctypes.c_void_p, ci, i64, P(f32), P(i32), P(i64),
                                            P(i64), ci, ci, P(f64), P(u8), P(f64), P(i32), ci]),
                "ora_plan_segments": (ci, [P(i64), P(i64), ci, P(u32), P(u32), i64, P(i64), P(i64)]),
                "ora_expand_pools_and_append_tail": (None, [P(i32), i64, P(i64), ci, ci, ci, P(i32)]),
                "ora_c128_rows_to_cache": (None, [P(u8), i64, P(f32), P(i64), i64, ci, ci]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------- formats
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_from_double(x: float) -> int:
    return int(lib().ora_bf16_from_double(float(x)))


def e4m3_encode(x: float) -> int:
    return int(lib().ora_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(lib().ora_e4m3_decode(int(c)))


def pow2_ceil(v: float) -> float:
    return float(lib().ora_pow2_ceil(float(v)))


def hadamard128_exact(x: np.ndarray) -> np.ndarray:
    """Orthonormal Sylvester Hadamard-128 of a vector, dense product in double."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(128, np.float64)
    lib().ora_hadamard128_exact(_p(x, ctypes.c_double), _p(out, ctypes.c_double))
    return out


def hadamard128_fp32(x: np.ndarray) -> np.ndarray:
    """The fp32 butterfly reading of the rotation (spans 1..64 ascending, then * fp32(1/sqrt(128)))."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(128, np.float32)
    lib().ora_hadamard128_fp32(_p(x, ctypes.c_float), _p(out, ctypes.c_float))
    return out


def rotate_bf16(xb: np.ndarray) -> np.ndarray:
    """yb = bf16(H128_fp32(xb)) for each row of a bf16-bits array [..., 128]."""
    xb = np.ascontiguousarray(xb, dtype=np.uint16).reshape(-1, 128)
    yb = np.empty_like(xb)
    L = lib()
    for r in range(xb.shape[0]):
        L.ora_rotate_bf16(_p(xb[r], ctypes.c_uint16), _p(yb[r], ctypes.c_uint16))
    return yb


def quantize_rows(yb: np.ndarray, round_scale: bool):
    """Absmax FP8 quantisation of bf16-bits rows [..., D] -> (codes uint8, scales float32)."""
    yb = np.ascontiguousarray(yb, dtype=np.uint16)
    D = yb.shape[-1]
    rows = yb.reshape(-1, D)
    q = np.empty(rows.shape, np.uint8)
    sc = np.empty(rows.shape[0], np.float32)
    L = lib()
    for r in range(rows.shape[0]):
        s = ctypes.c_float()
        L.ora_quantize_row(_p(rows[r], ctypes.c_uint16), D, int(round_scale),
                           _p(q[r], ctypes.c_uint8), ctypes.byref(s))
        sc[r] = s.value
    return q.reshape(yb.shape), sc.reshape(yb.shape[:-1])


def pool_compress(k: np.ndarray, s: np.ndarray, ape: np.ndarray, round_scale: bool):
    """One pool from fp32 keys/scores [P, D] (D=128) -> dict of x, xb, yb, q, scale."""
    k = np.ascontiguousarray(k, np.float32)
    s = np.ascontiguousarray(s, np.float32)
    ape = np.ascontiguousarray(ape, np.float32)
    P, D = k.shape
    assert D == 128
    x = np.empty(D, np.float64)
    xb = np.empty(D, np.uint16)
    yb = np.empty(D, np.uint16)
    q = np.empty(D, np.uint8)
    sc = ctypes.c_float()
    lib().ora_pool_compress(_p(k, ctypes.c_float), _p(s, ctypes.c_float), _p(ape, ctypes.c_float),
                            P, D, int(round_scale), _p(x, ctypes.c_double), _p(xb, ctypes.c_uint16),
                            _p(yb, ctypes.c_uint16), _p(q, ctypes.c_uint8), ctypes.byref(sc))
    return {"x": x, "xb": xb, "yb": yb, "q": q, "scale": np.float32(sc.value)}


# --------------------------------------------------------- pooled (kpool)
def kpool_compress(cache, page_size, slot_k, slot_score, ape, loc, write_mask=None,
                   write_cache=True, return_compressed=False, round_scale=True, taps=False,
                   threads=None):
    """[KPOOL] one-shot pooled compression; updates ``cache`` (uint8 [pages, ps, D+4]) in place.

    slot_k / slot_score: bf16 bits uint16 [n, P, D]; ape float32 [P, D]; loc int64 [n].
    Returns dict with optional 'q', 'scale', 'x', 'xb', 'yb'.
    """
    n, P, D = slot_k.shape
    slot_k = np.ascontiguousarray(slot_k, np.uint16)
    slot_score = np.ascontiguousarray(slot_score, np.uint16)
    ape = np.ascontiguousarray(ape, np.float32)
    loc = np.ascontiguousarray(loc, np.int64)
    wm = None if write_mask is None else np.ascontiguousarray(write_mask, np.uint8)
    res = {}
    q = sc = tx = txb = tyb = None
    if return_compressed:
        q = res["q"] = np.zeros((n, D), np.uint8)
        sc = res["scale"] = np.zeros(n, np.float32)
    if taps:
        tx = res["x"] = np.full((n, D), np.nan, np.float64)
        txb = res["xb"] = np.zeros((n, D), np.uint16)
        tyb = res["yb"] = np.zeros((n, D), np.uint16)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    lib().ora_kpool_compress(_p(cache, ctypes.c_uint8), cache.shape[0], page_size,
                             _p(slot_k, ctypes.c_uint16), _p(slot_score, ctypes.c_uint16),
                             _p(ape, ctypes.c_float), _p(loc, ctypes.c_int64), _p(wm, ctypes.c_uint8),
                             int(write_cache), _p(q, ctypes.c_uint8), _p(sc, ctypes.c_float), n, P, D,
                             int(round_scale), _p(tx, ctypes.c_double), _p(txb, ctypes.c_uint16),
                             _p(tyb, ctypes.c_uint16), threads or default_threads())
    return res


def kpool_decode_update(cache, page_size, ring, tail_slot_mapping, slot_mapping, positions, key,
                        score, ape, round_scale=True, taps=False, threads=None):
    """[KPOOL] ordered decode/verify update; updates ``cache`` and ``ring`` in place.

    ring: bf16 bits uint16 [blocks, 2, P, D]; index arrays int32 [B, N];
    key/score bf16 bits uint16 [B, N, D]; ape float32 [P, D].
    Taps (rows = flattened token index, NaN/0 where no pool closed).
    """
    B, N, D = key.shape
    P = ring.shape[2]
    for a in (cache, ring):
        assert a.flags.c_contiguous
    tsm = np.ascontiguousarray(tail_slot_mapping, np.int32)
    sm = np.ascontiguousarray(slot_mapping, np.int32)
    pos = np.ascontiguousarray(positions, np.int32)
    key = np.ascontiguousarray(key, np.uint16)
    score = np.ascontiguousarray(score, np.uint16)
    ape = np.ascontiguousarray(ape, np.float32)
    res = {}
    tx = txb = tyb = None
    if taps:
        tx = res["x"] = np.full((B * N, D), np.nan, np.float64)
        txb = res["xb"] = np.zeros((B * N, D), np.uint16)
        tyb = res["yb"] = np.zeros((B * N, D), np.uint16)
    lib().ora_kpool_decode_update(_p(cache, ctypes.c_uint8), cache.shape[0], page_size,
                                  _p(ring, ctypes.c_uint16), ring.shape[0], _p(tsm, ctypes.c_int32),
                                  _p(sm, ctypes.c_int32), _p(pos, ctypes.c_int32),
                                  _p(key, ctypes.c_uint16), _p(score, ctypes.c_uint16),
                                  _p(ape, ctypes.c_float), B, N, P, D, int(round_scale),
                                  _p(tx, ctypes.c_double), _p(txb, ctypes.c_uint16),
                                  _p(tyb, ctypes.c_uint16), threads or default_threads())
    return res


def kpool_seed_tail(ring, key, score, tslot):
    """[KPOOL] tail-ring seed from a prefill batch; updates ``ring`` in place."""
    n, D = key.shape
    P = ring.shape[2]
    key = np.ascontiguousarray(key, np.uint16)
    score = np.ascontiguousarray(score, np.uint16)
    tslot = np.ascontiguousarray(tslot, np.int32)
    lib().ora_kpool_seed_tail(_p(ring, ctypes.c_uint16), ring.shape[0], _p(key, ctypes.c_uint16),
                              _p(score, ctypes.c_uint16), _p(tslot, ctypes.c_int32), n, P, D)


def expand_pools_and_append_tail(pool_ids, seq_lens, P):
    """[KPOOL] pool -> token index expansion with the tail appended; int32 [rows, G*P + P - 1].

    pool_ids int32 [rows, G]: a row-strided view (contiguous rows of a wider
    array) is passed with its own row stride."""
    pool_ids = np.asarray(pool_ids)
    if pool_ids.dtype != np.int32 or pool_ids.ndim != 2 or pool_ids.strides[1] != 4 or pool_ids.strides[0] % 4 \
            or pool_ids.strides[0] < 4 * pool_ids.shape[1]:
        pool_ids = np.ascontiguousarray(pool_ids, np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, np.int64)
    rows, groups = pool_ids.shape
    stride = pool_ids.strides[0] // 4 if rows > 1 else groups
    out = np.empty((rows, groups * P + P - 1), np.int32)
    lib().ora_expand_pools_and_append_tail(_p(pool_ids, ctypes.c_int32), stride, _p(seq_lens, ctypes.c_int64),
                                           rows, groups, P, _p(out, ctypes.c_int32))
    return out


# ------------------------------------------------------------- online c128
def _in_dtype(x):
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:
        return 1
    raise TypeError("input must be float32 or bf16 bits (uint16)")


def c128_decode(state, inp, ape, indices, seq_lens, threads=None):
    """[C128] online decode.  state float32 [slots, 3, D] (read only here); inp [B, 2D].

    Returns (out [B, D] f64, new_state [B, 3, D] f64, closed [B] bool).
    """
    state = np.ascontiguousarray(state, np.float32)
    inp = np.ascontiguousarray(inp)
    ape = np.ascontiguousarray(ape, np.float32)
    indices = np.ascontiguousarray(indices, np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, np.int32)
    B = inp.shape[0]
    D = inp.shape[1] // 2
    out = np.empty((B, D), np.float64)
    ns = np.empty((B, 3, D), np.float64)
    closed = np.empty(B, np.int32)
    lib().ora_c128_decode(_p(state, ctypes.c_float), inp.ctypes.data_as(ctypes.c_void_p), _in_dtype(inp),
                          _p(ape, ctypes.c_float), _p(indices, ctypes.c_int32),
                          _p(seq_lens, ctypes.c_int32), B, D, _p(out, ctypes.c_double),
                          _p(ns, ctypes.c_double), _p(closed, ctypes.c_int32),
                          threads or default_threads())
    return out, ns, closed.astype(bool)


def c128_prefill(state, inp, ape, load_indices, seq_lens, extend_lens, threads=None):
    """[C128] online prefill without a plan.

    Returns (out [T, D] f64 (NaN where unwritten), out_written [T] bool,
             final_state [B, 3, D] f64, state_written [B] bool).
    """
    state = np.ascontiguousarray(state, np.float32)
    inp = np.ascontiguousarray(inp)
    ape = np.ascontiguousarray(ape, np.float32)
    load_indices = np.ascontiguousarray(load_indices, np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, np.int64)
    extend_lens = np.ascontiguousarray(extend_lens, np.int64)
    T = inp.shape[0]
    D = inp.shape[1] // 2
    B = seq_lens.shape[0]
    out = np.full((T, D), np.nan, np.float64)
    written = np.zeros(T, np.uint8)
    fs = np.full((B, 3, D), np.nan, np.float64)
    sw = np.zeros(B, np.int32)
    lib().ora_c128_prefill(_p(state, ctypes.c_float), inp.ctypes.data_as(ctypes.c_void_p), _in_dtype(inp),
                           T, _p(ape, ctypes.c_float), _p(load_indices, ctypes.c_int32),
                           _p(seq_lens, ctypes.c_int64), _p(extend_lens, ctypes.c_int64), B, D,
                           _p(out, ctypes.c_double), _p(written, ctypes.c_uint8),
                           _p(fs, ctypes.c_double), _p(sw, ctypes.c_int32),
                           threads or default_threads())
    return out, written.astype(bool), fs, sw.astype(bool)


def plan_segments(seq_lens, extend_lens, cap=None):
    """Brute-force segmenter -> (compress [nc, 4] uint32, write [nw, 4] uint32).

    Rows are {ragged_id, batch_id, position, window_len} of each segment's last token.
    """
    seq_lens = np.ascontiguousarray(seq_lens, np.int64)
    extend_lens = np.ascontiguousarray(extend_lens, np.int64)
    B = seq_lens.shape[0]
    if cap is None:
        cap = int(extend_lens.sum()) + 1
    c = np.zeros((cap, 4), np.uint32)
    w = np.zeros((cap, 4), np.uint32)
    nc = ctypes.c_int64()
    nw = ctypes.c_int64()
    rc = lib().ora_plan_segments(_p(seq_lens, ctypes.c_int64), _p(extend_lens, ctypes.c_int64), B,
                                 _p(c, ctypes.c_uint32), _p(w, ctypes.c_uint32), cap, ctypes.byref(nc),
                                 ctypes.byref(nw))
    if rc != 0:
        raise ValueError("plan capacity exceeded")
    return c[: nc.value].copy(), w[: nw.value].copy()


def c128_rows_to_cache(cache, page_size, rows, locs, round_scale=True):
    """Store fp32 rows [n, D] into the paged FP8 cache (uint8 [pages, page_size,
    D + 4*D/128], updated in place), 128-channel block by block through the
    pooled output stage; rows with a negative location are skipped."""
    rows = np.ascontiguousarray(rows, dtype=np.float32)
    locs = np.ascontiguousarray(locs, dtype=np.int64)
    n, D = rows.shape
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[2] == D + 4 * (D // 128)
    lib().ora_c128_rows_to_cache(_p(cache, ctypes.c_uint8), int(page_size), _p(rows, ctypes.c_float),
                                 _p(locs, ctypes.c_int64), n, D, int(bool(round_scale)))
    return cache
