"""Seeded synthetic inputs for the five measured workloads.

This module only draws random numbers and lays out index arrays the way a
serving engine hands them over (tail slots, cache locations, ragged lengths);
it contains none of the compression arithmetic.  Both the CUDA path and the
CPU oracle are fed from it.  Every generator takes a ``device`` (tensors are
drawn there with a torch.Generator seeded by ``seed``) and size overrides so
that tests can run the same recipe at smaller sizes.

Workloads (sizes are the defaults):
  tiny_pooled     4 requests x 64 tokens, P=16, D=128, empty ring, 16 pools
  pooled_decode   512 requests x 4 verify tokens, P=16, D=128, start positions
                  U[0, 32768), prefilled ring, 5% padded entries
  c128_decode     2048 requests, D=512 fp32, 4096-slot state pool, seq_lens
                  U[1, 131072], random mid-chunk states
  c128_prefill    64 requests, D=512 fp32, prefix U[0, 16384], extend
                  U[1, 8192], ragged layout
  long_context    8 requests x 131072 tokens, zero prefix, D=512 bf16 with
                  Student-t (nu=3) scores; plus the pooled P=16, D=128 path on
                  the same token count
"""
from __future__ import annotations

import torch

BF16 = torch.bfloat16
F32 = torch.float32


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, scale=1.0, dtype=F32):
    x = torch.randn(shape, generator=g, device=device, dtype=F32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def _randint(lo, hi_inclusive, shape, g, device):
    return torch.randint(lo, hi_inclusive + 1, shape, generator=g, device=device, dtype=torch.int64)


def student_t(shape, nu3_gen, device):
    """Student-t draws with nu = 3: Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3)."""
    z = torch.randn(shape, generator=nu3_gen, device=device, dtype=F32)
    v = torch.zeros(shape, device=device, dtype=F32)
    for _ in range(3):
        w = torch.randn(shape, generator=nu3_gen, device=device, dtype=F32)
        v.addcmul_(w, w)
    return z / torch.sqrt(v / 3.0)


def random_states(num_slots, D, g, device):
    """Random running states (max | sum | kv) of partially filled chunks.

    max ~ N(1.5, 0.5), sum ~ U[1, 128] (the max token contributes 1, at most
    127 others contribute up to 1 each), kv ~ N(0, 0.3).
    """
    st = torch.empty((num_slots, 3, D), device=device, dtype=F32)
    st[:, 0] = _randn((num_slots, D), g, device) * 0.5 + 1.5
    st[:, 1] = torch.rand((num_slots, D), generator=g, device=device, dtype=F32) * 127.0 + 1.0
    st[:, 2] = _randn((num_slots, D), g, device, 0.3)
    return st


def prior_chunk_tokens(seq_lens, D, seed, device="cpu", dtype=F32):
    """Virtual earlier tokens of each request's current 128-token chunk: the
    new token of request b sits at chunk position p_b = (seq_lens[b] - 1) % 128,
    so p_b tokens (kv | score ~ N(0, 1)) came before it in its chunk.  They are
    laid out request after request in one ragged array [sum p_b, 2D]; a
    caller builds a consistent running state from them.  Returns (rows, p)."""
    seq = torch.as_tensor(seq_lens, dtype=torch.int64).cpu()
    p = (seq - 1) % 128
    g = _gen(device, seed)
    rows = _randn((int(p.sum()), 2 * D), g, device, dtype=dtype)
    return rows, p


# ---------------------------------------------------------------- pooled P=16
def tiny_pooled(device="cpu", seed=0, B=4, N=64, P=16, D=128, page_size=64):
    """B requests with positions 0..N-1 each; request b uses tail block b and
    cache locations b*(N/P) + pos/P; the ring starts empty (zeros)."""
    g = _gen(device, seed)
    key = _randn((B, N, D), g, device, dtype=BF16)
    score = _randn((B, N, D), g, device, dtype=BF16)
    ape = _randn((P, D), g, device, 0.1, dtype=BF16).to(F32)
    pos = torch.arange(N, device=device, dtype=torch.int64).expand(B, N)
    req = torch.arange(B, device=device, dtype=torch.int64)[:, None]
    tslot = req * P + pos % P
    loc = torch.where(pos % P == P - 1, req * (N // P) + pos // P, torch.full_like(pos, -1))
    rows = max(1, B * (N // P))
    pages = (rows + page_size - 1) // page_size
    out = {
        "key": key, "score": score, "ape": ape,
        "positions": pos.to(torch.int32).contiguous(),
        "tail_slot_mapping": tslot.to(torch.int32).contiguous(),
        "slot_mapping": loc.to(torch.int32).contiguous(),
        "ring": torch.zeros((B, 2, P, D), device=device, dtype=BF16),
        "kv_cache": torch.zeros((pages, page_size, D + 4), device=device, dtype=torch.uint8),
        "page_size": page_size, "P": P, "D": D, "B": B, "N": N,
    }
    if N % P == 0:
        # the same tokens as one-shot pools: [B * N/P, P, D], cache location = pool index
        out["slot_k"] = key.reshape(B * (N // P), P, D).contiguous()
        out["slot_score"] = score.reshape(B * (N // P), P, D).contiguous()
        out["loc"] = torch.arange(B * (N // P), device=device, dtype=torch.int64)
    return out


def pooled_decode(device="cpu", seed=0, B=512, N=4, P=16, D=128, max_start=32768,
                  pad_frac=0.05, page_size=64):
    """Decode/verify batch: request b's N tokens sit at positions start_b + t
    (start_b ~ U[0, max_start)), it owns tail block perm[b] of a ring that is
    prefilled with N(0,1) keys and scores, and its pool p has cache location
    b * (max_start/P + 1) + p.  Each (request, token) entry is padded
    (all three index arrays -1) with probability pad_frac."""
    g = _gen(device, seed)
    key = _randn((B, N, D), g, device, dtype=BF16)
    score = _randn((B, N, D), g, device, dtype=BF16)
    ape = _randn((P, D), g, device, 0.1, dtype=BF16).to(F32)
    ring = _randn((B, 2, P, D), g, device, dtype=BF16)
    blocks = torch.randperm(B, generator=g, device=device)
    start = torch.randint(0, max_start, (B,), generator=g, device=device, dtype=torch.int64)
    pos = start[:, None] + torch.arange(N, device=device, dtype=torch.int64)[None, :]
    pools_per_req = max_start // P + (N + P - 1) // P
    req = torch.arange(B, device=device, dtype=torch.int64)[:, None]
    tslot = blocks[:, None] * P + pos % P
    loc = torch.where(pos % P == P - 1, req * pools_per_req + pos // P, torch.full_like(pos, -1))
    pad = torch.rand((B, N), generator=g, device=device) < pad_frac
    neg = torch.full_like(pos, -1)
    rows = B * pools_per_req
    pages = (rows + page_size - 1) // page_size
    return {
        "key": key, "score": score, "ape": ape, "ring": ring,
        "positions": torch.where(pad, neg, pos).to(torch.int32).contiguous(),
        "tail_slot_mapping": torch.where(pad, neg, tslot).to(torch.int32).contiguous(),
        "slot_mapping": torch.where(pad, neg, loc).to(torch.int32).contiguous(),
        "kv_cache": torch.zeros((pages, page_size, D + 4), device=device, dtype=torch.uint8),
        "page_size": page_size, "P": P, "D": D, "B": B, "N": N,
    }


# ------------------------------------------------------------ online c128
def c128_decode(device="cpu", seed=0, B=2048, D=512, num_slots=4096, max_seq=131072, dtype=F32):
    """Decode batch: request b owns slot indices[b] (distinct, drawn from a
    permutation of num_slots), its new token is the seq_lens[b]-th of its
    sequence (seq_lens ~ U[1, max_seq]); input rows kv | score ~ N(0, 1)."""
    g = _gen(device, seed)
    state = random_states(num_slots, D, g, device)
    inp = _randn((B, 2 * D), g, device, dtype=dtype)
    ape = _randn((128, D), g, device, 0.1)
    indices = torch.randperm(num_slots, generator=g, device=device)[:B].to(torch.int32)
    seq_lens = _randint(1, max_seq, (B,), g, device).to(torch.int32)
    return {"state": state, "input": inp, "ape": ape, "indices": indices.contiguous(),
            "seq_lens": seq_lens.contiguous(), "out": torch.zeros((B, D), device=device, dtype=F32),
            "B": B, "D": D}


def c128_prefill(device="cpu", seed=0, B=64, D=512, max_prefix=16384, max_extend=8192,
                 num_slots=None, dtype=F32, score_dist="normal", zero_prefix=False):
    """Prefill batch: request b has prefix_b ~ U[0, max_prefix] cached tokens
    (a random partial state in slot indices[b]) and extend_b ~ U[1, max_extend]
    new tokens laid out back to back in the ragged input [sum(extend), 2D].
    Scores are N(0, 1) or Student-t(3)."""
    g = _gen(device, seed)
    num_slots = num_slots or 2 * B
    if zero_prefix:
        prefix = torch.zeros((B,), dtype=torch.int64)
        extend = torch.full((B,), max_extend, dtype=torch.int64)
    else:
        gh = _gen("cpu", seed)  # lengths are host data
        prefix = torch.randint(0, max_prefix + 1, (B,), generator=gh, dtype=torch.int64)
        extend = torch.randint(1, max_extend + 1, (B,), generator=gh, dtype=torch.int64)
    T = int(extend.sum())
    state = random_states(num_slots, D, g, device)
    kv = _randn((T, D), g, device)
    if score_dist == "student_t":
        sc = student_t((T, D), g, device)
    else:
        sc = _randn((T, D), g, device)
    inp = torch.cat([kv, sc], dim=1).to(dtype).contiguous()
    del kv, sc
    ape = _randn((128, D), g, device, 0.1)
    indices = torch.randperm(num_slots, generator=g, device=device)[:B].to(torch.int32).contiguous()
    return {"state": state, "input": inp, "ape": ape, "indices": indices,
            "seq_lens": (prefix + extend), "extend_lens": extend, "num_tokens": T,
            "out": torch.zeros((T, D), device=device, dtype=F32), "B": B, "D": D}


def long_context(device="cpu", seed=0, B=8, T=131072, D=512, P=16, Dp=128, page_size=64):
    """Long-context prefill sweep: B requests x T tokens from position 0.
    c128 part: bf16 [B*T, 2D] with N(0,1) kv and Student-t(3) scores, fp32 state.
    Pooled part: the same token count as B*T/P one-shot pools of [P, Dp] bf16
    keys (N(0,1)) and Student-t(3) scores; pool p is written at cache location p."""
    c = c128_prefill(device, seed, B=B, D=D, max_extend=T, dtype=BF16, score_dist="student_t",
                     zero_prefix=True, num_slots=B)
    g = _gen(device, seed + 1)
    n_pools = B * T // P
    slot_k = _randn((n_pools, P, Dp), g, device, dtype=BF16)
    slot_score = student_t((n_pools, P, Dp), g, device).to(BF16)
    ape_p = _randn((P, Dp), g, device, 0.1, dtype=BF16).to(F32)
    pages = (n_pools + page_size - 1) // page_size
    c.update({
        "slot_k": slot_k, "slot_score": slot_score, "ape_pool": ape_p,
        "loc": torch.arange(n_pools, device=device, dtype=torch.int64),
        "kv_cache": torch.zeros((pages, page_size, Dp + 4), device=device, dtype=torch.uint8),
        "page_size": page_size, "n_pools": n_pools, "P": P, "Dp": Dp,
    })
    return c
