"""GPU parity of the pooled (P <= 16, D = 128) path against the CPU oracle.

Source: vLLM page "kpool_compress" (_kpool_decode_update_batched_kernel,
_kpool_softmax_rotate_write_cache_kernel, _kpool_tail_seed_kernel).  Every
call goes through the C ABI (libckv.so) via the ctypes binding.

Bit-exactness is checked stage by stage (the oracle's rotation fed the GPU's
bf16 row must give the GPU's rotated row; the oracle's quantiser fed that
must give the GPU's codes and scale) and end to end (rows whose bf16 pooled
value agrees are identical; the pooled fp32 value is within tolerance).
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_rel, bf16_bits, bf16_flip_check, bf16_values, cache_rows, f32, u8

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


@pytest.fixture(params=[1, 2], ids=["warp_per_pool", "bulk_pipeline"])
def cvariant(request, ck):
    """Run a one-shot compression test with each kernel."""
    prev = ck.ckv_kpool_compress_set_variant(request.param)
    yield request.param
    ck.ckv_kpool_compress_set_variant(prev)


_E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def e4m3_values(codes):
    """Decoded OCP e4m3 values of uint8 codes (torch's float8_e4m3fn table)."""
    return _E4M3[np.asarray(codes, np.uint8)]


def ora_bf16_bits(x):
    """bf16 round-to-nearest-even of fp32 values (torch CPU cast), as bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_rows(ora, gpu_x, gpu_xb, gpu_yb, gpu_q, gpu_s, ref, round_scale, what):
    """Stage-wise and end-to-end comparison of pooled rows.

    The chain x -> bf16 -> rotation -> bf16 -> FP8 is checked link by link:
    x within the tolerance; the GPU's bf16 row is the round-to-nearest-even of
    its own x; it differs from the oracle's bf16 row only in channels where a
    rounding boundary lies between the two x values, no more often than the
    measured fp32 error makes likely (bf16_flip_check); the oracle's rotation
    of the GPU's bf16 row is the GPU's rotated row and the oracle's quantiser
    of that gives the GPU's codes and scale, bit for bit.  So rows whose bf16
    row agrees have the oracle's codes and scale exactly, and every other row
    is the exact image of a legitimately rounded bf16 row.  Returns the
    number of rows with a flipped bf16 channel."""
    assert_close_rel(gpu_x, ref["x"], what + " x")
    np.testing.assert_array_equal(ora.rotate_bf16(gpu_xb), gpu_yb, err_msg=what + " rotation stage")
    q2, s2 = ora.quantize_rows(gpu_yb, round_scale)
    np.testing.assert_array_equal(q2, gpu_q, err_msg=what + " quant stage codes")
    np.testing.assert_array_equal(s2.view(np.uint32), gpu_s.view(np.uint32), err_msg=what + " quant stage scales")
    same = np.all(gpu_xb == ref["xb"], axis=1)
    np.testing.assert_array_equal(gpu_q[same], ref["q"][same], err_msg=what + " codes (same xb rows)")
    np.testing.assert_array_equal(gpu_s[same].view(np.uint32), ref["scale"][same].view(np.uint32))
    np.testing.assert_array_equal(ora_bf16_bits(gpu_x), gpu_xb, err_msg=what + " bf16 rounding stage")
    rows, _, _ = bf16_flip_check(gpu_x, gpu_xb, ref["x"], ref["xb"], what)
    check_dequantised(gpu_xb, gpu_yb, gpu_q, gpu_s, ref, what)
    return rows


def _bf16_half_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


def _e4m3_half_quantum(t):
    """Half the spacing of e4m3 values around |t| (3 mantissa bits; subnormal spacing 2^-9)."""
    a = np.maximum(np.abs(t), 2.0 ** -6)
    return np.exp2(np.floor(np.log2(a)) - 4)


def check_dequantised(gpu_xb, gpu_yb, gpu_q, gpu_s, ref, what):
    """End to end in value space, with bounds derived per element: the rotated
    rows differ by no more than the rotation of the bf16 difference (its 1-norm
    over sqrt(128)) plus the two bf16 roundings and the fp32 butterfly's
    rounding; the dequantised codes differ by no more than that plus half an
    e4m3 step of each side at its own scale."""
    xg, xr = bf16_values(gpu_xb), bf16_values(ref["xb"])
    yg, yr = bf16_values(gpu_yb), bf16_values(ref["yb"])
    dx = np.abs(xg - xr).sum(axis=1, keepdims=True) / np.sqrt(128.0)
    top = np.maximum(np.abs(yg).max(axis=1, keepdims=True), np.abs(yr).max(axis=1, keepdims=True))
    bound_y = dx * (1 + 1e-6) + _bf16_half_ulp(yg) + _bf16_half_ulp(yr) + 2.0 ** -20 * top
    assert np.all(np.abs(yg - yr) <= bound_y), what + " rotated rows"
    sg = gpu_s.astype(np.float64)[:, None]
    sr = ref["scale"].astype(np.float64)[:, None]
    dq_g, dq_r = e4m3_values(gpu_q) * sg, e4m3_values(ref["q"]) * sr
    bound_q = np.abs(yg - yr) + sg * _e4m3_half_quantum(yg / sg) + sr * _e4m3_half_quantum(yr / sr)
    assert np.all(np.abs(dq_g - dq_r) <= bound_q * (1 + 1e-6)), what + " dequantised rows"


# ------------------------------------------------------------------ one-shot
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("round_scale", [True, False])
def test_kpool_compress_vs_oracle(cvariant, ck, ora, P, round_scale):
    from compressed_kv_attention_gated_gb300 import synth

    n = 203  # several CTAs of 8 pools and a ragged tail
    g = torch.Generator().manual_seed(100 + P)
    slot_k = (torch.randn((n, P, D), generator=g)).to(torch.bfloat16)
    slot_s = (torch.randn((n, P, D), generator=g) * 2).to(torch.bfloat16)
    ape = (torch.randn((P, D), generator=g) * 0.1)
    ps = 64
    pages = (n + ps - 1) // ps + 1
    loc = torch.randperm(pages * ps, generator=g)[:n].to(torch.int64)
    cache0 = torch.full((pages, ps, D + 4), 0x5A, dtype=torch.uint8)
    dev = "cuda"
    cache = cache0.to(dev)
    out_q = torch.zeros((n, D), dtype=torch.uint8, device=dev)
    out_s = torch.zeros((n,), dtype=torch.float32, device=dev)
    tx = torch.zeros((n, D), dtype=torch.float32, device=dev)
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_compress(slot_k.to(dev), slot_s.to(dev), ape.to(dev), kv_cache=cache, loc=loc.to(dev),
                          out_fp8=out_q, out_scale=out_s, round_scale=round_scale, tap_x=tx, tap_xb=txb,
                          tap_yb=tyb, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_cache = u8(cache0).copy()
    ref = ora.kpool_compress(ref_cache, ps, bf16_bits(slot_k), bf16_bits(slot_s), f32(ape), loc.numpy(),
                             return_compressed=True, round_scale=round_scale, taps=True)
    gq, gs = u8(out_q), f32(out_s)
    check_rows(ora, f32(tx), bf16_bits(txb), bf16_bits(tyb), gq, gs, ref, round_scale,
               f"one-shot P={P} round={round_scale} variant={cvariant}")
    # the cache holds the same rows at loc, and nothing else changed
    gcache = u8(cache)
    cq, cs = cache_rows(gcache, ps, D, loc.numpy())
    np.testing.assert_array_equal(cq, gq)
    np.testing.assert_array_equal(cs.view(np.uint32), gs.view(np.uint32))
    rq, rs = cache_rows(ref_cache, ps, D, loc.numpy())
    mask = np.ones(gcache.size, bool)
    flat = np.arange(gcache.size).reshape(gcache.shape)
    for l in loc.numpy():
        page, tok = divmod(int(l), ps)
        base = page * ps * (D + 4)
        mask[base + tok * D: base + tok * D + D] = False
        mask[base + ps * D + 4 * tok: base + ps * D + 4 * tok + 4] = False
    assert np.all(gcache.reshape(-1)[mask] == 0x5A), "bytes outside the written rows changed"


@pytest.mark.parametrize("ps", [1, 48, 100])
def test_kpool_page_sizes(cvariant, ck, ora, ps):
    """Cache pages of 1 row (a shift by 0) and of 48 or 100 rows (not powers of
    two: the kernels divide instead of shifting): the one-shot rows against the
    oracle stage by stage, each stored exactly at its location's page and row
    with every other byte untouched; the decode with the same page size."""
    from compressed_kv_attention_gated_gb300 import synth

    n, P = 777, 16
    g = torch.Generator().manual_seed(ps)
    slot_k = torch.randn((n, P, D), generator=g).to(torch.bfloat16)
    slot_s = torch.randn((n, P, D), generator=g).to(torch.bfloat16)
    ape = torch.randn((P, D), generator=g) * 0.1
    pages = (n + ps - 1) // ps + 2
    loc = torch.randperm(pages * ps, generator=g)[:n].to(torch.int64)
    cache0 = torch.full((pages, ps, D + 4), 0x5A, dtype=torch.uint8)
    dev = "cuda"
    cache = cache0.to(dev)
    out_q = torch.zeros((n, D), dtype=torch.uint8, device=dev)
    out_s = torch.zeros((n,), dtype=torch.float32, device=dev)
    tx = torch.zeros((n, D), device=dev)
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_compress(slot_k.to(dev), slot_s.to(dev), ape.to(dev), kv_cache=cache, loc=loc.to(dev),
                          out_fp8=out_q, out_scale=out_s, tap_x=tx, tap_xb=txb, tap_yb=tyb, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = ora.kpool_compress(u8(cache0).copy(), ps, bf16_bits(slot_k), bf16_bits(slot_s), f32(ape), loc.numpy(),
                             return_compressed=True, taps=True)
    gq, gs = u8(out_q), f32(out_s)
    check_rows(ora, f32(tx), bf16_bits(txb), bf16_bits(tyb), gq, gs, ref, True, f"one-shot page_size={ps}")
    gcache = u8(cache)
    cq, cs = cache_rows(gcache, ps, D, loc.numpy())
    np.testing.assert_array_equal(cq, gq)
    np.testing.assert_array_equal(cs.view(np.uint32), gs.view(np.uint32))
    rest = gcache.reshape(-1).copy()
    for l in loc.numpy():
        page, tok = divmod(int(l), ps)
        base = page * ps * (D + 4)
        rest[base + tok * D: base + tok * D + D] = 0x5A
        rest[base + ps * D + 4 * tok: base + ps * D + 4 * tok + 4] = 0x5A
    assert np.all(rest == 0x5A), "bytes outside the written rows changed"
    d = synth.pooled_decode("cpu", seed=ps, B=64, max_start=2048, page_size=ps)
    gpu = _run_decode(ck, d, True)
    _compare_decode(ora, d, gpu, _oracle_decode(ora, d, True), True, f"decode page_size={ps}")


def test_kpool_compress_worked_bf16_tie(cvariant, ck):
    """The hand-worked pool of the oracle pins (P = 2, equal weights, keys (1, 1)
    in channel 0 and (1, 1 - 2^-8) in channel 1): x = 1 - 2^-9 in channel 1 is
    a bf16 tie that goes to 1, so the rotation gives 2c in even channels and 0
    in odd ones; power-of-two scale 2^-11, codes 0x7B and 0x00.  On the GPU the
    equal weights are ex2(0) = 1 exactly and the mean is exact, so the codes are
    exact too."""
    n, P = 3, 2  # three copies of the pool
    k = torch.zeros((n, P, D))
    k[:, :, 0] = 1.0
    k[:, 0, 1], k[:, 1, 1] = 1.0, 1.0 - 2.0 ** -8
    z = torch.zeros((n, P, D), dtype=torch.bfloat16)
    dev = "cuda"
    out_q = torch.zeros((n, D), dtype=torch.uint8, device=dev)
    out_s = torch.zeros((n,), dtype=torch.float32, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_compress(k.to(torch.bfloat16).to(dev), z.to(dev), torch.zeros((P, D), device=dev),
                          write_cache=False, out_fp8=out_q, out_scale=out_s, round_scale=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q = u8(out_q)
    assert np.all(q[:, 0::2] == 0x7B) and np.all(q[:, 1::2] == 0x00)
    assert np.all(f32(out_s) == 2.0 ** -11)


def test_kpool_compress_write_mask_and_cache_only(cvariant, ck, ora):
    n, P = 77, 16
    g = torch.Generator().manual_seed(7)
    slot_k = torch.randn((n, P, D), generator=g).to(torch.bfloat16)
    slot_s = torch.randn((n, P, D), generator=g).to(torch.bfloat16)
    ape = torch.randn((P, D), generator=g) * 0.1
    wm = torch.rand((n,), generator=g) < 0.6
    ps = 16
    pages = (n + ps - 1) // ps
    loc = torch.arange(n, dtype=torch.int64)
    cache0 = torch.full((pages, ps, D + 4), 0xC3, dtype=torch.uint8)
    cache = cache0.cuda()
    tx = torch.full((n, D), float("nan"), device="cuda")
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device="cuda")
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device="cuda")
    ck.ckv_kpool_compress(slot_k.cuda(), slot_s.cuda(), ape.cuda(), kv_cache=cache, loc=loc.cuda(),
                          write_mask=wm.cuda(), tap_x=tx, tap_xb=txb, tap_yb=tyb)
    torch.cuda.synchronize()
    ref_cache = u8(cache0).copy()
    ref = ora.kpool_compress(ref_cache, ps, bf16_bits(slot_k), bf16_bits(slot_s), f32(ape), loc.numpy(),
                             write_mask=wm.numpy().astype(np.uint8), taps=True)
    g_cache = u8(cache)
    gq, gs = cache_rows(g_cache, ps, D, loc.numpy())
    rq, rs = cache_rows(ref_cache, ps, D, loc.numpy())
    w = wm.numpy()
    assert np.all(gq[~w] == 0xC3)
    assert np.all(np.isnan(f32(tx)[~w])), "masked pools computed nothing"
    sub = {"x": ref["x"][w], "xb": ref["xb"][w], "yb": ref["yb"][w], "q": rq[w], "scale": rs[w]}
    check_rows(ora, f32(tx)[w], bf16_bits(txb)[w], bf16_bits(tyb)[w], gq[w], gs[w], sub, True,
               f"write mask variant={cvariant}")


def test_kpool_compress_bad_loc_flags_and_skips(cvariant, ck):
    n, P = 16, 16
    slot = torch.randn((n, P, D), device="cuda").to(torch.bfloat16)
    ape = torch.zeros((P, D), device="cuda")
    ps = 16
    cache = torch.full((1, ps, D + 4), 7, dtype=torch.uint8, device="cuda")
    loc = torch.arange(n, dtype=torch.int64, device="cuda")
    loc[3] = ps  # one past the end
    loc[5] = -2
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_kpool_compress(slot, slot, ape, kv_cache=cache, loc=loc, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x4
    c = u8(cache).reshape(-1)
    assert np.all(c[3 * D:4 * D] == 7) and np.all(c[5 * D:6 * D] == 7)
    assert not np.all(c[4 * D:5 * D] == 7)


@pytest.mark.parametrize("n,masked", [(9001, False), (12007, True)])
def test_kpool_compress_many_pools_per_warp(cvariant, ck, ora, n, masked):
    """More pools than warps in the persistent grid, so every warp reuses its
    stages several times (and skips masked pools)."""
    P = 16
    g = torch.Generator().manual_seed(n)
    slot_k = torch.randn((n, P, D), generator=g).to(torch.bfloat16)
    slot_s = (torch.randn((n, P, D), generator=g) * 2).to(torch.bfloat16)
    ape = torch.randn((P, D), generator=g) * 0.1
    ps = 64
    pages = (n + ps - 1) // ps
    loc = torch.randperm(pages * ps, generator=g)[:n].to(torch.int64)
    wm = (torch.rand((n,), generator=g) < 0.7) if masked else None
    cache0 = torch.full((pages, ps, D + 4), 0x11, dtype=torch.uint8)
    cache = cache0.cuda()
    tx = torch.zeros((n, D), dtype=torch.float32, device="cuda")
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device="cuda")
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device="cuda")
    kw = {}
    if not masked:
        kw["out_fp8"] = torch.zeros((n, D), dtype=torch.uint8, device="cuda")
        kw["out_scale"] = torch.zeros((n,), dtype=torch.float32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_kpool_compress(slot_k.cuda(), slot_s.cuda(), ape.cuda(), kv_cache=cache, loc=loc.cuda(),
                          write_mask=None if wm is None else wm.cuda(), tap_x=tx, tap_xb=txb, tap_yb=tyb,
                          err_word=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_cache = u8(cache0).copy()
    ref = ora.kpool_compress(ref_cache, ps, bf16_bits(slot_k), bf16_bits(slot_s), f32(ape), loc.numpy(),
                             write_mask=None if wm is None else wm.numpy().astype(np.uint8), taps=True)
    w = np.ones(n, bool) if wm is None else wm.numpy()
    gq, gs = cache_rows(u8(cache), ps, D, loc.numpy())
    rq, rs = cache_rows(ref_cache, ps, D, loc.numpy())
    assert np.all(gq[~w] == 0x11)
    sub = {"x": ref["x"][w], "xb": ref["xb"][w], "yb": ref["yb"][w], "q": rq[w], "scale": rs[w]}
    check_rows(ora, f32(tx)[w], bf16_bits(txb)[w], bf16_bits(tyb)[w], gq[w], gs[w], sub, True,
               f"many pools n={n} masked={masked} variant={cvariant}")
    if not masked:
        np.testing.assert_array_equal(u8(kw["out_fp8"]), gq)


# -------------------------------------------------------------- decode update
def _run_decode(ck, d, round_scale, taps=True):
    dev = "cuda"
    B, N = d["B"], d["N"]
    cache = d["kv_cache"].to(dev)
    ring = d["ring"].to(dev)
    tx = torch.full((B * N, D), float("nan"), device=dev) if taps else None
    txb = torch.zeros((B * N, D), dtype=torch.bfloat16, device=dev) if taps else None
    tyb = torch.zeros((B * N, D), dtype=torch.bfloat16, device=dev) if taps else None
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_decode_update(cache, ring, d["tail_slot_mapping"].to(dev), d["slot_mapping"].to(dev),
                               d["positions"].to(dev), d["key"].to(dev), d["score"].to(dev), d["ape"].to(dev),
                               round_scale=round_scale, tap_x=tx, tap_xb=txb, tap_yb=tyb, err_word=err)
    torch.cuda.synchronize()
    return cache, ring, tx, txb, tyb, int(err.item())


def _oracle_decode(ora, d, round_scale):
    cache = u8(d["kv_cache"]).copy()
    ring = bf16_bits(d["ring"]).copy()
    ref = ora.kpool_decode_update(cache, d["page_size"], ring, d["tail_slot_mapping"].cpu().numpy(),
                                  d["slot_mapping"].cpu().numpy(), d["positions"].cpu().numpy(),
                                  bf16_bits(d["key"]), bf16_bits(d["score"]), f32(d["ape"]),
                                  round_scale=round_scale, taps=True)
    return cache, ring, ref


def _compare_decode(ora, d, gpu, oref, round_scale, what):
    cache, ring, tx, txb, tyb, err = gpu
    rcache, rring, ref = oref
    assert err == 0
    np.testing.assert_array_equal(bf16_bits(ring), rring, err_msg=what + " ring")
    sm = d["slot_mapping"].cpu().numpy().reshape(-1)
    pos = d["positions"].cpu().numpy().reshape(-1)
    P = d["P"]
    closing = np.nonzero((sm >= 0) & (pos >= 0) & (pos % P == P - 1))[0]
    assert len(closing) > 0
    gq, gs = cache_rows(u8(cache), d["page_size"], D, sm[closing])
    sub = {k: v[closing] for k, v in ref.items()}
    rq, rs = cache_rows(rcache, d["page_size"], D, sm[closing])
    sub["q"], sub["scale"] = rq, rs
    ndiff = check_rows(ora, f32(tx)[closing], bf16_bits(txb)[closing], bf16_bits(tyb)[closing], gq, gs, sub,
                       round_scale, what)
    # everything but the closing rows is untouched on both sides
    g = u8(cache).reshape(-1).copy()
    r = rcache.reshape(-1).copy()
    ps = d["page_size"]
    for l in sm[closing]:
        page, tok = divmod(int(l), ps)
        base = page * ps * (D + 4)
        for arr in (g, r):
            arr[base + tok * D: base + tok * D + D] = 0
            arr[base + ps * D + 4 * tok: base + ps * D + 4 * tok + 4] = 0
    np.testing.assert_array_equal(g, r, err_msg=what + " untouched cache bytes")
    return len(closing), ndiff


@pytest.mark.parametrize("round_scale", [True, False])
def test_kpool_decode_tiny_in_order_matches_oracle_and_one_shot(ck, ora, round_scale):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.tiny_pooled("cpu", seed=0)
    gpu = _run_decode(ck, d, round_scale)
    oref = _oracle_decode(ora, d, round_scale)
    n, _ = _compare_decode(ora, d, gpu, oref, round_scale, f"tiny decode round={round_scale}")
    assert n == 16
    # the same 16 pools through the one-shot kernel give bit-identical cache rows
    cache2 = d["kv_cache"].cuda()
    ck.ckv_kpool_compress(d["slot_k"].cuda(), d["slot_score"].cuda(), d["ape"].cuda(), kv_cache=cache2,
                          loc=d["loc"].cuda(), round_scale=round_scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(cache2), u8(gpu[0]))


@pytest.mark.parametrize("round_scale", [True, False])
def test_kpool_decode_verify_batch_full_size(ck, ora, round_scale):
    """512 requests x 4 verify tokens, prefilled ring, 5% padding (full size)."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.pooled_decode("cpu", seed=0 if round_scale else 1)
    gpu = _run_decode(ck, d, round_scale)
    oref = _oracle_decode(ora, d, round_scale)
    n, ndiff = _compare_decode(ora, d, gpu, oref, round_scale, f"decode/verify 512x4 round={round_scale}")
    assert n > 50


@pytest.mark.parametrize("P", [1, 4, 16])
def test_kpool_decode_long_sequences_and_across_calls(ck, ora, P):
    """N > P tokens per call (several closings per request) and a pool that is
    filled over several calls: the ring carries the stashes between calls."""
    from compressed_kv_attention_gated_gb300 import synth

    B, total = 5, 3 * P + 5
    d = synth.tiny_pooled("cpu", seed=3, B=B, N=total, P=P)
    # shuffle tail blocks so requests do not own block b
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(1))
    pos = d["positions"].to(torch.int64)
    d["tail_slot_mapping"] = (perm[:, None] * P + pos % P).to(torch.int32)
    ring_g = d["ring"].cuda()
    cache_g = d["kv_cache"].cuda()
    rcache = u8(d["kv_cache"]).copy()
    rring = bf16_bits(d["ring"]).copy()
    cuts = [0, 1, P + 2, total]
    taps_g, taps_r, closing_locs = [], [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = {k: d[k][:, a:b].contiguous() for k in ("tail_slot_mapping", "slot_mapping", "positions", "key", "score")}
        n_tok = B * (b - a)
        tx = torch.full((n_tok, D), float("nan"), device="cuda")
        txb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device="cuda")
        tyb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device="cuda")
        ck.ckv_kpool_decode_update(cache_g, ring_g, sl["tail_slot_mapping"].cuda(), sl["slot_mapping"].cuda(),
                                   sl["positions"].cuda(), sl["key"].cuda(), sl["score"].cuda(), d["ape"].cuda(),
                                   tap_x=tx, tap_xb=txb, tap_yb=tyb)
        r = ora.kpool_decode_update(rcache, d["page_size"], rring, sl["tail_slot_mapping"].numpy(),
                                    sl["slot_mapping"].numpy(), sl["positions"].numpy(), bf16_bits(sl["key"]),
                                    bf16_bits(sl["score"]), f32(d["ape"]), taps=True)
        sm = sl["slot_mapping"].numpy().reshape(-1)
        pos = sl["positions"].numpy().reshape(-1)
        closing = np.nonzero((sm >= 0) & (pos >= 0) & (pos % P == P - 1))[0]
        taps_g.append((tx, txb, tyb, closing))
        taps_r.append({k: v[closing] for k, v in r.items()})
        closing_locs.append(sm[closing])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(ring_g), rring)
    locs = np.concatenate(closing_locs)
    assert len(locs) == (total // P) * B
    gq, gs = cache_rows(u8(cache_g), d["page_size"], D, locs)
    rq, rs = cache_rows(rcache, d["page_size"], D, locs)
    gx = np.concatenate([f32(t[0])[t[3]] for t in taps_g])
    gxb = np.concatenate([bf16_bits(t[1])[t[3]] for t in taps_g])
    gyb = np.concatenate([bf16_bits(t[2])[t[3]] for t in taps_g])
    ref = {k: np.concatenate([t[k] for t in taps_r]) for k in ("x", "xb", "yb")}
    ref["q"], ref["scale"] = rq, rs
    check_rows(ora, gx, gxb, gyb, gq, gs, ref, True, f"across calls P={P}")


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_kpool_decode_random_calls(ck, ora, P):
    """Random small calls in sequence on one ring and cache: random request
    counts and token counts per call (several pool closings per request and
    per group of four tokens when P is small), random padding anywhere, random
    tail blocks, positions that continue across calls, both FP8 scales.  Ring
    bit-exact after every call; every closing row checked stage by stage."""
    rng = np.random.default_rng(1000 + P)
    B, blocks, ps = 9, 12, 8
    ring0 = torch.from_numpy(rng.standard_normal((blocks, 2, P, D)).astype(np.float32)).to(torch.bfloat16)
    ring_g = ring0.cuda()
    rring = bf16_bits(ring0).copy()
    cap = 64
    cache0 = torch.full(((B * cap + ps - 1) // ps, ps, D + 4), 0x29, dtype=torch.uint8)
    cache_g = cache0.cuda()
    rcache = u8(cache0).copy()
    ape = torch.from_numpy((rng.standard_normal((P, D)) * 0.1).astype(np.float32))
    block_of = rng.permutation(blocks)[:B]
    next_pos = rng.integers(0, 3 * P, B)
    for call in range(6):
        N = int(rng.integers(1, 3 * P + 3))
        pos = next_pos[:, None] + np.arange(N)[None, :]
        next_pos = next_pos + N
        pad = rng.random((B, N)) < 0.15
        ts = block_of[:, None] * P + pos % P
        sm = np.where(pos % P == P - 1, np.arange(B)[:, None] * cap + (pos // P) % cap, -1)
        ts_pad, sm_pad, pos_pad = (np.where(pad, -1, x).astype(np.int32) for x in (ts, sm, pos))
        # a few padded-slot cases: a token keeps its position but has no cache location
        nosm = (rng.random((B, N)) < 0.05) & ~pad
        sm_pad = np.where(nosm, -1, sm_pad).astype(np.int32)
        key = torch.from_numpy(rng.standard_normal((B, N, D)).astype(np.float32)).to(torch.bfloat16)
        score = torch.from_numpy((rng.standard_normal((B, N, D)) * 2).astype(np.float32)).to(torch.bfloat16)
        round_scale = bool(call % 2)
        n_tok = B * N
        tx = torch.full((n_tok, D), float("nan"), device="cuda")
        txb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device="cuda")
        tyb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros((1,), dtype=torch.int32, device="cuda")
        t = lambda x: torch.from_numpy(x).cuda()
        ck.ckv_kpool_decode_update(cache_g, ring_g, t(ts_pad), t(sm_pad), t(pos_pad), key.cuda(), score.cuda(),
                                   ape.cuda(), round_scale=round_scale, tap_x=tx, tap_xb=txb, tap_yb=tyb,
                                   use_pdl=bool(call % 3 == 0), err_word=err)
        r = ora.kpool_decode_update(rcache, ps, rring, ts_pad, sm_pad, pos_pad, bf16_bits(key), bf16_bits(score),
                                    f32(ape), round_scale=round_scale, taps=True)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        np.testing.assert_array_equal(bf16_bits(ring_g), rring, err_msg=f"ring after call {call}")
        fsm, fpos = sm_pad.reshape(-1), pos_pad.reshape(-1)
        closing = np.nonzero((fsm >= 0) & (fpos >= 0) & (fpos % P == P - 1))[0]
        if len(closing) == 0:
            continue
        gq, gs = cache_rows(u8(cache_g), ps, D, fsm[closing])
        rq, rs = cache_rows(rcache, ps, D, fsm[closing])
        sub = {k: v[closing] for k, v in r.items()}
        sub["q"], sub["scale"] = rq, rs
        check_rows(ora, f32(tx)[closing], bf16_bits(txb)[closing], bf16_bits(tyb)[closing], gq, gs, sub,
                   round_scale, f"random calls P={P} call={call}")
        assert np.all(np.isnan(f32(tx)[np.setdiff1d(np.arange(n_tok), closing)])), "taps of non-closing tokens"


def test_kpool_decode_strided_key_score(ck, ora):
    """Key and score rows as views of one fused per-token buffer (batch stride
    N * 3 * 128 + 64, token stride 3 * 128 elements): the C ABI takes both
    strides; the result equals the oracle's on contiguous copies."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.pooled_decode("cpu", seed=21, B=96, N=5)
    B, N = d["B"], d["N"]
    buf = torch.randn((B, N * 3 * D + 64), dtype=torch.float32).to(torch.bfloat16)
    fused = buf[:, :N * 3 * D].view(B, N, 3, D)
    fused[:, :, 1] = d["key"]
    fused[:, :, 2] = d["score"]
    gbuf = buf.cuda()
    gf = gbuf[:, :N * 3 * D].view(B, N, 3, D)
    gk, gsc = gf[:, :, 1], gf[:, :, 2]
    assert gk.stride() == (N * 3 * D + 64, 3 * D, 1) and not gk.is_contiguous()
    dev = "cuda"
    cache, ring = d["kv_cache"].to(dev), d["ring"].to(dev)
    tx = torch.full((B * N, D), float("nan"), device=dev)
    txb = torch.zeros((B * N, D), dtype=torch.bfloat16, device=dev)
    tyb = torch.zeros((B * N, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_decode_update(cache, ring, d["tail_slot_mapping"].to(dev), d["slot_mapping"].to(dev),
                               d["positions"].to(dev), gk, gsc, d["ape"].to(dev), tap_x=tx, tap_xb=txb, tap_yb=tyb,
                               use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    oref = _oracle_decode(ora, d, True)
    n, _ = _compare_decode(ora, d, (cache, ring, tx, txb, tyb, int(err.item())), oref, True, "strided key/score")
    assert n > 10


def test_kpool_decode_golden_gating_and_block_clamp(ck):
    """The hand-derived pooled-decode fixture (closing token with a negative
    tail slot reads ring block 0 and stashes nothing; closing slot without a
    cache location only stashes; open slot with a negative tail slot does
    nothing; a stash lands in its position's slot of its tail slot's block)
    through the C ABI."""
    from test_oracle_pins import _KD_GOLDEN as fx, kpool_decode_golden_check, kpool_decode_golden_inputs

    a = kpool_decode_golden_inputs(fx)
    dev = "cuda"
    t16 = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    cache = torch.from_numpy(a["cache"]).to(dev)
    ring = t16(a["ring"])
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_decode_update(cache, ring, torch.from_numpy(a["tail_slot_mapping"]).to(dev),
                               torch.from_numpy(a["slot_mapping"]).to(dev), torch.from_numpy(a["positions"]).to(dev),
                               t16(a["key"]), t16(a["score"]), torch.from_numpy(a["ape"]).to(dev), round_scale=True,
                               err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kpool_decode_golden_check(fx, u8(cache), bf16_bits(ring))


def test_kpool_decode_bad_block_flags(ck):
    B, N, P = 2, 1, 16
    ring = torch.zeros((1, 2, P, D), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 16, D + 4), dtype=torch.uint8, device="cuda")
    tsm = torch.tensor([[5 * P + 3], [0 * P + 4]], dtype=torch.int32, device="cuda")  # block 5 does not exist
    sm = torch.full((B, N), -1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([[3], [4]], dtype=torch.int32, device="cuda")
    key = torch.ones((B, N, D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_kpool_decode_update(cache, ring, tsm, sm, pos, key, key, torch.zeros((P, D), device="cuda"), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x2
    r = bf16_bits(ring)
    assert np.all(r[0, 0, 4] == 0x3F80) and np.all(r[0, 0, 3] == 0)


def test_kpool_decode_bad_cache_location_flags_and_stashes(ck):
    """A closing token whose cache location is past the cache: the cache-location
    bit is set, no cache byte changes, the token is still stashed, and the
    other request of the call closes its pool normally."""
    P = 16
    B, N = 2, 1
    ring = torch.zeros((2, 2, P, D), dtype=torch.bfloat16, device="cuda")
    ps = 16
    cache = torch.full((1, ps, D + 4), 0x37, dtype=torch.uint8, device="cuda")
    tsm = torch.tensor([[0 * P + 15], [1 * P + 15]], dtype=torch.int32, device="cuda")
    sm = torch.tensor([[ps], [3]], dtype=torch.int32, device="cuda")  # request 0: one past the end
    pos = torch.tensor([[15], [31]], dtype=torch.int32, device="cuda")
    key = torch.full((B, N, D), 2.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_kpool_decode_update(cache, ring, tsm, sm, pos, key, key, torch.zeros((P, D), device="cuda"), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0x4
    c = u8(cache).reshape(-1)
    row3 = c[3 * D:4 * D]
    assert not np.all(row3 == 0x37), "request 1's pool was not written"
    c2 = c.copy()
    c2[3 * D:4 * D] = 0x37
    c2[ps * D + 12:ps * D + 16] = 0x37
    assert np.all(c2 == 0x37), "bytes other than request 1's row and scale changed"
    r = bf16_bits(ring)
    assert np.all(r[0, 0, 15] == 0x4000) and np.all(r[0, 1, 15] == 0x4000), "request 0's token was not stashed"


def _seed_case(P, lens, seed):
    g = torch.Generator().manual_seed(seed)
    blocks = torch.randperm(len(lens), generator=g)
    ts, first = [], []
    for r, n in enumerate(lens):
        ts.append(blocks[r] * P + torch.arange(n) % P)
        first.append(torch.arange(n) < P)
    tslot = torch.cat(ts).to(torch.int32)
    n = tslot.numel()
    # padded entries only among a request's first P tokens: a padded entry
    # further in would make the token P places before it a tail token too, and
    # two tokens would write one ring slot (a race the method leaves undefined)
    pad = (torch.rand((n,), generator=g) < 0.05) & torch.cat(first)
    tslot[pad] = -1
    key = torch.randn((n, D), generator=g).to(torch.bfloat16)
    score = torch.randn((n, D), generator=g).to(torch.bfloat16)
    ring0 = torch.randn((len(lens), 2, P, D), generator=g).to(torch.bfloat16)
    return tslot, key, score, ring0


def test_kpool_seed_tail_vs_oracle(ck, ora):
    P = 16
    tslot, key, score, ring0 = _seed_case(P, [37, 5, 16, 0, 130], 5)
    ring = ring0.cuda()
    ck.ckv_kpool_seed_tail(ring, key.cuda(), score.cuda(), tslot.cuda())
    torch.cuda.synchronize()
    rring = bf16_bits(ring0).copy()
    ora.kpool_seed_tail(rring, bf16_bits(key), bf16_bits(score), tslot.numpy())
    np.testing.assert_array_equal(bf16_bits(ring), rring)


@pytest.mark.parametrize("misaligned", [False, True])
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_kpool_seed_tail_many_requests(ck, ora, P, misaligned):
    """Several CTAs of tokens with a ragged end; a slot map that starts 4 bytes
    past a 16-byte boundary takes the element-wise load path."""
    r = np.random.default_rng(P)
    lens = [int(x) for x in r.integers(0, 300, 97)] + [3001, 1, P - 1 if P > 1 else 1]
    tslot, key, score, ring0 = _seed_case(P, lens, 100 + P)
    ring = ring0.cuda()
    ts = tslot.cuda()
    if misaligned:
        buf = torch.empty((tslot.numel() + 1,), dtype=torch.int32, device="cuda")
        buf[1:] = ts
        ts = buf[1:]
        assert ts.data_ptr() % 16 != 0
    ck.ckv_kpool_seed_tail(ring, key.cuda(), score.cuda(), ts)
    torch.cuda.synchronize()
    rring = bf16_bits(ring0).copy()
    ora.kpool_seed_tail(rring, bf16_bits(key), bf16_bits(score), tslot.numpy())
    np.testing.assert_array_equal(bf16_bits(ring), rring)


@pytest.mark.parametrize("P", [4, 16])
def test_kpool_prefill_seed_decode_continuity(ck, ora, P):
    """Prefill -> decode on the pooled path (vLLM page kpool_compress:
    kpool_compress_and_write_cache for the prefill's complete pools,
    kpool_seed_tail_cache / _kpool_tail_seed_kernel for the ring, then
    _kpool_decode_update_batched_kernel for the decode tokens).  The decode
    tokens close the pool that straddles the prefill/decode boundary and the
    next one.  Every cache row must equal the one-shot compression of that
    pool's tokens taken straight from the whole sequence (staged FP8 checks),
    and the ring must equal the oracle's after each step."""
    B = 6
    lens = [37, 16, 5, 64, 1, 50] if P == 16 else [9, 4, 2, 16, 1, 14]
    N = 2 * P + 3
    g = torch.Generator().manual_seed(60 + P)
    seq_k = [torch.randn((n + N, D), generator=g).to(torch.bfloat16) for n in lens]
    seq_s = [(torch.randn((n + N, D), generator=g) * 2).to(torch.bfloat16) for n in lens]
    ape = torch.randn((P, D), generator=g) * 0.1
    blocks = torch.randperm(B, generator=g)
    cap = (max(lens) + N) // P + 1  # cache rows per request: row b * cap + pool index
    ps = 16
    pages = (B * cap + ps - 1) // ps
    cache0 = torch.full((pages, ps, D + 4), 0x6B, dtype=torch.uint8)
    ring0 = torch.randn((B, 2, P, D), generator=g).to(torch.bfloat16)  # stale contents
    dev = "cuda"
    cache, ring = cache0.to(dev), ring0.to(dev)
    rcache, rring = u8(cache0).copy(), bf16_bits(ring0).copy()
    err = torch.zeros((1,), dtype=torch.int32, device=dev)

    # 1. the prefill's complete pools, one-shot
    full = [(b, p) for b in range(B) for p in range(lens[b] // P)]
    pk = torch.stack([seq_k[b][p * P:(p + 1) * P] for b, p in full])
    pscore = torch.stack([seq_s[b][p * P:(p + 1) * P] for b, p in full])
    ploc = torch.tensor([b * cap + p for b, p in full], dtype=torch.int64)
    n1 = len(full)
    tx1 = torch.zeros((n1, D), device=dev)
    txb1 = torch.zeros((n1, D), dtype=torch.bfloat16, device=dev)
    tyb1 = torch.zeros((n1, D), dtype=torch.bfloat16, device=dev)
    ck.ckv_kpool_compress(pk.to(dev), pscore.to(dev), ape.to(dev), kv_cache=cache, loc=ploc.to(dev), tap_x=tx1,
                          tap_xb=txb1, tap_yb=tyb1, err_word=err)
    ora.kpool_compress(rcache, ps, bf16_bits(pk), bf16_bits(pscore), f32(ape), ploc.numpy())

    # 2. the ring seeded from the prefill batch (requests back to back)
    tslot = torch.cat([blocks[b] * P + torch.arange(n) % P for b, n in enumerate(lens)]).to(torch.int32)
    pre_k = torch.cat([seq_k[b][:n] for b, n in enumerate(lens)])
    pre_s = torch.cat([seq_s[b][:n] for b, n in enumerate(lens)])
    ck.ckv_kpool_seed_tail(ring, pre_k.to(dev), pre_s.to(dev), tslot.to(dev), err_word=err)
    ora.kpool_seed_tail(rring, bf16_bits(pre_k), bf16_bits(pre_s), tslot.numpy())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(ring), rring, err_msg="ring after the seed")

    # 3. N decode tokens per request in two calls
    taps = []
    for a, b_ in ((0, P - 1), (P - 1, N)):
        pos = torch.tensor([[lens[b] + t for t in range(a, b_)] for b in range(B)], dtype=torch.int64)
        ts = (blocks[:, None] * P + pos % P).to(torch.int32)
        sm = torch.where(pos % P == P - 1, torch.arange(B)[:, None] * cap + pos // P, -1).to(torch.int32)
        key = torch.stack([seq_k[b][lens[b] + a:lens[b] + b_] for b in range(B)])
        score = torch.stack([seq_s[b][lens[b] + a:lens[b] + b_] for b in range(B)])
        n_tok = B * (b_ - a)
        tx = torch.full((n_tok, D), float("nan"), device=dev)
        txb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device=dev)
        tyb = torch.zeros((n_tok, D), dtype=torch.bfloat16, device=dev)
        ck.ckv_kpool_decode_update(cache, ring, ts.to(dev), sm.to(dev), pos.to(torch.int32).to(dev), key.to(dev),
                                   score.to(dev), ape.to(dev), tap_x=tx, tap_xb=txb, tap_yb=tyb, err_word=err)
        ora.kpool_decode_update(rcache, ps, rring, ts.numpy(), sm.numpy(), pos.to(torch.int32).numpy(),
                                bf16_bits(key), bf16_bits(score), f32(ape))
        flat_sm = sm.numpy().reshape(-1)
        taps.append((tx, txb, tyb, np.nonzero(flat_sm >= 0)[0], flat_sm[flat_sm >= 0]))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bf16_bits(ring), rring, err_msg="ring after the decode calls")

    # every complete pool of the whole sequence, one-shot from its own tokens
    allp = [(b, p) for b in range(B) for p in range((lens[b] + N) // P)]
    wk = torch.stack([seq_k[b][p * P:(p + 1) * P] for b, p in allp])
    ws = torch.stack([seq_s[b][p * P:(p + 1) * P] for b, p in allp])
    wloc = np.array([b * cap + p for b, p in allp], np.int64)
    wcache = u8(cache0).copy()
    ref = ora.kpool_compress(wcache, ps, bf16_bits(wk), bf16_bits(ws), f32(ape), wloc, taps=True)
    assert sum(len(t[4]) for t in taps) == len(allp) - n1 and len(allp) - n1 >= 2 * B
    # GPU rows in the order of allp: the prefill's pools, then the decode closings
    gx = {int(l): r for l, r in zip(ploc.numpy(), f32(tx1))}
    gxb = {int(l): r for l, r in zip(ploc.numpy(), bf16_bits(txb1))}
    gyb = {int(l): r for l, r in zip(ploc.numpy(), bf16_bits(tyb1))}
    for tx, txb, tyb, rows, locs in taps:
        for r, l in zip(rows, locs):
            gx[int(l)], gxb[int(l)], gyb[int(l)] = f32(tx)[r], bf16_bits(txb)[r], bf16_bits(tyb)[r]
    gq, gs = cache_rows(u8(cache), ps, D, wloc)
    rq, rs = cache_rows(wcache, ps, D, wloc)
    ref["q"], ref["scale"] = rq, rs
    check_rows(ora, np.stack([gx[int(l)] for l in wloc]), np.stack([gxb[int(l)] for l in wloc]),
               np.stack([gyb[int(l)] for l in wloc]), gq, gs, ref, True, f"prefill-seed-decode P={P}")
    # nothing but those rows was written
    g = u8(cache).reshape(-1).copy()
    for l in wloc:
        page, tok = divmod(int(l), ps)
        base = page * ps * (D + 4)
        g[base + tok * D: base + tok * D + D] = 0x6B
        g[base + ps * D + 4 * tok: base + ps * D + 4 * tok + 4] = 0x6B
    assert np.all(g == 0x6B)


# ------------------------------------------------- pool -> token expansion
@pytest.mark.parametrize("P", [1, 4, 16])
def test_expand_pools_and_append_tail_vs_oracle(ck, ora, P):
    """Index work: bit-exact against the oracle (vLLM page kpool_compress,
    expand_pools_and_append_tail), including invalid pools, strided rows and a
    row count above the grid's y limit."""
    g = torch.Generator().manual_seed(P)
    for rows, groups in ((3, 5), (70000, 2)):
        full = torch.randint(-1, 5000, (rows, groups + 3), generator=g, dtype=torch.int32)
        ids = full[:, :groups]  # row stride groups + 3
        seq = torch.randint(0, 80000, (rows,), generator=g, dtype=torch.int64)
        out = ck.ckv_expand_pools_and_append_tail(full.cuda()[:, :groups], seq.cuda(), P)
        torch.cuda.synchronize()
        ref = ora.expand_pools_and_append_tail(ids.numpy(), seq.numpy(), P)
        np.testing.assert_array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("P", [3, 5, 12, 1000, 1024])
def test_expand_any_pool_size_and_most_groups(ck, ora, P):
    """Pool sizes that are not a power of two take the kernel's division path
    (column -> pool by a 32-bit division); rows of 2048 pool ids (the most a
    call accepts) with P up to 1024 are the widest rows.  Bit-exact against
    the oracle."""
    g = torch.Generator().manual_seed(1000 + P)
    for rows, groups in ((7, 5), (3, 2048)):
        ids = torch.randint(-1, 2000, (rows, groups), generator=g, dtype=torch.int32)
        seq = torch.randint(0, groups * P + P, (rows,), generator=g, dtype=torch.int64)
        out = ck.ckv_expand_pools_and_append_tail(ids.cuda(), seq.cuda(), P)
        torch.cuda.synchronize()
        ref = ora.expand_pools_and_append_tail(ids.numpy(), seq.numpy(), P)
        np.testing.assert_array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("P", [1, 4, 16])
def test_expand_output_off_16_byte_boundary(ck, ora, P, offset):
    """The output starts 4, 8 or 12 bytes past a 16-byte boundary: every row's
    columns before its first 16-byte boundary and after its last one are
    written one by one, the rest four at a time; the element before the output
    and the one after it keep their canary."""
    g = torch.Generator().manual_seed(P * 10 + offset)
    for rows, groups in ((5, 3), (1000, 7), (33, 64)):
        ids = torch.randint(-1, 900, (rows, groups), generator=g, dtype=torch.int32)
        seq = torch.randint(0, 20000, (rows,), generator=g, dtype=torch.int64)
        cols = groups * P + P - 1
        big = torch.full((rows * cols + 8,), -7, dtype=torch.int32, device="cuda")
        out = big[offset:offset + rows * cols].view(rows, cols)
        assert out.data_ptr() % 16 == 4 * offset
        ck.ckv_expand_pools_and_append_tail(ids.cuda(), seq.cuda(), P, out=out)
        torch.cuda.synchronize()
        ref = ora.expand_pools_and_append_tail(ids.numpy(), seq.numpy(), P)
        np.testing.assert_array_equal(out.cpu().numpy(), ref)
        b = big.cpu().numpy()
        assert np.all(b[:offset] == -7) and np.all(b[offset + rows * cols:] == -7)
