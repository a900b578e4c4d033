"""c128 rows with the FP8 output stage (ckv_c128_online_decode_fp8,
ckv_c128_online_prefill_fp8): the sglang c128_online.cuh page's compressed
rows taken, 128-channel block by block, through the vLLM kpool_compress
page's output stage into a paged FP8 cache.

For every call: the state and fp32 rows equal the plain call's bit for bit;
every byte of the cache equals the oracle's store of the GPU's own fp32 rows
(bf16, Hadamard-128, bf16 and absmax FP8 are deterministic given the fp32
row, so this is exact), bytes of other rows keep their canary; leaving out
the fp32 rows gives the same cache; a bad location is flagged and skipped.
End to end, against the oracle's store of its OWN rows: every 128-channel
block whose bf16 rounding agrees has identical codes and scale, and the
blocks that differ are bounded by the bf16 flips the fp32 error explains."""
import numpy as np
import pytest
import torch

from helpers import assert_close_rel, bf16_bits, bf16_flip_check, f32, report, u8

pytestmark = pytest.mark.gpu
CANARY = 0x5A


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


@pytest.fixture(params=[1, 2], ids=["cta_per_segment", "tma_pipeline"])
def variant(request, ck):
    prev = ck.ckv_c128_prefill_set_variant(request.param)
    yield request.param
    ck.ckv_c128_prefill_set_variant(prev)


def _cache(rows, D, ps=16):
    pages = (rows + ps - 1) // ps + 1
    return torch.full((pages, ps, D + 4 * (D // 128)), CANARY, dtype=torch.uint8), ps


def _expect(ora, cache0, ps, rows, locs, round_scale):
    ref = u8(cache0).copy()
    ora.c128_rows_to_cache(ref, ps, rows, locs, round_scale=round_scale)
    return ref


def _input_np(t):
    return bf16_bits(t) if t.dtype == torch.bfloat16 else f32(t)


def _bf16_of(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _block_bytes(cache, ps, D, loc, j):
    """(codes, scale bits) of 128-channel block j of the row at loc."""
    nb = D // 128
    flat = cache.reshape(-1)
    page, tok = divmod(int(loc), ps)
    base = page * ps * (D + 4 * nb)
    codes = flat[base + tok * D + 128 * j: base + tok * D + 128 * j + 128]
    sc = flat[base + ps * D + 4 * (tok * nb + j): base + ps * D + 4 * (tok * nb + j) + 4]
    return codes, sc


def check_vs_oracle_rows(ora, gpu_cache, cache0, ps, gpu_rows, ref_rows, locs, round_scale, what):
    """The GPU's FP8 cache against the oracle's store of the oracle's own rows:
    identical bytes on every block whose bf16 rounding agrees; flips bounded."""
    D = gpu_rows.shape[1]
    nb = D // 128
    r32 = np.asarray(ref_rows, np.float32)
    ref = _expect(ora, cache0, ps, r32, locs, round_scale)
    xg, xr = _bf16_of(gpu_rows), _bf16_of(r32)
    bf16_flip_check(gpu_rows, xg, r32, xr, what)
    same = np.all((xg == xr).reshape(len(locs), nb, 128), axis=2)
    for i, loc in enumerate(locs):
        for j in range(nb):
            gc, gsc = _block_bytes(gpu_cache, ps, D, loc, j)
            rc, rsc = _block_bytes(ref, ps, D, loc, j)
            if same[i, j]:
                assert np.array_equal(gc, rc) and np.array_equal(gsc, rsc), (what, i, j)
    report(what + " blocks", blocks=int(same.size), blocks_differing_bf16=int((~same).sum()))


@pytest.mark.parametrize("round_scale", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [128, 256, 512])
def test_decode_fp8(ck, ora, D, dtype, round_scale):
    from compressed_kv_attention_gated_gb300 import synth

    B = 301
    d = synth.c128_decode("cpu", seed=D + 2 * (dtype == torch.bfloat16), B=B, D=D, num_slots=700, dtype=dtype)
    seq = d["seq_lens"].clone()
    seq[::3] = (seq[::3] // 128 + 1) * 128  # a third of the requests close their chunk
    d["seq_lens"] = seq
    closed = ((seq.numpy().astype(np.int64) - 1) % 128) == 127
    g = torch.Generator().manual_seed(D)
    cache0, ps = _cache(2 * B, D)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=g)[:B].to(torch.int64)
    dev = "cuda"
    args = [d["input"].to(dev), None, d["ape"].to(dev), d["indices"].to(dev), d["seq_lens"].to(dev)]
    # plain call
    st_p = d["state"].to(dev).clone()
    out_p = torch.zeros((B, D), device=dev)
    ck.ckv_c128_online_decode(st_p, args[0], out_p, *args[2:])
    # FP8 stage with and without the fp32 rows
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    st_f, out_f, cache = d["state"].to(dev).clone(), torch.zeros((B, D), device=dev), cache0.to(dev)
    ck.ckv_c128_online_decode_fp8(st_f, args[0], out_f, *args[2:], cache, cache_loc.to(dev),
                                  round_scale=round_scale, use_pdl=True, err_word=err)
    st_n, cache_n = d["state"].to(dev).clone(), cache0.to(dev)
    ck.ckv_c128_online_decode_fp8(st_n, args[0], None, *args[2:], cache_n, cache_loc.to(dev),
                                  round_scale=round_scale, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(f32(st_f).view(np.uint32), f32(st_p).view(np.uint32))
    assert np.array_equal(f32(st_n).view(np.uint32), f32(st_p).view(np.uint32))
    assert np.array_equal(f32(out_f)[closed].view(np.uint32), f32(out_p)[closed].view(np.uint32))
    out_ref, _, cl = ora.c128_decode(f32(d["state"]), _input_np(d["input"]), f32(d["ape"]), d["indices"].numpy(),
                                     d["seq_lens"].numpy())
    assert np.array_equal(cl, closed) and closed.sum() > 50
    assert_close_rel(f32(out_f)[closed], out_ref[closed], "closing rows")
    ref = _expect(ora, cache0, ps, f32(out_f)[closed], cache_loc.numpy()[closed], round_scale)
    np.testing.assert_array_equal(u8(cache), ref)
    np.testing.assert_array_equal(u8(cache_n), ref)
    check_vs_oracle_rows(ora, u8(cache), cache0, ps, f32(out_f)[closed], out_ref[closed], cache_loc.numpy()[closed],
                         round_scale, f"c128 decode fp8 D={D} {dtype} round={round_scale}")


@pytest.mark.parametrize("round_scale", [True, False])
@pytest.mark.parametrize("closing", ["workload", "third"])
def test_decode_fp8_full_size(ck, ora, closing, round_scale):
    """The full-size decode batch (2048 requests, D = 512, fp32, 4096 slots)
    in the launch the bench times (FP8 rows only, PDL): the requests' own
    sequence lengths (about 16 closing), or a third of them closing.  States
    equal the plain call's bit for bit; the cache holds exactly the oracle's
    store of the GPU's rows (from a separate plain call) and every other byte
    keeps its canary; end to end against the oracle's own rows."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=5)
    B, D = d["B"], d["D"]
    if closing == "third":
        seq = d["seq_lens"].clone()
        seq[::3] = (seq[::3] // 128 + 1) * 128
        d["seq_lens"] = seq
    closed = ((d["seq_lens"].numpy().astype(np.int64) - 1) % 128) == 127
    cache0, ps = _cache(B, D, ps=64)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=torch.Generator().manual_seed(9))[:B].to(torch.int64)
    dev = "cuda"
    args = [d["input"].to(dev), None, d["ape"].to(dev), d["indices"].to(dev), d["seq_lens"].to(dev)]
    st_p, out_p = d["state"].to(dev).clone(), torch.zeros((B, D), device=dev)
    ck.ckv_c128_online_decode(st_p, args[0], out_p, *args[2:])
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    st_n, cache = d["state"].to(dev).clone(), cache0.to(dev)
    ck.ckv_c128_online_decode_fp8(st_n, args[0], None, *args[2:], cache, cache_loc.to(dev),
                                  round_scale=round_scale, use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and closed.sum() >= 8
    assert np.array_equal(f32(st_n).view(np.uint32), f32(st_p).view(np.uint32))
    rows = f32(out_p)[closed]
    np.testing.assert_array_equal(u8(cache), _expect(ora, cache0, ps, rows, cache_loc.numpy()[closed], round_scale))
    out_ref, _, cl = ora.c128_decode(f32(d["state"]), _input_np(d["input"]), f32(d["ape"]), d["indices"].numpy(),
                                     d["seq_lens"].numpy())
    assert np.array_equal(cl, closed)
    assert_close_rel(rows, out_ref[closed], "closing rows")
    check_vs_oracle_rows(ora, u8(cache), cache0, ps, rows, out_ref[closed], cache_loc.numpy()[closed], round_scale,
                         f"c128 decode fp8 full size closing={closing} round={round_scale}")


@pytest.mark.parametrize("ps", [1, 48])
def test_fp8_page_sizes(variant, ck, ora, ps):
    """Cache pages of 1 row (a shift by 0) and of 48 rows (not a power of two:
    the page comes from a division): decode and prefill rows stored exactly
    where the oracle's store of the GPU's own rows puts them."""
    from compressed_kv_attention_gated_gb300 import synth

    D, B = 512, 301
    d = synth.c128_decode("cpu", seed=40 + ps, B=B, D=D, num_slots=700)
    seq = d["seq_lens"].clone()
    seq[::3] = (seq[::3] // 128 + 1) * 128
    d["seq_lens"] = seq
    closed = ((seq.numpy().astype(np.int64) - 1) % 128) == 127
    cache0, ps = _cache(B, D, ps=ps)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=torch.Generator().manual_seed(ps))[:B].to(torch.int64)
    dev = "cuda"
    args = [d["input"].to(dev), None, d["ape"].to(dev), d["indices"].to(dev), d["seq_lens"].to(dev)]
    out = torch.zeros((B, D), device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    cache = cache0.to(dev)
    ck.ckv_c128_online_decode_fp8(d["state"].to(dev).clone(), args[0], out, *args[2:], cache, cache_loc.to(dev),
                                  err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and closed.sum() > 50
    np.testing.assert_array_equal(u8(cache), _expect(ora, cache0, ps, f32(out)[closed], cache_loc.numpy()[closed],
                                                     True))
    dp = synth.c128_prefill("cpu", seed=50 + ps, B=11, D=D, max_prefix=700, max_extend=900)
    T = dp["num_tokens"]
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(dp["seq_lens"], dp["extend_lens"])
    rows = cp[:nc].view(torch.int32).view(-1, 4)[:, 0].numpy().astype(np.int64)
    cache0, _ = _cache(T, D, ps=ps)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=torch.Generator().manual_seed(ps + 1))[:T].to(torch.int64)
    out_p, cache = torch.zeros((T, D), device=dev), cache0.to(dev)
    _prefill(ck, dp, cp, wp, nc, nw, out_p, cache, cache_loc, True, True, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and nc > 10
    np.testing.assert_array_equal(u8(cache), _expect(ora, cache0, ps, f32(out_p)[rows], cache_loc.numpy()[rows], True))


def _prefill(ck, d, cp, wp, nc, nw, out, cache, cache_loc, round_scale, use_pdl, err, fp8=True):
    dev = "cuda"
    state = d["state"].to(dev).clone()
    common = (state, d["input"].to(dev), out, d["ape"].to(dev), d["indices"].to(dev), cp.to(dev), nc,
              wp.to(dev), nw)
    if fp8:
        ck.ckv_c128_online_prefill_fp8(*common, cache, cache_loc.to(dev), round_scale=round_scale, use_pdl=use_pdl,
                                       err_word=err)
    else:
        ck.ckv_c128_online_prefill(*common, use_pdl=use_pdl, err_word=err)
    return state


@pytest.mark.parametrize("use_pdl", [False, True])
@pytest.mark.parametrize("round_scale", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [128, 256, 512])
def test_prefill_fp8(variant, ck, ora, D, dtype, round_scale, use_pdl):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=7 + D, B=11, D=D, max_prefix=700, max_extend=900, dtype=dtype)
    T = d["num_tokens"]
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
    rows = cp[:nc].view(torch.int32).view(-1, 4)[:, 0].numpy().astype(np.int64)
    cache0, ps = _cache(T, D)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=torch.Generator().manual_seed(D))[:T].to(torch.int64)
    dev = "cuda"
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    out_p = torch.zeros((T, D), device=dev)
    st_p = _prefill(ck, d, cp, wp, nc, nw, out_p, None, None, round_scale, use_pdl, err, fp8=False)
    out_f, cache = torch.zeros((T, D), device=dev), cache0.to(dev)
    st_f = _prefill(ck, d, cp, wp, nc, nw, out_f, cache, cache_loc, round_scale, use_pdl, err)
    cache_n = cache0.to(dev)
    st_n = _prefill(ck, d, cp, wp, nc, nw, None, cache_n, cache_loc, round_scale, use_pdl, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and nc > 10
    for st in (st_f, st_n):
        assert np.array_equal(f32(st).view(np.uint32), f32(st_p).view(np.uint32))
    assert np.array_equal(f32(out_f)[rows].view(np.uint32), f32(out_p)[rows].view(np.uint32))
    ref = _expect(ora, cache0, ps, f32(out_f)[rows], cache_loc.numpy()[rows], round_scale)
    np.testing.assert_array_equal(u8(cache), ref)
    np.testing.assert_array_equal(u8(cache_n), ref)
    out_ref, written, _, _ = ora.c128_prefill(f32(d["state"]), _input_np(d["input"]), f32(d["ape"]),
                                              d["indices"].numpy(), d["seq_lens"].numpy(), d["extend_lens"].numpy())
    assert np.array_equal(np.nonzero(written)[0], np.sort(rows))
    check_vs_oracle_rows(ora, u8(cache), cache0, ps, f32(out_f)[rows], out_ref[rows], cache_loc.numpy()[rows],
                         round_scale, f"c128 prefill fp8 D={D} {dtype} round={round_scale} pdl={use_pdl} "
                                      f"variant={variant}")


def test_prefill_fp8_long_context_full(ck, ora):
    """8 x 131,072 bf16 tokens (8192 compress rows, TMA pipeline by default)."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.long_context("cuda", seed=3)
    T = d["num_tokens"]
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
    rows = np.arange(127, T, 128)
    cache0, ps = _cache(nc, 512, ps=64)
    cache_loc = torch.full((T,), -1, dtype=torch.int64)
    cache_loc[torch.from_numpy(rows)] = torch.randperm(nc, generator=torch.Generator().manual_seed(1))
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = torch.zeros((T, 512), device="cuda")
    cache = cache0.cuda()
    ck.ckv_c128_online_prefill_fp8(d["state"], d["input"], out, d["ape"], d["indices"], cp.cuda(), nc, wp.cuda(), nw,
                                   cache, cache_loc.cuda(), use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g = f32(out.index_select(0, torch.from_numpy(rows).cuda()))
    ref = _expect(ora, cache0, ps, g, cache_loc.numpy()[rows], True)
    np.testing.assert_array_equal(u8(cache), ref)
    out_ref, written, _, _ = ora.c128_prefill(f32(d["state"]), bf16_bits(d["input"]), f32(d["ape"]),
                                              d["indices"].cpu().numpy(), d["seq_lens"].numpy(),
                                              d["extend_lens"].numpy())
    assert np.array_equal(np.nonzero(written)[0], rows)
    check_vs_oracle_rows(ora, u8(cache), cache0, ps, g, out_ref[rows], cache_loc.numpy()[rows], True,
                         "c128 prefill fp8 long context 8x131072")


@pytest.mark.parametrize("D", [128, 256, 512])
def test_fp8_bad_location_flagged_and_skipped(ck, ora, D):
    """D = 128 stages the closing rows per CTA; D = 256 and 512 quantise from
    the request's registers: both skip and flag an out-of-range location."""
    from compressed_kv_attention_gated_gb300 import synth

    B = 64
    d = synth.c128_decode("cpu", seed=5, B=B, D=D, num_slots=128)
    d["seq_lens"] = torch.full((B,), 128, dtype=torch.int32)  # every request closes
    cache0, ps = _cache(B, D)
    cache_loc = torch.arange(B, dtype=torch.int64)
    cache_loc[3] = -2
    cache_loc[7] = cache0.shape[0] * ps  # one past the end
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out, cache = torch.zeros((B, D), device="cuda"), cache0.cuda()
    ck.ckv_c128_online_decode_fp8(d["state"].cuda().clone(), d["input"].cuda(), out, d["ape"].cuda(),
                                  d["indices"].cuda(), d["seq_lens"].cuda(), cache, cache_loc.cuda(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0x4  # CKV_DEVERR_CACHE_LOC
    good = np.ones(B, bool)
    good[[3, 7]] = False
    ref = _expect(ora, cache0, ps, f32(out)[good], cache_loc.numpy()[good], True)
    np.testing.assert_array_equal(u8(cache), ref)


def test_counted_fp8_captured_with_device_planner(variant, ck, ora):
    """Device planner + counted FP8 prefill captured in one CUDA graph and
    replayed: identical to the host-planned FP8 call, cache equal to the oracle's."""
    from compressed_kv_attention_gated_gb300 import synth

    D = 256
    d = synth.c128_prefill("cpu", seed=43, B=23, D=D, max_prefix=900, max_extend=1500)
    T = d["num_tokens"]
    dev = "cuda"
    seq, ext = d["seq_lens"].to(dev), d["extend_lens"].to(dev)
    cp = torch.empty((T, 16), dtype=torch.uint8, device=dev)
    wp = torch.empty((T, 16), dtype=torch.uint8, device=dev)
    cnt = torch.zeros((2,), dtype=torch.int32, device=dev)
    cache0, ps = _cache(T, D)
    cache_loc = torch.randperm(cache0.shape[0] * ps, generator=torch.Generator().manual_seed(3))[:T].to(torch.int64)
    inp, ape, idx, loc = d["input"].to(dev), d["ape"].to(dev), d["indices"].to(dev), cache_loc.to(dev)
    state0 = d["state"].to(dev)
    state, out, cache = state0.clone(), torch.zeros((T, D), device=dev), cache0.to(dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)

    def body():
        ck.ckv_plan_online_prefill_device(seq, ext, T, compress_plan=cp, write_plan=wp, counts=cnt, err_word=err)
        ck.ckv_c128_online_prefill_counted_fp8(state, inp, out, ape, idx, cp, wp, cnt, cache, loc, use_pdl=True,
                                               err_word=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        body()  # set-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    state.copy_(state0)
    out.zero_()
    cache.copy_(cache0.to(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        body()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # host-planned FP8 call on fresh buffers
    hcp, hwp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
    out_h, cache_h = torch.zeros((T, D), device=dev), cache0.to(dev)
    st_h = _prefill(ck, d, hcp, hwp, nc, nw, out_h, cache_h, cache_loc, True, True, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = hcp[:nc].view(torch.int32).view(-1, 4)[:, 0].numpy().astype(np.int64)
    assert np.array_equal(f32(state).view(np.uint32), f32(st_h).view(np.uint32))
    assert np.array_equal(f32(out)[rows].view(np.uint32), f32(out_h)[rows].view(np.uint32))
    np.testing.assert_array_equal(u8(cache), u8(cache_h))
    ref = _expect(ora, cache0, ps, f32(out)[rows], cache_loc.numpy()[rows], True)
    np.testing.assert_array_equal(u8(cache), ref)
