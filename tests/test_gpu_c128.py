"""GPU parity of the online c128 path (decode, prefill, planner) against the CPU oracle.

Source: sglang page "deepseek_v4/c128_online.cuh" (flash_c128_online_decode,
flash_c128_online_prefill, run_prefill, plan_online_prefill_host).  Every
call goes through the C ABI (libckv.so) via the ctypes binding.

Outputs the method does not define (decode rows of requests that do not
close a chunk, prefill rows not named by a compress segment) are filled with
a canary before the call and must still hold it afterwards; state slots not
written by a call must be bit-identical afterwards.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_abs, assert_close_rel, bf16_bits, f32

pytestmark = pytest.mark.gpu
CANARY = -12345.0


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


@pytest.fixture(params=[1, 2], ids=["cta_per_segment", "tma_pipeline"])
def variant(request, ck):
    """Run a prefill test with each compress-pass kernel."""
    prev = ck.ckv_c128_prefill_set_variant(request.param)
    yield request.param
    ck.ckv_c128_prefill_set_variant(prev)


def _np_input(t):
    return bf16_bits(t) if t.dtype == torch.bfloat16 else f32(t)


# ------------------------------------------------------------------ decode
def _decode_gpu(ck, d, use_pdl=False):
    state = d["state"].cuda().clone()
    out = torch.full((d["B"], d["D"]), CANARY, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_decode(state, d["input"].cuda(), out, d["ape"].cuda(), d["indices"].cuda(),
                              d["seq_lens"].cuda(), use_pdl=use_pdl, err_word=err)
    torch.cuda.synchronize()
    return f32(state), f32(out), int(err.item())


def _check_decode(ora, d, g_state, g_out):
    state0 = f32(d["state"])
    idx = d["indices"].cpu().numpy()
    out_ref, ns_ref, closed = ora.c128_decode(state0, _np_input(d["input"]), f32(d["ape"]), idx,
                                              d["seq_lens"].cpu().numpy())
    assert closed.any() or len(idx) < 200
    if closed.any():
        assert_close_rel(g_out[closed], out_ref[closed], "closing rows")
    assert np.all(g_out[~closed] == CANARY), "rows of non-closing requests were written"
    open_ = ~closed
    gs = g_state[idx[open_]]
    assert_close_abs(gs[:, 0], ns_ref[open_, 0], what="max")
    assert_close_rel(gs[:, 1], ns_ref[open_, 1], "sum")
    assert_close_rel(gs[:, 2], ns_ref[open_, 2], "kv")
    untouched = np.ones(state0.shape[0], bool)
    untouched[idx[open_]] = False
    np.testing.assert_array_equal(g_state[untouched].view(np.uint32), state0[untouched].view(np.uint32))
    return int(closed.sum())


def test_c128_decode_full_size(ck, ora):
    """2048 requests, D=512 fp32, 4096-slot pool, seq_lens U[1, 131072]."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=0)
    # make sure chunk positions 0 and 127 both occur
    d["seq_lens"][:8] = torch.tensor([1, 128, 129, 256, 2, 127, 131072, 131071], dtype=torch.int32)
    g_state, g_out, err = _decode_gpu(ck, d)
    assert err == 0
    assert _check_decode(ora, d, g_state, g_out) >= 3


def test_c128_decode_full_size_states_from_prior_tokens(ck, ora):
    """Full size (2048 requests, D=512, 4096 slots) with every touched slot
    holding the state of its chunk's earlier tokens: p = (seq_len - 1) % 128
    virtual tokens drawn like the input, reduced by the oracle's two-pass.  The
    closing rows must then equal a two-pass over all 128 tokens of the chunk,
    and the new states the two-pass over its p + 1 tokens (sglang page
    c128_online.cuh, flash_c128_online_decode; consistent initial states)."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=11)
    D, B = d["D"], d["B"]
    d["seq_lens"][:4] = torch.tensor([128, 1, 2, 131072], dtype=torch.int32)
    seq = d["seq_lens"].numpy().astype(np.int64)
    prior, p = synth.prior_chunk_tokens(seq, D, seed=12)
    p = p.numpy()
    ape = f32(d["ape"])
    idx = d["indices"].numpy()
    chunk0 = seq - 1 - p  # position of the chunk's first token
    has = p > 0
    zeros = np.zeros((1, 3, D), np.float32)
    _, _, fs, sw = ora.c128_prefill(zeros, f32(prior), ape, np.zeros(int(has.sum()), np.int32),
                                    chunk0[has] + p[has], p[has])
    assert sw.all()
    state = d["state"].clone()
    state[torch.from_numpy(idx[has]).long()] = torch.from_numpy(fs.astype(np.float32))
    d["state"] = state
    g_state, g_out, err = _decode_gpu(ck, d)
    assert err == 0
    n_closed = _check_decode(ora, d, g_state, g_out)
    assert n_closed >= 5
    # the whole chunk so far (prior tokens, then the new one) as one prefill segment per request
    starts = np.concatenate([[0], np.cumsum(p)])
    full = np.concatenate([np.concatenate([f32(prior)[starts[b]:starts[b + 1]], f32(d["input"])[b:b + 1]])
                           for b in range(B)])
    out2, written, fs2, sw2 = ora.c128_prefill(zeros, full, ape, np.zeros(B, np.int32), seq, p + 1)
    last = np.cumsum(p + 1) - 1
    closed = p == 127
    assert np.all(written[last] == closed) and np.all(sw2 == ~closed)
    assert_close_rel(g_out[closed], out2[last[closed]], "closing rows vs two-pass over the chunk")
    gs = g_state[idx[~closed]]
    assert_close_abs(gs[:, 0], fs2[~closed, 0], what="max vs two-pass")
    assert_close_rel(gs[:, 1], fs2[~closed, 1], "sum vs two-pass")
    assert_close_rel(gs[:, 2], fs2[~closed, 2], "kv vs two-pass")


@pytest.mark.parametrize("D", [128, 256, 512])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("use_pdl", [False, True])
def test_c128_decode_dims_dtypes(ck, ora, D, dtype, use_pdl):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=D, B=301, D=D, num_slots=700, max_seq=1000, dtype=dtype)
    d["seq_lens"][:4] = torch.tensor([1, 128, 256, 129], dtype=torch.int32)
    g_state, g_out, err = _decode_gpu(ck, d, use_pdl)
    assert err == 0
    _check_decode(ora, d, g_state, g_out)


def test_c128_decode_chunk_equals_two_pass(ck, ora):
    """128 decode calls over one chunk give the two-pass softmax of the chunk."""
    D = 256
    g = torch.Generator().manual_seed(3)
    k = torch.randn((128, D), generator=g)
    s = torch.randn((128, D), generator=g) * 3
    ape = (torch.randn((128, D), generator=g) * 0.1).cuda()
    state = torch.zeros((2, 3, D), device="cuda")
    idx = torch.tensor([1], dtype=torch.int32, device="cuda")
    out = torch.full((1, D), CANARY, device="cuda")
    for t in range(128):
        inp = torch.cat([k[t], s[t]])[None].cuda()
        ck.ckv_c128_online_decode(state, inp, out, ape, idx, torch.tensor([384 + t + 1], dtype=torch.int32,
                                                                           device="cuda"))
    torch.cuda.synchronize()
    z = s.double() + ape.cpu().double()
    w = torch.exp(z - z.max(0).values)
    ref = (w * k.double()).sum(0) / w.sum(0)
    assert_close_rel(f32(out)[0], ref.numpy(), "chunk via decode")


def test_c128_decode_bad_indices_flag(ck):
    D = 128
    state = torch.zeros((4, 3, D), device="cuda")
    inp = torch.ones((3, 2 * D), device="cuda")
    out = torch.zeros((3, D), device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_decode(state, inp, out, torch.zeros((128, D), device="cuda"),
                              torch.tensor([0, 9, 1], dtype=torch.int32, device="cuda"),
                              torch.tensor([5, 5, 0], dtype=torch.int32, device="cuda"), err_word=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & 0x1 and e & 0x10
    st = f32(state)
    assert np.all(st[1] == 0) and np.all(st[2:] == 0) and not np.all(st[0] == 0)


# ------------------------------------------------------------------ prefill
def _plan_rows(t, n):
    return t[:n].view(torch.int32).view(-1, 4).numpy().astype(np.uint32)


def _prefill_gpu(ck, d, pad=False, use_pdl=False, load_indices=None, state=None):
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"], pad_for_graph=pad)
    state = (d["state"] if state is None else state).cuda().clone()
    T, D = d["num_tokens"], d["D"]
    out = torch.full((T, D), CANARY, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_prefill(state, d["input"].cuda(), out, d["ape"].cuda(), d["indices"].cuda(), cp.cuda(), nc,
                               wp.cuda(), nw, load_indices=None if load_indices is None else load_indices.cuda(),
                               use_pdl=use_pdl, err_word=err)
    torch.cuda.synchronize()
    return state, out, int(err.item()), (cp, wp, nc, nw)


def _check_prefill(ora, d, g_state, g_out, load_indices=None, state0=None):
    state0 = f32(d["state"] if state0 is None else state0)
    idx = d["indices"].cpu().numpy()
    lidx = idx if load_indices is None else load_indices.cpu().numpy()
    ref_out, written, fs, sw = ora.c128_prefill(state0, _np_input(d["input"]), f32(d["ape"]), lidx,
                                                d["seq_lens"].numpy(), d["extend_lens"].numpy())
    go = f32(g_out)
    assert_close_rel(go[written], ref_out[written], "compressed rows")
    assert np.all(go[~written] == CANARY), "rows outside compress segments were written"
    gs = f32(g_state)
    assert_close_abs(gs[idx[sw], 0], fs[sw, 0], what="max")
    assert_close_rel(gs[idx[sw], 1], fs[sw, 1], "sum")
    assert_close_rel(gs[idx[sw], 2], fs[sw, 2], "kv")
    untouched = np.ones(state0.shape[0], bool)
    untouched[idx[sw]] = False
    np.testing.assert_array_equal(gs[untouched].view(np.uint32), state0[untouched].view(np.uint32))
    return int(written.sum()), int(sw.sum())


def test_planner_matches_oracle_segmenter(ck, ora):
    from compressed_kv_attention_gated_gb300 import synth

    for seed in range(5):
        d = synth.c128_prefill("cpu", seed=seed, B=17, D=128, max_prefix=700, max_extend=600)
        cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
        rc, rw = ora.plan_segments(d["seq_lens"].numpy(), d["extend_lens"].numpy())
        np.testing.assert_array_equal(_plan_rows(cp, nc), rc)
        np.testing.assert_array_equal(_plan_rows(wp, nw), rw)


@pytest.mark.parametrize("use_pdl", [False, True])
@pytest.mark.parametrize("D", [128, 256, 512])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_c128_prefill_small(variant, ck, ora, D, dtype, use_pdl):
    """With use_pdl the write pass reads its tokens before waiting for the
    compress pass, which reads the same state slots the write pass stores."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=D + (dtype == torch.bfloat16), B=9, D=D, max_prefix=500,
                           max_extend=450, dtype=dtype)
    g_state, g_out, err, _ = _prefill_gpu(ck, d, use_pdl=use_pdl)
    assert err == 0
    nrows, nstates = _check_prefill(ora, d, g_state, g_out)
    assert nrows > 0 and nstates > 0


@pytest.mark.parametrize("use_pdl", [False, True])
@pytest.mark.parametrize("pad", [False, True])
def test_c128_prefill_full_size(variant, ck, ora, use_pdl, pad):
    """64 requests, prefix U[0,16384], extend U[1,8192], D=512 fp32 (about 262K tokens)."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=0)
    g_state, g_out, err, plans = _prefill_gpu(ck, d, pad=pad, use_pdl=use_pdl)
    assert err == 0
    nrows, nstates = _check_prefill(ora, d, g_state, g_out)
    assert nrows > 1000 and nstates > 30


def test_c128_prefill_full_size_states_from_prior_tokens(ck, ora):
    """Full size (64 requests, prefix U[0,16384], extend U[1,8192], D=512 fp32)
    with each request's slot holding the state of its prefix's last, partial
    chunk: p = prefix % 128 virtual prior tokens drawn like the input
    (synth.prior_chunk_tokens), reduced by the oracle's two-pass.  Every
    compressed row must then equal a two-pass over all 128 tokens of its chunk
    (the prior ones included for the first chunk) and every new state the
    two-pass over its chunk's tokens (sglang page c128_online.cuh,
    flash_c128_online_prefill; consistent initial states)."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=12)
    D, B = d["D"], d["B"]
    seq = d["seq_lens"].numpy().astype(np.int64)
    ext = d["extend_lens"].numpy().astype(np.int64)
    prefix = seq - ext
    prior, p = synth.prior_chunk_tokens(torch.from_numpy(prefix + 1), D, seed=13)
    p = p.numpy()
    assert np.array_equal(p, prefix % 128) and (p > 0).sum() > 50
    ape = f32(d["ape"])
    idx = d["indices"].numpy()
    zeros = np.zeros((1, 3, D), np.float32)
    has = p > 0
    _, _, fs, sw = ora.c128_prefill(zeros, f32(prior), ape, np.zeros(int(has.sum()), np.int32), prefix[has],
                                    p[has])
    assert sw.all()
    state = d["state"].clone()
    state[torch.from_numpy(idx[has]).long()] = torch.from_numpy(fs.astype(np.float32))
    d["state"] = state
    g_state, g_out, err, _ = _prefill_gpu(ck, d, use_pdl=True)
    assert err == 0
    nrows, nstates = _check_prefill(ora, d, g_state, g_out)
    assert nrows > 1000 and nstates > 30
    # every request from the start of its prefix's last chunk, in one piece
    pstart = np.concatenate([[0], np.cumsum(p)])
    estart = np.concatenate([[0], np.cumsum(ext)])
    inp = f32(d["input"])
    full = np.concatenate([np.concatenate([f32(prior)[pstart[b]:pstart[b + 1]], inp[estart[b]:estart[b + 1]]])
                           for b in range(B)])
    out2, written2, fs2, sw2 = ora.c128_prefill(zeros, full, ape, np.zeros(B, np.int32), seq, p + ext)
    fstart = np.concatenate([[0], np.cumsum(p + ext)])
    # GPU ragged row estart[b] + i is row fstart[b] + p[b] + i of the whole-chunk layout
    rows = np.concatenate([np.arange(ext[b]) + estart[b] for b in range(B)])
    frows = np.concatenate([np.arange(ext[b]) + fstart[b] + p[b] for b in range(B)])
    go = f32(g_out)
    wr = written2[frows]
    assert wr.sum() == nrows
    assert_close_rel(go[rows[wr]], out2[frows[wr]], "compressed rows vs two-pass over whole chunks")
    gs = f32(g_state)
    assert np.array_equal(sw2, ~((seq % 128) == 0))
    assert_close_abs(gs[idx[sw2], 0], fs2[sw2, 0], what="max vs two-pass")
    assert_close_rel(gs[idx[sw2], 1], fs2[sw2, 1], "sum vs two-pass")
    assert_close_rel(gs[idx[sw2], 2], fs2[sw2, 2], "kv vs two-pass")


# (prefix, extend) pairs on every chunk boundary: first token of a chunk,
# last token of a chunk, exactly one chunk, one past it, single tokens, spans
# of many chunks, and segments ending on position 127 with nothing to write
BOUNDARY_CASES = [(0, 1), (0, 127), (0, 128), (0, 129), (127, 1), (127, 2), (126, 2), (128, 128), (1, 255),
                  (255, 1), (256, 384), (100, 28), (100, 29), (383, 1), (0, 1024), (64, 640), (511, 130)]


@pytest.mark.parametrize("use_pdl", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_c128_prefill_chunk_boundaries(variant, ck, ora, dtype, use_pdl):
    D = 128
    B = len(BOUNDARY_CASES)
    g = torch.Generator().manual_seed(31)
    pre = torch.tensor([c[0] for c in BOUNDARY_CASES], dtype=torch.int64)
    ext = torch.tensor([c[1] for c in BOUNDARY_CASES], dtype=torch.int64)
    T = int(ext.sum())
    st = torch.zeros((B, 3, D))
    st[:, 0] = torch.randn((B, D), generator=g)
    st[:, 1] = 1.0 + 10 * torch.rand((B, D), generator=g)
    st[:, 2] = torch.randn((B, D), generator=g)
    d = {"seq_lens": pre + ext, "extend_lens": ext, "input": torch.randn((T, 2 * D), generator=g).to(dtype),
         "ape": torch.randn((128, D), generator=g) * 0.1, "indices": torch.arange(B, dtype=torch.int32),
         "num_tokens": T, "D": D, "state": st}
    g_state, g_out, err, (cp, wp, nc, nw) = _prefill_gpu(ck, d, use_pdl=use_pdl)
    assert err == 0
    nrows, nstates = _check_prefill(ora, d, g_state, g_out)
    assert nc == nrows and nw == nstates


def test_c128_prefill_load_indices_differ(variant, ck, ora):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=11, B=12, D=256, max_prefix=400, max_extend=300, num_slots=40)
    g = torch.Generator().manual_seed(2)
    perm = torch.randperm(40, generator=g)
    d["indices"] = perm[:12].to(torch.int32)
    lidx = perm[12:24].to(torch.int32)
    g_state, g_out, err, _ = _prefill_gpu(ck, d, load_indices=lidx)
    assert err == 0
    _check_prefill(ora, d, g_state, g_out, load_indices=lidx)


def test_c128_prefill_then_decode_then_prefill(variant, ck, ora):
    """A sequence fed through prefill, decode steps and another prefill equals the
    oracle's chain (the running state is the only carried checkpoint)."""
    from compressed_kv_attention_gated_gb300 import synth

    D, B = 256, 3
    g = torch.Generator().manual_seed(9)
    ape = (torch.randn((128, D), generator=g) * 0.1)
    state_g = torch.zeros((B, 3, D), device="cuda")
    state_o = np.zeros((B, 3, D), np.float32)
    idx = torch.arange(B, dtype=torch.int32)
    seq = np.zeros(B, np.int64)
    for step, ext in enumerate([[100, 128, 5], None, None, [200, 1, 300], None]):
        if ext is None:  # one decode token per request
            inp = torch.randn((B, 2 * D), generator=g)
            seq += 1
            out = torch.full((B, D), CANARY, device="cuda")
            ck.ckv_c128_online_decode(state_g, inp.cuda(), out, ape.cuda(), idx.cuda(),
                                      torch.from_numpy(seq.astype(np.int32)).cuda())
            o_out, o_ns, closed = ora.c128_decode(state_o, f32(inp), f32(ape), idx.numpy(), seq.astype(np.int32))
            for b in range(B):
                if not closed[b]:
                    state_o[b] = o_ns[b]
            torch.cuda.synchronize()
            if closed.any():
                assert_close_rel(f32(out)[closed], o_out[closed], "decode rows")
        else:
            ext = np.array(ext, np.int64)
            seq += ext
            T = int(ext.sum())
            inp = torch.randn((T, 2 * D), generator=g)
            d = {"seq_lens": torch.from_numpy(seq.copy()), "extend_lens": torch.from_numpy(ext), "input": inp,
                 "ape": ape, "indices": idx, "num_tokens": T, "D": D, "state": torch.from_numpy(state_o.copy())}
            cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
            out = torch.full((T, D), CANARY, device="cuda")
            ck.ckv_c128_online_prefill(state_g, inp.cuda(), out, ape.cuda(), idx.cuda(), cp.cuda(), nc, wp.cuda(), nw)
            ref_out, written, fs, sw = ora.c128_prefill(state_o, f32(inp), f32(ape), idx.numpy(),
                                                        seq, ext)
            torch.cuda.synchronize()
            assert_close_rel(f32(out)[written], ref_out[written], "prefill rows")
            for b in range(B):
                if sw[b]:
                    state_o[b] = fs[b]
        live = np.array([(s % 128) != 0 for s in seq])
        gs = f32(state_g)
        assert_close_rel(gs[live, 2], state_o[live, 2], f"state kv after step {step}")


def test_c128_prefill_sentinels_and_bad_plans(variant, ck):
    D = 128
    T = 300
    state = torch.zeros((2, 3, D), device="cuda")
    inp = torch.randn((T, 2 * D), device="cuda")
    out = torch.full((T, D), CANARY, device="cuda")
    ape = torch.zeros((128, D), device="cuda")
    idx = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    # sentinel (skipped), window 0, compress entry not at a chunk end,
    # batch out of range, ragged row past the input
    plan = torch.tensor(np.array([[0xFFFFFFFF] * 4, [127, 0, 127, 0], [126, 0, 126, 127], [127, 5, 127, 128],
                                  [400, 0, 127, 128]], np.uint32).view(np.int32)).cuda()
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    empty = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_prefill(state, inp, out, ape, idx, plan, 5, empty, 0, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0x8
    assert np.all(f32(out) == CANARY)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_c128_prefill_masked_rows_do_not_leak(variant, ck, ora, dtype):
    """Rows outside a segment carry weight 0 (sglang page: padded kv is zeroed so
    that 0 * NaN never happens).  One request's input rows are NaN and +inf; the
    TMA boxes and token batches of its neighbours overlap them, yet every other
    request's rows and states must equal the oracle's."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=23, B=10, D=256, max_prefix=300, max_extend=90, dtype=dtype)
    ext = d["extend_lens"].numpy()
    starts = np.concatenate([[0], np.cumsum(ext)[:-1]])
    bad = 4
    x = d["input"].clone()
    x[starts[bad]:starts[bad] + ext[bad], :d["D"]] = float("nan")
    x[starts[bad]:starts[bad] + ext[bad], d["D"]:] = float("inf")
    d["input"] = x
    g_state, g_out, err, (cp, wp, nc, nw) = _prefill_gpu(ck, d)
    assert err == 0
    idx = d["indices"].numpy()
    ref_out, written, fs, sw = ora.c128_prefill(f32(d["state"]), _np_input(x), f32(d["ape"]), idx,
                                                d["seq_lens"].numpy(), d["extend_lens"].numpy())
    owner = np.repeat(np.arange(len(ext)), ext)
    rows = written & (owner != bad)
    assert rows.sum() > 0
    assert_close_rel(f32(g_out)[rows], ref_out[rows], "rows of clean requests")
    keep = sw & (np.arange(len(ext)) != bad)
    gs = f32(g_state)
    assert_close_abs(gs[idx[keep], 0], fs[keep, 0], what="max")
    assert_close_rel(gs[idx[keep], 1], fs[keep, 1], "sum")
    assert_close_rel(gs[idx[keep], 2], fs[keep, 2], "kv")
