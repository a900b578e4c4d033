"""Buffers whose element or byte offsets pass 2^31: state slots, ring blocks
and cache rows near the top of multi-GB pools.  Each case is a small problem
of the ordinary tests moved to the top of a large buffer (the indices shifted
by a fixed amount), so the oracle runs on the small problem and the GPU's
results, read back from the large buffer at the shifted places, must match it
exactly as in the ordinary tests; everything below the shifted region stays
untouched.  About 13 GB of device memory at most, one case at a time."""
import numpy as np
import pytest
import torch

from helpers import assert_close_abs, assert_close_rel, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_c128_decode_state_slots_past_2_31_floats(ck, ora):
    """D = 512 (1536 floats a slot): slot 2^21 starts at float 3.2e9."""
    from compressed_kv_attention_gated_gb300 import synth

    B, D = 96, 512
    base = 1 << 21
    d = synth.c128_decode("cpu", seed=31, B=B, D=D, num_slots=B)
    d["seq_lens"][:4] = torch.tensor([1, 128, 129, 131072], dtype=torch.int32)
    idx = d["indices"].numpy().astype(np.int64)
    big = torch.zeros((base + B, 3, D), device="cuda")  # 12.9 GB
    big[base:] = d["state"].cuda()
    out = torch.full((B, D), -7.0, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_decode(big, d["input"].cuda(), out, d["ape"].cuda(),
                              torch.from_numpy(idx + base).to(torch.int32).cuda(), d["seq_lens"].cuda(),
                              use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not bool(big[:base].any()), "slots below the shifted ones were written"
    g_state, g_out = f32(big[base:]), f32(out)
    del big
    _free()
    out_ref, ns_ref, closed = ora.c128_decode(f32(d["state"]), f32(d["input"]), f32(d["ape"]), idx,
                                              d["seq_lens"].numpy())
    assert closed.any() and not closed.all()
    assert_close_rel(g_out[closed], out_ref[closed], "closing rows")
    assert np.all(g_out[~closed] == -7.0)
    open_ = ~closed
    gs = g_state[idx[open_]]
    assert_close_abs(gs[:, 0], ns_ref[open_, 0], what="max")
    assert_close_rel(gs[:, 1], ns_ref[open_, 1], "sum")
    assert_close_rel(gs[:, 2], ns_ref[open_, 2], "kv")
    s0 = f32(d["state"])
    np.testing.assert_array_equal(g_state[idx[closed]].view(np.uint32), s0[idx[closed]].view(np.uint32))


@pytest.mark.parametrize("variant", [1, 2], ids=["cta_per_segment", "tma_pipeline"])
def test_c128_prefill_state_slots_past_2_31_floats(ck, ora, variant):
    """Prefill segments whose stored partial and final state sit at slots
    2^21 and above (load and store indices shifted)."""
    from compressed_kv_attention_gated_gb300 import synth

    D = 512
    base = 1 << 21
    d = synth.c128_prefill("cpu", seed=32, B=8, D=D, max_prefix=400, max_extend=600, num_slots=16)
    nslots = d["state"].shape[0]
    idx = d["indices"].numpy().astype(np.int64)
    big = torch.zeros((base + nslots, 3, D), device="cuda")
    big[base:] = d["state"].cuda()
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
    T = d["num_tokens"]
    out = torch.full((T, D), -7.0, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    prev = ck.ckv_c128_prefill_set_variant(variant)
    try:
        ck.ckv_c128_online_prefill(big, d["input"].cuda(), out, d["ape"].cuda(),
                                   torch.from_numpy(idx + base).to(torch.int32).cuda(), cp.cuda(), nc, wp.cuda(), nw,
                                   use_pdl=True, err_word=err)
        torch.cuda.synchronize()
    finally:
        ck.ckv_c128_prefill_set_variant(prev)
    assert int(err.item()) == 0 and nc > 0
    assert not bool(big[:base].any()), "slots below the shifted ones were written"
    g_state, g_out = f32(big[base:]), f32(out)
    del big
    _free()
    ref_out, written, fs, sw = ora.c128_prefill(f32(d["state"]), f32(d["input"]), f32(d["ape"]), idx,
                                                d["seq_lens"].numpy(), d["extend_lens"].numpy())
    assert_close_rel(g_out[written], ref_out[written], "compressed rows")
    assert np.all(g_out[~written] == -7.0)
    assert_close_abs(g_state[idx[sw], 0], fs[sw, 0], what="max")
    assert_close_rel(g_state[idx[sw], 1], fs[sw, 1], "sum")
    assert_close_rel(g_state[idx[sw], 2], fs[sw, 2], "kv")


@pytest.mark.parametrize("round_scale", [True, False])
def test_kpool_decode_ring_and_cache_past_2_31(ck, ora, round_scale):
    """Tail blocks from 2^19 (ring element offset 2^31 and up, a 4.3 GB ring)
    and cache rows from 2^24 (byte offset 2.2e9 and up, a 2.2 GB cache): the
    pooled decode's ring and cache, read back at the shifted places, match the
    oracle on the unshifted problem as in the ordinary decode tests."""
    from compressed_kv_attention_gated_gb300 import synth
    from test_gpu_kpool import D, _compare_decode, _oracle_decode

    d = synth.pooled_decode("cpu", seed=33, B=48, max_start=4096)
    P, ps, B = d["P"], d["page_size"], d["B"]
    base_block, base_loc = 1 << 19, 1 << 24  # base_loc a whole number of pages
    pages = d["kv_cache"].shape[0]
    tsm, sm = d["tail_slot_mapping"], d["slot_mapping"]
    big_tsm = torch.where(tsm >= 0, tsm + base_block * P, tsm)
    big_sm = torch.where(sm >= 0, sm + base_loc, sm)
    dev = "cuda"
    ring = torch.zeros((base_block + B, 2, P, D), dtype=torch.bfloat16, device=dev)
    ring[base_block:] = d["ring"].to(dev)
    cache = torch.zeros((base_loc // ps + pages, ps, D + 4), dtype=torch.uint8, device=dev)
    n = B * d["N"]
    tx = torch.full((n, D), float("nan"), device=dev)
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_decode_update(cache, ring, big_tsm.to(dev), big_sm.to(dev), d["positions"].to(dev),
                               d["key"].to(dev), d["score"].to(dev), d["ape"].to(dev), round_scale=round_scale,
                               tap_x=tx, tap_xb=txb, tap_yb=tyb, use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    assert not bool(ring[:base_block].view(torch.int16).any()), "ring blocks below the shifted ones were written"
    assert not bool(cache[:base_loc // ps].any()), "cache pages below the shifted ones were written"
    gpu = (cache[base_loc // ps:].cpu(), ring[base_block:].cpu(), tx, txb, tyb, int(err.item()))
    del ring, cache
    _free()
    n_closing, _ = _compare_decode(ora, d, gpu, _oracle_decode(ora, d, round_scale), round_scale,
                                   f"pooled decode at large offsets round={round_scale}")
    assert n_closing > 0


@pytest.mark.parametrize("variant", [1, 2], ids=["warp_per_pool", "bulk_pipeline"])
def test_kpool_compress_pools_past_2_31_elements(ck, ora, variant):
    """2^20 + 4096 one-shot pools (4.3 GB of keys, the same of scores): the
    rows of pools past 2^20 start past element 2^31.  Sampled pools at the
    top and the bottom against the oracle, stage by stage (as in the ordinary
    one-shot tests)."""
    from test_gpu_kpool import D, check_rows
    from helpers import bf16_bits

    P = 16
    n = (1 << 20) + 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(34)
    dev = "cuda"
    slot_k = torch.randn((n, P, D), generator=g, device=dev, dtype=torch.bfloat16)
    slot_s = torch.randn((n, P, D), generator=g, device=dev, dtype=torch.bfloat16) * 2
    ape = torch.randn((P, D), generator=g, device=dev) * 0.1
    out_q = torch.zeros((n, D), dtype=torch.uint8, device=dev)
    out_s = torch.zeros((n,), dtype=torch.float32, device=dev)
    tx = torch.zeros((n, D), device=dev)
    txb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    tyb = torch.zeros((n, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    prev = ck.ckv_kpool_compress_set_variant(variant)
    try:
        ck.ckv_kpool_compress(slot_k, slot_s, ape, write_cache=False, out_fp8=out_q, out_scale=out_s, tap_x=tx,
                              tap_xb=txb, tap_yb=tyb, err_word=err)
        torch.cuda.synchronize()
    finally:
        ck.ckv_kpool_compress_set_variant(prev)
    assert int(err.item()) == 0
    pick = torch.cat([torch.arange(8), torch.randperm(n - (1 << 20), generator=torch.Generator().manual_seed(35))[:40]
                      + (1 << 20), torch.tensor([n - 1])]).to(dev)
    sk, ss = bf16_bits(slot_k[pick]), bf16_bits(slot_s[pick])
    gx, gxb, gyb = f32(tx[pick]), bf16_bits(txb[pick]), bf16_bits(tyb[pick])
    gq, gs = out_q[pick].cpu().numpy(), f32(out_s[pick])
    ape_h = f32(ape)
    del slot_k, slot_s, out_q, out_s, tx, txb, tyb
    _free()
    m = len(pick)
    ref = ora.kpool_compress(np.zeros((1, 1, D + 4), np.uint8), 1, sk, ss, ape_h, np.zeros(m, np.int64),
                             write_cache=False, return_compressed=True, taps=True)
    check_rows(ora, gx, gxb, gyb, gq, gs, ref, True, f"one-shot pools past 2^31 variant={variant}")


@pytest.mark.parametrize("variant", [1, 2], ids=["cta_per_segment", "tma_pipeline"])
def test_c128_prefill_tokens_past_2_31_elements(ck, ora, variant):
    """One request of 2^21 + 2^17 bf16 tokens from position 0 (a 4.6 GB
    input: the rows past token 2^21 start past element 2^31).  Every chunk is
    a whole compress segment, so each sampled row is the oracle's two-pass
    over its own 128 tokens."""
    from compressed_kv_attention_gated_gb300 import synth
    from helpers import bf16_bits

    D = 512
    T = (1 << 21) + (1 << 17)
    d = synth.c128_prefill("cuda", seed=36, B=1, D=D, max_extend=T, zero_prefix=True, num_slots=1,
                           dtype=torch.bfloat16, score_dist="student_t")
    assert d["num_tokens"] == T
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"].cpu(), d["extend_lens"].cpu())
    assert nc == T // 128 and nw == 0
    out = torch.full((T, D), -7.0, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    prev = ck.ckv_c128_prefill_set_variant(variant)
    try:
        ck.ckv_c128_online_prefill(d["state"], d["input"], out, d["ape"], d["indices"], cp.cuda(), nc, wp.cuda(), nw,
                                   use_pdl=True, err_word=err)
        torch.cuda.synchronize()
    finally:
        ck.ckv_c128_prefill_set_variant(prev)
    assert int(err.item()) == 0
    chunks = torch.cat([torch.arange(4), torch.randperm(T // 128 - (1 << 14),
                                                        generator=torch.Generator().manual_seed(37))[:24] + (1 << 14),
                        torch.tensor([T // 128 - 1])])
    ape = f32(d["ape"])
    zero = np.zeros((1, 3, D), np.float32)
    for c in chunks.tolist():
        rows = d["input"][128 * c:128 * c + 128]
        ref, w, _, _ = ora.c128_prefill(zero, bf16_bits(rows), ape, np.zeros(1, np.int32), np.array([128]),
                                        np.array([128]))
        assert w[127] and not w[:127].any()
        assert_close_rel(f32(out[128 * c + 127])[None], ref[127][None], f"chunk {c}")
    written = (out.view(T // 128, 128, D)[:, :127] != -7.0).any()
    assert not bool(written), "rows other than the chunk ends were written"


def test_kpool_seed_tail_tokens_and_blocks_past_2_31(ck, ora):
    """2^24 padded prefill tokens (tail slot -1) in front of a small seed
    problem, whose key and score rows then start at element 2^31, with its
    tail blocks shifted to 2^19 and up (ring element offset 2^31 and up)."""
    from test_gpu_kpool import D, _seed_case
    from helpers import bf16_bits

    P = 16
    lens = [37, 5, 300, 16, 1, 129]
    tslot, key, score, ring0 = _seed_case(P, lens, 38)
    base_tok, base_block = 1 << 24, 1 << 19
    n = tslot.numel()
    dev = "cuda"
    big_ts = torch.full((base_tok + n,), -1, dtype=torch.int32, device=dev)
    big_ts[base_tok:] = torch.where(tslot >= 0, tslot + base_block * P, tslot).to(dev)
    big_key = torch.empty((base_tok + n, D), dtype=torch.bfloat16, device=dev)  # 4.3 GB, read only at the end
    big_score = torch.empty((base_tok + n, D), dtype=torch.bfloat16, device=dev)
    big_key[base_tok:] = key.to(dev)
    big_score[base_tok:] = score.to(dev)
    ring = torch.zeros((base_block + len(lens), 2, P, D), dtype=torch.bfloat16, device=dev)
    ring[base_block:] = ring0.to(dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ck.ckv_kpool_seed_tail(ring, big_key, big_score, big_ts, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not bool(ring[:base_block].view(torch.int16).any()), "ring blocks below the shifted ones were written"
    got = bf16_bits(ring[base_block:])
    del big_key, big_score, ring
    _free()
    rring = bf16_bits(ring0).copy()
    ora.kpool_seed_tail(rring, bf16_bits(key), bf16_bits(score), tslot.numpy())
    np.testing.assert_array_equal(got, rring)


def test_expand_output_past_2_31_elements(ck, ora):
    """65,600 rows of 2048 pool ids with P = 16: an 8.6 GB output whose rows
    from row 65,507 on start past element 2^31.  Sampled rows against the
    oracle."""
    rows, groups, P = 65600, 2048, 16
    g = torch.Generator(device="cuda")
    g.manual_seed(39)
    ids = torch.randint(-1, 1 << 20, (rows, groups), generator=g, device="cuda", dtype=torch.int32)
    seq = torch.randint(0, groups * P + P, (rows,), generator=g, device="cuda", dtype=torch.int64)
    out = ck.ckv_expand_pools_and_append_tail(ids, seq, P)
    torch.cuda.synchronize()
    cols = groups * P + P - 1
    assert (rows - 1) * cols > 2 ** 31
    pick = torch.cat([torch.arange(4), torch.arange(rows - 96, rows)]).to("cuda")
    got = out[pick].cpu().numpy()
    del out
    _free()
    ref = ora.expand_pools_and_append_tail(ids[pick].cpu().numpy(), seq[pick].cpu().numpy(), P)
    np.testing.assert_array_equal(got, ref)
