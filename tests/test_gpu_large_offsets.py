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
