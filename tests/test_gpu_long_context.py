"""Full-size parity of the long-context prefill workload (8 x 131,072 tokens).

The c128 part (D = 512, bf16 kv | Student-t scores, zero prefix) runs through
the host planner and ckv_c128_online_prefill; the pooled part (65,536 pools of
P = 16, D = 128) through ckv_kpool_compress -- the same calls and launch
configuration as the measured serving step.  Every written row is compared
with the CPU oracle (sglang page "deepseek_v4/c128_online.cuh"; vLLM page
"kpool_compress").
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_rel, bf16_bits, cache_rows, f32, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


@pytest.fixture(scope="module")
def lc(ck):
    from compressed_kv_attention_gated_gb300 import synth

    return synth.long_context("cuda", seed=3)


def test_long_context_c128_prefill_full(ck, ora, lc):
    d = lc
    cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
    assert nc == 8 * 1024 and nw == 0
    out = torch.full_like(d["out"], -7.0)
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_prefill(d["state"], d["input"], out, d["ape"], d["indices"], cp.cuda(), nc, wp.cuda(), nw,
                               err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = torch.arange(127, d["num_tokens"], 128, device="cuda")
    g = f32(out.index_select(0, rows))
    ref_out, written, fs, sw = ora.c128_prefill(f32(d["state"]), bf16_bits(d["input"]), f32(d["ape"]),
                                                d["indices"].cpu().numpy(), d["seq_lens"].numpy(),
                                                d["extend_lens"].numpy())
    assert written.sum() == 8 * 1024 and np.array_equal(np.nonzero(written)[0], rows.cpu().numpy())
    assert_close_rel(g, ref_out[written], "long-context compressed rows")
    # nothing else was written
    mask = torch.ones(d["num_tokens"], dtype=torch.bool, device="cuda")
    mask[rows] = False
    assert bool((out[mask] == -7.0).all())
    assert not sw.any()


def test_long_context_pooled_full(ck, ora, lc):
    from test_gpu_kpool import check_rows

    d = lc
    n = d["n_pools"]
    cache = torch.zeros_like(d["kv_cache"])
    tx = torch.zeros((n, 128), dtype=torch.float32, device="cuda")
    txb = torch.zeros((n, 128), dtype=torch.bfloat16, device="cuda")
    tyb = torch.zeros((n, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_kpool_compress(d["slot_k"], d["slot_score"], d["ape_pool"], kv_cache=cache, loc=d["loc"], tap_x=tx,
                          tap_xb=txb, tap_yb=tyb, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_cache = np.zeros(tuple(d["kv_cache"].shape), np.uint8)
    ref = ora.kpool_compress(ref_cache, d["page_size"], bf16_bits(d["slot_k"]), bf16_bits(d["slot_score"]),
                             f32(d["ape_pool"]), d["loc"].cpu().numpy(), taps=True)
    locs = np.arange(n)
    gq, gs = cache_rows(u8(cache), d["page_size"], 128, locs)
    rq, rs = cache_rows(ref_cache, d["page_size"], 128, locs)
    sub = {"x": ref["x"], "xb": ref["xb"], "yb": ref["yb"], "q": rq, "scale": rs}
    check_rows(ora, f32(tx), bf16_bits(txb), bf16_bits(tyb), gq, gs, sub, True, "long-context pools 65536")
