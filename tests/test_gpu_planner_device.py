"""Device-side prefill planner and the prefill that reads its counts on the device.

Source: sglang page "deepseek_v4/c128_online.cuh" (plan_online_prefill_host,
OnlinePrefillPlan, run_prefill).  The device planner must produce exactly the
host planner's entries (which the CPU tests pin to the oracle's brute-force
segmenter and to hand-derived plans); the counted prefill must match the CPU
oracle; and both must work inside a captured CUDA graph, replayed on new
lengths without any host round trip.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_abs, assert_close_rel, f32

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
    prev = ck.ckv_c128_prefill_set_variant(request.param)
    yield request.param
    ck.ckv_c128_prefill_set_variant(prev)


def _rows(t, n):
    return t[:n].cpu().contiguous().view(torch.int32).view(-1, 4).numpy().astype(np.uint32)


@pytest.mark.parametrize("pad", [False, True])
def test_device_planner_matches_host_planner(ck, ora, pad):
    rng = np.random.default_rng(0)
    for trial in range(41):
        B = int(rng.integers(1, 40)) if trial < 38 else int(rng.integers(1500, 3000)) if trial < 40 else 8192
        ext = rng.integers(1, 700, B)
        pre = rng.integers(0, 900, B)
        seq = torch.from_numpy((pre + ext).astype(np.int64))
        ex = torch.from_numpy(ext.astype(np.int64))
        hc, hw, hnc, hnw = ck.ckv_plan_online_prefill(seq, ex, pad_for_graph=pad)
        err = torch.zeros((1,), dtype=torch.int32, device="cuda")
        dc, dw, cnt = ck.ckv_plan_online_prefill_device(seq.cuda(), ex.cuda(), int(ext.sum()), pad_for_graph=pad,
                                                        err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        c = cnt.cpu().numpy()
        assert (c[0], c[1]) == (hnc, hnw)
        np.testing.assert_array_equal(_rows(dc, hnc), _rows(hc, hnc))
        np.testing.assert_array_equal(_rows(dw, hnw), _rows(hw, hnw))
        if not pad:
            rc, rw = ora.plan_segments(seq.numpy(), ex.numpy())
            np.testing.assert_array_equal(_rows(dc, hnc), rc)
            np.testing.assert_array_equal(_rows(dw, hnw), rw)


@pytest.mark.parametrize("seq,ext,nt", [([10], [0], 0), ([10], [11], 11), ([300, 5], [200, 3], 204)])
def test_device_planner_rejects_bad_lengths(ck, seq, ext, nt):
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    cnt = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    ck.ckv_plan_online_prefill_device(torch.tensor(seq, device="cuda"), torch.tensor(ext, device="cuda"), nt,
                                      counts=cnt, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0x8
    assert cnt.cpu().tolist() == [0, 0]


def _oracle_check(ora, state0, inp, ape, idx, seq, ext, g_state, g_out):
    ref_out, written, fs, sw = ora.c128_prefill(f32(state0), f32(inp), f32(ape), idx.cpu().numpy(), seq.numpy(),
                                                ext.numpy())
    go = f32(g_out)
    assert_close_rel(go[written], ref_out[written], "compressed rows")
    assert np.all(go[~written] == CANARY)
    gs = f32(g_state)
    i = idx.cpu().numpy()
    assert_close_abs(gs[i[sw], 0], fs[sw, 0], what="max")
    assert_close_rel(gs[i[sw], 2], fs[sw, 2], "kv")


@pytest.mark.parametrize("pad", [False, True])
def test_counted_prefill_matches_oracle(variant, ck, ora, pad):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_prefill("cpu", seed=41, B=23, D=256, max_prefix=900, max_extend=1500)
    T = d["num_tokens"]
    cp, wp, cnt = ck.ckv_plan_online_prefill_device(d["seq_lens"].cuda(), d["extend_lens"].cuda(), T,
                                                    pad_for_graph=pad)
    state = d["state"].cuda().clone()
    out = torch.full((T, d["D"]), CANARY, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_c128_online_prefill_counted(state, d["input"].cuda(), out, d["ape"].cuda(), d["indices"].cuda(), cp, wp,
                                       cnt, use_pdl=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _oracle_check(ora, d["state"], d["input"], d["ape"], d["indices"], d["seq_lens"], d["extend_lens"], state, out)


def test_graph_captured_plan_and_prefill(variant, ck, ora):
    """Planner + prefill captured once in a CUDA graph, replayed on two length sets
    (same batch size and token count) written into the captured input buffers."""
    D, B, T = 256, 6, 3000
    g = torch.Generator().manual_seed(77)
    seq_d = torch.zeros((B,), dtype=torch.int64, device="cuda")
    ext_d = torch.zeros((B,), dtype=torch.int64, device="cuda")
    inp = torch.zeros((T, 2 * D), device="cuda")
    ape = (torch.randn((128, D), generator=g) * 0.1).cuda()
    state = torch.zeros((2 * B, 3, D), device="cuda")
    idx = torch.arange(B, dtype=torch.int32, device="cuda") * 2
    out = torch.zeros((T, D), device="cuda")
    cp = torch.empty((T, 16), dtype=torch.uint8, device="cuda")
    wp = torch.empty((T, 16), dtype=torch.uint8, device="cuda")
    cnt = torch.zeros((2,), dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")

    def set_lengths(seed):
        r = np.random.default_rng(seed)
        cuts = np.sort(r.choice(np.arange(1, T), B - 1, replace=False))
        ext = np.diff(np.concatenate([[0], cuts, [T]])).astype(np.int64)
        pre = r.integers(0, 500, B).astype(np.int64)
        seq_d.copy_(torch.from_numpy(pre + ext))
        ext_d.copy_(torch.from_numpy(ext))
        x = torch.randn((T, 2 * D), generator=torch.Generator().manual_seed(seed))
        inp.copy_(x)
        st = torch.zeros((2 * B, 3, D))
        st[:, 0] = torch.randn((2 * B, D), generator=torch.Generator().manual_seed(seed + 1))
        st[:, 1] = 1.0 + 10 * torch.rand((2 * B, D), generator=torch.Generator().manual_seed(seed + 2))
        st[:, 2] = torch.randn((2 * B, D), generator=torch.Generator().manual_seed(seed + 3))
        state.copy_(st)
        out.fill_(CANARY)
        return torch.from_numpy(pre + ext), torch.from_numpy(ext), x, st

    def body():
        ck.ckv_plan_online_prefill_device(seq_d, ext_d, T, compress_plan=cp, write_plan=wp, counts=cnt, err_word=err)
        ck.ckv_c128_online_prefill_counted(state, inp, out, ape, idx, cp, wp, cnt, use_pdl=True, err_word=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    set_lengths(1)
    with torch.cuda.stream(s):
        body()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        body()
    for seed in (2, 3):
        seq, ext, x, st = set_lengths(seed)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _oracle_check(ora, st, x, ape.cpu(), idx, seq, ext, state, out)
