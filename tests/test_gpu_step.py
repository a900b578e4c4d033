"""The serving step in the launch configuration the benchmark times.

bench.py's timed step runs the five calls chained by programmatic dependent
launch, the two decode calls on a second stream concurrent with the three
prefill calls (the fp32 prefill's write pass reading its tokens before the
compress pass ends).  This test runs one such step on the full-size synthetic
workload and requires every output to equal, bit for bit, the same step run
call by call in plain stream order (the configuration the per-call full-size
tests compare with the CPU oracle); the c128 decode rows are also compared
with the oracle here."""
import numpy as np
import pytest
import torch

from helpers import assert_close_abs, assert_close_rel, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def steps():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    import compressed_kv_attention_gated_gb300 as ck

    ck.load()
    dev = torch.device("cuda", 0)
    timed, plain = bench.Step(dev, seed=0), bench.Step(dev, seed=0)
    state0 = timed.cd["state"].clone()
    # as in the timed loop: decode calls on their own stream, everything PDL-chained
    stream, dstream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    start = torch.cuda.Event()
    with torch.cuda.stream(stream):
        start.record(stream)
        dstream.wait_event(start)
        with torch.cuda.stream(dstream):
            timed.call(0, True)
            timed.call(1, True)
        for i in range(2, 5):
            timed.call(i, True)
    # reference: one call at a time, stream order, no programmatic launch
    torch.cuda.synchronize()
    for i in range(5):
        plain.call(i, False)
        torch.cuda.synchronize()
    assert int(timed.err.item()) == 0 and int(plain.err.item()) == 0
    return timed, plain, state0


def _same(a, b):
    return a.shape == b.shape and torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _rows(step, key):
    cpl, nc = step.plans[key][4], step.plans[key][1]
    return cpl[:nc].view(torch.int32).view(-1, 4)[:, 0].to(torch.int64).to(step.dev)


def test_step_pooled_decode_identical(steps):
    timed, plain, _ = steps
    assert _same(timed.pd["kv_cache"], plain.pd["kv_cache"])
    assert _same(timed.pd["ring"], plain.pd["ring"])


def test_step_c128_decode_identical_and_vs_oracle(steps, ora):
    timed, plain, state0 = steps
    cd = timed.cd
    p = (cd["seq_lens"].cpu().numpy().astype(np.int64) - 1) % 128
    closed = torch.from_numpy(np.nonzero(p == 127)[0]).to(timed.dev)
    assert _same(timed.cd["state"], plain.cd["state"])
    assert _same(cd["out"].index_select(0, closed), plain.cd["out"].index_select(0, closed))
    idx = cd["indices"].cpu().numpy()
    out_ref, ns_ref, cl = ora.c128_decode(f32(state0), f32(cd["input"]), f32(cd["ape"]), idx,
                                          cd["seq_lens"].cpu().numpy())
    assert np.array_equal(np.nonzero(cl)[0], closed.cpu().numpy())
    assert_close_rel(f32(cd["out"])[cl], out_ref[cl], "closing rows")
    gs = f32(cd["state"])[idx[~cl]]
    assert_close_abs(gs[:, 0], ns_ref[~cl, 0], what="max")
    assert_close_rel(gs[:, 1], ns_ref[~cl, 1], "sum")
    assert_close_rel(gs[:, 2], ns_ref[~cl, 2], "kv")


def test_step_prefills_identical(steps):
    timed, plain, _ = steps
    for key, name in (("cp", "cp"), ("lc", "lc")):
        rows = _rows(timed, key)
        a, b = getattr(timed, name), getattr(plain, name)
        assert _same(a["out"].index_select(0, rows), b["out"].index_select(0, rows)), key
        assert _same(a["state"], b["state"]), key


def test_step_pooled_one_shot_identical(steps):
    timed, plain, _ = steps
    assert _same(timed.lc["kv_cache"], plain.lc["kv_cache"])
