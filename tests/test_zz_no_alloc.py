"""The allocation-free distinct-id check, ckv_check_distinct_noalloc.

Some callers cannot give the check a scratch buffer: a serving engine that has
reserved nearly all HBM for its paged KV cache and owns every byte through its
own pool, or a loop that must not call cudaMalloc because cudaMalloc may
synchronise the device.  For them the check keeps its bitmap in a static
device array inside the library, shared by every call.  These tests compare
it with ckv_check_distinct (caller scratch) on calls made two in a row, so a
bitmap left over from the previous call would show up as a false repeat.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

DISTINCT = 0x40
MAX_RANGE = 1 << 21


def test_noalloc_rejects_range_beyond_its_bitmap():
    """CPU: a range above 2^21 ids, a missing or misaligned error word are
    refused during argument checking, before anything is launched."""
    from compressed_kv_attention_gated_gb300 import build, ckv

    build.build()
    L = ckv.load()
    one = ctypes.c_void_p(16)  # aligned dummy pointer, never dereferenced
    assert L.ckv_check_distinct_noalloc(one, 4, 10, MAX_RANGE + 1, one, None) == 2
    assert L.ckv_check_distinct_noalloc(one, 4, 10, MAX_RANGE, None, None) == 1
    assert L.ckv_check_distinct_noalloc(one, 3, 10, 64, one, None) == 2
    # a misaligned error word is refused like in every other entry point
    assert L.ckv_check_distinct_noalloc(one, 4, 10, 64, ctypes.c_void_p(18), None) == 4


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


def _with_scratch(ck, ids, id_range):
    scratch = torch.full(((id_range + 31) // 32,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_check_distinct(ids, id_range, scratch, err)
    return err


def _noalloc(ck, ids, id_range):
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_check_distinct_noalloc(ids, id_range, err)
    return err


def _cases():
    rng = np.random.default_rng(21)
    perm = rng.permutation(4096).astype(np.int64)
    rep = perm.copy()
    rep[-1] = rep[7]
    big = rng.choice(MAX_RANGE, 200000, replace=False).astype(np.int64)
    big_rep = big.copy()
    big_rep[123456] = big_rep[5]
    pad = perm.copy()
    pad[::3] = -1
    out = perm.copy()
    out[100] = 4096
    return [
        ("slots", perm, 4096, torch.int32),
        ("same slots again", perm, 4096, torch.int32),   # a stale bitmap would flag every id
        ("one repeat", rep, 4096, torch.int64),
        ("full range, distinct", big, MAX_RANGE, torch.int64),
        ("small range after the full one", np.arange(64)[::-1].copy(), 64, torch.int32),
        ("full range, one repeat", big_rep, MAX_RANGE, torch.int32),
        ("padding", pad, 4096, torch.int32),
        ("out of range", out, 4096, torch.int64),
        ("empty", perm[:0], 4096, torch.int32),
    ]


@pytest.mark.gpu
def test_noalloc_matches_scratch_entry_on_calls_in_a_row(ck):
    cases = _cases()
    for (name_a, ids_a, r_a, dt_a), (name_b, ids_b, r_b, dt_b) in zip(cases, cases[1:]):
        a = torch.from_numpy(ids_a).to(dt_a).cuda()
        b = torch.from_numpy(ids_b).to(dt_b).cuda()
        # two allocation-free calls back to back on one stream, no sync between them
        na, nb = _noalloc(ck, a, r_a), _noalloc(ck, b, r_b)
        sa, sb = _with_scratch(ck, a, r_a), _with_scratch(ck, b, r_b)
        torch.cuda.synchronize()
        assert int(na.item()) == int(sa.item()), name_a
        assert int(nb.item()) == int(sb.item()), name_b
    expected = {"one repeat": DISTINCT, "full range, one repeat": DISTINCT, "out of range": DISTINCT}
    for name, ids, r, dt in cases:
        got = _noalloc(ck, torch.from_numpy(ids).to(dt).cuda(), r)
        torch.cuda.synchronize()
        assert int(got.item()) == expected.get(name, 0), name


@pytest.mark.gpu
def test_noalloc_rejects_oversize_range(ck):
    ids = torch.arange(10, dtype=torch.int32, device="cuda")
    with pytest.raises(ck.CkvError) as e:
        _noalloc(ck, ids, MAX_RANGE + 1)
    assert e.value.status == 2


@pytest.mark.gpu
def test_noalloc_on_each_device(ck):
    """The bitmap's device address is looked up per device: on every GPU of
    the machine (one at a time, that device current) the allocation-free call
    agrees with the scratch one.  With one GPU this is the first device only."""
    n_dev = torch.cuda.device_count()
    perm = np.random.default_rng(5).permutation(20000).astype(np.int64)
    rep = perm.copy()
    rep[-1] = rep[3]
    for dev in range(n_dev):
        with torch.cuda.device(dev):
            for ids_np, want in ((perm, 0), (rep, DISTINCT)):
                ids = torch.from_numpy(ids_np).to(f"cuda:{dev}")
                na = torch.zeros((1,), dtype=torch.int32, device=f"cuda:{dev}")
                ck.ckv_check_distinct_noalloc(ids, 20000, na)
                sa = torch.zeros((1,), dtype=torch.int32, device=f"cuda:{dev}")
                scratch = torch.full(((20000 + 31) // 32,), -1, dtype=torch.int32, device=f"cuda:{dev}")
                ck.ckv_check_distinct(ids, 20000, scratch, sa)
                torch.cuda.synchronize(dev)
                assert int(na.item()) == int(sa.item()) == want, dev
