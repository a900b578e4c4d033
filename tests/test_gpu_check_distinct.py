"""Debug check of the caller contract (distinct state slots, cache locations,
tail blocks): the device bitmap check against numpy's own duplicate count."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DISTINCT = 0x40


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


def _expected(ids, id_range):
    v = ids[ids >= 0]
    return bool((v >= id_range).any() or np.unique(v).size != v.size)


def _run(ck, ids_np, id_range, dtype, scratch=None):
    ids = torch.from_numpy(ids_np.astype(np.int64)).to(dtype).cuda()
    if scratch is None:
        scratch = torch.full(((id_range + 31) // 32,), -1, dtype=torch.int32, device="cuda")  # stale bits
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ck.ckv_check_distinct(ids, id_range, scratch, err)
    torch.cuda.synchronize()
    return int(err.item())


@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
def test_check_distinct_vs_numpy(ck, dtype):
    rng = np.random.default_rng(3)
    for trial in range(60):
        id_range = int(rng.integers(1, 200000))
        n = int(rng.integers(0, min(id_range, 50000) + 1))
        ids = rng.permutation(id_range)[:n].astype(np.int64)
        kind = trial % 4
        if kind == 1 and n >= 2:  # one planted repeat
            i, j = rng.choice(n, 2, replace=False)
            ids[j] = ids[i]
        elif kind == 2 and n >= 1:  # padding entries are ignored
            ids[rng.random(n) < 0.3] = -1
        elif kind == 3 and n >= 1:  # one id out of range
            ids[int(rng.integers(0, n))] = id_range + int(rng.integers(0, 5))
        got = _run(ck, ids, id_range, dtype)
        assert got == (DISTINCT if _expected(ids, id_range) else 0), (trial, kind, n, id_range)


def test_check_distinct_workload_ids(ck):
    """The state slots of the 2048-request decode batch and the cache locations
    of the pooled decode batch are distinct; a slot list with one repeat is not."""
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=0)
    idx = d["indices"].numpy().astype(np.int64)
    assert _run(ck, idx, 4096, torch.int32) == 0
    bad = idx.copy()
    bad[-1] = bad[0]
    assert _run(ck, bad, 4096, torch.int32) == DISTINCT
    p = synth.pooled_decode("cpu", seed=0)
    loc = p["slot_mapping"].numpy().reshape(-1).astype(np.int64)
    rows = p["kv_cache"].shape[0] * p["page_size"]
    assert _run(ck, loc, rows, torch.int32) == 0
    blocks = (p["tail_slot_mapping"].numpy().max(axis=1) // p["P"]).astype(np.int64)  # one block per request
    assert _run(ck, blocks, p["ring"].shape[0], torch.int64) == 0


def test_check_distinct_reuses_scratch(ck):
    """Two calls in a row on one scratch buffer: the second starts from a clean bitmap."""
    scratch = torch.zeros((4,), dtype=torch.int32, device="cuda")
    assert _run(ck, np.arange(100), 128, torch.int64, scratch) == 0
    assert _run(ck, np.arange(100)[::-1].copy(), 128, torch.int64, scratch) == 0
    assert _run(ck, np.array([5, 7, 5]), 128, torch.int64, scratch) == DISTINCT
