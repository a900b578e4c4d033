"""CPU-only checks of the C ABI: the library loads, exports every symbol that
include/ckv.h declares, rejects bad arguments before launching anything, and
its host planner agrees with the oracle's brute-force segmenter and with the
hand-derived plans (sglang page "deepseek_v4/c128_online.cuh",
plan_online_prefill_host / OnlinePrefillPlan).  No compute call here touches
a GPU: each one returns during argument validation."""
import ctypes
import json
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_kv_attention_gated_gb300 import build, ckv

    build.build()
    return ckv.load()


def test_exports_every_declared_symbol(lib):
    hdr = open(os.path.join(ROOT, "include", "ckv.h")).read()
    names = set(re.findall(r"^\s*(?:ckv_status|const char\*|int32_t)\s+(ckv_\w+)\s*\(", hdr, re.M))
    assert {"ckv_kpool_decode_update", "ckv_kpool_compress", "ckv_c128_online_decode",
            "ckv_c128_online_prefill", "ckv_plan_online_prefill"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert lib.ckv_abi_version() == 1
    for s in range(7):
        assert lib.ckv_status_string(s)


def test_plan_entry_is_16_bytes():
    hdr = open(os.path.join(ROOT, "include", "ckv.h")).read()
    body = re.search(r"typedef struct ckv_plan_entry \{(.*?)\}", hdr, re.S).group(1)
    assert re.findall(r"uint32_t (\w+);", body) == ["ragged_id", "batch_id", "position", "window_len"]


def _nulls(n):
    return [None] * n


def test_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    one = P(16)  # a non-null, aligned dummy pointer that is never dereferenced
    # decode: unsupported D, bad dtype, null pointers, misaligned pointer, empty batch
    assert lib.ckv_c128_online_decode(one, 4, one, 0, one, one, one, one, 3, 100, 0, None, None) == 2
    assert lib.ckv_c128_online_decode(one, 4, one, 7, one, one, one, one, 3, 128, 0, None, None) == 3
    assert lib.ckv_c128_online_decode(None, 4, one, 0, one, one, one, one, 3, 128, 0, None, None) == 1
    assert lib.ckv_c128_online_decode(P(20), 4, one, 0, one, one, one, one, 3, 128, 0, None, None) == 4
    assert lib.ckv_c128_online_decode(None, 4, None, 0, None, None, None, None, 0, 128, 0, None, None) == 0
    # latency probe: bad hop count, warps, null rows for two hops, misaligned out
    assert lib.ckv_latency_probe(5, one, one, 4, one, 8, 4, 0, None) == 2
    assert lib.ckv_latency_probe(4, one, one, 4096, one, 8, 4, 0, None) == 2  # decode pattern: >= 16 warps
    assert lib.ckv_latency_probe(4, one, one, 63, one, 64, 4, 0, None) == 2   # ... and >= 64 rows
    assert lib.ckv_latency_probe(3, one, one, 4096, one, 8, 4, 0, None) == 2  # first-hop mode: >= 16 warps
    assert lib.ckv_latency_probe(3, one, one, 8, one, 64, 4, 0, None) == 2    # ... and >= 9 rows
    assert lib.ckv_latency_probe(3, one, None, 4096, one, 64, 4, 0, None) == 1
    assert lib.ckv_latency_probe(2, one, one, 4, one, 0, 4, 0, None) == 2
    assert lib.ckv_latency_probe(0, one, one, 4, one, (1 << 30) + 1, 4, 0, None) == 2  # grid size
    assert lib.ckv_latency_probe(1, one, one, 4, one, 8, 33, 0, None) == 2
    assert lib.ckv_latency_probe(2, one, None, 4, one, 8, 4, 0, None) == 1
    assert lib.ckv_latency_probe(1, None, None, 0, one, 8, 4, 0, None) == 1
    assert lib.ckv_latency_probe(2, one, one, 4, P(20), 8, 4, 0, None) == 4
    # prefill: empty plans is a no-op, null plan with a count is rejected
    assert lib.ckv_c128_online_prefill(one, 4, one, 0, 10, one, one, one, None, 2, None, 0, None, 0, 512, 0,
                                       None, None) == 0
    assert lib.ckv_c128_online_prefill(one, 4, one, 0, 10, one, one, one, None, 2, None, 3, None, 0, 512, 0,
                                       None, None) == 1
    # kpool: D must be 128, P a power of two <= 16, something must be requested
    assert lib.ckv_kpool_compress(one, 1, 16, one, one, one, one, None, 1, None, None, 4, 16, 64, 1,
                                  None, None, None, 0, None, None) == 2
    assert lib.ckv_kpool_compress(one, 1, 16, one, one, one, one, None, 1, None, None, 4, 3, 128, 1,
                                  None, None, None, 0, None, None) == 2
    assert lib.ckv_kpool_compress(one, 1, 16, one, one, one, one, None, 0, None, None, 4, 16, 128, 1,
                                  None, None, None, 0, None, None) == 2
    assert lib.ckv_kpool_compress(one, 1, 16, one, one, one, one, one, 1, one, one, 4, 16, 128, 1,
                                  None, None, None, 0, None, None) == 2  # mask + returned rows
    assert lib.ckv_kpool_decode_update(one, 1, 16, one, 1, one, one, one, one, 512, 100, one, 512, 128, one,
                                       2, 4, 16, 128, 1, None, None, None, 0, None, None) == 4  # stride not 16 B
    assert lib.ckv_kpool_decode_update(one, 1, 16, one, 1, one, one, one, one, 512, 128, one, 512, 128, one,
                                       0, 4, 16, 128, 1, None, None, None, 0, None, None) == 0  # empty batch
    assert lib.ckv_kpool_seed_tail(one, 1, one, one, one, 5, 16, 96, None, None) == 2
    # element alignment of the index arrays and of the error word (a misaligned
    # typed pointer would fault on the device): rejected on the host
    odd = P(18)
    assert lib.ckv_c128_online_decode(one, 4, one, 0, one, one, odd, one, 3, 128, 0, None, None) == 4
    assert lib.ckv_c128_online_decode(one, 4, one, 0, one, one, one, one, 3, 128, 0, odd, None) == 4
    assert lib.ckv_c128_online_prefill(one, 4, one, 0, 10, one, one, odd, None, 2, one, 3, None, 0, 512, 0,
                                       None, None) == 4
    assert lib.ckv_kpool_seed_tail(one, 1, one, one, odd, 5, 16, 128, None, None) == 4
    assert lib.ckv_kpool_decode_update(one, 1, 16, one, 1, odd, one, one, one, 512, 128, one, 512, 128, one,
                                       2, 4, 16, 128, 1, None, None, None, 0, None, None) == 4
    assert lib.ckv_expand_pools_and_append_tail(odd, 4, one, 2, 4, 16, one, 0, None) == 4
    # distinct-id check: id width, range, scratch size, required pointers, alignment
    chk = lib.ckv_check_distinct
    chk.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int64, P, P]
    assert chk(one, 2, 10, 64, one, 2, one, None) == 2       # id_bytes must be 4 or 8
    assert chk(one, 4, 10, 0, one, 2, one, None) == 2        # empty range
    assert chk(one, 4, 10, 1 << 41, one, 1 << 36, one, None) == 2  # range above 2^40
    assert chk(one, 4, 10, 65, one, 2, one, None) == 2       # 65 ids need 3 scratch words
    assert chk(one, 4, -1, 64, one, 2, one, None) == 2
    assert chk(one, 4, 10, 64, None, 2, one, None) == 1      # scratch required
    assert chk(one, 4, 10, 64, one, 2, None, None) == 1      # err_word required
    assert chk(None, 4, 10, 64, one, 2, one, None) == 1      # ids required when n > 0
    assert chk(P(18), 4, 10, 64, one, 2, one, None) == 4     # int32 ids 4-byte aligned
    assert chk(P(20), 8, 10, 64, one, 2, one, None) == 4     # int64 ids 8-byte aligned


def _plan(lib, seq, ext, pad=False, num_tokens=None):
    from compressed_kv_attention_gated_gb300 import ckv

    return ckv.ckv_plan_online_prefill(torch.tensor(seq, dtype=torch.int64), torch.tensor(ext, dtype=torch.int64),
                                       num_tokens=num_tokens, pad_for_graph=pad)


def _rows(t, n):
    return t[:n].view(torch.int32).view(-1, 4).numpy().astype(np.uint32)


def test_planner_golden(lib):
    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "plan_examples.json")))["cases"]
    for c in cases:
        cp, wp, nc, nw = _plan(lib, c["seq_lens"], c["extend_lens"])
        assert _rows(cp, nc).tolist() == c["compress"], c["name"]
        assert _rows(wp, nw).tolist() == c["write"], c["name"]


def test_planner_vs_oracle_brute_force(lib, ora):
    rng = np.random.default_rng(0)
    for _ in range(400):
        B = int(rng.integers(1, 4))
        ext = rng.integers(1, 301, B)
        pre = rng.integers(0, 301, B)
        cp, wp, nc, nw = _plan(lib, (pre + ext).tolist(), ext.tolist())
        rc, rw = ora.plan_segments(pre + ext, ext)
        np.testing.assert_array_equal(_rows(cp, nc), rc)
        np.testing.assert_array_equal(_rows(wp, nw), rw)


def test_planner_graph_padding(lib):
    cp, wp, nc, nw = _plan(lib, [300, 5], [200, 3], pad=True)
    assert nc == nw == 203
    c = _rows(cp, nc)
    w = _rows(wp, nw)
    assert c[:2].tolist() == [[27, 0, 127, 28], [155, 0, 255, 128]]
    assert np.all(c[2:] == 0xFFFFFFFF)
    assert w[:2].tolist() == [[199, 0, 299, 44], [202, 1, 4, 3]]
    assert np.all(w[2:] == 0xFFFFFFFF)


@pytest.mark.parametrize("seq,ext,nt", [([10], [0], 0), ([10], [11], 11), ([10], [5], 6), ([2 ** 33], [5], 5)])
def test_planner_rejects_bad_lengths(lib, seq, ext, nt):
    from compressed_kv_attention_gated_gb300 import ckv

    with pytest.raises(ckv.CkvError) as e:
        _plan(lib, seq, ext, num_tokens=nt)
    assert e.value.status == 5


def test_binding_refuses_cpu_tensors(lib):
    from compressed_kv_attention_gated_gb300 import ckv

    x = torch.zeros((4, 256))
    with pytest.raises(ValueError):
        ckv.ckv_c128_online_decode(torch.zeros((4, 3, 128)), x, torch.zeros((4, 128)), torch.zeros((128, 128)),
                                   torch.zeros(4, dtype=torch.int32), torch.ones(4, dtype=torch.int32))


def test_binding_rejects_tensors_off_the_current_device(monkeypatch):
    """The binding refuses tensors spread over several CUDA devices, or on a
    device other than the current one, before anything reaches the library (a
    kernel on one device given another device's pointers would fault)."""
    import types

    import torch

    from compressed_kv_attention_gated_gb300 import ckv

    def fake(index):
        return types.SimpleNamespace(is_cuda=True, device=types.SimpleNamespace(index=index))

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    ckv._cuda("f", fake(0), None, fake(0))  # one device, the current one
    with pytest.raises(ValueError, match="several CUDA devices"):
        ckv._cuda("f", fake(0), fake(1))
    with pytest.raises(ValueError, match="not on the current CUDA device"):
        ckv._cuda("f", fake(1), fake(1))
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        ckv._cuda("f", torch.zeros(1))
