"""Failure detection on the GPU without faulting it.

Every pipeline wait in the TMA / bulk-copy kernels is bounded by wall time.
Here a wait is made to run out on purpose (an mbarrier that nothing
completes, limited to 20 ms): the kernel must record CKV_DEVERR_TIMEOUT in
the error word and return, and the context must stay usable afterwards.
Bad indices are covered in the parity tests (they set error bits and skip the
access)."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(ck_lib):
    ck = ck_lib
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    t0 = time.time()
    ck.ckv_wait_timeout_selftest(err, limit_us=20000)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(err.item()) == 0x20
    assert dt < 10.0
    # the context is still healthy: a normal call works afterwards
    x = torch.arange(16, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 120.0


def test_selftest_rejects_bad_limits(ck_lib):
    ck = ck_lib
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(ck.CkvError):
        ck.ckv_wait_timeout_selftest(err, limit_us=0)
    with pytest.raises(ck.CkvError):
        ck.ckv_wait_timeout_selftest(err, limit_us=3_000_000)


@pytest.fixture(scope="module")
def ck_lib():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck
