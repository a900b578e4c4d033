"""ckv_latency_probe: the latency-floor kernels behind the decode measurements
do the memory work they claim.  Two hops: each warp copies the row its index
names (out of range: the warp writes nothing); one hop: each warp writes its
index word to the first 4 bytes of its output row; the first-hop mode: lane
0's exclusive or of the 12 index words and 8 row words it loaded; the
decode-pattern mode: the 8 row words of every lane stored to the warp's
kilobyte, and lane 0's exclusive or of all it loaded, closing warp pairs'
block words included; zero hops: nothing."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


@pytest.mark.parametrize("warps_per_cta", [1, 4, 32])
def test_probe_hops_copy_what_they_claim(ck, warps_per_cta):
    g = torch.Generator().manual_seed(warps_per_cta)
    n, nrows = 777, 4096
    idx = torch.randperm(nrows, generator=g)[:n].to(torch.int32)
    idx[5], idx[9] = -1, nrows  # skipped by the second hop
    rows = torch.randint(0, 256, (nrows, 256), generator=g, dtype=torch.uint8)
    dev = "cuda"
    d_idx, d_rows = idx.to(dev), rows.to(dev)
    out2 = torch.full((n, 256), 0xEE, dtype=torch.uint8, device=dev)
    out1 = torch.full((n, 256), 0xEE, dtype=torch.uint8, device=dev)
    out0 = torch.full((n, 256), 0xEE, dtype=torch.uint8, device=dev)
    ck.ckv_latency_probe(2, n, d_idx, d_rows, out2, warps_per_cta=warps_per_cta, use_pdl=True)
    ck.ckv_latency_probe(1, n, d_idx, d_rows, out1, warps_per_cta=warps_per_cta)
    ck.ckv_latency_probe(0, n, d_idx, d_rows, out0, warps_per_cta=warps_per_cta)
    torch.cuda.synchronize()
    o2, o1, o0 = out2.cpu().numpy(), out1.cpu().numpy(), out0.cpu().numpy()
    ok = (idx >= 0) & (idx < nrows)
    np.testing.assert_array_equal(o2[ok.numpy()], rows.numpy()[idx[ok].numpy()])
    assert np.all(o2[~ok.numpy()] == 0xEE)
    np.testing.assert_array_equal(o1[:, :4].copy().view(np.int32)[:, 0], idx.numpy())
    assert np.all(o1[:, 4:] == 0xEE)
    assert np.all(o0 == 0xEE)


@pytest.mark.parametrize("n", [16, 1024, 777])
def test_probe_first_hop_mode(ck, n):
    g = torch.Generator().manual_seed(n)
    nrows = 4096
    idx = torch.randint(-2**31, 2**31 - 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    rows = torch.randint(0, 256, (nrows, 256), generator=g, dtype=torch.uint8)
    out = torch.full((n, 256), 0xEE, dtype=torch.uint8, device="cuda")
    ck.ckv_latency_probe(3, n, idx.cuda(), rows.cuda(), out, warps_per_cta=2, use_pdl=True)
    torch.cuda.synchronize()
    iw = idx.numpy()
    rw = rows.numpy().view(np.uint32).reshape(-1)
    want = np.empty(n, np.uint32)
    for w in range(n):
        b0 = min(w & ~3, n - 16)
        acc = np.uint32(iw[w])
        for q in range(1, 12):
            acc ^= np.uint32(iw[b0 + ((q * 7) & 15)])
        base = (w * 8) % (nrows * 64 - 512)  # lane 0's words: the ones it stores
        for q in range(8):
            acc ^= rw[base + q * 64]
        want[w] = acc
    o = out.cpu().numpy()
    np.testing.assert_array_equal(o[:, :4].copy().view(np.uint32)[:, 0], want)
    assert np.all(o[:, 4:] == 0xEE)


@pytest.mark.parametrize("n,nrows", [(16, 64), (1024, 16384), (778, 100)])
def test_probe_decode_pattern_mode(ck, n, nrows):
    g = torch.Generator().manual_seed(n + nrows)
    idx = torch.randint(-5, nrows + 5, (n,), generator=g, dtype=torch.int32)  # some out of range
    rows = torch.randint(0, 256, (nrows, 256), generator=g, dtype=torch.uint8)
    out = torch.full((4 * n, 256), 0xEE, dtype=torch.uint8, device="cuda")
    ck.ckv_latency_probe(4, n, idx.cuda(), rows.cuda(), out, warps_per_cta=2, use_pdl=True)
    torch.cuda.synchronize()
    iw = idx.numpy()
    rw = rows.numpy().view(np.uint32).reshape(-1)
    o = out.cpu().numpy().view(np.uint32).reshape(n, 256)
    blocks = nrows // 32
    for w in range(n):
        first = ((w >> 1) * 512) % (nrows * 64 - 512) + (w & 1) * 32
        want = np.array([rw[first + q * 64 + lane] for q in range(8) for lane in range(32)], np.uint32)
        b0 = min(w & ~3, n - 16)
        acc = np.uint32(iw[w])
        for q in range(1, 12):
            acc ^= np.uint32(iw[b0 + ((q * 7) & 15)])
        for q in range(8):
            acc ^= rw[first + q * 64]
        r = int(iw[w])
        if ((w >> 1) & 3) == 0 and 0 <= r < nrows:
            blk = min(r >> 5, blocks - 1) * 2048 + (w & 1) * 32
            for q in list(range(15)) + list(range(16, 31)):
                acc ^= rw[blk + q * 64]
        want[0] = acc
        np.testing.assert_array_equal(o[w], want)
