"""Out-of-bounds write check without a sanitizer: every buffer a call writes
is a view into a larger canary-filled allocation, with 4 KB guard bands on
both sides; after the call the guard bands must be untouched.  Covers every
entry point that writes device memory, at sizes with ragged ends."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
GUARD = 4096  # bytes on each side (a multiple of 16: views stay aligned)
BYTE = 0xA5


@pytest.fixture(scope="module")
def ck():
    import compressed_kv_attention_gated_gb300 as ck

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ck.load()
    return ck


class Guarded:
    """A tensor of `shape`/`dtype` living between two canary bands."""

    def __init__(self, shape, dtype, init=None):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), BYTE, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self):
        r = self.raw.cpu().numpy()
        return bool(np.all(r[:GUARD] == BYTE) and np.all(r[GUARD + self.n:] == BYTE))


def test_guard_c128_decode_and_fp8(ck):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.c128_decode("cpu", seed=1, B=333, D=512, num_slots=400)
    d["seq_lens"][::2] = 128
    st = Guarded(d["state"].shape, torch.float32, d["state"])
    out = Guarded((333, 512), torch.float32, torch.zeros(333, 512))
    cache = Guarded((7, 64, 512 + 16), torch.uint8, torch.zeros(7, 64, 528, dtype=torch.uint8))
    loc = torch.randperm(7 * 64)[:333].to(torch.int64).cuda()
    args = (d["input"].cuda(), out.t, d["ape"].cuda(), d["indices"].cuda(), d["seq_lens"].cuda())
    ck.ckv_c128_online_decode(st.t, *args)
    ck.ckv_c128_online_decode_fp8(st.t, *args, cache.t, loc)
    torch.cuda.synchronize()
    assert st.intact() and out.intact() and cache.intact()


@pytest.mark.parametrize("variant", [1, 2])
def test_guard_c128_prefill_and_fp8(ck, variant):
    from compressed_kv_attention_gated_gb300 import synth

    prev = ck.ckv_c128_prefill_set_variant(variant)
    try:
        d = synth.c128_prefill("cpu", seed=2, B=13, D=512, max_prefix=600, max_extend=700, dtype=torch.bfloat16)
        T = d["num_tokens"]
        cp, wp, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
        st = Guarded(d["state"].shape, torch.float32, d["state"])
        out = Guarded((T, 512), torch.float32, torch.zeros(T, 512))
        pages = T // 64 + 2
        cache = Guarded((pages, 64, 528), torch.uint8, torch.zeros(pages, 64, 528, dtype=torch.uint8))
        loc = torch.randperm(pages * 64)[:T].to(torch.int64).cuda()
        common = (d["input"].cuda(), out.t, d["ape"].cuda(), d["indices"].cuda(), cp.cuda(), nc, wp.cuda(), nw)
        ck.ckv_c128_online_prefill(st.t, *common, use_pdl=True)
        ck.ckv_c128_online_prefill_fp8(st.t, *common, cache.t, loc, use_pdl=True)
        cpd = Guarded((T, 16), torch.uint8)
        wpd = Guarded((T, 16), torch.uint8)
        cnt = Guarded((2,), torch.int32)
        ck.ckv_plan_online_prefill_device(d["seq_lens"].cuda(), d["extend_lens"].cuda(), T, compress_plan=cpd.t,
                                          write_plan=wpd.t, counts=cnt.t, pad_for_graph=True)
        ck.ckv_c128_online_prefill_counted_fp8(st.t, d["input"].cuda(), out.t, d["ape"].cuda(), d["indices"].cuda(),
                                               cpd.t, wpd.t, cnt.t, cache.t, loc)
        torch.cuda.synchronize()
        for g in (st, out, cache, cpd, wpd, cnt):
            assert g.intact()
    finally:
        ck.ckv_c128_prefill_set_variant(prev)


@pytest.mark.parametrize("variant", [1, 2])
def test_guard_kpool_compress(ck, variant):
    prev = ck.ckv_kpool_compress_set_variant(variant)
    try:
        n, P, D = 5003, 16, 128
        g = torch.Generator().manual_seed(3)
        k = torch.randn((n, P, D), generator=g).to(torch.bfloat16).cuda()
        s = torch.randn((n, P, D), generator=g).to(torch.bfloat16).cuda()
        ape = (torch.randn((P, D), generator=g) * 0.1).cuda()
        pages = n // 64 + 2
        cache = Guarded((pages, 64, D + 4), torch.uint8, torch.zeros(pages, 64, D + 4, dtype=torch.uint8))
        loc = torch.randperm(pages * 64, generator=g)[:n].to(torch.int64).cuda()
        q = Guarded((n, D), torch.uint8)
        sc = Guarded((n,), torch.float32)
        tx = Guarded((n, D), torch.float32)
        ck.ckv_kpool_compress(k, s, ape, kv_cache=cache.t, loc=loc, out_fp8=q.t, out_scale=sc.t, tap_x=tx.t)
        torch.cuda.synchronize()
        for gd in (cache, q, sc, tx):
            assert gd.intact()
    finally:
        ck.ckv_kpool_compress_set_variant(prev)


def test_guard_kpool_decode_seed_expand(ck):
    from compressed_kv_attention_gated_gb300 import synth

    d = synth.pooled_decode("cpu", seed=4, B=97)
    cache = Guarded(d["kv_cache"].shape, torch.uint8, d["kv_cache"])
    ring = Guarded(d["ring"].shape, torch.bfloat16, d["ring"])
    ck.ckv_kpool_decode_update(cache.t, ring.t, d["tail_slot_mapping"].cuda(), d["slot_mapping"].cuda(),
                               d["positions"].cuda(), d["key"].cuda(), d["score"].cuda(), d["ape"].cuda())
    # tail seed: 97 requests of 61 tokens
    per = 61
    key = torch.randn((97 * per, 128)).to(torch.bfloat16).cuda()
    score = torch.randn((97 * per, 128)).to(torch.bfloat16).cuda()
    tslot = (torch.arange(97)[:, None] * 16 + torch.arange(per)[None, :] % 16).reshape(-1).to(torch.int32).cuda()
    ck.ckv_kpool_seed_tail(ring.t, key, score, tslot)
    # expansion: 1001 rows of 37 pools
    ids = torch.randint(-1, 500, (1001, 37), dtype=torch.int32).cuda()
    seq = torch.randint(0, 9000, (1001,), dtype=torch.int64).cuda()
    out = Guarded((1001, 37 * 16 + 15), torch.int32)
    ck.ckv_expand_pools_and_append_tail(ids, seq, 16, out=out.t)
    torch.cuda.synchronize()
    assert cache.intact() and ring.intact() and out.intact()


def test_guard_check_distinct(ck):
    ids = torch.randperm(5000).to(torch.int32).cuda()
    scratch = Guarded(((5000 + 31) // 32,), torch.int32)
    err = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32))
    ck.ckv_check_distinct(ids, 5000, scratch.t, err.t)
    ck.ckv_check_distinct_noalloc(ids, 5000, err.t)
    torch.cuda.synchronize()
    assert scratch.intact() and err.intact() and int(err.t.item()) == 0
