"""Pins of the CPU oracle to facts fixed outside it.

Each test checks an oracle function against something other than itself: a
hand-derived fixture (tests/golden), a closed form, an invariant of the
mathematics, a library routine (scipy's Hadamard matrix, torch's float8 and
bfloat16 casts) or brute force.  They run on the CPU only.

Sources: vLLM page "kpool_compress" (pooled path), sglang page
"deepseek_v4/c128_online.cuh" (online c128 path and its plan).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_round(x):
    return _bf16_bits(x).astype(np.uint32).__lshift__(16).view(np.float32)


# --------------------------------------------------------------------- formats
def test_bf16_matches_torch_cast_on_fp32(ora):
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000).astype(np.float32),
        # exact ties between two bf16 neighbours (low 16 bits = 0x8000)
        (rng.integers(0x0080, 0x7F00, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, 1.17e-38], np.float32),
        # around the largest bf16 value (2 - 2^-7) * 2^127: below the midpoint to
        # 2^128 it stays finite, from the midpoint on it rounds to infinity
        np.array([3.3895e38, 3.3960e38, 3.3962e38, 3.4e38, -3.4e38], np.float32),
    ])
    vals = vals[np.isfinite(vals)]
    ref = _bf16_bits(vals)
    got = np.array([ora.bf16_from_double(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)
    assert ora.bf16_from_double(3.4e38) == 0x7F80 and ora.bf16_from_double(-3.4e38) == 0xFF80
    assert ora.bf16_from_double(float(np.ldexp(255.0, 120))) == 0x7F7F  # the largest finite value itself
    h = ora.bf16_from_double(float("nan"))
    assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0  # a NaN pattern


def test_bf16_from_double_is_nearest(ora):
    # brute force: the result is the closest bf16 value, ties to an even mantissa
    allb = np.arange(0, 0x7F80, dtype=np.uint32)
    allv = (allb << 16).view(np.float32).astype(np.float64)
    rng = np.random.default_rng(1)
    xs = rng.uniform(-4, 4, 3000)
    for x in xs:
        h = ora.bf16_from_double(x)
        a = abs(x)
        i = np.searchsorted(allv, a)
        cand = [j for j in (i - 1, i) if 0 <= j < len(allv)]
        dist = [abs(allv[j] - a) for j in cand]
        best = [cand[k] for k in range(len(cand)) if dist[k] == min(dist)]
        if len(best) > 1:
            best = [j for j in best if j % 2 == 0]
        assert (h & 0x7FFF) == best[0]
        assert (h >> 15) == (1 if x < 0 else 0)


def _e4m3_table(ora):
    codes = np.arange(256)
    vals = np.array([ora.e4m3_decode(int(c)) for c in codes])
    return codes, vals


def test_e4m3_decode_known_points(ora):
    # OCP E4M3: max 448 at 0x7E, min normal 2^-6 at 0x08, min subnormal 2^-9 at 0x01, NaN at 0x7F
    assert ora.e4m3_decode(0x7E) == 448.0
    assert ora.e4m3_decode(0xFE) == -448.0
    assert ora.e4m3_decode(0x08) == 2.0 ** -6
    assert ora.e4m3_decode(0x01) == 2.0 ** -9
    assert ora.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert ora.e4m3_decode(0x38) == 1.0
    assert math.isnan(ora.e4m3_decode(0x7F))
    vals = np.array([ora.e4m3_decode(c) for c in range(256)])
    torch_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(np.nan_to_num(vals, nan=1e9), np.nan_to_num(torch_vals, nan=1e9))


def test_e4m3_encode_exhaustive_bf16_vs_brute_force(ora):
    codes, vals = _e4m3_table(ora)
    finite = ~np.isnan(vals)
    fcodes, fvals = codes[finite], vals[finite]
    xs = (np.arange(0, 65536, dtype=np.uint32) << 16).view(np.float32)
    xs = xs[np.isfinite(xs)]
    for x in xs:
        c = ora.e4m3_encode(float(x))
        a = min(abs(float(x)), 448.0)  # saturation
        pos = fvals >= 0
        cand_codes = fcodes[pos & ((fcodes & 0x80) == 0)]
        cand_vals = fvals[pos & ((fcodes & 0x80) == 0)]
        d = np.abs(cand_vals - a)
        best = cand_codes[d == d.min()]
        if len(best) > 1:
            best = best[best % 2 == 0]
        assert (c & 0x7F) == int(best[0]), (x, c, best)
        if c & 0x7F:
            assert (c >> 7) == (1 if x < 0 else 0)


def test_e4m3_round_trip_and_torch_cast(ora):
    for c in range(256):
        v = ora.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert ora.e4m3_encode(v) == c
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-1, 1, 20000) * 2.0 ** -6]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([ora.e4m3_encode(float(x)) for x in xs], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_pow2_ceil(ora):
    for e in range(-30, 30):
        assert ora.pow2_ceil(2.0 ** e) == 2.0 ** e
    rng = np.random.default_rng(3)
    for v in rng.uniform(1e-7, 10.0, 2000).astype(np.float32):
        r = ora.pow2_ceil(float(v))
        m, ex = math.frexp(r)
        assert m == 0.5  # a power of two
        assert r / 2 < v <= r


# -------------------------------------------------------------------- Hadamard
def test_hadamard_exact_matches_scipy(ora):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128).astype(np.float64) / math.sqrt(128.0)
    rng = np.random.default_rng(4)
    for _ in range(20):
        x = rng.standard_normal(128)
        np.testing.assert_allclose(ora.hadamard128_exact(x), H @ x, rtol=0, atol=1e-12)


def test_hadamard_exact_closed_forms(ora):
    c = 1.0 / math.sqrt(128.0)
    e0 = np.zeros(128)
    e0[0] = 1.0
    np.testing.assert_allclose(ora.hadamard128_exact(e0), np.full(128, c), atol=1e-15)
    ones = np.ones(128)
    np.testing.assert_allclose(ora.hadamard128_exact(ones), math.sqrt(128.0) * e0, atol=1e-12)
    rng = np.random.default_rng(5)
    x = rng.standard_normal(128)
    y = ora.hadamard128_exact(x)
    np.testing.assert_allclose(ora.hadamard128_exact(y), x, atol=1e-12)  # involution
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12          # Parseval
    # row 5 of the Sylvester matrix: signs (-1)^popcount(5 & j)
    e5 = np.zeros(128)
    e5[5] = 1.0
    col = ora.hadamard128_exact(e5)
    expect = np.array([(-1) ** bin(5 & j).count("1") for j in range(128)]) * c
    np.testing.assert_allclose(col, expect, atol=1e-15)


def test_hadamard_fp32_butterfly_vs_exact(ora):
    rng = np.random.default_rng(6)
    for _ in range(200):
        x = _bf16_round(rng.standard_normal(128).astype(np.float32) * 0.3)
        y32 = ora.hadamard128_fp32(x).astype(np.float64)
        ye = ora.hadamard128_exact(x.astype(np.float64))
        assert np.max(np.abs(y32 - ye)) <= 1e-6 * max(1.0, np.max(np.abs(ye)))
        back = ora.hadamard128_fp32(y32.astype(np.float32)).astype(np.float64)
        assert np.max(np.abs(back - x)) <= 2e-6 * max(1.0, np.max(np.abs(x)))


def test_hadamard_fp32_rounding_path_worked_example(ora):
    """The fp32 rotation's rounding path (butterfly spans 1, 2, ..., 64 in
    ascending order, each (u + v, u - v) rounded to fp32 to nearest even, then
    one multiply by fp32(1/sqrt(128))), worked by hand on x = (1, 2^-24,
    2^-23, 0, ..., 0):
      span 1: 1 + 2^-24 is a tie between 1 and 1 + 2^-23 -> 1 (even);
              1 - 2^-24 exact; 2^-23 + 0 = 2^-23 - 0 = 2^-23;
      span 2: 1 + 2^-23 and 1 - 2^-23 exact; (1 - 2^-24) + 2^-23 = 1 + 2^-24,
              a tie -> 1; (1 - 2^-24) - 2^-23 = 1 - 3 * 2^-24 exact;
      spans 4..64 pair every value with a zero: output i is the value at i % 4.
    Spans in the other order would round the first output to 1 + 2^-22 instead
    (span 2 first gives 1 + 2^-23 and 2^-24, whose sum is a tie -> 1 + 2^-22),
    and the exact transform gives (1 + 3 * 2^-24) / sqrt(128)."""
    x = np.zeros(128, np.float32)
    x[0], x[1], x[2] = 1.0, 2.0 ** -24, 2.0 ** -23
    before_scale = np.array([1 + 2.0 ** -23, 1.0, 1 - 2.0 ** -23, 1 - 3 * 2.0 ** -24], np.float32)
    c = np.float32(1.0 / math.sqrt(128.0))
    want = np.tile(before_scale * c, 32)  # one fp32 multiply per value
    np.testing.assert_array_equal(ora.hadamard128_fp32(x), want)


# ------------------------------------------------------------------- quantise
def test_quantize_scale_invariants(ora):
    rng = np.random.default_rng(7)
    for round_scale in (True, False):
        for _ in range(200):
            y = _bf16_round(rng.standard_normal(128).astype(np.float32) * rng.uniform(0.01, 30))
            yb = _bf16_bits(y)
            q, sc = ora.quantize_rows(yb, round_scale)
            absmax = max(np.max(np.abs(y)), np.float32(1e-4))
            dec = np.array([ora.e4m3_decode(int(c)) for c in q])
            if round_scale:
                m, _ = math.frexp(float(sc))
                assert m == 0.5
                assert 224.0 < absmax / sc <= 448.0 * (1 + 1e-6)
            else:
                assert abs(sc - absmax / 448.0) <= 1e-6 * sc
                assert np.max(np.abs(dec)) == 448.0
            # every code is the nearest e4m3 value to y/scale (within half a quantum)
            t = np.clip(y / sc, -448, 448)
            quantum = np.where(np.abs(t) < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 1e-30))) - 3))
            assert np.all(np.abs(dec - t) <= quantum / 2 * (1 + 1e-6))


def _fp32_nearest(q):
    """The fp32 value nearest to the positive rational q (ties to even), exactly."""
    from fractions import Fraction

    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    assert -126 <= e < 128  # normal range
    ulp = Fraction(2) ** (e - 23)
    n, r = divmod(q, ulp)
    if r * 2 > ulp or (r * 2 == ulp and n % 2 == 1):
        n += 1
    return n * ulp


def _e4m3_nearest_code(t):
    """The e4m3 code nearest to the non-negative rational t < 2^-6 (the
    subnormal range, quantum 2^-9; ties to even)."""
    from fractions import Fraction

    q = Fraction(1, 512)
    n, r = divmod(t, q)
    if r * 2 > q or (r * 2 == q and n % 2 == 1):
        n += 1
    return int(n)  # subnormal codes are the multiple itself (8 = the smallest normal, code 0x08)


@pytest.mark.parametrize("am_bits,y_bits", [(0x3F84, 0x3784), (0x3F98, 0x3798), (0x3FA3, 0x37A3)])
def test_quantize_linear_scale_divides(ora, am_bits, y_bits):
    """The quotient q = y / scale is one IEEE fp32 division.  The row holds its
    absmax a and one element y = a * 2^-16, so y / scale lies within an fp32
    ulp of the e4m3 midpoint 3.5 * 2^-9: fp32(y / scale) and fp32(y *
    fp32(1 / scale)) round to different codes.  The expected code and scale
    are computed here with exact rational arithmetic."""
    from fractions import Fraction

    def bf16(bits):
        return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))

    a, y = bf16(am_bits), bf16(y_bits)
    inv448 = _fp32_nearest(Fraction(1, 448))
    scale = _fp32_nearest(a * inv448)
    want = _e4m3_nearest_code(_fp32_nearest(y / scale))
    other = _e4m3_nearest_code(_fp32_nearest(y * _fp32_nearest(1 / scale)))
    assert want != other  # the case tells the two apart
    row = np.zeros(128, np.uint16)
    row[0], row[1] = am_bits, y_bits
    q, sc = ora.quantize_rows(row, False)
    assert Fraction(float(sc)) == scale
    assert int(q[1]) == want and int(q[0]) == 0x7E  # the absmax itself maps to 448


def test_quantize_floor_on_zero_row(ora):
    q, sc = ora.quantize_rows(np.zeros(128, np.uint16), True)
    assert sc == ora.pow2_ceil(np.float32(1e-4) * np.float32(1.0 / 448.0))
    assert np.all(q == 0)


# --------------------------------------------------------------- pool softmax
def _pool(ora, k, s, ape, rs=True):
    return ora.pool_compress(k, s, ape, rs)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "pool_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_pool_golden(ora, case):
    P = case["P"]
    k = np.repeat(np.array(case["keys"], np.float32)[:, None], 128, 1)
    s = np.repeat(np.array(case["scores"], np.float32)[:, None], 128, 1)
    ape = np.repeat(np.array(case["ape"], np.float32)[:, None], 128, 1)
    r = _pool(ora, k, s, ape, True)
    np.testing.assert_allclose(r["x"], case["x"], rtol=0, atol=1e-6)
    assert np.all(r["xb"] == case["xb"])
    if "yb0" in case:
        assert r["yb"][0] == case["yb0"] and np.all(r["yb"][1:] == 0)
        assert r["scale"] == case["round"]["scale"] and r["q"][0] == case["round"]["q0"]
        assert np.all(r["q"][1:] == 0)
        r2 = _pool(ora, k, s, ape, False)
        absmax = ora.bf16_to_float(case["yb0"]) if hasattr(ora, "bf16_to_float") else 28.25
        assert abs(r2["scale"] - 28.25 * case["linear"]["scale_over_absmax"]) < 1e-8
        assert r2["q"][0] == case["linear"]["q0"]


def test_pool_rotation_takes_the_bf16_rounded_output(ora):
    """Worked by hand: P = 2 with equal weights (scores and bias 0), keys
    (1, 1) in channel 0 and (1, 1 - 2^-8) in channel 1 (both bf16), zeros
    elsewhere: x = (1, 1 - 2^-9, 0, ...), and 1 - 2^-9 is a bf16 tie between
    1 - 2^-8 and 1 that goes to 1 (even mantissa), so xb = (1, 1, 0, ...).
    The rotation of xb is 2c in even channels and 0 in odd ones (c =
    fp32(1/sqrt(128))): yb even = bf16(2c) = 0.1767578125, power-of-two scale
    2^-11, 0.1767578125 * 2^11 = 362 -> e4m3 352, code 0x7B; odd codes 0x00.
    Rotating the unrounded x instead would leave 2^-9 c in the odd channels."""
    k = np.zeros((2, 128), np.float32)
    k[:, 0] = 1.0
    k[0, 1], k[1, 1] = 1.0, 1.0 - 2.0 ** -8
    z = np.zeros((2, 128), np.float32)
    r = _pool(ora, k, z, z, True)
    assert r["x"][1] == 1.0 - 2.0 ** -9 and r["xb"][1] == 0x3F80
    assert np.all(r["yb"][1::2] == 0) and np.all(r["q"][0::2] == 0x7B) and np.all(r["q"][1::2] == 0x00)
    assert r["scale"] == 2.0 ** -11


def test_pool_equal_scores_give_mean(ora):
    rng = np.random.default_rng(8)
    for P in (1, 2, 4, 8, 16):
        k = _bf16_round(rng.standard_normal((P, 128)).astype(np.float32))
        s = np.repeat(rng.standard_normal((1, 128)).astype(np.float32), P, 0)
        ape = np.repeat(rng.standard_normal((1, 128)).astype(np.float32) * 0.1, P, 0)
        r = _pool(ora, k, s, ape)
        np.testing.assert_allclose(r["x"], k.astype(np.float64).mean(0), atol=1e-12)


def test_pool_dominant_score_and_bias(ora):
    rng = np.random.default_rng(9)
    for P in (2, 4, 16):
        for jstar in (0, P // 2, P - 1):
            k = _bf16_round(rng.standard_normal((P, 128)).astype(np.float32))
            s = rng.standard_normal((P, 128)).astype(np.float32)
            s[jstar] += 60.0
            ape = (rng.standard_normal((P, 128)) * 0.1).astype(np.float32)
            r = _pool(ora, k, s, ape)
            np.testing.assert_allclose(r["x"], k[jstar], atol=1e-12)
            # same selection made by the position bias alone (catches a wrong ape row)
            s2 = np.zeros((P, 128), np.float32)
            ape2 = np.zeros((P, 128), np.float32)
            ape2[jstar] = 60.0
            r2 = _pool(ora, k, s2, ape2)
            np.testing.assert_allclose(r2["x"], k[jstar], atol=1e-12)


def test_pool_p1_identity(ora):
    rng = np.random.default_rng(10)
    k = _bf16_round(rng.standard_normal((1, 128)).astype(np.float32))
    r = _pool(ora, k, rng.standard_normal((1, 128)).astype(np.float32), np.zeros((1, 128), np.float32))
    np.testing.assert_array_equal(r["x"], k[0].astype(np.float64))
    np.testing.assert_array_equal(r["xb"], _bf16_bits(k[0]))


def test_pool_two_slot_logistic_closed_form(ora):
    # P=2: x = k0 * sigma(z0 - z1) + k1 * sigma(z1 - z0), sigma the logistic function
    rng = np.random.default_rng(11)
    k = rng.standard_normal((2, 128)).astype(np.float32)
    s = (rng.standard_normal((2, 128)) * 3).astype(np.float32)
    ape = (rng.standard_normal((2, 128)) * 0.1).astype(np.float32)
    z = s.astype(np.float64) + ape
    sig = 1.0 / (1.0 + np.exp(-(z[0] - z[1])))
    expect = k[0] * sig + k[1] * (1.0 - sig)
    np.testing.assert_allclose(_pool(ora, k, s, ape)["x"], expect, atol=1e-12)


def test_pool_brute_force_small_chunks(ora):
    # every assignment of keys and scores from {-1, 0, 1} for P <= 3 (one per channel),
    # plus permutation / shift / affine invariances and convexity.
    import itertools

    for P in (2, 3):
        combos = list(itertools.product((-1.0, 0.0, 1.0), repeat=2 * P))
        for start in range(0, len(combos), 128):
            chunk = combos[start:start + 128]
            chunk = chunk + [chunk[-1]] * (128 - len(chunk))
            arr = np.array(chunk, np.float32).T  # [2P, 128]
            k, s = arr[:P], arr[P:]
            ape = np.zeros((P, 128), np.float32)
            x = _pool(ora, k, s, ape)["x"]
            # closed form without the max shift: weights e^{s_j} / sum e^{s_i}
            w = np.exp(s.astype(np.float64))
            expect = (w * k).sum(0) / w.sum(0)
            np.testing.assert_allclose(x, expect, atol=1e-14)
    rng = np.random.default_rng(12)
    P = 16
    # bf16-valued inputs so that the shifted / scaled copies below are exact in fp32
    k = _bf16_round(rng.standard_normal((P, 128)).astype(np.float32))
    s = _bf16_round((rng.standard_normal((P, 128)) * 2).astype(np.float32))
    ape = _bf16_round((rng.standard_normal((P, 128)) * 0.1).astype(np.float32))
    x = _pool(ora, k, s, ape)["x"]
    perm = rng.permutation(P)
    np.testing.assert_allclose(_pool(ora, k[perm], s[perm], ape[perm])["x"], x, atol=1e-12)
    np.testing.assert_allclose(_pool(ora, k, s, ape + np.float32(3.0))["x"], x, atol=1e-12)
    np.testing.assert_allclose(_pool(ora, 2 * k + 1, s, ape)["x"], 2 * x + 1, atol=1e-12)
    assert np.all(x <= k.max(0) + 1e-12) and np.all(x >= k.min(0) - 1e-12)


# ------------------------------------------------------------ pooled kernels
def _rand_bf16(rng, shape, scale=1.0):
    return _bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def test_kpool_compress_cache_layout(ora):
    # one pool written at loc: the FP8 row sits at page*ps*(D+4) + tok*D, the fp32 scale
    # at byte page*ps*(D+4) + ps*D + 4*tok; nothing else changes.
    rng = np.random.default_rng(13)
    P, D, ps, pages = 16, 128, 64, 3
    k = _rand_bf16(rng, (1, P, D))
    s = _rand_bf16(rng, (1, P, D))
    ape = (rng.standard_normal((P, D)) * 0.1).astype(np.float32)
    for loc in (0, 63, 64, 130):
        cache = np.full((pages, ps, D + 4), 0xAB, np.uint8)
        r = ora.kpool_compress(cache, ps, k, s, ape, np.array([loc]), return_compressed=True)
        flat = cache.reshape(-1)
        page, tok = divmod(loc, ps)
        row0 = page * ps * (D + 4) + tok * D
        sc0 = page * ps * (D + 4) + ps * D + 4 * tok
        np.testing.assert_array_equal(flat[row0:row0 + D], r["q"][0])
        assert flat[sc0:sc0 + 4].view(np.float32)[0] == r["scale"][0]
        mask = np.ones(flat.size, bool)
        mask[row0:row0 + D] = False
        mask[sc0:sc0 + 4] = False
        assert np.all(flat[mask] == 0xAB)


def test_kpool_compress_codes_without_cache_write(ora):
    """write_cache off: the cache is untouched and the returned codes and
    scales are those a cache write would have stored."""
    rng = np.random.default_rng(43)
    P, D, ps, n = 16, 128, 8, 5
    k = _rand_bf16(rng, (n, P, D))
    s = _rand_bf16(rng, (n, P, D))
    ape = (rng.standard_normal((P, D)) * 0.1).astype(np.float32)
    loc = np.arange(n, dtype=np.int64)
    c0 = np.full((1, ps, D + 4), 0x3C, np.uint8)
    r = ora.kpool_compress(c0, ps, k, s, ape, loc, write_cache=False, return_compressed=True)
    assert np.all(c0 == 0x3C)
    c1 = np.full((1, ps, D + 4), 0x3C, np.uint8)
    ora.kpool_compress(c1, ps, k, s, ape, loc)
    flat = c1.reshape(-1)
    for i in range(n):
        np.testing.assert_array_equal(flat[i * D:(i + 1) * D], r["q"][i])
        assert flat[ps * D + 4 * i:ps * D + 4 * i + 4].view(np.float32)[0] == r["scale"][i]


def test_kpool_compress_write_mask(ora):
    rng = np.random.default_rng(14)
    P, D, ps = 16, 128, 64
    n = 8
    k = _rand_bf16(rng, (n, P, D))
    s = _rand_bf16(rng, (n, P, D))
    ape = (rng.standard_normal((P, D)) * 0.1).astype(np.float32)
    loc = np.arange(n, dtype=np.int64)
    wm = np.array([1, 0, 1, 1, 0, 0, 1, 0], np.uint8)
    c1 = np.zeros((1, ps, D + 4), np.uint8)
    ora.kpool_compress(c1, ps, k, s, ape, loc, write_mask=wm)
    c2 = np.zeros((1, ps, D + 4), np.uint8)
    ora.kpool_compress(c2, ps, k[wm == 1], s[wm == 1], ape, loc[wm == 1])
    np.testing.assert_array_equal(c1, c2)


def _decode_case(rng, B, positions_start, N, P=16, D=128, ring_blocks=None):
    ring_blocks = ring_blocks or B
    blocks = rng.permutation(ring_blocks)[:B]
    pos = positions_start[:, None] + np.arange(N)[None, :]
    tslot = (blocks[:, None] * P + pos % P).astype(np.int32)
    loc = np.where(pos % P == P - 1, np.arange(B)[:, None] * 4096 + pos // P, -1).astype(np.int32)
    return blocks, pos.astype(np.int32), tslot, loc


def test_kpool_decode_matches_one_shot_from_empty_ring(ora):
    # N = 64 tokens from position 0 per request: 4 pools each, all built in one call
    rng = np.random.default_rng(15)
    B, N, P, D, ps = 4, 64, 16, 128, 64
    blocks, pos, tslot, loc = _decode_case(rng, B, np.zeros(B, np.int64), N)
    loc = np.where(pos % P == P - 1, np.arange(B)[:, None] * 4 + pos // P, -1).astype(np.int32)
    key = _rand_bf16(rng, (B, N, D))
    score = _rand_bf16(rng, (B, N, D))
    ape = _bf16_round((rng.standard_normal((P, D)) * 0.1).astype(np.float32))
    ring = np.zeros((B, 2, P, D), np.uint16)
    cache = np.zeros((1, ps, D + 4), np.uint8)
    ora.kpool_decode_update(cache, ps, ring, tslot, loc, pos, key, score, ape)
    cache2 = np.zeros_like(cache)
    slot_k = key.reshape(B * 4, P, D)
    slot_s = score.reshape(B * 4, P, D)
    ora.kpool_compress(cache2, ps, slot_k, slot_s, ape, np.arange(B * 4, dtype=np.int64))
    np.testing.assert_array_equal(cache, cache2)
    # the ring now holds each request's last pool, slot by slot
    for b in range(B):
        np.testing.assert_array_equal(ring[blocks[b], 0], key[b, -P:])
        np.testing.assert_array_equal(ring[blocks[b], 1], score[b, -P:])


def test_kpool_decode_pool_across_calls_uses_fresh_stashes(ora):
    # a pool filled over three calls must compress the stashed tokens of those calls,
    # not stale ring contents (ordering/gating regression named on the kpool page)
    rng = np.random.default_rng(16)
    P, D, ps = 16, 128, 64
    key = _rand_bf16(rng, (1, P, D))
    score = _rand_bf16(rng, (1, P, D))
    ape = (rng.standard_normal((P, D)) * 0.1).astype(np.float32)
    ring = _rand_bf16(rng, (2, 2, P, D))  # stale garbage
    cache = np.zeros((1, ps, D + 4), np.uint8)
    for lo, hi in ((0, 6), (6, 11), (11, 16)):
        pos = np.arange(lo, hi, dtype=np.int32)[None, :]
        tslot = (1 * P + pos % P).astype(np.int32)
        loc = np.where(pos % P == P - 1, 5, -1).astype(np.int32)
        ora.kpool_decode_update(cache, ps, ring, tslot, loc, pos, key[:, lo:hi], score[:, lo:hi], ape)
    ref = ora.pool_compress(_bf16_round_bits(key[0]), _bf16_round_bits(score[0]), ape, True)
    flat = cache.reshape(-1)  # linear page layout: rows at tok*D, scales after ps*D bytes
    np.testing.assert_array_equal(flat[5 * D:6 * D], ref["q"])
    assert flat[ps * D + 20:ps * D + 24].view(np.float32)[0] == ref["scale"]


def _bf16_round_bits(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_kpool_decode_padding_is_inert(ora):
    rng = np.random.default_rng(17)
    B, N, P, D, ps = 3, 4, 16, 128, 64
    ring = _rand_bf16(rng, (B, 2, P, D))
    ring0 = ring.copy()
    cache = np.zeros((1, ps, D + 4), np.uint8)
    neg = -np.ones((B, N), np.int32)
    ora.kpool_decode_update(cache, ps, ring, neg, neg, neg, _rand_bf16(rng, (B, N, D)),
                            _rand_bf16(rng, (B, N, D)), np.zeros((P, D), np.float32))
    np.testing.assert_array_equal(ring, ring0)
    assert np.all(cache == 0)


_KD_GOLDEN = json.load(open(os.path.join(GOLDEN, "kpool_decode_examples.json")))


def kpool_decode_golden_inputs(fx, D=128):
    """Arrays of the pooled-decode fixture: one token per request."""
    P = fx["P"]
    ring = np.zeros((len(fx["ring"]["key"]), 2, P, D), np.float32)
    ring[:, 0] = np.array(fx["ring"]["key"], np.float32)[:, :, None]
    ring[:, 1] = np.array(fx["ring"]["score"], np.float32)[:, :, None]
    toks = fx["tokens"]
    col = lambda name: np.array([[t[name]] for t in toks], np.int32)
    key = np.array([[np.full(D, t["key"])] for t in toks], np.float32)
    score = np.array([[np.full(D, t["score"])] for t in toks], np.float32)
    ape = np.repeat(np.array(fx["ape"], np.float32)[:, None], D, 1)
    cache = np.full((fx["pages"], fx["page_size"], D + 4), fx["canary"], np.uint8)
    return {"ring": _bf16_bits(ring), "tail_slot_mapping": col("tail_slot"), "slot_mapping": col("slot_mapping"),
            "positions": col("position"), "key": _bf16_bits(key), "score": _bf16_bits(score), "ape": ape,
            "cache": cache}


def kpool_decode_golden_check(fx, cache, ring, D=128):
    """The cache and ring after the fixture's call, against the hand-derived values."""
    P, ps = fx["P"], fx["page_size"]
    e = fx["expect"]
    flat = cache.reshape(-1)
    page, tok = divmod(e["cache"]["loc"], ps)
    row0 = page * ps * (D + 4) + tok * D
    sc0 = page * ps * (D + 4) + ps * D + 4 * tok
    assert flat[row0] == e["cache"]["q0"]
    assert np.all(flat[row0 + 1:row0 + D] == e["cache"]["q_rest"])
    assert flat[sc0:sc0 + 4].view(np.float32)[0] == e["cache"]["scale"]
    rest = np.ones(flat.size, bool)
    rest[row0:row0 + D] = False
    rest[sc0:sc0 + 4] = False
    assert np.all(flat[rest] == fx["canary"]), "only the closing row's bytes change"
    want = np.zeros((len(e["ring_key"]), 2, P, D), np.float32)
    want[:, 0] = np.array(e["ring_key"], np.float32)[:, :, None]
    want[:, 1] = np.array(e["ring_score"], np.float32)[:, :, None]
    np.testing.assert_array_equal(ring, _bf16_bits(want))


def test_kpool_decode_golden_gating_and_block_clamp(ora):
    """Hand-derived: a closing token whose tail slot is negative still closes
    its pool, from ring block 0 (block = max(tail_slot, 0) // P), and stashes
    nothing; a token at the closing slot without a cache location only stashes;
    an open slot with a negative tail slot changes nothing; a token is stashed
    in its position's slot of its tail slot's block."""
    fx = _KD_GOLDEN
    a = kpool_decode_golden_inputs(fx)
    ring, cache = a["ring"].copy(), a["cache"].copy()
    ora.kpool_decode_update(cache, fx["page_size"], ring, a["tail_slot_mapping"], a["slot_mapping"],
                            a["positions"], a["key"], a["score"], a["ape"], round_scale=True)
    kpool_decode_golden_check(fx, cache, ring)


def test_kpool_seed_tail_selects_last_pool(ora):
    # two requests of 21 and 7 prefill tokens; request r's tail block is r; a token is
    # seeded iff it is among its request's last P tokens
    rng = np.random.default_rng(18)
    P, D = 16, 128
    lens = [21, 7]
    tslot = np.concatenate([r * P + np.arange(n) % P for r, n in enumerate(lens)]).astype(np.int32)
    n = len(tslot)
    key = _rand_bf16(rng, (n, D))
    score = _rand_bf16(rng, (n, D))
    ring = np.zeros((2, 2, P, D), np.uint16)
    ora.kpool_seed_tail(ring, key, score, tslot)
    seeded = np.zeros((2, P), bool)
    for i in range(n):
        r = 0 if i < lens[0] else 1
        idx_in_req = i if r == 0 else i - lens[0]
        if idx_in_req >= lens[r] - P:
            np.testing.assert_array_equal(ring[r, 0, tslot[i] % P], key[i])
            np.testing.assert_array_equal(ring[r, 1, tslot[i] % P], score[i])
            seeded[r, tslot[i] % P] = True
    assert np.all(ring[0][:, ~seeded[0]] == 0) and np.all(ring[1][:, ~seeded[1]] == 0)


# ---------------------------------------------------------------- online c128
_C128_GOLDEN = json.load(open(os.path.join(GOLDEN, "c128_examples.json")))["cases"]


@pytest.mark.parametrize("case", [c for c in _C128_GOLDEN if "state_after" in c], ids=lambda c: c["name"])
def test_c128_golden_two_tokens(ora, case):
    """fp32 and bf16 input rows (the bf16 case pins the oracle's bf16 branch)."""
    D = 128
    state = np.zeros((1, 3, D), np.float32)
    ape = np.zeros((128, D), np.float32)
    for t, (kk, ss) in enumerate(zip(case["keys"], case["scores"])):
        inp = np.concatenate([np.full(D, kk, np.float32), np.full(D, ss, np.float32)])[None]
        if case["dtype"] == "bf16":
            inp = _bf16_bits(inp)
        out, ns, closed = ora.c128_decode(state, inp, ape, np.array([0]), np.array([t + 1]))
        np.testing.assert_allclose(ns[0, :, 0], case["state_after"][t], rtol=1e-6, atol=1e-6)
        assert np.all(ns[0] == ns[0, :, :1])  # every channel alike
        state[0] = ns[0].astype(np.float32)


def test_c128_golden_equal_logits_full_chunk(ora):
    """Keys 0..127 under equal logits: after 127 tokens the state is (c, 127,
    63); the 128th token closes the chunk with the mean 63.5.  The same chunk
    as one prefill segment emits the same row.  Both input types."""
    case = next(c for c in _C128_GOLDEN if "closing_kv" in c)
    D = 128
    keys = np.arange(128, dtype=np.float32)
    for dtype in ("f32", "bf16"):
        for logit in (0.0, -3.5):
            ape = np.zeros((128, D), np.float32)
            state = np.zeros((1, 3, D), np.float32)
            for t in range(128):
                inp = np.concatenate([np.full(D, keys[t], np.float32), np.full(D, logit, np.float32)])[None]
                if dtype == "bf16":
                    inp = _bf16_bits(inp)
                out, ns, closed = ora.c128_decode(state, inp, ape, np.array([0]), np.array([128 * 3 + t + 1]))
                assert closed[0] == (t == 127)
                if t == 126:
                    np.testing.assert_allclose(ns[0, :, 0], [logit, 127.0, 63.0], rtol=1e-12, atol=1e-12)
                if t < 127:
                    state[0] = ns[0].astype(np.float32)
            np.testing.assert_allclose(out[0], case["closing_kv"], rtol=0, atol=1e-12)
            chunk = np.concatenate([np.repeat(keys[:, None], D, 1), np.full((128, D), logit, np.float32)], 1)
            if dtype == "bf16":
                chunk = _bf16_bits(chunk)
            pout, w, _, sw = ora.c128_prefill(np.zeros((1, 3, D), np.float32), chunk, ape, np.array([0]),
                                              np.array([128]), np.array([128]))
            assert w[127] and w.sum() == 1 and not sw[0]
            np.testing.assert_allclose(pout[127], case["closing_kv"], rtol=0, atol=1e-12)


def _two_pass(k, z):
    """Softmax-weighted mean of rows k under logits z (both [n, D]), computed
    straight from the definition in double: (max, sum, kv)."""
    k = np.asarray(k, np.float64)
    z = np.asarray(z, np.float64)
    m = z.max(0)
    w = np.exp(z - m)
    return m, w.sum(0), (w * k).sum(0) / w.sum(0)


def test_c128_decode_merge_equals_two_pass_over_prior_tokens(ora):
    """A slot whose state is the two-pass (max, sum, kv) of p virtual tokens at
    chunk positions 0..p-1 (built here in numpy), updated with one token at
    position p, equals the two-pass over all p+1 tokens; at p = 127 the emitted
    row does and the slot is left alone.  Pins the merge branch of the decode."""
    rng = np.random.default_rng(40)
    D = 128
    ps = [1, 2, 17, 63, 64, 100, 126, 127]
    B = len(ps)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    k = rng.standard_normal((B, 128, D)).astype(np.float32)
    s = (rng.standard_normal((B, 128, D)) * 2).astype(np.float32)
    z = s.astype(np.float64) + ape
    state = np.zeros((2 * B, 3, D), np.float32)
    slots = rng.permutation(2 * B)[:B]
    for b, p in enumerate(ps):
        m, sm, kv = _two_pass(k[b, :p], z[b, :p])
        state[slots[b]] = np.stack([m, sm, kv]).astype(np.float32)
    inp = np.stack([np.concatenate([k[b, p], s[b, p]]) for b, p in enumerate(ps)])
    seq = np.array([128 * (b + 2) + p + 1 for b, p in enumerate(ps)])
    out, ns, closed = ora.c128_decode(state, inp, ape, slots.astype(np.int32), seq)
    for b, p in enumerate(ps):
        # the stored state is fp32: compare with the two-pass over the fp32-rounded prior
        m, sm, kv = _two_pass(k[b, :p + 1], z[b, :p + 1])
        assert closed[b] == (p == 127)
        np.testing.assert_allclose(ns[b, 2], kv, rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(ns[b, 0], m, rtol=0, atol=1e-6)
        # the sum is relative to the running max: equal up to the fp32 rounding of the prior state
        np.testing.assert_allclose(ns[b, 1], sm, rtol=1e-6)
        if p == 127:
            np.testing.assert_allclose(out[b], kv, rtol=1e-6, atol=1e-6)


def test_c128_prefill_merge_equals_two_pass_over_prior_tokens(ora):
    """Prefill of a request whose first extend token sits mid-chunk: the slot
    holds the two-pass (max, sum, kv) of the chunk's p earlier (virtual) tokens,
    built here in numpy.  The closing row of that chunk must equal the two-pass
    over all 128 of its tokens, later chunks the two-pass over their own
    tokens, and the trailing partial chunk's new state the two-pass over its
    tokens (merged with the prior when the extend ends in the first chunk).
    Pins the prefill's merge with a stored partial directly."""
    rng = np.random.default_rng(41)
    D = 128
    cases = [(37, 91), (37, 400), (5, 20), (127, 1), (127, 130), (64, 64), (1, 300)]  # (p, extend)
    B = len(cases)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    chunk0 = 128 * np.arange(1, B + 1)  # request b's prior chunk starts at position chunk0[b]
    state = np.zeros((2 * B, 3, D), np.float32)
    load = rng.permutation(2 * B)[:B].astype(np.int32)
    toks_k, toks_s, rows = [], [], []
    seq, ext = [], []
    for b, (p, e) in enumerate(cases):
        n = p + e
        k = rng.standard_normal((n, D)).astype(np.float32)
        s = (rng.standard_normal((n, D)) * 2).astype(np.float32)
        m, sm, kv = _two_pass(k[:p], s[:p].astype(np.float64) + ape[:p])
        state[load[b]] = np.stack([m, sm, kv]).astype(np.float32)
        toks_k.append(k)
        toks_s.append(s)
        rows.append(np.concatenate([k[p:], s[p:]], 1))
        seq.append(chunk0[b] + n)
        ext.append(e)
    inp = np.concatenate(rows, 0)
    out, written, fs, sw = ora.c128_prefill(state, inp, ape, load, np.array(seq), np.array(ext))
    base = 0
    for b, (p, e) in enumerate(cases):
        n = p + e
        k, s = toks_k[b], toks_s[b]
        z = s.astype(np.float64) + ape[np.arange(n) % 128]
        # chunks of this request in local token numbering (local 0 = chunk position 0)
        for c0 in range(0, n, 128):
            c1 = min(n, c0 + 128)
            m, sm, kv = _two_pass(k[c0:c1], z[c0:c1])
            if c1 - c0 == 128:
                r = base + (c1 - 1 - p)  # ragged row of the closing token
                assert written[r]
                np.testing.assert_allclose(out[r], kv, rtol=1e-6, atol=1e-6)
            else:
                assert sw[b]
                np.testing.assert_allclose(fs[b, 2], kv, rtol=1e-6, atol=1e-6)
                np.testing.assert_allclose(fs[b, 0], m, rtol=0, atol=1e-6)
                np.testing.assert_allclose(fs[b, 1], sm, rtol=1e-6)
        if n % 128 == 0:
            assert not sw[b]
        assert written[base:base + e].sum() == n // 128
        base += e


@pytest.mark.parametrize("fn", ["decode", "prefill"])
def test_c128_bf16_input_equals_widened_fp32(ora, fn):
    """The bf16 input branch reads each value as its exact fp32 widening: the
    same rows given as bf16 bits and as fp32 give identical results."""
    rng = np.random.default_rng(42)
    D = 256
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    state = rng.standard_normal((64, 3, D)).astype(np.float32)
    state[:, 1] = np.abs(state[:, 1]) + 1
    if fn == "decode":
        B = 40
        bits = _bf16_bits(rng.standard_normal((B, 2 * D)).astype(np.float32) * 3)
        idx = rng.permutation(64)[:B].astype(np.int32)
        seq = rng.integers(1, 5000, B)
        seq[:3] = [1, 128, 129]
        r_b = ora.c128_decode(state, bits, ape, idx, seq)
        r_f = ora.c128_decode(state, _bf16_round_bits(bits), ape, idx, seq)
    else:
        ext = np.array([300, 5, 128, 77])
        seq = ext + np.array([0, 60, 128, 200])
        bits = _bf16_bits(rng.standard_normal((int(ext.sum()), 2 * D)).astype(np.float32) * 3)
        idx = rng.permutation(64)[:4].astype(np.int32)
        r_b = ora.c128_prefill(state, bits, ape, idx, seq, ext)
        r_f = ora.c128_prefill(state, _bf16_round_bits(bits), ape, idx, seq, ext)
    for a, b in zip(r_b, r_f):
        np.testing.assert_array_equal(np.nan_to_num(a, nan=7.0), np.nan_to_num(b, nan=7.0))


def test_c128_decode_chunk_equals_two_pass(ora):
    # 128 single-token updates from chunk position 0 == a two-pass softmax over the chunk
    rng = np.random.default_rng(19)
    D = 256
    k = rng.standard_normal((128, D)).astype(np.float32)
    s = (rng.standard_normal((128, D)) * 2).astype(np.float32)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    state = np.zeros((1, 3, D), np.float32)
    seq0 = 128 * 7  # chunk starts at seq_len-1 = 896
    for t in range(128):
        inp = np.concatenate([k[t], s[t]])[None]
        out, ns, closed = ora.c128_decode(state, inp, ape, np.array([0]), np.array([seq0 + t + 1]))
        assert closed[0] == (t == 127)
        if t == 0:
            np.testing.assert_array_equal(ns[0, 1], 1.0)
            np.testing.assert_array_equal(ns[0, 2], k[0])
        if t < 127:
            state[0] = ns[0]
    z = s.astype(np.float64) + ape
    w = np.exp(z - z.max(0))
    ref = (w * k).sum(0) / w.sum(0)
    np.testing.assert_allclose(out[0], ref, rtol=2e-6, atol=2e-6)
    # and the oracle's own prefill path (two-pass over the chunk) agrees
    inp_all = np.concatenate([k, s], 1)
    pout, written, fs, sw = ora.c128_prefill(np.zeros((1, 3, D), np.float32), inp_all, ape,
                                             np.array([0]), np.array([seq0 + 128]), np.array([128]))
    assert written[127] and written.sum() == 1 and not sw[0]
    np.testing.assert_allclose(pout[127], out[0], rtol=2e-6, atol=2e-6)


def test_c128_decode_position_from_seq_len_minus_one(ora):
    # seq_len % 128 == 0 means the token sits at chunk position 127 and closes the chunk;
    # seq_len % 128 == 1 means position 0 and starts a new chunk from this token alone
    D = 128
    rng = np.random.default_rng(20)
    state = rng.standard_normal((2, 3, D)).astype(np.float32)
    state[:, 1] = np.abs(state[:, 1]) + 1
    inp = rng.standard_normal((2, 2 * D)).astype(np.float32)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    out, ns, closed = ora.c128_decode(state, inp, ape, np.array([0, 1]), np.array([256, 257]))
    assert closed[0] and not closed[1]
    np.testing.assert_array_equal(ns[1, 0], inp[1, D:].astype(np.float64) + ape[0])
    np.testing.assert_array_equal(ns[1, 2], inp[1, :D])


def test_c128_prefill_split_equals_whole(ora):
    # prefill of a request in several extend pieces, chaining the partial state through the
    # slot, equals a single extend (checkpoint/resume of the running state)
    rng = np.random.default_rng(21)
    D = 128
    T = 700
    prefix = 37
    k = rng.standard_normal((T, D)).astype(np.float32)
    s = (rng.standard_normal((T, D)) * 2).astype(np.float32)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    inp = np.concatenate([k, s], 1)
    # prior partial state for positions [0, 37) built by the oracle from virtual tokens
    pk = rng.standard_normal((prefix, D)).astype(np.float32)
    psc = rng.standard_normal((prefix, D)).astype(np.float32)
    _, _, fs0, sw0 = ora.c128_prefill(np.zeros((1, 3, D), np.float32), np.concatenate([pk, psc], 1), ape,
                                      np.array([0]), np.array([prefix]), np.array([prefix]))
    st0 = fs0.astype(np.float32)
    whole_out, whole_w, whole_fs, _ = ora.c128_prefill(st0, inp, ape, np.array([0]),
                                                       np.array([prefix + T]), np.array([T]))
    cuts = [0, 1, 91, 92, 219, 500, 640, T]
    st = st0.copy()
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, w, fs, sw = ora.c128_prefill(st, inp[a:b], ape, np.array([0]), np.array([prefix + b]),
                                        np.array([b - a]))
        for r in np.nonzero(w)[0]:
            assert whole_w[a + r]
            np.testing.assert_allclose(o[r], whole_out[a + r], rtol=1e-5, atol=1e-5)
        if sw[0]:
            st = fs.astype(np.float32)
    np.testing.assert_allclose(st[0], whole_fs[0], rtol=1e-5, atol=1e-5)


def test_c128_prefill_emits_exactly_at_chunk_position_127(ora):
    # c128 page, flash_c128_online_prefill: a chunk closes at its 128th token
    # (chunk position 127), which emits the row; a request whose last token sits
    # anywhere else (126 included) leaves its running state in the slot instead
    rng = np.random.default_rng(24)
    D = 128
    ends = [125, 126, 127, 128, 129, 254, 255, 256, 383]  # sequence lengths around chunk ends
    B = len(ends)
    seq = np.array(ends, np.int64)
    ext = np.array([int(rng.integers(1, e + 1)) for e in ends], np.int64)
    T = int(ext.sum())
    inp = rng.standard_normal((T, 2 * D)).astype(np.float32)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    state = rng.standard_normal((B, 3, D)).astype(np.float32)
    state[:, 1] = np.abs(state[:, 1]) + 1.0
    out, w, fs, sw = ora.c128_prefill(state, inp, ape, np.arange(B), seq, ext)
    pos = np.concatenate([np.arange(s - e, s) for s, e in zip(seq, ext)])
    w, sw = w.astype(bool), sw.astype(bool)
    np.testing.assert_array_equal(w, pos % 128 == 127)
    np.testing.assert_array_equal(sw, (seq - 1) % 128 != 127)
    # the values go where the flags say: emitted rows and stored states are
    # finite, rows of tokens that emit nothing are left unwritten (NaN)
    assert np.all(np.isfinite(out[w])) and np.all(np.isnan(out[~w]))
    assert np.all(np.isfinite(fs[sw]))


def test_c128_prefill_single_token_window(ora):
    D = 128
    rng = np.random.default_rng(22)
    inp = rng.standard_normal((1, 2 * D)).astype(np.float32)
    ape = (rng.standard_normal((128, D)) * 0.1).astype(np.float32)
    _, w, fs, sw = ora.c128_prefill(np.zeros((1, 3, D), np.float32), inp, ape, np.array([0]),
                                    np.array([129]), np.array([1]))
    assert sw[0] and not w.any()
    np.testing.assert_array_equal(fs[0, 0], inp[0, D:].astype(np.float64) + ape[0])
    np.testing.assert_array_equal(fs[0, 1], 1.0)
    np.testing.assert_array_equal(fs[0, 2], inp[0, :D])


# -------------------------------------------------------------- segmenter
@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "plan_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_segmenter_golden(ora, case):
    c, w = ora.plan_segments(np.array(case["seq_lens"]), np.array(case["extend_lens"]))
    assert c.tolist() == case["compress"]
    assert w.tolist() == case["write"]


def test_segmenter_invariants_brute_force(ora):
    rng = np.random.default_rng(23)
    for _ in range(300):
        B = int(rng.integers(1, 4))
        ext = rng.integers(1, 301, B)
        pre = rng.integers(0, 301, B)
        seq = pre + ext
        c, w = ora.plan_segments(seq, ext)
        cover = np.zeros(int(ext.sum()), int)
        base = np.concatenate([[0], np.cumsum(ext)])
        for kind, rows in (("c", c.astype(np.int64)), ("w", w.astype(np.int64))):
            for rid, b, pos, wl in rows:
                assert 1 <= wl <= 128
                first_pos = pos - wl + 1
                assert first_pos // 128 == pos // 128
                assert (pos % 128 == 127) == (kind == "c")
                assert pre[b] <= first_pos and pos < seq[b]
                assert rid - (pos - pre[b]) == base[b]
                cover[rid - wl + 1: rid + 1] += 1
        assert np.all(cover == 1)
        assert np.all(np.bincount(w[:, 1], minlength=B) <= 1) if len(w) else True


# ---------------------------------------------------- pool -> token expansion
@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "expand_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_expand_golden(ora, case):
    out = ora.expand_pools_and_append_tail(np.array(case["pool_ids"]), np.array(case["seq_lens"]), case["P"])
    assert out.tolist() == case["out"]
    # the same ids as the first columns of wider rows (row stride G + 3, junk
    # in the extra columns) give the same output
    ids = np.array(case["pool_ids"], np.int32).reshape(len(case["seq_lens"]), -1)
    wide = np.full((ids.shape[0], ids.shape[1] + 3), 12345, np.int32)
    wide[:, :ids.shape[1]] = ids
    out = ora.expand_pools_and_append_tail(wide[:, :ids.shape[1]], np.array(case["seq_lens"]), case["P"])
    assert out.tolist() == case["out"]


def test_expand_invariants(ora):
    rng = np.random.default_rng(30)
    for P in (1, 2, 4, 16):
        rows, G = 7, 5
        ids = rng.integers(-1, 50, (rows, G)).astype(np.int32)
        seq = rng.integers(0, 900, rows)
        out = ora.expand_pools_and_append_tail(ids, seq, P)
        assert out.shape == (rows, G * P + P - 1)
        for r in range(rows):
            hist = out[r, :G * P].reshape(G, P)
            for g in range(G):
                if ids[r, g] < 0:
                    assert np.all(hist[g] == -1)
                else:  # P consecutive ids starting at a multiple of P
                    assert hist[g, 0] % P == 0 and np.all(np.diff(hist[g]) == 1) and hist[g, 0] // P == ids[r, g]
            tail = out[r, G * P:]
            real = tail[tail >= 0]
            # the tail is exactly the tokens after the last full pool, in order, then -1s
            assert real.tolist() == list(range((seq[r] // P) * P, seq[r]))
            assert np.all(tail[len(real):] == -1)


# ------------------------------------------- c128 rows -> paged FP8 cache
def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _e4m3(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("round_scale", [False, True])
def test_c128_rows_to_cache_golden(ora, round_scale):
    """Block j of the row is (j+1)·e_0: its rotation is the constant (j+1)/sqrt(128)
    in every channel, so every code of the block is one value and the block's
    scale follows from that constant alone.  Row at location 5 of a
    4-row-per-page cache: page 1, row 1; scales of row 1 at footer 4..7."""
    D, ps = 512, 4
    cache = np.zeros((2, ps, D + 16), np.uint8)
    row = np.zeros((1, D), np.float32)
    for j in range(4):
        row[0, 128 * j] = j + 1
    ora.c128_rows_to_cache(cache, ps, row, np.array([5]), round_scale=round_scale)
    c = np.float32(1.0 / np.sqrt(128.0))
    expect = cache.copy() * 0
    for j in range(4):
        y = _bf16(np.float32(j + 1) * c)  # the fp32 butterfly of e_0 is exact; one multiply, then bf16
        v = np.float32(y * np.float32(1.0 / 448.0))
        scale = np.float32(2.0 ** np.ceil(np.log2(np.float64(v)))) if round_scale else v
        q = _e4m3(np.clip(np.float32(y / scale), -448, 448))
        page = expect[1].reshape(-1)  # a page: 4 rows of D code bytes, then 4 x 4 fp32 scales
        page[1 * D + 128 * j:1 * D + 128 * j + 128] = q
        page[ps * D + 4 * (4 * 1 + j):ps * D + 4 * (4 * 1 + j) + 4] = np.array([scale], np.float32).view(np.uint8)
    np.testing.assert_array_equal(cache, expect)
    if not round_scale:
        assert np.all(cache[1].reshape(-1)[D:2 * D] == 0x7E)  # 448, the largest e4m3 value
    # a row with a negative location is skipped: nothing changes
    before = cache.copy()
    ora.c128_rows_to_cache(cache, ps, row * 3, np.array([-1]), round_scale=round_scale)
    np.testing.assert_array_equal(cache, before)


def test_c128_rows_to_cache_rounds_the_row_to_bf16_first(ora):
    """Worked by hand, D = 128, power-of-two scale: the row (1, 1 - 2^-9, 0,
    ..., 0) rounds to bf16 (1, 1) (1 - 2^-9 is a tie between 1 - 2^-8 and 1;
    1 has the even mantissa), so the rotation is 2c in even channels and 0 in
    odd ones (c = fp32(1/sqrt(128))).  bf16(2c) = 0.1767578125 is the absmax;
    absmax/448 = 3.95e-4 gives the scale 2^-11; 0.1767578125 * 2^11 = 362
    rounds to the e4m3 value 352 = 1.375 * 2^8, code 0x7B; the odd channels are
    +0, code 0x00.  Without the first rounding the odd channels would hold
    2^-9 c and a nonzero code."""
    D, ps = 128, 1
    cache = np.full((1, ps, D + 4), 0xAB, np.uint8)
    row = np.zeros((1, D), np.float32)
    row[0, 0], row[0, 1] = 1.0, 1.0 - 2.0 ** -9
    ora.c128_rows_to_cache(cache, ps, row, np.array([0]), round_scale=True)
    codes = cache[0, 0, :D]
    assert np.all(codes[0::2] == 0x7B) and np.all(codes[1::2] == 0x00)
    assert cache[0, 0, D:].view(np.float32)[0] == 2.0 ** -11


@pytest.mark.parametrize("round_scale", [False, True])
def test_c128_rows_to_cache_inverse_rotation(ora, round_scale):
    """Decoding the codes, scaling them and applying the inverse of the
    orthonormal Hadamard matrix (itself) recovers each 128-block of the row to
    FP8 precision; a wrong rotation order, block offset or scale index would not."""
    from scipy.linalg import hadamard

    rng = np.random.default_rng(7)
    D, ps, n = 256, 8, 10
    rows = (rng.standard_normal((n, D)) * np.repeat(rng.uniform(0.01, 30, (n, D // 128)), 128, axis=1))
    rows = rows.astype(np.float32)
    locs = rng.permutation(3 * ps)[:n].astype(np.int64)
    cache = np.zeros((3, ps, D + 8), np.uint8)
    ora.c128_rows_to_cache(cache, ps, rows, locs, round_scale=round_scale)
    H = hadamard(128) / np.sqrt(128.0)
    flat = cache.reshape(3, -1)
    for r in range(n):
        page, tok = divmod(int(locs[r]), ps)
        codes = flat[page, tok * D:tok * D + D]
        deq = torch.tensor(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        scales = flat[page, ps * D + 4 * tok * 2: ps * D + 4 * tok * 2 + 8].view(np.float32)
        for j in range(2):
            x = rows[r, 128 * j:128 * j + 128].astype(np.float64)
            back = H @ (deq[128 * j:128 * j + 128] * scales[j])
            assert np.linalg.norm(back - x) <= 0.08 * np.linalg.norm(x), (r, j)
