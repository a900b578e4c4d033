"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a copy of oracle/ckv_oracle.cpp (a dropped
term, a wrong sign or index, a wrong rounding, a skipped branch), builds it
with the oracle's own flags, and runs tests/test_oracle_pins.py against that
build (CKV_ORACLE_SO): the pins must fail.  A control build of the unchanged
source must pass.  CPU only; the planted mistakes stay in temporary files."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ckv_oracle.cpp")

# (what the mistake is, text in the oracle, text that replaces it)
MUTANTS = [
    ("bf16 rounding truncates instead of rounding to nearest even",
     "double r = std::nearbyint(std::ldexp(a, -qexp));  // ties to even (default mode)",
     "double r = std::trunc(std::ldexp(a, -qexp));"),
    ("e4m3 ties round away from zero",
     "double r = std::ldexp(std::nearbyint(std::ldexp(a, -qexp)), qexp);",
     "double r = std::ldexp(std::round(std::ldexp(a, -qexp)), qexp);"),
    ("power-of-two scale doubles exact powers of two",
     "if (f == 0.5) return v;                             // already a power of two",
     ""),
    ("Hadamard sign pattern flipped",
     "acc += parity ? -in[j] : in[j];",
     "acc += parity ? in[j] : -in[j];"),
    ("fp32 rotation scaled by 1/128 instead of 1/sqrt(128)",
     "const float c = static_cast<float>(1.0 / std::sqrt(128.0));",
     "const float c = static_cast<float>(1.0 / 128.0);"),
    ("power-of-two and linear scales swapped",
     "const float scale = round_scale ? pow2_ceil(v) : v;",
     "const float scale = round_scale ? v : pow2_ceil(v);"),
    ("linear scale: multiply by the reciprocal instead of dividing",
     "float t = bf16_to_float(yb[d]) / scale;",
     "float t = bf16_to_float(yb[d]) * (1.0f / scale);"),
    ("absmax floor 1e-3 instead of 1e-4",
     "absmax = std::max(absmax, 1e-4f);",
     "absmax = std::max(absmax, 1e-3f);"),
    ("position bias left out of the pool weights",
     "const double w = std::exp(static_cast<double>(s[j * D + d]) + ape[j * D + d] - mx);",
     "const double w = std::exp(static_cast<double>(s[j * D + d]) - mx);"),
    ("cache scale stored at the wrong footer offset",
     "std::memcpy(base + page_size * D + 4 * tok, &scale, 4);",
     "std::memcpy(base + page_size * D + tok, &scale, 4);"),
    ("a closing token with a negative tail slot does not close its pool",
     "const bool pos_valid = loc >= 0 && pos >= 0;",
     "const bool pos_valid = loc >= 0 && pos >= 0 && tslot >= 0;"),
    ("c128 decode: stored partial weighted by e^(m - m1)",
     "const double w1 = s1 * std::exp(m1 - m);",
     "const double w1 = s1 * std::exp(m - m1);"),
    ("c128 decode: chunk position from seq_len instead of seq_len - 1",
     "const int p = (seq_lens[b] - 1) % 128;",
     "const int p = seq_lens[b] % 128;"),
    ("bf16 input read as raw integers",
     "return bf16_to_float(static_cast<const uint16_t*>(p)[i]);",
     "return static_cast<const uint16_t*>(p)[i];"),
    ("prefill: stored partial never merged",
     "if (starts_mid) {",
     "if (false && starts_mid) {"),
    ("prefill: merge drops the segment's own sum",
     "const double w1 = s1 * std::exp(m1 - M), w2 = s * std::exp(m - M);",
     "const double w1 = s1 * std::exp(m1 - M), w2 = std::exp(m - M);"),
    ("segmenter: window length one too long",
     "dst[3] = static_cast<uint32_t>(len);",
     "dst[3] = static_cast<uint32_t>(len + 1);"),
    ("tail seed ignores the tail block of the token P ahead",
     "if (ahead >= 0 && ahead / P == blk) continue;",
     "if (ahead >= 0) continue;"),
    ("pool expansion treats pool id 0 as invalid",
     "o[g * P + k] = id >= 0 ? static_cast<int32_t>(id * P + k) : -1;",
     "o[g * P + k] = id > 0 ? static_cast<int32_t>(id * P + k) : -1;"),
    ("Hadamard fp32 butterflies in descending span order",
     "  for (int h = 1; h < 128; h <<= 1) {\n    for (int i = 0; i < 128; ++i) {\n      if (i & h) continue;",
     "  for (int h = 64; h >= 1; h >>= 1) {\n    for (int i = 0; i < 128; ++i) {\n      if (i & h) continue;"),
    ("prefill emits a row at chunk position 126",
     "if (last % 128 == 127) {",
     "if (last % 128 >= 126) {"),
    ("pooled decode stashes at the tail slot's own offset",
     "std::memcpy(kring + slot * D, kcur, D * 2);",
     "std::memcpy(kring + (std::max(tslot, 0) % P) * D, kcur, D * 2);"),
    ("pooled path: the pool output enters the rotation without its bf16 rounding",
     "  // D == 128 for the rotation (checked by the callers).\n  float xf[128], yf[128];\n"
     "  for (int d = 0; d < 128; ++d) xf[d] = bf16_to_float(xb[d]);",
     "  // D == 128 for the rotation (checked by the callers).\n  float xf[128], yf[128];\n"
     "  for (int d = 0; d < 128; ++d) xf[d] = static_cast<float>(x[d]);"),
    ("c128 FP8 store: the row enters the rotation without its bf16 rounding",
     "for (int d = 0; d < 128; ++d) xf[d] = bf16_to_float(bf16_from_double(rows[r * D + 128 * j + d]));",
     "for (int d = 0; d < 128; ++d) xf[d] = static_cast<float>(rows[r * D + 128 * j + d]);"),
    ("pool expansion reads the ids with the group count as row stride",
     "const int64_t id = pool_ids[r * stride + g];",
     "const int64_t id = pool_ids[r * groups + g];"),
    ("c128 FP8 store: block scales laid out block-major",
     "std::memcpy(base + page_size * D + 4 * (tok * blocks + j), &scale, 4);",
     "std::memcpy(base + page_size * D + 4 * (j * page_size + tok), &scale, 4);"),
]


def _build(tmp_path, source, name):
    import oracle

    cpp = tmp_path / f"{name}.cpp"
    cpp.write_text(source)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["g++", *oracle.CFLAGS, str(cpp), "-o", str(so)], check=True)
    return str(so)


def _run_pins(so):
    env = dict(os.environ, CKV_ORACLE_SO=so)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _outcome(tmp_dir, name, source):
    path = tmp_dir / name
    path.mkdir()
    r = _run_pins(_build(path, source, name))
    return r.returncode, r.stdout[-1500:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every planted mistake (and the unchanged control) built and run against
    the pins, several at a time; keyed by the mistake's description."""
    from concurrent.futures import ThreadPoolExecutor

    src = open(SRC).read()
    jobs = {"control": src}
    for what, old, new in MUTANTS:
        if src.count(old) == 1:
            jobs[what] = src.replace(old, new)
    tmp = tmp_path_factory.mktemp("mutants")
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {what: ex.submit(_outcome, tmp, f"m{i}", source) for i, (what, source) in enumerate(jobs.items())}
        return {what: f.result() for what, f in futs.items()}


def test_control_build_passes_the_pins(outcomes):
    rc, out = outcomes["control"]
    assert rc == 0, out


@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, what, old, new):
    assert open(SRC).read().count(old) == 1, f"the oracle no longer contains the mutated line: {old}"
    rc, out = outcomes[what]
    assert rc == 1, f"the pins did not catch: {what}\n{out}"
