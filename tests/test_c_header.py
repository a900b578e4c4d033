"""The C ABI from C: include/ckv.h compiles as strict C11 with warnings as
errors, a C program links libckv.so and calls it.  CPU only: the program runs
the host planner on the hand-derived plans of tests/golden/plan_examples.json
(sglang page "deepseek_v4/c128_online.cuh", plan_online_prefill_host) and
checks argument validation of the device entry points, which returns before
anything is launched."""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "ckv.h"

int main(int argc, char** argv) {
  /* argv: B, then B (seq_len, extend_len) pairs */
  if (argc < 2) return 4;
  uint32_t B = (uint32_t)atoi(argv[1]);
  if (B > 8 || argc < 2 + 2 * (int)B) return 4;
  int64_t seq[8], ext[8];
  uint32_t T = 0;
  for (uint32_t b = 0; b < B; ++b) {
    seq[b] = atoll(argv[2 + 2 * b]);
    ext[b] = atoll(argv[3 + 2 * b]);
    T += (uint32_t)ext[b];
  }
  ckv_plan_entry cp[4096], wp[4096];
  uint32_t nc = 0, nw = 0;
  ckv_status s = ckv_plan_online_prefill(seq, ext, B, T, cp, wp, 0, &nc, &nw);
  if (s != CKV_OK) { printf("status %d %s\n", s, ckv_status_string(s)); return 1; }
  printf("abi %d\n", ckv_abi_version());
  for (uint32_t i = 0; i < nc; ++i)
    printf("c %u %u %u %u\n", cp[i].ragged_id, cp[i].batch_id, cp[i].position, cp[i].window_len);
  for (uint32_t i = 0; i < nw; ++i)
    printf("w %u %u %u %u\n", wp[i].ragged_id, wp[i].batch_id, wp[i].position, wp[i].window_len);
  /* validation happens before any launch: no GPU is touched */
  if (ckv_c128_online_decode(0, 4, 0, CKV_F32, 0, 0, 0, 0, 3, 100, 0, 0, 0) != CKV_ERR_SHAPE) return 2;
  if (ckv_check_distinct_noalloc((void*)16, 4, 10, CKV_NOALLOC_MAX_RANGE + 1, (int32_t*)16, 0) != CKV_ERR_SHAPE)
    return 3;
  return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    from compressed_kv_attention_gated_gb300 import build

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = build.build()
    d = tmp_path_factory.mktemp("capi")
    src = d / "main.c"
    src.write_text("#include <stdlib.h>\n" + PROGRAM)
    exe = d / "main"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", os.path.dirname(lib), "-lckv",
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True, capture_output=True, text=True)
    return str(exe)


def test_c_program_plans_match_golden(program):
    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "plan_examples.json")))["cases"]
    for c in cases:
        args = [str(len(c["seq_lens"]))]
        for s, e in zip(c["seq_lens"], c["extend_lens"]):
            args += [str(s), str(e)]
        r = subprocess.run([program, *args], capture_output=True, text=True, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
        assert r.returncode == 0, (c["name"], r.stdout, r.stderr)
        lines = r.stdout.split("\n")
        assert lines[0] == "abi 1"
        got_c = [[int(x) for x in l.split()[1:]] for l in lines if l.startswith("c ")]
        got_w = [[int(x) for x in l.split()[1:]] for l in lines if l.startswith("w ")]
        assert got_c == c["compress"], c["name"]
        assert got_w == c["write"], c["name"]
