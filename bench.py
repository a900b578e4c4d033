#!/usr/bin/env python
"""Throughput of gated-softmax KV compression on GB300.

One step is one pass of the whole hot path over one batch of synthetic,
device-resident input, in the order a serving engine would issue it:

  1. pooled decode/verify update   512 requests x 4 tokens, P=16, D=128
  2. online c128 decode            2048 requests, D=512 fp32
  3. online c128 prefill           64 requests (prefix U[0,16384], extend
                                   U[1,8192], ~262K tokens), D=512 fp32
  4. online c128 prefill           8 x 131072 tokens, D=512 bf16, Student-t scores
  5. pooled one-shot compression   the same 1,048,576 tokens as 65,536 pools
                                   of P=16, D=128 bf16

The metric is compressed-KV tokens per second: every input token consumed by
one of the five calls counts once per call.  Alongside: per-kernel time,
algorithmic bytes, achieved HBM GB/s and its fraction of the measured peak;
the roofline of the dominant kernel; an end-to-end number through the same
C-ABI calls with host-resident inputs (H2D copies and the D2H of the
compressed rows inside the timed region); and the CPU oracle timed on a
bounded sample of the same step on this machine's host cores.

The step's working set (~3.7 GB) is far larger than the 126 MB L2, and every
call streams gigabytes between two uses of the same buffer, so no input is
L2-resident when its kernel starts.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica of the step (independent
requests, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed-KV tokens/s and achieved HBM GB/s (% of GB300 peak), decode & prefill"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("serving step: pooled decode/verify B=512 N=4 P=16 D=128 + c128 decode B=2048 D=512 fp32 + "
            "c128 prefill 64 req (prefix U[0,16384], extend U[1,8192]) D=512 fp32 + long-context prefill "
            "8x131072 D=512 bf16 (Student-t scores) + pooled one-shot 65536 pools P=16 D=128 bf16")

# DRAM traffic (read + write bytes) per launch of the dominant kernel from one
# ncu capture of a 131,072-token case, scaled by tokens to the 8 x 131,072-token
# launch; `src` is a hash of the kernel's source files at capture time: any
# later change to them turns the figure into null.
NCU_TRAFFIC = {
    "c128_online_prefill_bf16": {"bytes_per_launch": 2173.3e6, "files": ["prefill_tma.cu", "ckv_tma.cuh", "ckv_fp8.cuh",
                                                                         "ckv_device.cuh"],
                                 "src": "d0f27c2178d63d8f"},
}


# ------------------------------------------------------------------ helpers
def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _src_hash(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "compressed_kv_attention_gated_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, device_index=0):
        self.samples, self.reasons, self.ok = [], 0, False
        self.max_mhz = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device_index)
            uuid = str(getattr(props, "uuid", ""))
            if uuid:
                u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                rc = self.nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h))
            else:
                rc = 1
            if rc != 0:
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if rc != 0:
                return
            m = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        get_reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if get_reasons(self.h, ctypes.byref(r)) == 0:
                self.reasons |= r.value & ~0x1
            time.sleep(0.002)

    def __enter__(self):
        self.stop = False
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self.stop = True
        if self.ok:
            self.t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        names = [n for b, n in self.REASONS.items() if self.reasons & b]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ------------------------------------------------------------ algorithmic bytes
def kpool_decode_bytes(pd):
    """(bytes, real tokens, closing pools) of one pooled decode/verify call."""
    pos = pd["positions"].cpu().numpy()
    ts = pd["tail_slot_mapping"].cpu().numpy()
    sm = pd["slot_mapping"].cpu().numpy()
    P, D = pd["P"], pd["D"]
    real = int((pos >= 0).sum())
    stash = int(((pos >= 0) & (ts >= 0)).sum())
    closes = int(((sm >= 0) & (pos >= 0) & (pos % P == P - 1)).sum())
    b = real * 2 * D * 2 + pos.size * 12 + stash * 2 * D * 2 + closes * ((P - 1) * 2 * D * 2 + D + 4) + P * D * 4
    return b, real, closes


def c128_decode_bytes(cd):
    """(bytes, closing requests) of one online c128 decode call."""
    D = cd["D"]
    es = cd["input"].element_size()
    p = (cd["seq_lens"].cpu().numpy().astype(np.int64) - 1) % 128
    b = cd["B"] * (2 * D * es + 8) + int((p != 0).sum()) * 3 * D * 4 + int((p != 127).sum()) * 3 * D * 4 + \
        int((p == 127).sum()) * D * 4 + 128 * D * 4
    return b, int((p == 127).sum())


# ------------------------------------------------------------ the workload
class Step:
    """Device-resident inputs of one step plus the five C-ABI calls."""

    def __init__(self, device, seed=0, scale=1):
        import compressed_kv_attention_gated_gb300 as ck
        from compressed_kv_attention_gated_gb300 import synth

        self.ck = ck
        self.dev = device
        self.err = torch.zeros((1,), dtype=torch.int32, device=device)
        # 1. pooled decode/verify
        self.pd = synth.pooled_decode(device, seed=seed)
        # 2. c128 decode
        self.cd = synth.c128_decode(device, seed=seed + 1)
        # 3. c128 prefill, fp32
        self.cp = synth.c128_prefill(device, seed=seed + 2)
        # 4 + 5. long context, bf16 c128 + pooled one-shot
        self.lc = synth.long_context(device, seed=seed + 3, T=131072 // scale)
        self.plans = {}
        for k, d in (("cp", self.cp), ("lc", self.lc)):
            cpl, wpl, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
            self.plans[k] = (cpl[:max(nc, 1)].to(device), nc, wpl[:max(nw, 1)].to(device), nw, cpl, wpl)
        self.names = ["kpool_decode_update", "c128_online_decode", "c128_online_prefill_f32",
                      "c128_online_prefill_bf16", "kpool_compress"]
        self._accounting()

    # -- calls -------------------------------------------------------------
    nvtx = False  # --nvtx: an NVTX range named after the C entry point around each call
    round_scale = True  # FP8 scale of the pooled decode call: power of two, or linear when False

    def call(self, i, pdl=False):
        """Call i of the step; with pdl every launch is a programmatic dependent
        launch on its predecessor (each kernel still waits for it on the device
        before touching memory, but its launch overlaps the predecessor's tail)."""
        if self.nvtx:
            torch.cuda.nvtx.range_push(self.names[i])
            try:
                return self._call(i, pdl)
            finally:
                torch.cuda.nvtx.range_pop()
        return self._call(i, pdl)

    def _call(self, i, pdl):
        ck, pd, cd, cp, lc = self.ck, self.pd, self.cd, self.cp, self.lc
        if i == 0:
            ck.ckv_kpool_decode_update(pd["kv_cache"], pd["ring"], pd["tail_slot_mapping"], pd["slot_mapping"],
                                       pd["positions"], pd["key"], pd["score"], pd["ape"],
                                       round_scale=self.round_scale, use_pdl=pdl, err_word=self.err)
        elif i == 1:
            ck.ckv_c128_online_decode(cd["state"], cd["input"], cd["out"], cd["ape"], cd["indices"], cd["seq_lens"],
                                      use_pdl=pdl, err_word=self.err)
        elif i == 2:
            c, nc, w, nw = self.plans["cp"][:4]
            ck.ckv_c128_online_prefill(cp["state"], cp["input"], cp["out"], cp["ape"], cp["indices"], c, nc, w, nw,
                                       use_pdl=pdl, err_word=self.err)
        elif i == 3:
            c, nc, w, nw = self.plans["lc"][:4]
            ck.ckv_c128_online_prefill(lc["state"], lc["input"], lc["out"], lc["ape"], lc["indices"], c, nc, w, nw,
                                       use_pdl=pdl, err_word=self.err)
        elif i == 4:
            ck.ckv_kpool_compress(lc["slot_k"], lc["slot_score"], lc["ape_pool"], kv_cache=lc["kv_cache"],
                                  loc=lc["loc"], round_scale=True, use_pdl=pdl, err_word=self.err)

    def launches(self):
        n = 0
        n += 1  # kpool decode
        n += 1  # c128 decode
        for k in ("cp", "lc"):
            _, nc, _, nw = self.plans[k][:4]
            n += (nc > 0) + (nw > 0)
        n += 1  # kpool compress
        return n

    # -- algorithmic bytes and tokens per call ------------------------------
    def _accounting(self):
        pd, cd = self.pd, self.cd
        b0, real, closes = kpool_decode_bytes(pd)
        b1, n_out = c128_decode_bytes(cd)

        def prefill_bytes(d, key):
            cpl, wpl = self.plans[key][4], self.plans[key][5]
            nc, nw = self.plans[key][1], self.plans[key][3]
            D_ = d["D"]
            es = d["input"].element_size()
            b = d["num_tokens"] * 2 * D_ * es + 128 * D_ * 4
            for rows, n, is_w in ((cpl, nc, False), (wpl, nw, True)):
                if n == 0:
                    continue
                r = rows[:n].view(torch.int32).view(-1, 4).numpy().astype(np.int64)
                mid = ((r[:, 2] % 128) + 1 - r[:, 3]) != 0
                b += n * 16 + int(mid.sum()) * (3 * D_ * 4 + 4)
                b += n * (3 * D_ * 4 + 4) if is_w else n * D_ * 4
            return b

        b2 = prefill_bytes(self.cp, "cp")
        b3 = prefill_bytes(self.lc, "lc")
        lc = self.lc
        b4 = lc["n_pools"] * (2 * lc["P"] * lc["Dp"] * 2 + 8 + lc["Dp"] + 4) + lc["P"] * lc["Dp"] * 4
        self.bytes = [b0, b1, b2, b3, b4]
        self.tokens = [real, cd["B"], self.cp["num_tokens"], lc["num_tokens"], lc["n_pools"] * lc["P"]]
        self.rows = [closes, n_out, self.plans["cp"][1], self.plans["lc"][1], lc["n_pools"]]
        self.units = {
            "kpool_decode_update": "per real token 512 B key+score read + 512 B ring stash + 12 B indices; per "
                                   "closing pool 15x512 B ring read + 132 B cache row; + ape 8 KB",
            "c128_online_decode": "per request 4096 B input + 8 B indices + 6144 B state read (chunk pos != 0) + "
                                  "6144 B state write (pos != 127) or 2048 B output (pos == 127); + ape 256 KB",
            "c128_online_prefill_f32": "per token 4096 B (kv|score fp32); per compress row 2048 B; per write entry "
                                       "6148 B; per mid-chunk segment 6148 B state read; 16 B per plan; + ape 256 KB",
            "c128_online_prefill_bf16": "per token 2048 B (kv|score bf16); per compress row 2048 B; 16 B per plan; "
                                        "+ ape 256 KB",
            "kpool_compress": "per pool 8192 B key+score read + 8 B loc + 132 B cache row; + ape 8 KB",
        }


# ------------------------------------------------------------ e2e (host I/O)
class HostIO:
    """Pinned host copies of every per-step input, and gathers of the results."""

    def __init__(self, step: Step):
        self.s = step
        dev = step.dev
        self.pairs = []  # (pinned host tensor, device tensor)
        self.groups = [[] for _ in range(5)]  # the pairs each call reads, in call order

        def add(call, t):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            self.pairs.append((h, t))
            self.groups[call].append((h, t))

        pd, cd, cp, lc = step.pd, step.cd, step.cp, step.lc
        for k in ("key", "score", "tail_slot_mapping", "slot_mapping", "positions"):
            add(0, pd[k])
        for k in ("input", "indices", "seq_lens"):
            add(1, cd[k])
        for k in ("input", "indices"):
            add(2, cp[k])
        add(3, lc["input"])
        for k in ("slot_k", "slot_score", "loc"):
            add(4, lc[k])
        # host planner output goes straight into pinned buffers
        self.plan_host = {}
        for key, d in (("cp", cp), ("lc", lc)):
            T = d["num_tokens"]
            self.plan_host[key] = (torch.empty((T, 16), dtype=torch.uint8, pin_memory=True),
                                   torch.empty((T, 16), dtype=torch.uint8, pin_memory=True))
        self.h2d_bytes = sum(h.numel() * h.element_size() for h, _ in self.pairs)
        # results to read back: closing decode rows, compressed prefill rows, written cache rows
        sm = pd["slot_mapping"].cpu().numpy().reshape(-1)
        pos = pd["positions"].cpu().numpy().reshape(-1)
        P, D, ps = pd["P"], pd["D"], pd["page_size"]
        locs = sm[(sm >= 0) & (pos >= 0) & (pos % P == P - 1)]
        idx = []
        for l in locs:
            page, tok = divmod(int(l), ps)
            base = page * ps * (D + 4)
            idx.extend(range(base + tok * D, base + tok * D + D))
            idx.extend(range(base + ps * D + 4 * tok, base + ps * D + 4 * tok + 4))
        self.g_pd = torch.tensor(idx, dtype=torch.int64, device=dev)
        p = (cd["seq_lens"].cpu().numpy().astype(np.int64) - 1) % 128
        self.g_cd = torch.tensor(np.nonzero(p == 127)[0], dtype=torch.int64, device=dev)
        self.g_cp = self._rows(step.plans["cp"])
        self.g_lc = self._rows(step.plans["lc"])
        self.outs = []
        for n in (self.g_pd.numel(), (self.g_cd.numel(), cd["D"]), (self.g_cp.numel(), cp["D"]),
                  (self.g_lc.numel(), lc["D"])):
            shape = (n,) if isinstance(n, int) else n
            dt = torch.uint8 if isinstance(n, int) else torch.float32
            self.outs.append(torch.empty(shape, dtype=dt, pin_memory=True))
        self.outs.append(torch.empty(lc["kv_cache"].shape, dtype=torch.uint8, pin_memory=True))
        self.d2h_bytes = sum(o.numel() * o.element_size() for o in self.outs)

    def _rows(self, plan):
        cpl, nc = plan[4], plan[1]
        r = cpl[:nc].view(torch.int32).view(-1, 4)[:, 0].to(torch.int64)
        return r.to(self.s.dev)

    def h2d(self, stream, copy_streams):
        """Host-to-device copies of the step's inputs.  Tensors above 64 MB are
        split in equal byte ranges over the copy streams (one DMA stream alone
        does not fill the host link); the compute stream then waits for them."""
        big = 64 << 20
        k = 0
        for h, dv in self.pairs:
            nb = h.numel() * h.element_size()
            if nb <= big or len(copy_streams) < 2:
                dv.copy_(h, non_blocking=True)
                continue
            hb = h.view(-1).view(torch.uint8)
            db = dv.view(-1).view(torch.uint8)
            n = len(copy_streams)
            step_b = (nb + n - 1) // n
            for i, cs in enumerate(copy_streams):
                lo, hi = i * step_b, min(nb, (i + 1) * step_b)
                if lo >= hi:
                    continue
                cs.wait_stream(stream)
                with torch.cuda.stream(cs):
                    db[lo:hi].copy_(hb[lo:hi], non_blocking=True)
                k += 1
        for cs in copy_streams:
            stream.wait_stream(cs)

    def _issue(self, pairs, copy_streams, rr):
        """Enqueue the copies of one call's inputs on the copy streams (small
        tensors round-robin, tensors above 64 MB split in equal byte ranges over
        all of them); returns the streams used."""
        big = 64 << 20
        n = len(copy_streams)
        used = []
        for h, dv in pairs:
            nb = h.numel() * h.element_size()
            if nb <= big:
                cs = copy_streams[rr[0] % n]
                rr[0] += 1
                with torch.cuda.stream(cs):
                    dv.copy_(h, non_blocking=True)
                used.append(cs)
                continue
            hb = h.view(-1).view(torch.uint8)
            db = dv.view(-1).view(torch.uint8)
            step_b = (nb + n - 1) // n
            for i, cs in enumerate(copy_streams):
                lo, hi = i * step_b, min(nb, (i + 1) * step_b)
                if lo < hi:
                    with torch.cuda.stream(cs):
                        db[lo:hi].copy_(hb[lo:hi], non_blocking=True)
                    used.append(cs)
        return list({id(c): c for c in used}.values())

    def run_step(self, stream=None, copy_streams=()):
        """One step from host memory: the host planner writes the plans into
        pinned buffers, every call's inputs are copied in call order on the copy
        streams, and each call starts as soon as its own inputs have arrived (so
        it runs under the copies of the calls after it); its results are
        gathered and read back right after it."""
        s = self.s
        ck = s.ck
        stream = stream or torch.cuda.current_stream()
        groups = [list(g) for g in self.groups]
        for call, key, d in ((2, "cp", s.cp), (3, "lc", s.lc)):
            hc, hw = self.plan_host[key]
            _, _, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"], compress_plan=hc, write_plan=hw)
            dc, _, dw, _ = s.plans[key][:4]
            if nc:
                groups[call].append((hc[:nc], dc[:nc]))
            if nw:
                groups[call].append((hw[:nw], dw[:nw]))
        cstreams = list(copy_streams) or [stream]
        for cs in cstreams:
            cs.wait_stream(stream)  # the previous step's kernels are done with the input buffers
        ready = []
        rr = [0]
        for g in groups:
            evs = []
            for cs in self._issue(g, cstreams, rr):
                ev = torch.cuda.Event()
                ev.record(cs)
                evs.append(ev)
            ready.append(evs)
        gathers = [lambda: self.outs[0].copy_(s.pd["kv_cache"].view(-1).index_select(0, self.g_pd), non_blocking=True),
                   lambda: self.outs[1].copy_(s.cd["out"].index_select(0, self.g_cd), non_blocking=True),
                   lambda: self.outs[2].copy_(s.cp["out"].index_select(0, self.g_cp), non_blocking=True),
                   lambda: self.outs[3].copy_(s.lc["out"].index_select(0, self.g_lc), non_blocking=True),
                   lambda: self.outs[4].copy_(s.lc["kv_cache"], non_blocking=True)]
        for i in range(5):
            for ev in ready[i]:
                stream.wait_event(ev)
            s.call(i)
            gathers[i]()


# --------------------------------------------------------- CPU oracle sample
def oracle_sample(budget_s=15.0, threads=None):
    """Time the CPU oracle on a bounded sample of each of the five calls (the
    sample grows with budget_s), on `threads` host threads (default: every
    core).  Returns (per-call (seconds, tokens), threads, sample description)."""
    import oracle
    from compressed_kv_attention_gated_gb300 import synth

    threads = threads or os.cpu_count() or 1

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    res = {}
    # 1. pooled decode (full size)
    d = synth.pooled_decode("cpu", seed=0)
    real = int((d["positions"] >= 0).sum())
    cache = d["kv_cache"].numpy().copy()
    ring = bits(d["ring"]).copy()
    t0 = time.perf_counter()
    oracle.kpool_decode_update(cache, d["page_size"], ring, d["tail_slot_mapping"].numpy(), d["slot_mapping"].numpy(),
                               d["positions"].numpy(), bits(d["key"]), bits(d["score"]), d["ape"].numpy(),
                               threads=threads)
    res["kpool_decode_update"] = (time.perf_counter() - t0, real)
    # 2. c128 decode (full size)
    d = synth.c128_decode("cpu", seed=1)
    t0 = time.perf_counter()
    oracle.c128_decode(d["state"].numpy(), d["input"].numpy(), d["ape"].numpy(), d["indices"].numpy(),
                       d["seq_lens"].numpy(), threads=threads)
    res["c128_online_decode"] = (time.perf_counter() - t0, 2048)
    # 3. c128 prefill fp32: a sample of requests with the same length distribution
    nreq = max(2, int(budget_s * 2))
    d = synth.c128_prefill("cpu", seed=2, B=min(64, nreq))
    t0 = time.perf_counter()
    oracle.c128_prefill(d["state"].numpy(), d["input"].numpy(), d["ape"].numpy(), d["indices"].numpy(),
                        d["seq_lens"].numpy(), d["extend_lens"].numpy(), threads=threads)
    res["c128_online_prefill_f32"] = (time.perf_counter() - t0, d["num_tokens"])
    # 4 + 5. long context: a sample of one request's tokens
    T = 2048 * max(1, int(budget_s / 5))  # tokens per request; 8 requests as in the workload
    d = synth.long_context("cpu", seed=3, B=8, T=T)
    T = 8 * T
    t0 = time.perf_counter()
    oracle.c128_prefill(d["state"].numpy(), bits(d["input"]), d["ape"].numpy(), d["indices"].numpy(),
                        d["seq_lens"].numpy(), d["extend_lens"].numpy(), threads=threads)
    res["c128_online_prefill_bf16"] = (time.perf_counter() - t0, T)
    cache = d["kv_cache"].numpy().copy()
    t0 = time.perf_counter()
    oracle.kpool_compress(cache, d["page_size"], bits(d["slot_k"]), bits(d["slot_score"]), d["ape_pool"].numpy(),
                          d["loc"].numpy(), threads=threads)
    res["kpool_compress"] = (time.perf_counter() - t0, T)
    sample = (f"oracle timed per call on: pooled decode 512x4 (full), c128 decode 2048 (full), c128 prefill "
              f"{min(64, nreq)} requests fp32 ({res['c128_online_prefill_f32'][1]} tokens), long-context 8 requests, "
              f"{T} tokens (bf16 c128 + pooled); per-token cost scaled to one full step")
    return res, threads, sample


def cpu_step_estimate(res, step_tokens):
    """Seconds the oracle would need for one full step, from per-token costs."""
    names = ["kpool_decode_update", "c128_online_decode", "c128_online_prefill_f32", "c128_online_prefill_bf16",
             "kpool_compress"]
    total = 0.0
    for n, tok in zip(names, step_tokens):
        t, s = res[n]
        total += t / s * tok
    return total


# ------------------------------------------------------------------- main
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seed(rank):
    """Seed of a rank's replica: ranks process independent requests."""
    return 1000 * rank


def whole_job_value(tokens_per_step, ws, steps, max_elapsed_ms):
    """Tokens all ranks processed divided by the slowest rank's time (tokens/s)."""
    return tokens_per_step * ws * steps / (max_elapsed_ms / 1e3)


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle itself, each step a bounded sample."""
    if rank != 0:
        return
    import oracle
    from compressed_kv_attention_gated_gb300 import synth

    oracle.build()
    threads = os.cpu_count() or 1

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    # one bounded sample of the step, in the step's token proportions (scaled down)
    pd = synth.pooled_decode("cpu", seed=0, B=64)
    cd = synth.c128_decode("cpu", seed=1, B=256)
    cp = synth.c128_prefill("cpu", seed=2, B=1, max_extend=2048)
    lc = synth.long_context("cpu", seed=3, B=1, T=8192)
    tokens = int((pd["positions"] >= 0).sum()) + 256 + cp["num_tokens"] + 2 * 8192

    def one():
        cache = pd["kv_cache"].numpy().copy()
        ring = bits(pd["ring"]).copy()
        oracle.kpool_decode_update(cache, pd["page_size"], ring, pd["tail_slot_mapping"].numpy(),
                                   pd["slot_mapping"].numpy(), pd["positions"].numpy(), bits(pd["key"]),
                                   bits(pd["score"]), pd["ape"].numpy(), threads=threads)
        oracle.c128_decode(cd["state"].numpy(), cd["input"].numpy(), cd["ape"].numpy(), cd["indices"].numpy(),
                           cd["seq_lens"].numpy(), threads=threads)
        oracle.c128_prefill(cp["state"].numpy(), cp["input"].numpy(), cp["ape"].numpy(), cp["indices"].numpy(),
                            cp["seq_lens"].numpy(), cp["extend_lens"].numpy(), threads=threads)
        oracle.c128_prefill(lc["state"].numpy(), bits(lc["input"]), lc["ape"].numpy(), lc["indices"].numpy(),
                            lc["seq_lens"].numpy(), lc["extend_lens"].numpy(), threads=threads)
        c2 = lc["kv_cache"].numpy().copy()
        oracle.kpool_compress(c2, lc["page_size"], bits(lc["slot_k"]), bits(lc["slot_score"]), lc["ape_pool"].numpy(),
                              lc["loc"].numpy(), threads=threads)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    v = tokens * args.steps / el
    sample = (f"per step: pooled decode 64 req x 4 tok, c128 decode 256 req, c128 prefill 1 req "
              f"({cp['num_tokens']} tok fp32), long-context 8192 tok bf16 c128 + 512 pools")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "reference": "CPU oracle (plain C++, double precision) on host cores",
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_case(args):
    """One kernel on its own input (profiling target).  Prints the per-call time:
    median over 5 replays of a CUDA graph of --steps calls, divided by --steps."""
    import compressed_kv_attention_gated_gb300 as ck
    from compressed_kv_attention_gated_gb300 import build as libbuild, synth

    libbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    n = args.case_tokens
    if args.case in ("prefill_f32", "prefill_bf16"):
        bf = args.case == "prefill_bf16"
        d = synth.c128_prefill(dev, seed=5, B=1, D=512, max_extend=n, zero_prefix=True, num_slots=1,
                               dtype=torch.bfloat16 if bf else torch.float32,
                               score_dist="student_t" if bf else "normal")
        cpl, wpl, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
        c, w = cpl[:max(nc, 1)].to(dev), wpl[:max(nw, 1)].to(dev)

        def call():
            ck.ckv_c128_online_prefill(d["state"], d["input"], d["out"], d["ape"], d["indices"], c, nc, w, nw,
                                       err_word=err)
        nbytes = n * 2 * 512 * d["input"].element_size() + nc * 2048
    elif args.case in ("prefill_bf16_fp8", "prefill_f32_fp8"):
        # the c128 prefill with the FP8 output stage only (no fp32 rows)
        bf = args.case == "prefill_bf16_fp8"
        d = synth.c128_prefill(dev, seed=5, B=1, D=512, max_extend=n, zero_prefix=True, num_slots=1,
                               dtype=torch.bfloat16 if bf else torch.float32,
                               score_dist="student_t" if bf else "normal")
        cpl, wpl, nc, nw = ck.ckv_plan_online_prefill(d["seq_lens"], d["extend_lens"])
        c, w = cpl[:max(nc, 1)].to(dev), wpl[:max(nw, 1)].to(dev)
        ps = 64
        cache = torch.zeros(((nc + ps - 1) // ps + 1, ps, 512 + 16), device=dev, dtype=torch.uint8)
        cache_loc = torch.full((n,), -1, device=dev, dtype=torch.int64)
        cache_loc[127::128] = torch.arange(nc, device=dev)

        def call():
            ck.ckv_c128_online_prefill_fp8(d["state"], d["input"], None, d["ape"], d["indices"], c, nc, w, nw, cache,
                                           cache_loc, err_word=err)
        nbytes = n * 2 * 512 * d["input"].element_size() + nc * (512 + 16 + 8 + 16)
    elif args.case == "c128_decode_fp8":
        d = synth.c128_decode(dev, seed=5)
        ps = 64
        cache = torch.zeros((2048 // ps + 1, ps, 512 + 16), device=dev, dtype=torch.uint8)
        cache_loc = torch.arange(2048, device=dev, dtype=torch.int64)

        def call():
            ck.ckv_c128_online_decode_fp8(d["state"], d["input"], None, d["ape"], d["indices"], d["seq_lens"], cache,
                                          cache_loc, err_word=err)
        nbytes = 2048 * (4096 + 2 * 6144)
    elif args.case == "kpool_compress":
        d = synth.long_context(dev, seed=5, B=1, T=n)

        def call():
            ck.ckv_kpool_compress(d["slot_k"], d["slot_score"], d["ape_pool"], kv_cache=d["kv_cache"], loc=d["loc"],
                                  err_word=err)
        nbytes = d["n_pools"] * (8192 + 140)
    elif args.case == "c128_decode":
        d = synth.c128_decode(dev, seed=5)

        def call():
            ck.ckv_c128_online_decode(d["state"], d["input"], d["out"], d["ape"], d["indices"], d["seq_lens"],
                                      err_word=err)
        nbytes = 2048 * (4096 + 2 * 6144)
    elif args.case == "kpool_decode":
        d = synth.pooled_decode(dev, seed=5)

        def call():
            ck.ckv_kpool_decode_update(d["kv_cache"], d["ring"], d["tail_slot_mapping"], d["slot_mapping"],
                                       d["positions"], d["key"], d["score"], d["ape"], err_word=err)
        nbytes = 2048 * 1024
    elif args.case == "seed_tail":
        # n prefill tokens over 64 requests, each request's last 16 tokens seeded
        B = 64
        per = n // B
        key = torch.randn((B * per, 128), device=dev).to(torch.bfloat16)
        score = torch.randn((B * per, 128), device=dev).to(torch.bfloat16)
        pos = torch.arange(per, device=dev, dtype=torch.int32)
        tslot = (torch.arange(B, device=dev, dtype=torch.int32)[:, None] * 16 + pos % 16).reshape(-1).contiguous()
        ring = torch.zeros((B, 2, 16, 128), device=dev, dtype=torch.bfloat16)

        def call():
            ck.ckv_kpool_seed_tail(ring, key, score, tslot, err_word=err)
        nbytes = B * 16 * 512 * 2 + tslot.numel() * 8
    elif args.case == "expand":
        # n rows of 128 selected pools (P = 16): a top-2048 token selection per row
        ids = torch.randint(-1, 4096, (n, 128), device=dev, dtype=torch.int32)
        seq = torch.randint(0, 65536, (n,), device=dev, dtype=torch.int64)
        out = torch.empty((n, 128 * 16 + 15), device=dev, dtype=torch.int32)

        def call():
            ck.ckv_expand_pools_and_append_tail(ids, seq, 16, out=out)
        nbytes = n * (128 * 4 + 8 + (128 * 16 + 15) * 4)
    elif args.case == "plan_device":
        # the 64-request prefill batch (prefix U[0,16384], extend U[1,8192]) planned on the device
        d = synth.c128_prefill("cpu", seed=2, B=64, D=128, max_extend=8192)
        T = d["num_tokens"]
        seq, ext = d["seq_lens"].to(dev), d["extend_lens"].to(dev)
        cp = torch.empty((T, 16), device=dev, dtype=torch.uint8)
        wp = torch.empty((T, 16), device=dev, dtype=torch.uint8)
        cnt = torch.zeros((2,), device=dev, dtype=torch.int32)

        def call():
            ck.ckv_plan_online_prefill_device(seq, ext, T, compress_plan=cp, write_plan=wp, counts=cnt, err_word=err)
        nbytes = 64 * 16 + (T // 128 + 128) * 16
    else:
        raise SystemExit(f"unknown case {args.case}")
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    # --steps calls captured in one CUDA graph, so that the host's per-call
    # launch cost (larger than these kernels) is not what gets timed
    stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(args.steps):
            call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        graph.replay()
        for _ in range(5):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) / args.steps * 1e3)
    us = float(np.median(times))
    print(json.dumps({"case": args.case, "tokens": n, "us_per_call": us, "approx_gbs": nbytes / us / 1e3,
                      "err": int(err.item())}))


def run_rotation(args):
    """--case c128_decode|kpool_decode|latency_floor0|1|2 --rotate: print
    rotation_timings() as one JSON line."""
    print(json.dumps(rotation_timings(args.case, args.steps, args.warmup, round_scale=not args.linear_scale,
                                      instances=args.instances)))


# Instances of a decode batch in one cold-timing graph, at least: the graph's
# own launch cost is spread over its calls, and with 17 calls (enough for 4 x
# L2 of the c128 decode) it still added a few percent to each.
kMinInstances = 64


def rotation_timings(case, replays=100, warmup=20, round_scale=True, instances=None):
    """Decode calls timed L2-cold and warm, each replayed from one CUDA graph.

    Cold: R independent instances of the batch (R x algorithmic bytes >= 4 x
    the L2 size, and R >= kMinInstances), one call on each, captured in order
    as one graph; every
    replay is bracketed by events and the median replay time / R is the time of
    one call that finds none of its data in L2.  Warm: a graph of one call on
    one instance (its data L2-resident after the first replay).  Both with and
    without programmatic dependent launch between the captured calls.

    c128 decode: before every replay (outside the events) each instance's
    state pool is restored from a pristine copy and a buffer of twice the L2
    size is written, so every timed call updates states it has never seen:
    its running max moves at the workload's own rate instead of never (a
    replay into states it already updated leaves every max unchanged).  The
    bytes it physically writes (the max-row sectors it leaves alone excluded)
    are reported beside the algorithmic bytes.  c128_decode_fp8: the same
    with the FP8 output stage instead of the fp32 rows, each instance writing
    its own cache rows.

    Pooled decode: the instances share one cache tensor, each writing its own
    rows (location r * B + b for request b of instance r); round_scale picks
    the power-of-two or the linear FP8 scale.

    latency_floor: the ckv_latency_probe kernels (0, 1 and 2 dependent global
    round trips per warp) in the pooled decode's launch shape, R instances of
    512 warps with an L2 flush before every replay: the floor under the pooled
    decode's cold time.  latency_floor<h>_r<rows> draws the second hop's rows
    from a buffer of <rows> x 256 B (default 512 rows); latency_floor3 is one
    round trip with the pooled decode's own first-hop loads (512 warps or more,
    9 rows or more); latency_floor4 the pooled decode's whole memory pattern
    without its arithmetic (64 rows or more; _r16384 gives the second hop a
    4 MB buffer like the ring).

    instances: a fixed instance count instead of the L2-sized one, with an L2
    flush before every replay (data cold, the instances' pages recently used)."""
    import math

    import compressed_kv_attention_gated_gb300 as ck
    from compressed_kv_attention_gated_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty((2 * l2,), dtype=torch.uint8, device=dev)
    restore = None
    extra = {}
    if case in ("c128_decode", "c128_decode_fp8"):
        first = synth.c128_decode(dev, seed=100)
        nbytes, closing = c128_decode_bytes(first)
        fp8 = case == "c128_decode_fp8"
        B, D = first["B"], first["D"]
        if fp8:
            # no fp32 output rows; per closing request its cache location and
            # FP8 row (D code bytes + one fp32 scale per 128 channels)
            nbytes += closing * (8 + D + 4 * (D // 128) - 4 * D)
        R = max(kMinInstances, math.ceil(4 * l2 / nbytes))
        if fp8:
            ps = 64
            cache = torch.zeros(((R * B + ps - 1) // ps, ps, D + 4 * (D // 128)), device=dev, dtype=torch.uint8)

        def make(r):
            d = first if r == 0 else synth.c128_decode(dev, seed=100 + r)
            d["state0"] = d["state"].clone()
            if fp8:
                d["cache_loc"] = torch.arange(r * B, (r + 1) * B, device=dev, dtype=torch.int64)
            return d

        def call(d, pdl):
            if fp8:
                ck.ckv_c128_online_decode_fp8(d["state"], d["input"], None, d["ape"], d["indices"], d["seq_lens"],
                                              cache, d["cache_loc"], round_scale=round_scale, use_pdl=pdl,
                                              err_word=err)
            else:
                ck.ckv_c128_online_decode(d["state"], d["input"], d["out"], d["ape"], d["indices"], d["seq_lens"],
                                          use_pdl=pdl, err_word=err)

        def restore(inst):
            for d in inst:
                d["state"].copy_(d["state0"])
    elif case == "kpool_decode":
        first = synth.pooled_decode(dev, seed=100)
        nbytes = kpool_decode_bytes(first)[0]
        B, ps = first["B"], first["page_size"]
        R = max(kMinInstances, math.ceil(4 * l2 / nbytes))
        cache = torch.zeros(((R * B + ps - 1) // ps, ps, first["D"] + 4), device=dev, dtype=torch.uint8)

        def make(r):
            d = first if r == 0 else synth.pooled_decode(dev, seed=100 + r)
            sm = d["slot_mapping"]
            req = torch.arange(B, device=dev, dtype=torch.int32)[:, None].expand_as(sm)
            d["slot_mapping"] = torch.where(sm >= 0, r * B + req, sm).contiguous()
            d["kv_cache"] = cache
            return d

        def call(d, pdl):
            ck.ckv_kpool_decode_update(d["kv_cache"], d["ring"], d["tail_slot_mapping"], d["slot_mapping"],
                                       d["positions"], d["key"], d["score"], d["ape"], round_scale=round_scale,
                                       use_pdl=pdl, err_word=err)
    elif case.startswith("latency_floor"):
        # same instance count as the pooled decode's cold timing; latency_floor<h>
        # or latency_floor<h>_w<warps>_c<warps per CTA> (default 512 warps, 4 per CTA)
        nbytes = kpool_decode_bytes(synth.pooled_decode("cpu", seed=100))[0]
        R = max(kMinInstances, math.ceil(4 * l2 / nbytes))
        parts = case[len("latency_floor"):].split("_")
        hops = int(parts[0])
        n = next((int(p[1:]) for p in parts[1:] if p.startswith("w")), 512)
        wpc = next((int(p[1:]) for p in parts[1:] if p.startswith("c")), 4)
        nrows = next((int(p[1:]) for p in parts[1:] if p.startswith("r")), n)
        g = torch.Generator(device=dev)
        g.manual_seed(7)

        def make(r):
            return {"idx": torch.randperm(nrows, generator=g, device=dev)[:n].to(torch.int32),
                    "rows": torch.randint(0, 255, (nrows, 256), generator=g, device=dev, dtype=torch.uint8),
                    "out": torch.zeros(((4 if hops == 4 else 1) * n, 256), device=dev, dtype=torch.uint8)}

        def call(d, pdl):
            ck.ckv_latency_probe(hops, n, d["idx"], d["rows"], d["out"], warps_per_cta=wpc, use_pdl=pdl)

        nbytes = {0: 0, 1: n * 8, 2: n * 516, 3: n * (48 + 1024 + 4),
                  4: n * (48 + 1024 + 1024 + 4) + (n // 4) * 3840}[hops]
    else:
        raise SystemExit("--rotate applies to --case c128_decode, c128_decode_fp8, kpool_decode or latency_floor<h>")
    if instances:
        R = int(instances)
    inst = [make(r) for r in range(R)]
    flush_each = restore is not None or case.startswith("latency_floor") or bool(instances)
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(dev)
    res = {"case": case, "mode": "rotate", "instances": R, "l2_bytes": l2, "bytes_per_call": nbytes,
           "replays": replays, "l2_flush_before_each_replay": flush_each}
    if case in ("kpool_decode", "c128_decode_fp8"):
        res["round_scale"] = bool(round_scale)

    def before(warm):
        # cold: every instance restored, then L2 flushed; warm: the one instance
        # restored (its state then sits in L2), nothing flushed
        if restore is not None:
            restore(inst[:1] if warm else inst)
        if flush_each and not warm:
            flush.zero_()

    def timed(graph, n_calls, warm=False):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t = []
        with torch.cuda.stream(stream):
            for _ in range(max(20, warmup)):
                before(warm)
                graph.replay()
            for _ in range(replays):
                before(warm)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                e1.synchronize()
                t.append(e0.elapsed_time(e1) * 1e3 / n_calls)
        return float(np.median(t))

    if case in ("c128_decode", "c128_decode_fp8"):
        # bytes the call physically writes: the max-row sectors (8 channels, 32
        # bytes) of open requests whose new maxima equal the stored ones are left
        # alone by the kernel
        with torch.cuda.stream(stream):
            restore(inst)
            d = inst[0]
            before_max = d["state"][:, 0].clone()
            call(d, False)
        stream.synchronize()
        p = (d["seq_lens"].to(torch.int64) - 1) % 128
        open_ = (p != 0) & (p != 127)
        rows = d["indices"].to(torch.int64)[open_]
        same = (d["state"][rows, 0].view(torch.int32) == before_max[rows].view(torch.int32))
        kept = int(same.view(same.shape[0], -1, 8).all(dim=2).sum())
        extra = {"max_sectors_left_alone": kept, "physical_bytes_per_call": nbytes - 32 * kept,
                 "max_moved_fraction": round(1.0 - float(same.float().mean()), 4) if rows.numel() else 0.0}
        res.update(extra)
    for pdl in (True, False):
        with torch.cuda.stream(stream):
            for d in inst:
                call(d, pdl)  # one-time set-up outside the capture
        stream.synchronize()
        cold = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cold, stream=stream):
            for d in inst:
                call(d, pdl)
        warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(warm, stream=stream):
            call(inst[0], pdl)
        tag = "pdl" if pdl else "no_pdl"
        us_cold = timed(cold, R)
        us_warm = timed(warm, 1, warm=True)
        res[tag] = {"us_per_call_cold": round(us_cold, 3), "gbs_cold": round(nbytes / us_cold / 1e3, 1),
                    f"frac_of_{peak_kind}_hbm": round(nbytes / us_cold / 1e3 / peak, 4),
                    "us_single_call_warm": round(us_warm, 3)}
        if "physical_bytes_per_call" in extra:
            res[tag]["gbs_cold_physical"] = round(extra["physical_bytes_per_call"] / us_cold / 1e3, 1)
            res[tag][f"frac_of_{peak_kind}_hbm_physical"] = round(
                extra["physical_bytes_per_call"] / us_cold / 1e3 / peak, 4)
        del cold, warm
    torch.cuda.synchronize()
    res["err"] = int(err.item())
    res["peak_gbs"] = peak
    del inst
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None,
                    help="profile one kernel alone: prefill_f32|prefill_bf16|prefill_f32_fp8|prefill_bf16_fp8|"
                         "kpool_compress|c128_decode|c128_decode_fp8|kpool_decode|seed_tail|expand|plan_device")
    ap.add_argument("--case-tokens", type=int, default=131072)
    ap.add_argument("--rotate", action="store_true",
                    help="with --case c128_decode|kpool_decode: L2-cold and warm per-call time from CUDA graph "
                         "replays over rotating instances (--steps replays, median)")
    ap.add_argument("--linear-scale", action="store_true",
                    help="with --case kpool_decode --rotate: the linear FP8 scale instead of the power-of-two one")
    ap.add_argument("--instances", type=int, default=None,
                    help="with --rotate: this many instances, L2 flushed before every replay")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nvtx", action="store_true",
                    help="NVTX range around each call (e.g. ncu --nvtx --nvtx-include 'c128_online_decode/')")
    ap.add_argument("--no-decode-cold", action="store_true",
                    help="skip the L2-cold CUDA-graph timing of the two decode calls")
    ap.add_argument("--no-pdl", action="store_true", help="plain stream order between the five calls")
    ap.add_argument("--no-overlap", action="store_true", help="run the decode calls on the prefill stream")
    ap.add_argument("--copy-streams", type=int, default=4, help="streams sharing the large H2D copies (e2e)")
    ap.add_argument("--prefill-variant", type=int, default=0,
                    help="compress-pass kernel: 0 auto, 1 one CTA per segment, 2 TMA pipeline")
    ap.add_argument("--kpool-variant", type=int, default=0,
                    help="pooled one-shot kernel: 0 auto, 1 one warp per pool, 2 bulk-copy pipeline")
    args = ap.parse_args()
    if args.impl == "ours":
        import compressed_kv_attention_gated_gb300 as ck
        from compressed_kv_attention_gated_gb300 import build as libbuild

        libbuild.build()
        ck.ckv_c128_prefill_set_variant(args.prefill_variant)
        ck.ckv_kpool_compress_set_variant(args.kpool_variant)
    if args.case:
        run_rotation(args) if args.rotate else run_case(args)
        return
    ws, rank, local = _dist()
    if ws > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, ws, rank)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    warmup = max(3, args.warmup)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from compressed_kv_attention_gated_gb300 import build as libbuild

    libbuild.build()
    step = Step(dev, seed=replica_seed(rank))
    step.nvtx = args.nvtx
    nk = len(step.names)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    pdl = not args.no_pdl
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for i in range(nk):
                step.call(i, pdl)
        stream.synchronize()
        assert int(step.err.item()) == 0, f"kernel error word {int(step.err.item()):#x}"
        K = args.steps
        # timed region: K whole steps.  The two decode calls (latency bound, their own
        # buffers) run on a second stream, overlapping the bandwidth-bound prefill
        # calls of the same step; launches on each stream are chained by
        # programmatic dependent launch.
        overlap = not args.no_overlap
        dstream = torch.cuda.Stream(dev) if overlap else stream
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_dec = torch.cuda.Event()
        _barrier(ws)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            e_start.record(stream)
            dstream.wait_event(e_start)
            for k in range(K):
                with torch.cuda.stream(dstream):
                    step.call(0, pdl)
                    step.call(1, pdl)
                for i in range(2, nk):
                    step.call(i, pdl)
            e_dec.record(dstream)
            stream.wait_event(e_dec)
            e_end.record(stream)
            stream.synchronize()
        _barrier(ws)
        elapsed_ms = e_start.elapsed_time(e_end)

        def run_steps(skip):
            """K steps launched exactly like the timed region, without call `skip`."""
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e_d = torch.cuda.Event()
            torch.cuda.synchronize()
            e0.record(stream)
            dstream.wait_event(e0)
            for _ in range(K):
                with torch.cuda.stream(dstream):
                    for i in (0, 1):
                        if i != skip:
                            step.call(i, pdl)
                for i in range(2, nk):
                    if i != skip:
                        step.call(i, pdl)
            e_d.record(dstream)
            stream.wait_event(e_d)
            e1.record(stream)
            stream.synchronize()
            return e0.elapsed_time(e1)

        # what each call adds to the launched step: the step's time minus the time
        # of the same step without that call (overlap and launch chaining included)
        full_again_ms = run_steps(None)
        marginal_ms = [(full_again_ms - run_steps(i)) / K for i in range(nk)]
        # breakdown: the same steps with an event between consecutive calls (an event
        # between two launches removes the programmatic overlap, so this loop is
        # timed on its own and used only to attribute time to the five calls).
        # Every other step of this loop runs the pooled decode with the linear FP8
        # scale instead of the power-of-two one, in the same place of the step.
        Kb = 2 * K
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(Kb)]
        torch.cuda.synchronize()
        for k in range(Kb):
            evs[k][0].record(stream)
            for i in range(nk):
                step.round_scale = (k % 2 == 0) or i != 0
                step.call(i, False)
                evs[k][i + 1].record(stream)
        step.round_scale = True
        stream.synchronize()
        breakdown_ms = statistics.mean(evs[k][0].elapsed_time(evs[k][nk]) for k in range(0, Kb, 2))
    per_kernel_ms = [statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(0, Kb, 2))
                     for i in range(nk)]
    linear_ms = statistics.mean(evs[k][0].elapsed_time(evs[k][1]) for k in range(1, Kb, 2))
    elapsed_ms = _max_over_ranks(elapsed_ms, ws, dev)
    ms_per_step = elapsed_ms / K
    tokens_step = sum(step.tokens)
    value = whole_job_value(tokens_step, ws, K, elapsed_ms)
    peak, peak_kind = _peaks()
    kernels = {}
    for i, n in enumerate(step.names):
        gbs = step.bytes[i] / (per_kernel_ms[i] / 1e3) / 1e9
        kernels[n] = {"us": round(per_kernel_ms[i] * 1e3, 2), "bytes": int(step.bytes[i]), "gbs": round(gbs, 1),
                      "frac_of_" + peak_kind + "_peak": round(gbs / peak, 4),
                      "us_in_step_marginal": round(marginal_ms[i] * 1e3, 2),
                      "frac_in_step_marginal": (round(step.bytes[i] / (marginal_ms[i] / 1e3) / 1e9 / peak, 4)
                                                if marginal_ms[i] > 0 else None),
                      "tokens": int(step.tokens[i]),
                      "compressed_rows": int(step.rows[i]),
                      "tokens_per_s": round(step.tokens[i] / (per_kernel_ms[i] / 1e3), 1)}
    kernels["kpool_decode_update_linear_scale"] = {
        "us": round(linear_ms * 1e3, 2), "bytes": int(step.bytes[0]),
        "frac_of_" + peak_kind + "_peak": round(step.bytes[0] / (linear_ms / 1e3) / 1e9 / peak, 4),
        "note": "the pooled decode call with the linear FP8 scale, timed in the same place of the step (not part "
                "of the step's tokens)"}
    kernels["c128_online_decode"]["note"] = (
        "every step replays the same tokens into the same slots, so after the first step no running max moves; "
        "decode_l2_cold times it on restored states")
    dom = max(range(nk), key=lambda i: per_kernel_ms[i])
    dom_gbs = step.bytes[dom] / (per_kernel_ms[dom] / 1e3) / 1e9
    tr = NCU_TRAFFIC.get(step.names[dom])
    traffic = tr["bytes_per_launch"] if tr and tr.get("src") == _src_hash(tr["files"]) else None
    roofline = {"bound": "hbm", "kernel": step.names[dom], "achieved": round(dom_gbs, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dom_gbs / peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": int(step.bytes[dom]), "unit_bytes": step.units[step.names[dom]]}
    step_gbs = sum(step.bytes) / (ms_per_step / 1e3) / 1e9

    # end to end through the same C-ABI calls, host-resident inputs
    e2e = None
    io = HostIO(step)
    Ke = args.e2e_steps or max(3, min(K, 20))
    copy_streams = [torch.cuda.Stream(dev) for _ in range(args.copy_streams)] if args.copy_streams > 1 else []
    with torch.cuda.stream(stream):
        io.run_step(stream, copy_streams)
        stream.synchronize()
        # the host link alone: the same H2D bytes, nothing else (best of 3)
        h2d_gbs = 0.0
        for _ in range(3):
            h0 = torch.cuda.Event(enable_timing=True)
            h1 = torch.cuda.Event(enable_timing=True)
            h0.record(stream)
            io.h2d(stream, copy_streams)
            h1.record(stream)
            h1.synchronize()
            h2d_gbs = max(h2d_gbs, io.h2d_bytes / (h0.elapsed_time(h1) / 1e3) / 1e9)
        _barrier(ws)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            io.run_step(stream, copy_streams)
            stream.synchronize()  # the host consumes the compressed rows every step
        e1.record(stream)
        e1.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), ws, dev)
    e2e = {"value": whole_job_value(tokens_step, ws, Ke, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(io.h2d_bytes),
           "d2h_bytes_per_step": int(io.d2h_bytes), "ms_per_step": e2e_ms / Ke, "steps": Ke,
           "h2d_only_gbs": round(h2d_gbs, 1), "copy_streams": max(1, len(copy_streams))}
    assert int(step.err.item()) == 0

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:  # the host baseline is an N = 1 figure
        res, threads, sample = oracle_sample(args.cpu_budget)
        est = cpu_step_estimate(res, step.tokens)
        cpu = {"value": tokens_step / est, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": sample,
               "per_call_s": {k: round(v[0], 4) for k, v in res.items()},
               "per_call_tokens": {k: int(v[1]) for k, v in res.items()}}
        # the same oracle on one thread, on a smaller sample
        res1, _, sample1 = oracle_sample(max(1.0, args.cpu_budget / 8), threads=1)
        cpu["single_thread"] = {"value": tokens_step / cpu_step_estimate(res1, step.tokens), "cores": 1,
                                "sample": sample1}

    decode_cold = None
    if rank == 0 and ws == 1 and not args.no_decode_cold:  # rotating instances on the one GPU
        decode_cold = {}
        for name, case, rs in (("kpool_decode_update", "kpool_decode", True),
                               ("kpool_decode_update_linear_scale", "kpool_decode", False),
                               ("c128_online_decode", "c128_decode", True),
                               ("c128_online_decode_fp8", "c128_decode_fp8", True),
                               ("latency_floor_2hops", "latency_floor2", True),
                               ("latency_floor_0hops", "latency_floor0", True),
                               ("latency_floor_decode_pattern", "latency_floor4_w1024_c2_r16384", True)):
            r = rotation_timings(case, round_scale=rs)
            e = {"instances": r["instances"], "bytes_per_call": r["bytes_per_call"],
                 "us_per_call_cold": r["pdl"]["us_per_call_cold"], "gbs_cold": r["pdl"]["gbs_cold"],
                 "frac": r["pdl"][f"frac_of_{peak_kind}_hbm"],
                 "us_single_call_warm": r["pdl"]["us_single_call_warm"], "err": r["err"]}
            for k in ("physical_bytes_per_call", "max_moved_fraction"):
                if k in r:
                    e[k] = r[k]
            if "gbs_cold_physical" in r["pdl"]:
                e["frac_physical"] = r["pdl"][f"frac_of_{peak_kind}_hbm_physical"]
            decode_cold[name] = e
        decode_cold["method"] = ("R instances (R x bytes per call >= 4 x L2, R >= 64), one call on each, captured in order "
                                 "in one CUDA graph with programmatic dependent launch; median of 100 replays / R. "
                                 "c128 decode: every state pool restored from a pristine copy and a 2 x L2 buffer "
                                 "written before each replay (outside the events); the fp8 entry stores FP8 rows "
                                 "instead of fp32 rows. latency_floor: the probe "
                                 "kernels (512 warps, 4 per CTA; the decode pattern: 1024 warps, 2 per CTA, the "
                                 "pooled decode's own launch shape, over a 4 MB row buffer), L2 flushed before each "
                                 "replay")

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded; shapes and distributions of the five workloads)",
            "config": {"workload": WORKLOAD, "tokens_per_step": int(tokens_step), "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (step working set ~3.7 GB >> 126 MB L2)"},
            "step_hbm_gbs": round(step_gbs, 1), "step_frac_of_peak": round(step_gbs / peak, 4),
            "launch_chaining": ("programmatic dependent launch" if pdl else "stream order") +
                               ("; decode calls on a second stream, concurrent with the prefill calls"
                                if overlap else "; one stream"),
            "breakdown_ms_per_step": round(breakdown_ms, 4),
            "per_call_timing": ("us / frac_of_*_peak: an event pair around each call in stream order (each event "
                                "breaks the launch chaining, so every call also pays a launch gap); "
                                "us_in_step_marginal: the chained step's time minus the same step's time without "
                                "that call (calls on the decode stream overlap the prefill stream, so theirs is "
                                "near zero)"),
            "kernels": kernels, "roofline": roofline, "clocks": clk.summary(),
            "gpu_launches": step.launches() * K, "e2e": e2e, "cpu_baseline": cpu, "decode_l2_cold": decode_cold,
        }), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
