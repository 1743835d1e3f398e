"""Benchmark: GEMM TFLOP/s of the tcgen05 swizzled GEMM on one GB300.

One step = one full GEMM of the workload (all hot-path stages: scale
rearrangement for block-scaled inputs, TMA ring, descriptor walk, tcgen05.mma,
tcgen05.ld epilogue), inputs already resident in HBM.  Default workload: bf16
M=N=K=8192 with CTA pairs (cta_group::2, 256x256 pair tiles), fp32
accumulation, bf16 output.  The other workloads -- block-scaled MXFP8
8192^3, bf16 4096^3 (A K-major, B MN-major, single CTAs), tf32 2048 x 2048 x
8192, f16-in / f16-accumulate 8192^3, block-scaled FP6 / MXFP4 / NVFP4 8192^3
and the HBM-bound 16 x 8192 x 8192 --
are measured the same way and reported under "secondary", and a ~1.5 s
back-to-back pass of the headline ("sustained") is compared with the
sustained cuBLAS figure, with the SM clock seen in that window.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Timing: CUDA events on the stream the kernels are launched on, W untimed
warm-up steps, then exactly K timed steps between a barrier +
synchronize on both sides; max over ranks.  A and B together exceed the
129 MB L2, so no flush is needed between steps.  Multi-GPU runs are
independent replicas (the GEMM needs no exchange): value = all ranks' FLOPs /
max time.  The reference arm times the float64 CPU oracle on a bounded row
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "GEMM TFLOP/s at 1 GB300 and % of dtype dense tensor peak (bf16/mxf8 8192^3)"
UNIT = "TFLOP/s"
IN_TYPE = {"f16": 0, "bf16": 1, "tf32": 2, "e4m3": 3, "e5m2": 4, "e3m2": 5, "e2m3": 6, "e2m1": 7, "nvf4": 8}
OUT = {"f32": 0, "f16": 1, "bf16": 2}
ACC = {"f32": 0, "f16": 1}
ESIZE = {"f16": 2, "bf16": 2, "tf32": 4, "e4m3": 1, "e5m2": 1, "e3m2": 0.75, "e2m3": 0.75, "e2m1": 0.5, "nvf4": 0.5}
# nominal dense tensor rate relative to bf16 (NVIDIA GB300 figures: tf32 1.1,
# bf16/fp16 2.25, fp8 4.5, fp4 13.5 PFLOP/s).  FP6 elements run on the FP8
# kind (kind::mxf8f6f4, one byte of shared memory per element) at the FP8
# rate; FP4 (MXFP4, NVFP4) on the packed FP4 kinds at the FP4 rate.
NOMINAL_RATIO = {"bf16": 1.0, "f16": 1.0, "tf32": 1.1 / 2.25, "e4m3": 2.0, "e5m2": 2.0, "e3m2": 2.0, "e2m3": 2.0,
                 "e2m1": 6.0, "nvf4": 6.0}
# NVIDIA's dense (no 2:4 sparsity) GB300 datasheet rates, TFLOP/s, for the
# MMA kind each format runs on
DATASHEET_DENSE_TFLOPS = {"bf16": 2250.0, "f16": 2250.0, "tf32": 1100.0, "e4m3": 4500.0, "e5m2": 4500.0,
                          "e3m2": 4500.0, "e2m3": 4500.0, "e2m1": 13500.0, "nvf4": 13500.0}
# Tensor-pipe rate of each MMA kind relative to kind::f16, as measured on this
# GPU (a pair of CTAs issuing M = 256, N = 256 MMAs back to back on zero
# operands: 128 cycles per MMA for f16 K = 16, mxf8f6f4 K = 32 and both FP4
# kinds K = 64).  The packed-FP4 kinds run at 4x, not the datasheet's 6x;
# reported beside the nominal fraction, which stays the roofline's peak.
MEASURED_PIPE_RATIO = {"e2m1": 4.0, "nvf4": 4.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "desc.cuh", "gemm_f16.cu", "gemm_tf32.cu", "gemm_mxf8.cu", "api.cu",
                  "splitk_reduce.cu", "gemm_chain.cu", "gemm_chain.cuh", "tmem_ldst.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "blackwell_tensor_core_swizzled_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    or None if there is none or the kernel sources changed since."""
    p = os.path.join(PROFILE_DIR, f"gemm_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_t or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_t.group(1))


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms in a thread."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []  # (host time, sm, max, power, hw, hwt, swt, swpc)
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            import torch
            props = torch.cuda.get_device_properties(self.dev)
            sel = []
            bus = getattr(props, "pci_bus_id", None)
            if bus is not None:
                sel = ["-i", f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:"
                             f"{getattr(props, 'pci_device_id', 0):02X}.0"]
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "20"] + sel, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True, bufsize=1)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), *parts[:7]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: nearest samples under load
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest samples to the timed region (shorter than the sampling period)"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ----------------------------------------------------------------- GPU arm

def to_dev(bits, torch):
    view = {np.dtype(np.uint8): np.uint8, np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}[bits.dtype]
    return torch.from_numpy(np.ascontiguousarray(bits).view(view)).cuda()


# tcg_gemm_args.epilogue for the device-timed calls (--epilogue): 0 auto,
# 1 .32x32b rows, 2 .16x256b fragments written with stmatrix
EPILOGUE = {"auto": 0, "rows": 1, "frag": 2}
_epilogue = 0


def run_workload(tcg, torch, w, steps, warmup, dist_ctx, measure_e2e=True):
    x = syn.make_inputs(w)
    M, N, K = w.M, w.N, w.K
    A = to_dev(x["A"], torch)
    B = to_dev(x["B"], torch)
    out_t = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.out]
    D = torch.empty((M, N), dtype=out_t, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    scaled = w.block_scaled
    a_maj = 0 if w.a_major == "k" else 1
    b_maj = 0 if w.b_major == "k" else 1
    if scaled:
        SFA = to_dev(x["SFA"], torch)
        SFB = to_dev(x["SFB"], torch)
        fmt = IN_TYPE[w.dtype]
        tn = tcg.tile_n(fmt, M, N, K, b_maj, w.cta_group)
        ia = torch.empty(tcg.scale_image_bytes(fmt, M, K, 128), dtype=torch.uint8, device="cuda")
        ib = torch.empty(tcg.scale_image_bytes(fmt, N, K, tn), dtype=torch.uint8, device="cuda")

    launches = [0]
    # Inputs of HBM-bound (skinny) workloads are not much larger than the
    # L2: flush it before every step by writing a 256 MiB buffer (outside the
    # GEMM's events; such workloads report the GEMM time, not the step time).
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if w.extra.get("bound") == "hbm" else None

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    trace_buf = torch.zeros((sms, 10), dtype=torch.int64, device="cuda")

    def step(ev_pair=None, trace=False):
        n = 0
        if flush is not None:
            flush.zero_()
        if scaled:
            tcg.prepare_scales_ab(fmt, SFA, M, ia, SFB, N, tn, ib, K, stream=sp)
            n += 1
            if ev_pair:
                ev_pair[0].record(stream)
            if trace:
                tcg.trace_next(trace_buf, sms)
            tcg.gemm(M, N, K, IN_TYPE[w.dtype], A, a_maj, x["lda"], B, b_maj, x["ldb"], D, OUT[w.out], N, ACC[w.acc],
                     SFA_img=ia, SFB_img=ib, cta_group=w.cta_group, stream=sp, epilogue=_epilogue)
        else:
            if ev_pair:
                ev_pair[0].record(stream)
            if trace:
                tcg.trace_next(trace_buf, sms)
            tcg.gemm(M, N, K, IN_TYPE[w.dtype], A, a_maj, x["lda"], B, b_maj, x["ldb"], D, OUT[w.out], N,
                     ACC[w.acc], cta_group=w.cta_group, stream=sp, epilogue=_epilogue)
        n += tcg.last_launch_count()
        if ev_pair:
            ev_pair[1].record(stream)
        launches[0] += n

    for _ in range(warmup):
        step()
    rc = tcg.check(sp)
    if rc != 0:
        raise RuntimeError(f"warm-up failed: {tcg.status_string(rc)} {tcg.last_error_string()}")

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    torch.cuda.synchronize()
    launches[0] = 0
    t_host0 = time.time()
    start.record(stream)
    for i in range(steps):
        # the last timed launch records its CTAs' globaltimer and SM cycle
        # counters at entry and exit: the SM clock it actually ran at
        step(kev[i], trace=(i == steps - 1))
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    dist_ctx.barrier()
    rc = tcg.check(sp)
    if rc != 0:
        raise RuntimeError(f"timed run failed: {tcg.status_string(rc)} {tcg.last_error_string()}")
    total_ms = start.elapsed_time(end)
    kernel_ms = float(np.mean([a.elapsed_time(b) for a, b in kev]))
    res = {"total_ms": total_ms, "kernel_ms": kernel_ms, "launches": launches[0], "t0": t_host0, "t1": t_host1,
           **kernel_clock(trace_buf)}

    if measure_e2e:
        # End to end through the C ABI: every step copies its inputs in from
        # pinned host memory, runs the GEMM and copies the result out.  Steps
        # are double buffered on three streams (upload, compute, download), so
        # the upload of step i+1 and the download of step i-1 overlap the GEMM
        # of step i, as a serving loop would run it.
        view = {np.dtype(np.uint8): np.uint8, np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}
        hA = torch.from_numpy(x["A"].view(view[x["A"].dtype])).pin_memory()
        hB = torch.from_numpy(x["B"].view(view[x["B"].dtype])).pin_memory()
        hD = [torch.empty((M, N), dtype=out_t).pin_memory() for _ in range(2)]
        e_steps = max(2, min(steps, 100))  # the same steps as the device-timed run (bounded)
        h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        dA = [A, torch.empty_like(A)]
        dB = [B, torch.empty_like(B)]
        dD = [D, torch.empty_like(D)]
        if scaled:
            hSFA = torch.from_numpy(x["SFA"]).pin_memory()
            hSFB = torch.from_numpy(x["SFB"]).pin_memory()
            h2d += hSFA.numel() + hSFB.numel()
            dSFA = [SFA, torch.empty_like(SFA)]
            dSFB = [SFB, torch.empty_like(SFB)]
        d2h = hD[0].numel() * hD[0].element_size()
        up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("up", "comp", "down")}
        started = [[False, False]]

        def e2e_step(i):
            bi = i % 2
            with torch.cuda.stream(up):
                if started[0][bi]:
                    up.wait_event(ev["comp"][bi])  # the GEMM of step i-2 has read this buffer
                dA[bi].copy_(hA, non_blocking=True)
                dB[bi].copy_(hB, non_blocking=True)
                if scaled:
                    dSFA[bi].copy_(hSFA, non_blocking=True)
                    dSFB[bi].copy_(hSFB, non_blocking=True)
                ev["up"][bi].record(up)
            comp.wait_event(ev["up"][bi])
            if started[0][bi]:
                comp.wait_event(ev["down"][bi])  # the result of step i-2 has left this buffer
            cs = comp.cuda_stream
            if scaled and w.dtype == "e4m3":
                tcg.gemm_mxf8_blockscaled(M, N, K, dA[bi], a_maj, x["lda"], dB[bi], b_maj, x["ldb"], dSFA[bi],
                                          dSFB[bi], dD[bi], OUT[w.out], N, ACC[w.acc], stream=cs)
            elif scaled and w.dtype == "e2m1":
                tcg.gemm_mxf4_blockscaled(M, N, K, dA[bi], a_maj, x["lda"], dB[bi], b_maj, x["ldb"], dSFA[bi],
                                          dSFB[bi], dD[bi], OUT[w.out], N, ACC[w.acc], stream=cs)
            elif scaled and w.dtype == "nvf4":
                tcg.gemm_nvf4_blockscaled(M, N, K, dA[bi], a_maj, x["lda"], dB[bi], b_maj, x["ldb"], dSFA[bi],
                                          dSFB[bi], dD[bi], OUT[w.out], N, ACC[w.acc], stream=cs)
            elif scaled and w.dtype in ("e3m2", "e2m3"):
                tcg.gemm_mxf6_blockscaled(IN_TYPE[w.dtype], M, N, K, dA[bi], a_maj, x["lda"], dB[bi], b_maj,
                                          x["ldb"], dSFA[bi], dSFB[bi], dD[bi], OUT[w.out], N, ACC[w.acc], stream=cs)
            elif scaled:
                tcg.gemm(M, N, K, IN_TYPE[w.dtype], dA[bi], a_maj, x["lda"], dB[bi], b_maj, x["ldb"], dD[bi],
                         OUT[w.out], N, ACC[w.acc], SFA=dSFA[bi], SFB=dSFB[bi], stream=cs)
            else:
                fn = {"f16": tcg.gemm_f16, "bf16": tcg.gemm_bf16, "tf32": tcg.gemm_tf32}[w.dtype]
                fn(M, N, K, dA[bi], a_maj, x["lda"], dB[bi], b_maj, x["ldb"], dD[bi], OUT[w.out], N, ACC[w.acc],
                   stream=cs)
            ev["comp"][bi].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev["comp"][bi])
                hD[bi].copy_(dD[bi], non_blocking=True)
                ev["down"][bi].record(down)
            started[0][bi] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        started[0] = [False, False]
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        es.record(up)
        for i in range(e_steps):
            e2e_step(i)
        for k in range(2):
            down.wait_event(ev["down"][k])
        ee.record(down)
        torch.cuda.synchronize()
        rc = tcg.check(comp.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"e2e run failed: {tcg.status_string(rc)}")
        res.update({"e2e_ms": es.elapsed_time(ee) / e_steps, "h2d": h2d, "d2h": d2h, "e2e_steps": e_steps})
    return res


# A timed region longer than this runs into the 1.4 kW power cap (the SM clock
# falls from ~2.0 to ~1.6 GHz within ~100 ms of back-to-back GEMMs), so it is
# compared with the sustained bf16 figure instead of the burst one.
SUSTAINED_AFTER_S = 0.05


OUT_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def roofline(w, kernel_ms, peaks, traffic, timed_s):
    if w.extra.get("bound") == "hbm":
        # skinny shapes stream B once: bound by HBM, reported in GB/s
        byts = ESIZE[w.dtype] * (w.M * w.K + w.N * w.K) + OUT_BYTES[w.out] * w.M * w.N
        achieved = byts / (kernel_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peaks['source']} HBM copy bandwidth",
                "kernel": "tcg::gemm_kernel + tcg::splitk_reduce_kernel (L2 flushed before each step)",
                "algorithmic_bytes_per_launch": byts}
    flops = 2.0 * w.M * w.N * w.K
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    ratio = NOMINAL_RATIO[w.dtype]
    regime = "sustained" if timed_s > SUSTAINED_AFTER_S else "burst"
    peak = (peaks["bf16_tflops_sustained"] if regime == "sustained" else peaks["bf16_tflops"]) * ratio
    src = (f"{peaks['source']} bf16 {regime} (timed region {timed_s * 1e3:.0f} ms)"
           + ("" if ratio == 1.0 else f" x nominal {w.dtype}/bf16 ratio {ratio:g}"))
    sheet = DATASHEET_DENSE_TFLOPS[w.dtype]
    line = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": src,
            "frac_of_datasheet_dense": round(achieved / sheet, 4),
            "datasheet_dense_peak": sheet,
            "kernel": "tcg::gemm_kernel", "algorithmic_flops_per_launch": flops}
    if w.dtype in MEASURED_PIPE_RATIO:
        mp = peak / ratio * MEASURED_PIPE_RATIO[w.dtype]
        line.update({"measured_pipe_peak": round(mp, 1), "frac_of_measured_pipe": round(achieved / mp, 4),
                     "measured_pipe_source": f"bf16 {regime} peak x the measured per-clock ratio "
                                             f"{MEASURED_PIPE_RATIO[w.dtype]:g} of this MMA kind"})
    return line


def kernel_clock(trace_buf):
    """The SM clock a traced launch ran at (tcg_trace_next slots 0/6 =
    globaltimer at entry / exit, 8/9 = clock64 next to them): median and
    range over its CTAs, in MHz."""
    tr = trace_buf.cpu().numpy()
    ok = (tr[:, 6] > tr[:, 0]) & (tr[:, 9] > tr[:, 8])
    ghz = (tr[ok, 9] - tr[ok, 8]) / (tr[ok, 6] - tr[ok, 0]) if ok.any() else np.array([])
    if not ghz.size:
        return {"kernel_sm_mhz": None, "kernel_sm_mhz_range": None}
    return {"kernel_sm_mhz": round(float(np.median(ghz)) * 1000, 1),
            "kernel_sm_mhz_range": [round(float(ghz.min()) * 1000, 1), round(float(ghz.max()) * 1000, 1)]}


def run_chain_workload(tcg, torch, w, steps, warmup):
    """Device-timed chained GEMM E = round(A.B1).B2 (tcg_gemm_chain): one
    launch per step, CUDA events around each.  Inputs (A and E larger than the
    L2) are resident on the device."""
    x = syn.make_chain_inputs(w)
    M, N1, N2, K = x["M"], x["N1"], x["N2"], x["K"]
    A, B1, B2 = (to_dev(x[k], torch) for k in ("A", "B1", "B2"))
    out_t = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.out]
    E = torch.empty((M, N2), dtype=out_t, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def call():
        tcg.gemm_chain(IN_TYPE[w.dtype], M, N1, N2, K, A, K, B1, K, B2, N1, E, OUT[w.out], N2, stream=sp)

    for _ in range(warmup):
        call()
    rc = tcg.check(sp)
    if rc != 0:
        raise RuntimeError(f"chain warm-up failed: {tcg.status_string(rc)} {tcg.last_error_string()}")
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    trace_buf = torch.zeros((sms, 10), dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    launches = 0
    t0 = time.time()
    for i in range(steps):
        kev[i][0].record(stream)
        if i == steps - 1:  # the last timed launch records the SM clock it ran at
            tcg.trace_next(trace_buf, sms)
        call()
        launches += tcg.last_launch_count()
        kev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    rc = tcg.check(sp)
    if rc != 0:
        raise RuntimeError(f"chain run failed: {tcg.status_string(rc)}")
    kernel_ms = float(np.mean([a.elapsed_time(b) for a, b in kev]))
    return {"kernel_ms": kernel_ms, "launches": launches, "t0": t0, "t1": t1, **kernel_clock(trace_buf),
            "flops": 2.0 * M * K * N1 + 2.0 * M * N1 * N2,
            "bytes": float(ESIZE[w.dtype] * (M * K + N1 * K + N2 * N1) + OUT_BYTES[w.out] * M * N2)}


def chain_roofline(w, r, peaks, traffic=None):
    """The chain's roofline is the larger of its tensor time (both products at
    the bf16 peak) and its HBM time (A, B1, B2 read and E written once)."""
    t_tensor = r["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = r["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t = r["kernel_ms"] * 1e-3
    if t_hbm >= t_tensor:
        achieved = r["bytes"] / t / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"{peaks['source']} HBM copy bandwidth (tensor time at the bf16 burst peak: "
                               f"{t_tensor * 1e6:.1f} us, HBM time {t_hbm * 1e6:.1f} us)",
                "kernel": "tcg::gemm_chain_kernel", "algorithmic_bytes_per_launch": r["bytes"],
                "algorithmic_flops_per_launch": r["flops"]}
    achieved = r["flops"] / t / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peaks["bf16_tflops"], 1),
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
            "peak_source": f"{peaks['source']} bf16 burst (HBM time {t_hbm * 1e6:.1f} us, tensor time "
                           f"{t_tensor * 1e6:.1f} us)",
            "kernel": "tcg::gemm_chain_kernel", "algorithmic_bytes_per_launch": r["bytes"],
            "algorithmic_flops_per_launch": r["flops"]}


# ----------------------------------------------------------------- CPU (oracle) arm

# seconds of host work in the CPU baseline reported beside the GPU numbers
CPU_BASELINE_S = 15.0

def oracle_inputs(w):
    import oracle
    oracle.build()
    return syn.make_inputs(w)


def oracle_sample(w, x, rows_n: int):
    """Time the float64 oracle on `rows_n` output rows (all N columns) of the
    workload (inputs `x` already generated); returns (TFLOP/s, seconds, threads)."""
    import oracle
    t = {"f16": oracle.F16, "bf16": oracle.BF16, "tf32": oracle.F32, "e4m3": oracle.E4M3, "e5m2": oracle.E5M2,
         "e3m2": oracle.E3M2, "e2m3": oracle.E2M3, "e2m1": oracle.E2M1, "nvf4": oracle.E2M1}[w.dtype]
    nv = w.dtype == "nvf4"
    rows = np.linspace(0, w.M - 1, rows_n).astype(np.int64)
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.gemm(w.M, w.N, w.K, x["A"], t, 0 if w.a_major == "k" else 1, x["lda"], x["B"], t,
                0 if w.b_major == "k" else 1, x["ldb"], SFA=x["SFA"], SFB=x["SFB"], rows=rows, nthreads=threads,
                sf_block=16 if nv else 32, sf_kind=oracle.SF_UE4M3 if nv else oracle.SF_E8M0)
    dt = time.perf_counter() - t0
    return 2.0 * rows_n * w.N * w.K / dt / 1e12, dt, threads


# ----------------------------------------------------------------- distributed

class DistCtx:
    """One process per GPU (torchrun's RANK / WORLD_SIZE / LOCAL_RANK), NCCL on
    the GPU by default; the CPU tests use the same class over gloo."""

    def __init__(self, n, backend: str = "nccl", device: str = "cuda"):
        self.n = n
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.device = device
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            if device == "cuda":
                torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())


def whole_job(dctx: DistCtx, flops_per_step: float, steps: int, local_ms: float):
    """Replicas: every rank runs the same steps; the job takes as long as the
    slowest rank (max over ranks), and its throughput counts every rank's
    work.  Returns (TFLOP/s of the whole job, the max time in ms)."""
    t = dctx.max(local_ms)
    return dctx.world * flops_per_step * steps / (t * 1e-3) / 1e12, t


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_8192_cta2",
                    choices=sorted(n for n, v in syn.WORKLOADS.items() if "chain_n1" not in v.extra))
    ap.add_argument("--secondary",
                    default="mxf8_8192,bf16_skinny_m16,bf16_4096_kmn_cta1,tf32_2048x2048x8192,f16acc_8192_cta2,"
                            "mxf6_e2m3_8192,mxf4_8192,nvf4_8192,chain_bf16_38912x256x4096",
                    help="comma list of extra workloads ('' for none)")
    ap.add_argument("--sustained-s", type=float, default=1.5,
                    help="length of the back-to-back sustained pass of the headline workload (0: skip)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle rows in the CPU baseline (0: 2 per thread)")
    ap.add_argument("--epilogue", default="auto", choices=sorted(EPILOGUE),
                    help="how 16-bit outputs leave TMEM in the device-timed calls (frag: .16x256b + stmatrix)")
    args = ap.parse_args()
    global _epilogue
    _epilogue = EPILOGUE[args.epilogue]
    w = syn.WORKLOADS[args.workload]

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        import oracle
        oracle.build()
        rows_n = args.cpu_rows or oracle.num_threads()
        x = oracle_inputs(w)
        vals = []
        for _ in range(max(args.warmup, 0)):
            oracle_sample(w, x, max(1, rows_n // 4))
        for _ in range(args.steps):
            v, dt, thr = oracle_sample(w, x, rows_n)
            vals.append((v, dt))
        value = float(np.median([v for v, _ in vals]))
        ms = float(np.mean([dt for _, dt in vals])) * 1e3
        sample = f"{rows_n} of {w.M} output rows (all {w.N} columns, K={w.K}) of {w.name} per step"
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                                                "in": w.dtype, "sample": sample},
                "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": thr, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dctx = DistCtx(args.gpus)
    if dctx.world == 1:
        torch.cuda.set_device(0)
    from blackwell_tensor_core_swizzled_gb300.build import build as build_lib
    build_lib()
    import blackwell_tensor_core_swizzled_gb300 as tcg

    peaks = measured_peaks()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    sustained = None
    try:
        res = run_workload(tcg, torch, w, args.steps, args.warmup, dctx)
        if args.sustained_s > 0:
            # Back-to-back headline GEMMs for ~1.5 s: long enough to reach the
            # power-capped clock, compared with the sustained cuBLAS figure,
            # with the clock record of that window.
            n_sus = max(args.steps, int(args.sustained_s / max(res["kernel_ms"] * 1e-3, 1e-6)))
            rs = run_workload(tcg, torch, w, n_sus, 0, dctx, measure_e2e=False)
            v_s, t_s = whole_job(dctx, 2.0 * w.M * w.N * w.K, n_sus, rs["total_ms"])
            rl_s = roofline(w, rs["total_ms"] / n_sus, peaks, None, rs["total_ms"] * 1e-3)
            sustained = {"value": round(v_s, 1), "unit": UNIT, "steps": n_sus, "ms_per_step": round(t_s / n_sus, 4),
                         "timed_s": round(rs["total_ms"] * 1e-3, 3), "frac": rl_s["frac"], "peak": rl_s["peak"],
                         "peak_source": rl_s["peak_source"], "frac_of_datasheet_dense": rl_s["frac_of_datasheet_dense"],
                         "clocks": {**sampler.summary(rs["t0"], rs["t1"]),
                                    "kernel_sm_mhz": rs["kernel_sm_mhz"],
                                    "kernel_sm_mhz_range": rs["kernel_sm_mhz_range"]}}
        sec = []
        for name in [s for s in args.secondary.split(",") if s and s != w.name]:
            ws = syn.WORKLOADS[name]
            if "chain_n1" in ws.extra:
                rc2 = run_chain_workload(tcg, torch, ws, args.steps, args.warmup)
                rl2 = chain_roofline(ws, rc2, peaks, profiled_traffic(name))
                # replicas: the whole job's throughput, timed by the slowest rank
                v2, t2 = whole_job(dctx, rc2["flops"], args.steps, rc2["kernel_ms"] * args.steps)
                sec.append({"workload": name, "value": round(v2, 1),
                            "unit": UNIT, "ms_per_step": round(t2 / args.steps, 4), "dtype": ws.dtype,
                            "gpu_launches": rc2["launches"], "kernel_sm_mhz": rc2["kernel_sm_mhz"], "roofline": rl2})
                continue
            r2 = run_workload(tcg, torch, ws, args.steps, args.warmup, dctx, measure_e2e=False)
            # steps of an hbm workload include an L2 flush: count the GEMM time only
            local = r2["kernel_ms"] * args.steps if ws.extra.get("bound") == "hbm" else r2["total_ms"]
            v2, t2 = whole_job(dctx, 2.0 * ws.M * ws.N * ws.K, args.steps, local)
            sec.append({"workload": name, "value": round(v2, 1),
                        "unit": UNIT, "ms_per_step": round(t2 / args.steps, 4), "dtype": ws.dtype,
                        "gpu_launches": r2["launches"], "kernel_sm_mhz": r2["kernel_sm_mhz"],
                        "roofline": roofline(ws, r2["kernel_ms"], peaks, profiled_traffic(name),
                                                    r2["total_ms"] * 1e-3)})
    finally:
        sampler.stop()
    clocks = sampler.summary(res["t0"], res["t1"])
    # the SM clock of the last timed launch, from its CTAs' own counters
    # (median and range over CTAs of cycles / nanoseconds between entry and exit)
    clocks["kernel_sm_mhz"] = res["kernel_sm_mhz"]
    clocks["kernel_sm_mhz_range"] = res["kernel_sm_mhz_range"]

    flops_step = 2.0 * w.M * w.N * w.K
    value, total_ms = whole_job(dctx, flops_step, args.steps, res["total_ms"])
    e2e_val, e2e_ms = whole_job(dctx, flops_step, 1, res["e2e_ms"])

    if dctx.rank != 0:
        return
    cpu = None
    if dctx.world == 1 or dctx.rank == 0:
        import oracle
        oracle.build()
        x_cpu = oracle_inputs(w)
        rows_n = args.cpu_rows or 2 * oracle.num_threads()
        v, dt, thr = oracle_sample(w, x_cpu, rows_n)
        if not args.cpu_rows and dt < CPU_BASELINE_S / 2:
            # a bounded sample of about CPU_BASELINE_S seconds, sized from the first
            rows_n = int(min(w.M, max(rows_n, rows_n * CPU_BASELINE_S / max(dt, 1e-3))))
            v, dt, thr = oracle_sample(w, x_cpu, rows_n)
        cpu = {"value": round(v, 6), "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"{rows_n} of {w.M} output rows (all {w.N} columns, K={w.K}) of {w.name}, "
                         f"{dt:.2f} s wall"}
    rl = roofline(w, res["kernel_ms"], peaks, profiled_traffic(w.name), res["total_ms"] * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dctx.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": w.dtype, "a_major": w.a_major,
                   "b_major": w.b_major, "acc": w.acc, "out": w.out, "cta_group": w.cta_group,
                   "l2": "inputs larger than L2 (no flush): A+B = "
                         f"{(w.M * w.K + w.N * w.K) * ESIZE[w.dtype] / 2**20:.0f} MiB",
                   "parallelism": f"replicas x{dctx.world}",
                   **({"epilogue": args.epilogue} if args.epilogue != "auto" else {})},
        "pct_of_measured_peak": round(100 * rl["frac"], 2),
        "pct_of_datasheet_dense_peak": (round(100 * rl["frac_of_datasheet_dense"], 2)
                                        if "frac_of_datasheet_dense" in rl else None),
        "roofline": rl,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"], "ms_per_step": round(e2e_ms, 3), "steps": res["e2e_steps"],
                "pipeline": "pinned host inputs in and result out every step; double buffered on upload / "
                            "compute / download streams"},
        "gpu_launches": res["launches"],
        "clocks": clocks,
        "sustained": sustained,
        "secondary": sec,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
