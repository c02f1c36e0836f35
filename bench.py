"""Benchmark of the NVFP4 block-scaled path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

Prints ONE JSON line.  The timed step is one NVFP4 block-scaled GEMM
D = alpha * (A*SFA)(B*SFB)^T on the square workload M = N = K = 8192 (codes
uniform over the 16 E2M1 codes, scales uniform over the E4M3 values 2^-4..2^4,
alpha uniform in [0.25, 4]), operands resident in HBM; L2 is flushed between
timed iterations.  `value` is TFLOP/s (2*M*N*K per step) summed over ranks.
Sub-measurements in the same line: the 16384^3 GEMM, the W4A16 decode GEMM
(weight GB/s, CUDA-graph replay over rotated weight copies larger than L2) and
the quantize / pack_scales producers (GB/s).

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload; its value is in the same unit.

Under torchrun (N > 1) every rank runs the same step on its own GPU (replicas,
weak scaling); rank 0 prints the line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOP/s at 8k/16k square, % of GB300 dense FP4 peak; W4A16 GB/s"
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense FP4 : BF16 tensor ratio (GB300)
P1_V1_8K_TFLOPS = 1476.0      # pages' 8192^3 NVFP4 GEMM (RTX PRO 6000, context only)
S_MAIN = 8192


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="skip the sub-measurements")
    ap.add_argument("--only", choices=["w4a16", "producers", "llm", "mma_ceiling", "cublaslt"], default=None,
                    help="run one sub-measurement alone and print its JSON (for profiling runs)")
    ap.add_argument("--w4a16-shapes", default=None,
                    help="with --only w4a16: comma-separated NxKxM list, e.g. 17408x5120x1")
    ap.add_argument("--llm-configs", default="0",
                    help="with --only llm: comma-separated GEMM configs to time (0 = automatic choice)")
    ap.add_argument("--llm-shapes", default=None,
                    help="with --only llm: comma-separated MxNxK list (default: every LLM layer shape)")
    return ap.parse_args()


def dist_setup(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def all_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_value(ms_max, steps, flops_per_step, world):
    """Whole-job TFLOP/s of `world` replicas that each ran `steps` steps, timed by the
    slowest rank (ms_max = that rank's summed step time)."""
    return world * steps * flops_per_step / (ms_max / 1e3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "10"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi needs a moment to start: wait for its first sample so that the
        # samples cover the timed region that follows
        t0 = time.time()
        while not self.samples and time.time() - t0 < 3.0:
            time.sleep(0.005)
        self.first = len(self.samples)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        self.last = len(self.samples)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        """Samples taken between the start and the end of the timed region (the timed
        launches are asynchronous: the region ends at the synchronisation)."""
        window = self.samples[getattr(self, "first", 0):getattr(self, "last", len(self.samples))]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[1]) for s in window if s[1].replace(".", "", 1).isdigit()]
        mx = [float(s[2]) for s in window if s[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in window for n, v in zip(names, s[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(window)}


def kernel_source_hash():
    """Hash of the pair kernel's code (its file, its schedule and the PTX helpers), comments and
    whitespace removed: the committed counters stay valid across comment edits and
    are dropped by any change to the code itself."""
    import re

    h = hashlib.sha256()
    for name in ("gemm_w4a4.cu", "pair_sched.h", "ptx.cuh"):
        with open(os.path.join(ROOT, "nvfp4_block_scaled_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ our arm

def gemm_operands(S, seed=0):
    import numpy as np
    import torch

    import nvfp4_block_scaled_gb300 as nv
    from synthetic import generators as G

    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=seed)
    alpha = G.alpha_uniform(seed)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    a, b = dev(A), dev(B)
    sfa, sfb = nv.pack_scales(dev(SFA), S), nv.pack_scales(dev(SFB), S)
    return (A, SFA, B, SFB, alpha), (a, sfa, b, sfb)


def time_gemm(S, steps, warmup, world, sampler=None):
    """Per-iteration CUDA-event time of nvfp4_gemm on S^3, L2 flushed in between."""
    import torch

    import nvfp4_block_scaled_gb300 as nv

    host, (a, sfa, b, sfb) = gemm_operands(S)
    alpha = host[4]
    D = torch.empty((S, S), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        nv.gemm(a, sfa, b, sfb, alpha, S, S, S, out=D)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush.zero_()                       # evict the operands from L2 (not timed)
        e0.record(stream)
        nv.gemm(a, sfa, b, sfb, alpha, S, S, S, out=D)
        e1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.stop()
    barrier(world)
    times = [e0.elapsed_time(e1) for e0, e1 in evs]
    err = nv.device_error()
    if err != 0:
        raise RuntimeError(f"device error {err}")
    return times, (host, D)


def time_gemm_e2e(S, steps, warmup, world=1):
    """Same GEMM end to end through the C ABI with host buffers: every step copies
    its A, B, SFA, SFB from pinned host memory to the device, runs the GEMM and
    copies D back to pinned host memory, all inside the timed region.  Steps are
    pipelined the way a serving loop would run them: host-to-device copies, GEMMs
    and device-to-host copies on three streams with two device buffer sets, so step
    i's result copy-out overlaps step i+1's copy-in and GEMM (stream events order
    each buffer set's reuse).  Returns (ms per step, h2d bytes, d2h bytes)."""
    import torch

    import nvfp4_block_scaled_gb300 as nv
    from synthetic import generators as G

    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0)
    alpha = G.alpha_uniform(0)
    # host-side packed scales (the layout the GEMM consumes) come from the GPU packer once
    sfa_p = nv.pack_scales(torch.from_numpy(SFA).cuda(), S).cpu()
    sfb_p = nv.pack_scales(torch.from_numpy(SFB).cuda(), S).cpu()
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hSFA = sfa_p.pin_memory()
    hSFB = sfb_p.pin_memory()
    hD = [torch.empty((S, S), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    bufs = [dict(A=torch.empty_like(hA, device="cuda"), B=torch.empty_like(hB, device="cuda"),
                 SFA=torch.empty_like(hSFA, device="cuda"), SFB=torch.empty_like(hSFB, device="cuda"),
                 D=torch.empty((S, S), dtype=torch.bfloat16, device="cuda")) for _ in range(2)]
    s_in, s_gemm, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inputs_free = [ev(), ev()]   # the GEMM that read set k has finished
    inputs_ready = [ev(), ev()]
    d_ready = [ev(), ev()]
    d_free = [ev(), ev()]        # set k's D has been copied out
    used = [False, False]

    def step(i):
        k = i % 2
        b = bufs[k]
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(inputs_free[k])
            b["A"].copy_(hA, non_blocking=True)
            b["B"].copy_(hB, non_blocking=True)
            b["SFA"].copy_(hSFA, non_blocking=True)
            b["SFB"].copy_(hSFB, non_blocking=True)
            inputs_ready[k].record(s_in)
        with torch.cuda.stream(s_gemm):
            s_gemm.wait_event(inputs_ready[k])
            if used[k]:
                s_gemm.wait_event(d_free[k])
            nv.gemm(b["A"], b["SFA"], b["B"], b["SFB"], alpha, S, S, S, out=b["D"], stream=s_gemm)
            inputs_free[k].record(s_gemm)
            d_ready[k].record(s_gemm)
        with torch.cuda.stream(s_out):
            s_out.wait_event(d_ready[k])
            hD[k].copy_(b["D"], non_blocking=True)
            d_free[k].record(s_out)
        used[k] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        step(warmup + i)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1) / steps
    h2d = hA.numel() + hB.numel() + hSFA.numel() + hSFB.numel()
    d2h = hD[0].numel() * 2
    return ms, h2d, d2h


W4A16_NK = [(5120, 5120), (17408, 5120), (5120, 17408)]
W4A16_M = (1, 8, 32, 72, 144, 1024)


def bench_w4a16(peaks, shapes=None):
    """W4A16 decode: weight GB/s over CUDA-graph replay of rotated weight copies, for
    nvfp4_w4a16_linear and nvfp4_w4a16_linear_streamk (keys prefixed streamk_) up to
    32 tokens and where the stream-K entry takes its tensor-core stream-K kernel
    (more than 256 tokens on a tile grid of less than 1.25 waves).
    shapes: list of (N, K, [M...]); default every (N, K) of W4A16_NK with every M of W4A16_M."""
    import numpy as np
    import torch

    import nvfp4_block_scaled_gb300 as nv
    from synthetic import generators as G

    out = {}
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    if shapes is None:
        shapes = [(N, K, W4A16_M) for (N, K) in W4A16_NK]
    for (N, K, Ms) in shapes:
        W = G.packed_codes_uniform(N, K, 0, "W")
        SW = G.scales_uniform_normal(N, K, 0, "SW")
        w0 = nv.w4a16_prepare(torch.from_numpy(W).cuda(), torch.from_numpy(SW).cuda())
        wbytes = nv.w4a16_prepared_bytes(N, K)
        copies = max(4, int(np.ceil(4 * l2 / wbytes)))
        ws = [w0.clone() for _ in range(copies)]
        sk_ws = torch.zeros(nv.w4a16_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")
        for M in Ms:
            x = torch.from_numpy(G.bf16_normal(M, K, 0, "x").view(np.int16)).cuda().view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            alg_bytes = wbytes + 2 * M * K + 2 * M * N
            calls = {"": lambda w, s=None: nv.w4a16_linear(x, w, 1.0, N, out=y, stream=s)}
            tiles = ((M + 255) // 256) * (N // 128)
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            if M <= 32 or (M > 256 and 4 * tiles < 5 * sms):
                calls["streamk_"] = lambda w, s=None: nv.w4a16_linear_streamk(x, w, 1.0, N, sk_ws, out=y, stream=s)
            cell = {}
            for prefix, call in calls.items():
                best, iso = _time_w4a16_call(call, ws)
                cell.update({prefix + "us": round(best, 3), prefix + "weight_GBps": round(wbytes / best / 1e3, 1),
                             prefix + "GBps": round(alg_bytes / best / 1e3, 1),
                             prefix + "hbm_frac": round(alg_bytes / best / 1e3 / peaks["hbm_gbs"], 3),
                             prefix + "tflops": round(2 * M * N * K / best / 1e6, 1),
                             prefix + "isolated_us": round(iso, 2)})
            out[f"M{M}_N{N}_K{K}"] = cell
        del ws
    return out


def _time_w4a16_call(call, ws):
    """(best per-call us over CUDA-graph replay of one call per weight copy, median
    isolated us): the graph replays back to back three times; an isolated call has no
    call before or after it and its weights are not in L2."""
    import statistics as st

    import torch

    for w in ws[:2]:
        call(w)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for w in ws:
                call(w, s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / len(ws)
        best = us if best is None else min(best, us)
    del g
    # a short device-side sleep queued first keeps the host's launch cost out of the
    # event interval, so the isolated number is the call's device time
    iso = []
    for i in range(min(len(ws), 8)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)
        e0.record()
        call(ws[i])
        e1.record()
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1) * 1e3)
    return best, st.median(iso)


LLM_M = (128, 1024, 8192)
LLM_NK = [(5120, 5120), (17408, 5120), (5120, 17408), (6144, 5120)]


def bench_llm(peaks, configs=(0,), shapes=None):
    """W4A4 GEMM on the LLM linear-layer shapes: activations N(0,1) and weights
    N(0,0.02) in BF16 (seeded device RNG), quantised by nvfp4_quantize with per-tensor
    scales, scales packed.  Per-call time from CUDA-graph replay of one call per
    rotated weight copy (copies totalling >= 4x L2, so each call reads its weight
    from HBM), for the automatic configuration and for nvfp4_gemm_streamk.  Each cell
    reports its roofline bound: max(2MNK / FP4 peak, bytes / HBM bandwidth)."""
    import math

    import torch

    import nvfp4_block_scaled_gb300 as nv

    peak_fp4 = peaks["bf16_tflops"] * FP4_OVER_BF16
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    gen = torch.Generator(device="cuda")
    out = {}
    if shapes is None:
        shapes = [(M, N, K) for M in LLM_M for (N, K) in LLM_NK]
    for (M, N, K) in shapes:
        gen.manual_seed(M * 7 + N * 3 + K)
        x = torch.randn((M, K), device="cuda", generator=gen).to(torch.bfloat16)
        w = (0.02 * torch.randn((N, K), device="cuda", generator=gen)).to(torch.bfloat16)
        gx = float(x.abs().max().float() / (6 * 448))
        gw = float(w.abs().max().float() / (6 * 448))
        A, SFA = nv.quantize(x, gx)
        B, SFB = nv.quantize(w, gw)
        A2, SP2 = nv.quantize_two_pass(x, gx) if K % 256 == 0 else (None, None)
        del x, w
        sfa, sfb = nv.pack_scales(SFA, K), nv.pack_scales(SFB, K)
        wbytes = B.numel() + sfb.numel()
        copies = min(64, max(2, math.ceil(4 * l2 / wbytes)))
        Bs = [B] + [B.clone() for _ in range(copies - 1)]
        sfbs = [sfb] + [sfb.clone() for _ in range(copies - 1)]
        D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        alpha = gx * gw
        flops = 2.0 * M * N * K
        nbytes = M * K // 2 + N * K // 2 + (M + N) * K // 16 + 2 * M * N
        t_tensor = flops / (peak_fp4 * 1e12) * 1e6
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        cell = {"bound": "tensor" if t_tensor >= t_hbm else "hbm",
                "roofline_us": round(max(t_tensor, t_hbm), 2), "copies": copies}
        ws = torch.zeros(nv.gemm_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")
        for cfg in list(configs) + ["streamk"] + (["two_pass"] if A2 is not None else []):
            def call(i, stream=None, cfg=cfg):
                if cfg == "streamk":
                    nv.gemm_streamk(A, sfa, Bs[i], sfbs[i], alpha, M, N, K, ws, out=D, stream=stream)
                elif cfg == "two_pass":
                    nv.gemm_two_pass(A2, SP2, Bs[i], sfbs[i], alpha, M, N, K, out=D, stream=stream)
                else:
                    nv.gemm(A, sfa, Bs[i], sfbs[i], alpha, M, N, K, out=D, config=cfg, stream=stream)
            for i in range(2):
                call(i)
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for i in range(copies):
                        call(i, s)
            torch.cuda.current_stream().wait_stream(s)
            g.replay()
            torch.cuda.synchronize()
            best = None
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / copies
                best = us if best is None else min(best, us)
            del g
            key = cfg if cfg in ("streamk", "two_pass") else ("auto" if cfg == 0 else f"config{cfg}")
            if cfg == "two_pass":
                # twice the MMA work; the activation operand is twice as large
                f2 = 2 * flops
                b2 = nbytes + M * K // 2 + M * K // 16
                r2 = max(f2 / (peak_fp4 * 1e12) * 1e6, b2 / (peaks["hbm_gbs"] * 1e9) * 1e6)
                cell[key] = {"us": round(best, 2), "tflops": round(f2 / best / 1e6, 1),
                             "roofline_us": round(r2, 2), "roofline_frac": round(r2 / best, 3)}
            else:
                cell[key] = {"us": round(best, 2), "tflops": round(flops / best / 1e6, 1),
                             "roofline_frac": round(max(t_tensor, t_hbm) / best, 3)}
        if 0 in configs:
            cell["auto_config"] = nv.gemm_config_name(nv.gemm_choose_config(M, N, K)).split(" ")[0]
        out[f"M{M}_N{N}_K{K}"] = cell
        del A, B, SFA, SFB, sfa, sfb, D, Bs, sfbs, ws, A2, SP2
    err = nv.device_error()
    if err != 0:
        raise RuntimeError(f"device error {err}")
    return out


def bench_producers(peaks):
    """quantize and pack_scales at 8192 x 5120: per-call time from CUDA-graph replay of
    one call per rotated input/output copy (copies totalling >= 4x L2, so every call
    reads from and writes to HBM; no host launch overhead inside the graph)."""
    import numpy as np
    import torch

    import nvfp4_block_scaled_gb300 as nv
    from synthetic import generators as G

    R, K = 8192, 5120
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    x0 = torch.from_numpy(G.bf16_normal(R, K, 0, "x").view(np.int16)).cuda().view(torch.bfloat16)
    g = 0.001
    res = {}

    def graph_time(calls, nbytes):
        for c in calls[:2]:
            c(None)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                for c in calls:
                    c(s)
        torch.cuda.current_stream().wait_stream(s)
        graph.replay()
        torch.cuda.synchronize()
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / len(calls)
            best = us if best is None else min(best, us)
        return {"workload": f"{R}x{K}", "us": round(best, 2), "GBps": round(nbytes / best / 1e3, 1),
                "hbm_frac": round(nbytes / best / 1e3 / peaks["hbm_gbs"], 3), "copies": len(calls)}

    # quantize: 2 B in, 0.5625 B out per element
    qbytes = R * K * 2 + R * K // 2 + R * K // 16
    n = max(2, int(np.ceil(4 * l2 / qbytes)))
    xs = [x0.clone() for _ in range(n)]
    codes = [torch.empty((R, K // 2), dtype=torch.uint8, device="cuda") for _ in range(n)]
    sfs = [torch.empty((R, K // 16), dtype=torch.uint8, device="cuda") for _ in range(n)]
    calls = [lambda st, i=i: nv.quantize(xs[i], g, codes[i], sfs[i], stream=st) for i in range(n)]
    res["quantize"] = graph_time(calls, qbytes)
    # fused quantize + pack: same reads, scales written in the packed layout
    sfps = [torch.empty(nv.packed_scales_bytes(R, K), dtype=torch.uint8, device="cuda") for _ in range(n)]
    calls = [lambda st, i=i: nv.quantize_packed(xs[i], g, codes[i], sfps[i], stream=st) for i in range(n)]
    res["quantize_packed"] = graph_time(calls, qbytes)
    # two-pass quantise: same reads, twice the codes and scales (packed) written
    tbytes = R * K * 2 + R * K + R * K // 8
    c2s = [torch.empty((R, K), dtype=torch.uint8, device="cuda") for _ in range(n)]
    s2s = [torch.empty(nv.packed_scales_bytes(R, 2 * K), dtype=torch.uint8, device="cuda") for _ in range(n)]
    calls = [lambda st, i=i: nv.quantize_two_pass(xs[i], g, c2s[i], s2s[i], stream=st) for i in range(n)]
    res["quantize_two_pass"] = graph_time(calls, tbytes)
    del xs, codes, sfps, c2s, s2s
    # pack_scales: 1 B in, 1 B out per scale
    pbytes = 2 * R * K // 16
    n = max(2, int(np.ceil(4 * l2 / pbytes)))
    srcs = [sfs[i % len(sfs)].clone() for i in range(n)]
    outs = [torch.empty(nv.packed_scales_bytes(R, K), dtype=torch.uint8, device="cuda") for _ in range(n)]
    calls = [lambda st, i=i: nv.pack_scales(srcs[i], K, outs[i], stream=st) for i in range(n)]
    res["pack_scales"] = graph_time(calls, pbytes)
    return res


def bench_mma_ceiling(iters=8192):
    """Back-to-back tcgen05 CTA-pair MMAs (M = N = 256, operands resident) per kind:
    the instruction ceiling the GEMM can reach, and the hardware's FP4 : BF16 ratio."""
    import nvfp4_block_scaled_gb300 as nv

    out = {}
    for kind in ("bf16", "fp8", "nvf4"):
        best = None
        for _ in range(3):
            tf, cyc = nv.mma_ceiling(kind, iters)
            if best is None or tf > best[0]:
                best = (tf, cyc)
        out[kind] = {"tflops": round(best[0], 1), "cycles_per_mma": round(best[1], 1)}
    out["nvf4_over_bf16"] = round(out["nvf4"]["tflops"] / out["bf16"]["tflops"], 3)
    return out


def bench_cublaslt(sizes=(S_MAIN,), steps=10):
    """The vendor library's NVFP4 GEMM on the headline's own operands, beside ours: a
    reference point, not part of the library's path.  cuBLASLt is reached through
    torch._scaled_mm with FP4 operands and E4M3 scales per 16 elements in the same
    128x4-atom layout that pack_scales writes; it has no alpha, so the bit-identity
    check compares both at alpha = 1.  Both are timed like the headline (CUDA events
    on the current stream, L2 flushed between iterations)."""
    import torch

    import nvfp4_block_scaled_gb300 as nv

    if not hasattr(torch, "float4_e2m1fn_x2"):
        return {"unavailable": f"PyTorch {torch.__version__} has no FP4 dtype"}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)

    out = {}
    for S in sizes:
        _, (a, sfa, b, sfb) = gemm_operands(S)
        a4, b4 = a.view(torch.float4_e2m1fn_x2), b.view(torch.float4_e2m1fn_x2).t()
        sa8, sb8 = sfa.view(torch.float8_e4m3fn), sfb.view(torch.float8_e4m3fn)
        D = torch.empty((S, S), dtype=torch.bfloat16, device="cuda")
        try:
            L = torch._scaled_mm(a4, b4, sa8, sb8, out_dtype=torch.bfloat16)
            torch.cuda.synchronize()
        except (RuntimeError, TypeError, ValueError) as e:
            out[str(S)] = {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}
            continue
        nv.gemm(a, sfa, b, sfb, 1.0, S, S, S, out=D)
        torch.cuda.synchronize()
        same = bool(torch.equal(D.view(torch.int16), L.view(torch.int16)))
        ms_lib = timed(lambda: torch._scaled_mm(a4, b4, sa8, sb8, out_dtype=torch.bfloat16))
        ms_ours = timed(lambda: nv.gemm(a, sfa, b, sfb, 1.0, S, S, S, out=D))
        tf = lambda ms: round(2.0 * S ** 3 / (ms / 1e3) / 1e12, 1)  # noqa: E731
        out[str(S)] = {"library_ms": round(ms_lib, 4), "library_tflops": tf(ms_lib), "ours_ms": round(ms_ours, 4),
                       "ours_tflops": tf(ms_ours), "ours_over_library": round(ms_lib / ms_ours, 3),
                       "bit_identical_at_alpha_1": same}
        del a, b, sfa, sfb, a4, b4, sa8, sb8, D, L
    return {"impl": "cuBLASLt through torch._scaled_mm (FP4 x FP4, E4M3 scale per 16, FP32 accumulate, BF16 out)",
            "torch": torch.__version__, "results": out}


def cpu_baseline_gemm(S, target_s=12.0, max_samples=1 << 16):
    """The oracle on a bounded sample of the S^3 workload: sampled outputs, each a full
    K-length dot product of dequantised rows (float64).  Returns TFLOP/s."""
    import numpy as np

    from oracle import nvfp4_oracle as O
    from synthetic import generators as G

    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0)
    alpha = G.alpha_uniform(0)
    rng = np.random.default_rng(7)
    n, total, elapsed = 64, 0, 0.0
    while elapsed < target_s and total < max_samples:
        rows, cols = rng.integers(0, S, n), rng.integers(0, S, n)
        t0 = time.perf_counter()
        O.gemm_at(A, SFA, B, SFB, alpha, rows, cols)
        elapsed += time.perf_counter() - t0
        total += n
        n = min(2 * n, 4096)
    tflops = total * 2 * S / elapsed / 1e12
    affinity = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info

        blas = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except ImportError:
        blas = affinity
    # Full-output oracle timings of the small square workloads (every output, float64).
    full = {}
    for Sf in (256, 2048):
        Af, SFAf, Bf, SFBf = G.gemm_square_inputs(Sf, Sf, Sf, seed=0)
        t0 = time.perf_counter()
        O.gemm(Af, SFAf, Bf, SFBf, alpha)
        dt = time.perf_counter() - t0
        full[str(Sf)] = {"s": round(dt, 4), "GFLOP/s": round(2 * Sf ** 3 / dt / 1e9, 2)}
    return {"value": tflops, "unit": "TFLOP/s", "cores": min(blas, affinity), "affinity_cores": affinity,
            "blas_threads": blas, "kind": "oracle",
            "sample": f"{total} sampled outputs of the {S}^3 GEMM (full K={S} dot products, float64), {elapsed:.1f} s",
            "full_output": full}


def run_ours(args):
    import torch

    rank, world = dist_setup(args)
    peaks = load_peaks()
    S = S_MAIN
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) if rank == 0 else None
    times, _ = time_gemm(S, args.steps, max(3, args.warmup), world, sampler)
    ms_rank = sum(times)
    ms_max = all_max(ms_rank, world)
    flops = 2.0 * S ** 3
    value = replicas_value(ms_max, args.steps, flops, world)
    avg_ms = statistics.mean(times)
    achieved = flops / (avg_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(value / world / P1_V1_8K_TFLOPS, 3), "dtype": "nvfp4 (e2m1 x ue4m3/16) -> fp32 acc -> bf16",
        "data": "synthetic",
        "config": {"workload": f"NVFP4 block-scaled GEMM M=N=K={S}, A MxK and B NxK K-major, E2M1 codes uniform, "
                               "one E4M3 scale per 16 K uniform over 2^-4..2^4, alpha U[0.25,4], BF16 out",
                   "M": S, "N": S, "K": S, "gemm_config": torch_config_name(S),
                   "l2": "flushed between timed iterations (512 MB write, untimed)",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(f"gemm_{S}"),
                     "peak_source": f"{peaks['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)"},
    }
    if rank == 0:
        line["clocks"] = sampler.summary() if sampler else None
        # the FP4 instruction ceiling measured on this GPU, beside the nominal peak
        ceil = bench_mma_ceiling()
        line["roofline"]["mma_ceiling"] = {"nvf4_tflops": ceil["nvf4"]["tflops"],
                                           "bf16_tflops": ceil["bf16"]["tflops"],
                                           "nvf4_over_bf16": ceil["nvf4_over_bf16"],
                                           "frac_of_nvf4_ceiling": round(achieved / ceil["nvf4"]["tflops"], 4)}
    if not args.quick:
        t16, _ = time_gemm(16384, 3, 2, world)
        line["gemm_16384"] = {"ms": round(statistics.mean(t16), 4),
                              "tflops": round(2 * 16384 ** 3 / (statistics.mean(t16) / 1e3) / 1e12, 1),
                              "frac_of_peak": round(2 * 16384 ** 3 / (statistics.mean(t16) / 1e3) / 1e12 / peak, 4)}
        # end to end on every rank (its own host buffers and GPU), timed by the slowest
        ms, h2d, d2h = time_gemm_e2e(S, 10, 3, world)
        ms_e2e = all_max(ms, world)
        line["e2e"] = {"value": round(replicas_value(ms_e2e, 1, flops, world), 1), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": world * h2d, "d2h_bytes_per_step": world * d2h,
                       "ms_per_step": round(ms_e2e, 3)}
        if rank == 0:
            line["w4a16"] = bench_w4a16(peaks)
            line["llm_w4a4"] = bench_llm(peaks)
            line["producers"] = bench_producers(peaks)
            line["cublaslt_same_operands"] = bench_cublaslt((S,))
            line["cpu_baseline"] = cpu_baseline_gemm(S)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def torch_config_name(S):
    import nvfp4_block_scaled_gb300 as nv

    return nv.gemm_config_name(nv.gemm_choose_config(S, S, S))


# ------------------------------------------------------------------ reference arm (the CPU oracle)

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    from oracle import nvfp4_oracle as O
    from synthetic import generators as G

    S = S_MAIN
    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0)
    alpha = G.alpha_uniform(0)
    rng = np.random.default_rng(11)
    n = 256  # sampled outputs per step (full K-length dot products)
    for _ in range(args.warmup):
        O.gemm_at(A, SFA, B, SFB, alpha, rng.integers(0, S, n), rng.integers(0, S, n))
    times = []
    for _ in range(args.steps):
        rows, cols = rng.integers(0, S, n), rng.integers(0, S, n)
        t0 = time.perf_counter()
        O.gemm_at(A, SFA, B, SFB, alpha, rows, cols)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * n * 2 * S / total / 1e12
    try:
        from threadpoolctl import threadpool_info

        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except ImportError:
        cores = len(os.sched_getaffinity(0))
    sample = f"{n} sampled outputs of the {S}^3 GEMM per step (float64 dot products over K={S})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"NVFP4 block-scaled GEMM M=N=K={S} (oracle on sampled outputs)", "M": S, "N": S,
                   "K": S},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_only(args):
    import torch  # noqa: F401

    peaks = load_peaks()
    if args.only == "w4a16":
        shapes = None
        if args.w4a16_shapes:
            shapes = []
            for item in args.w4a16_shapes.split(","):
                N, K, M = (int(v) for v in item.lower().split("x"))
                shapes.append((N, K, (M,)))
        out = bench_w4a16(peaks, shapes)
    elif args.only == "llm":
        shapes = None
        if args.llm_shapes:
            shapes = [tuple(int(v) for v in item.lower().split("x")) for item in args.llm_shapes.split(",")]
        out = bench_llm(peaks, tuple(int(c) for c in args.llm_configs.split(",")), shapes)
    elif args.only == "mma_ceiling":
        out = bench_mma_ceiling()
    elif args.only == "cublaslt":
        out = bench_cublaslt((S_MAIN, 16384))
    else:
        out = bench_producers(peaks)
    print(json.dumps({"only": args.only, "results": out}), flush=True)


def main():
    args = parse()
    if args.only is not None and args.impl == "ours":
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
