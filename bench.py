"""Benchmark of the W8A8 FP8 block-scaled linear layer on GB300.

One step = one pass of the whole hot path (per-token-group quantisation of
the activations, then the block-scaled GEMM) over one batch of the workload.
Default workload: "decode_block32" -- M in {1, 4, 16, 64} tokens against one
N=7168, K=2048 weight with [32,32] UE8M0 blocks and UE8M0 activation groups of
32, i.e. four quantise+GEMM pairs per step.  The metric is the GEMM family's
algorithmic bytes per second (Aq + As + Wq + Ws + D per GEMM, plus the quant
bytes x + codes + scales), with TFLOP/s alongside.

Timing: inputs resident in HBM; CUDA graphs of whole steps replayed on one
stream between CUDA events; the weights rotate over enough copies to exceed
twice the L2 size, so every step streams its weights from HBM.  `e2e` times
the same steps through the public API with the activation copied in from
pinned host memory and D read back to the host inside the timed region: each
step replays one CUDA graph holding the host-to-device copy of the step's
activations (one pinned buffer), the quantisation and GEMM calls of every linear
(largest M first) and each linear's device-to-host copy, issued on a copy stream
as soon as its GEMM is done, then waits for it on the host (the way a decode
loop runs).  `e2e.eager_ms_per_step` is the
same step issued call by call from Python.

`--impl reference` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload, on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fp8_block_scaled_sgq_gb300 import synth  # noqa: E402

METRIC = "block-scaled FP8 GEMM TFLOPS & GB/s vs GB300 roofline, M=1–8192; quant GB/s"
L2_BYTES = 129 * 2 ** 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The sources each workload's dominant kernel is compiled and planned from:
# its translation unit, the headers that reach it, and the host code that picks
# its tiles, splits and grid.  A workload not listed here hashes every source.
KERNEL_SOURCES = {
    "decode_block32": ["gemm_b32_32.cu", "gemm_kernel.cuh", "ptx.cuh", "quant_math.cuh", "sgq_internal.h",
                       "gemm_host.cu"],
}


def kernel_source_digest(workload: str | None = None) -> str:
    """sha256 over the CUDA sources of `workload`'s dominant kernel (all
    sources when it has no list), to tie ncu counters to the build they came from."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "fp8_block_scaled_sgq_gb300", "csrc")
    names = KERNEL_SOURCES.get(workload) or [n for n in os.listdir(d) if n.endswith((".cu", ".cuh", ".h"))]
    for name in sorted(names):
        h.update(name.encode())
        h.update(open(os.path.join(d, name), "rb").read())
    inc = os.path.join(ROOT, "include", "sgq.h")
    h.update(open(inc, "rb").read())
    return h.hexdigest()[:16]


# DRAM bytes (read + write) per launch of the dominant kernel, recorded by the
# profiling step (one ncu capture per workload) with the digest of the kernel
# sources it was taken on; a record for other sources reads as null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def measured_traffic(workload: str):
    """Bytes per launch for `workload` from the traffic record, or None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest = kernel_source_digest(workload)
    for line in open(TRAFFIC_FILE):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == workload and f[1] == digest:
            return int(f[2])
    return None


def workload_unit(cases):
    """("TFLOP/s", 1e12, "flops") for tensor-bound workloads, else ("GB/s", 1e9, "bytes")."""
    pk = peaks()
    ridge = 2.0 * pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    flops = sum(c.flops() for c in cases)
    gbytes = sum(c.gemm_bytes() for c in cases)
    return ("TFLOP/s", 1e12, "flops") if flops / gbytes > ridge else ("GB/s", 1e9, "bytes")


# ----------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str | None):
        self.index, self.path, self.proc = index, path, None

    def __enter__(self):
        try:
            out = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=out, stderr=subprocess.DEVNULL, text=True)
            self._out = out
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            o, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            o, _ = self.proc.communicate()
        if self.path:
            self._out.close()
            self.text = open(self.path).read()
        else:
            self.text = o or ""
        return False

    def summary(self):
        rows = []
        for line in self.text.strip().splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, _, flags in rows:
            for n, v in zip(names, flags):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------- our arm

def n_rotations(nbytes: float) -> int:
    """Copies of an operand of `nbytes` whose cycle exceeds twice the L2 size."""
    return max(2, math.ceil(2 * L2_BYTES / nbytes) + 1)


class GraphTimer:
    """CUDA graphs of library calls on one stream, timed with CUDA events.

    Each graph holds `reps` calls (call i uses operand set i % len(calls)); it is
    replayed once to warm up, then once between two events.  `launches` counts
    the library's kernels of every replay made (the graph's kernels, counted
    from the library's launch counter during capture, times its replays)."""

    def __init__(self, sgq, stream):
        self.sgq, self.stream, self.launches = sgq, stream, 0

    def capture(self, calls, reps):
        g = torch.cuda.CUDAGraph()
        n0 = self.sgq.sgq_launch_count()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                sp = torch.cuda.current_stream().cuda_stream
                for i in range(reps):
                    calls[i % len(calls)](sp)
        g.kernels = self.sgq.sgq_launch_count() - n0
        return g

    def replay_ms(self, g, reps, ws_=1):
        """(warm-up replay) then one timed replay; ms per call."""
        with torch.cuda.stream(self.stream):
            g.replay()
        self.stream.synchronize()
        barrier(ws_)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
        self.stream.synchronize()
        torch.cuda.synchronize()
        barrier(ws_)
        self.launches += 2 * g.kernels
        return e0.elapsed_time(e1) / reps

    def time(self, calls, reps, ws_=1):
        g = self.capture(calls, reps)
        ms = self.replay_ms(g, reps, ws_)
        del g
        return ms


def roofline_frac(flops: float, nbytes: float, us: float):
    """(bound, fraction) of min(FP8 peak, arithmetic intensity x HBM peak)."""
    pk = peaks()
    fp8 = 2.0 * pk["bf16_tflops"] * 1e12
    t_fp8, t_hbm = flops / fp8, nbytes / (pk["hbm_gbs"] * 1e9)
    return ("fp8" if t_fp8 > t_hbm else "hbm"), max(t_fp8, t_hbm) / (us * 1e-6)


# UE8M0 GEMMs from this M on, with a wave of 256 x 224 tiles, run on UE8M0
# scale bytes: the two-accumulator tiles read them directly (other plans would
# widen them to fp32 first, an extra step).
E8_MIN_M = 2048


def sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def gemm_cases(sgq, timer, device, reps, names):
    """The metric's GEMM configurations: the M = 1..8192 sweep (two weight
    shapes, both recipes) and the two prefill shapes; each timed as the GEMM
    alone and as quantisation + GEMM back to back ("pair")."""
    rows = []
    groups = {}
    for name in names:
        for c in synth.WORKLOADS[name]:
            groups.setdefault((c.N, c.K, c.blk_n, c.blk_k, c.ue8m0, c.seed), []).append(c)
    for (N, K, bn, bk, ue, seed), cs in groups.items():
        w = synth.weight(N, K, seed).to(device)
        wq0, ws0 = sgq.quant_weight_block(w, bn, bk, ue)
        del w
        wbytes = N * K + 4 * math.ceil(N / bn) * (K // bk)
        wrot = [(wq0, ws0)] + [(wq0.clone(), ws0.clone()) for _ in range(n_rotations(wbytes) - 1)]
        # UE8M0 bytes of the weight scales, converted once (the load-time step)
        werot = None
        for c in cs:
            x = c.x().to(device)
            # UE8M0 scales at prefill sizes travel as bytes: the quantiser
            # writes them, the GEMM reads them as they are (a quarter of the
            # fp32 scale bytes per stage, no conversion).  Elsewhere fp32 scales.
            e8 = (c.ue8m0 and c.M >= E8_MIN_M
                  and math.ceil(c.M / 256) * math.ceil(c.N / 224) >= sm_count())
            if e8 and werot is None:
                werot = [sgq.scales_to_ue8m0(ws) for _, ws in wrot]
            xq = torch.empty((c.M, c.K), dtype=torch.uint8, device=device)
            xs = torch.empty((c.M, c.K // c.group), dtype=torch.uint8 if e8 else torch.float32, device=device)
            d = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=device)
            sp0 = timer.stream.cuda_stream
            if e8:
                sgq.sgq_quant_token_group_ue8m0(x, c.M, c.K, c.group, xq, xs, sp0)
            else:
                sgq.sgq_quant_token_group(x, c.M, c.K, c.group, int(c.ue8m0), xq, xs, sp0)

            # the configurations' scales are UE8M0: the caller may promise powers of two
            fl = sgq.SGQ_GEMM_SCALES_POW2 if c.ue8m0 else sgq.SGQ_GEMM_DEFAULT

            def gemm(sp, r, c=c, xq=xq, xs=xs, d=d, fl=fl, e8=e8):
                if e8:
                    sgq.sgq_fp8_block_gemm_ue8m0(xq, xs, wrot[r][0], werot[r], d, c.M, c.N, c.K, c.blk_n, c.blk_k,
                                                 0, sp)
                else:
                    sgq.sgq_fp8_block_gemm_ex(xq, xs, wrot[r][0], wrot[r][1], d, c.M, c.N, c.K, c.blk_n, c.blk_k,
                                              fl, sp)

            def pair(sp, r, c=c, x=x, xq=xq, xs=xs, d=d, e8=e8):
                if e8:
                    sgq.sgq_quant_token_group_ue8m0(x, c.M, c.K, c.group, xq, xs, sp)
                else:
                    sgq.sgq_quant_token_group(x, c.M, c.K, c.group, int(c.ue8m0), xq, xs, sp)
                gemm(sp, r)
            sb = 1 if e8 else 4
            with torch.cuda.stream(timer.stream):
                gemm(sp0, 0)   # outside the capture: any first-use set-up happens here
            timer.stream.synchronize()
            for path, fn in (("gemm", gemm), ("pair", pair)):
                calls = [lambda sp, r=r, fn=fn: fn(sp, r) for r in range(len(wrot))]
                ms = timer.time(calls, reps)
                us = ms * 1e3
                nbytes = c.gemm_bytes(sb) + (c.quant_bytes(sb) if path == "pair" else 0.0)
                bound, frac = roofline_frac(c.flops(), nbytes, us)
                rows.append({"case": c.name, "path": path, "M": c.M, "N": c.N, "K": c.K,
                             "recipe": [1, c.blk_n, c.blk_k],
                             "flags": ("scales_pow2" if fl else "default") + (" ue8m0_bytes" if e8 else ""),
                             "us": round(us, 3),
                             "tflops": round(c.flops() / us / 1e6, 2), "gbs": round(nbytes / us / 1e3, 1),
                             "bound": bound, "frac": round(frac, 4)})
            del x, xq, xs, d
        del werot
        del wrot, wq0, ws0
        torch.cuda.empty_cache()
    return rows


QUANT_SHAPES = [(4096, 7168), (8192, 7168)]


def quant_cases(sgq, timer, device, reps):
    """sgq_quant_token_group alone at prefill sizes, both group sizes, UE8M0:
    GB/s of 2 B read + 1 B code + 4/g B scale per element (inputs rotated over
    more than twice the L2 size)."""
    rows = []
    for M, K in QUANT_SHAPES:
        x0 = synth.activation(M, K, seed=7).to(device)
        xr = [x0] + [x0.clone() for _ in range(n_rotations(2 * M * K) - 1)]
        for g in (128, 32):
            xq = torch.empty((M, K), dtype=torch.uint8, device=device)
            xs = torch.empty((M, K // g), dtype=torch.float32, device=device)
            calls = [lambda sp, x=x, g=g, xq=xq, xs=xs: sgq.sgq_quant_token_group(x, M, K, g, 1, xq, xs, sp)
                     for x in xr]
            us = timer.time(calls, reps) * 1e3
            nbytes = 2 * M * K + M * K + 4 * M * K / g
            rows.append({"case": f"quant_token_group_M{M}_K{K}_g{g}", "path": "quant", "M": M, "K": K,
                         "group": g, "us": round(us, 3), "gbs": round(nbytes / us / 1e3, 1), "bound": "hbm",
                         "frac": round(nbytes / us / 1e3 / peaks()["hbm_gbs"], 4)})
            del xq, xs
        # the byte-output quantiser (UE8M0 scale bytes), group 32
        xq = torch.empty((M, K), dtype=torch.uint8, device=device)
        xe = torch.empty((M, K // 32), dtype=torch.uint8, device=device)
        calls = [lambda sp, x=x: sgq.sgq_quant_token_group_ue8m0(x, M, K, 32, xq, xe, sp) for x in xr]
        us = timer.time(calls, reps) * 1e3
        nbytes = 2 * M * K + M * K + M * K / 32
        rows.append({"case": f"quant_token_group_ue8m0_M{M}_K{K}_g32", "path": "quant", "M": M, "K": K,
                     "group": 32, "us": round(us, 3), "gbs": round(nbytes / us / 1e3, 1), "bound": "hbm",
                     "frac": round(nbytes / us / 1e3 / peaks()["hbm_gbs"], 4)})
        del xq, xe, xr, x0
        torch.cuda.empty_cache()
    return rows


def build_problem(cases, device, n_rot):
    import fp8_block_scaled_sgq_gb300 as sgq
    c0 = cases[0]
    w = c0.w().to(device)
    wq, ws = sgq.quant_weight_block(w, c0.blk_n, c0.blk_k, c0.ue8m0)
    del w
    wrot = [(wq, ws)] + [(wq.clone(), ws.clone()) for _ in range(n_rot - 1)]
    per = []
    for c in cases:
        x = c.x().to(device)
        xq = torch.empty((c.M, c.K), dtype=torch.uint8, device=device)
        xs = torch.empty((c.M, c.K // c.group), dtype=torch.float32, device=device)
        d = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=device)
        per.append((c, x, xq, xs, d))
    return wrot, per


def step_fn(sgq, per, wsets, stream, gemm_only=False):
    """One step: quantisation + GEMM for every linear; linear j uses weight set
    wsets[j] (each GEMM of a step streams its own copy of the weights)."""
    for (c, x, xq, xs, d), (wq, ws) in zip(per, wsets):
        if not gemm_only:
            sgq.sgq_quant_token_group(x, c.M, c.K, c.group, c.ue8m0, xq, xs, stream)
        sgq.sgq_fp8_block_gemm(xq, xs, wq, ws, d, c.M, c.N, c.K, c.blk_n, c.blk_k, stream)


def fused_step_fn(sgq, per, wsets, stream):
    """The same layer through sgq_fp8_block_linear (one kernel per case at
    decode-sized M; codes and scales stay on chip)."""
    for (c, x, _, _, d), (wq, ws) in zip(per, wsets):
        sgq.sgq_fp8_block_linear(x, int(c.ue8m0), wq, ws, d, c.M, c.N, c.K, c.blk_n, c.blk_k, None, None, stream)


def fusable(cases):
    return all(c.M <= 64 and (c.K // c.blk_k) % 4 == 0 and c.K // c.blk_k >= (8 if c.blk_k == 128 else 16)
               for c in cases)


EXTRA_GEMM_WORKLOADS = ("sweep", "prefill_block128", "prefill_block32")


def run_ours(args, ws_, rank, local):
    import fp8_block_scaled_sgq_gb300 as sgq
    from fp8_block_scaled_sgq_gb300 import build as sgq_build
    if not os.path.exists(sgq_build.LIB):
        raise SystemExit("libsgq.so is not built; run __graft_entry__.build() first")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(ws_, "nccl")
    cases = synth.WORKLOADS[args.workload]
    if len({(c.N, c.K, c.blk_n, c.blk_k) for c in cases}) != 1:
        raise SystemExit("workload mixes weight shapes")
    c0 = cases[0]
    wbytes = c0.N * c0.K + 4 * math.ceil(c0.N / c0.blk_n) * (c0.K // c0.blk_k)
    n_rot = n_rotations(wbytes)
    wrot, per = build_problem(cases, device, n_rot)
    stream = torch.cuda.Stream(device)
    sptr = stream.cuda_stream
    timer = GraphTimer(sgq, stream)
    nl = len(per)

    def wsets(i):
        """Weight copies of step i: one per linear, cycling through all copies."""
        return [wrot[(i * nl + j) % n_rot] for j in range(nl)]

    gemm_bytes = sum(c.gemm_bytes() for c in cases)
    quant_bytes = sum(c.quant_bytes() for c in cases)
    step_bytes = gemm_bytes + quant_bytes
    step_flops = sum(c.flops() for c in cases)

    # warm-up outside capture (the first split-K call allocates the workspace)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step_fn(sgq, per, wsets(i), sptr)
    stream.synchronize()
    if sgq.sgq_device_status(sptr) != 0:
        raise SystemExit("device status not OK after warm-up")

    steps = args.steps
    graph = timer.capture([lambda sp, i=i: step_fn(sgq, per, wsets(i), sp) for i in range(n_rot)], steps)
    fused_graph = (timer.capture([lambda sp, i=i: fused_step_fn(sgq, per, wsets(i), sp) for i in range(n_rot)],
                                 steps) if fusable(cases) else None)
    # per linear: its GEMM alone, back to back, each call on the next weight copy
    case_graphs = [timer.capture([lambda sp, j=j, r=r: step_fn(sgq, per[j:j + 1], [wrot[r]], sp, gemm_only=True)
                                  for r in range(n_rot)], steps) for j in range(nl)]

    def preheat(seconds):
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            with torch.cuda.stream(stream):
                graph.replay()
            stream.synchronize()

    reps = max(20, steps)
    extra = []
    with ClockSampler(local, os.path.join(args.out_dir, f"clocks_rank{rank}.csv") if args.out_dir else None) as cs:
        preheat(args.preheat)
        ms_step = timer.replay_ms(graph, steps, ws_)
        ms_case = [timer.replay_ms(cg, steps, ws_) for cg in case_graphs]
        ms_fused = timer.replay_ms(fused_graph, steps, ws_) if fused_graph is not None else None
        if args.cases == "all" and ws_ == 1:
            extra = gemm_cases(sgq, timer, device, reps, EXTRA_GEMM_WORKLOADS)
            extra += quant_cases(sgq, timer, device, reps)
    clocks = cs.summary()
    gpu_launches = timer.launches
    ms_step = max_over_ranks(ms_step, ws_, device)
    ms_case = [max_over_ranks(t, ws_, device) for t in ms_case]
    ms_gemm = sum(ms_case)
    if ms_fused is not None:
        ms_fused = max_over_ranks(ms_fused, ws_, device)
    del graph, fused_graph, case_graphs

    # end to end through the public API: H2D of x, quant + GEMM, D2H of D, every
    # step.  The step's activations sit in one buffer (one H2D copy); each
    # linear's output goes back on a copy stream as soon as its GEMM is done,
    # largest first, so that the copies overlap the remaining linears.
    order = sorted(range(len(per)), key=lambda j: -per[j][0].M)
    x_sizes = [x.numel() for _, x, _, _, _ in per]
    d_sizes = [d.numel() for *_, d in per]
    hx = torch.cat([x.reshape(-1).cpu() for _, x, _, _, _ in per]).pin_memory()
    hd = torch.empty(sum(d_sizes), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=device)
    dd = torch.empty(sum(d_sizes), dtype=torch.bfloat16, device=device)
    per_e2e, hd_parts, ox, od = [], [], 0, 0
    for (c, x, xq, xs, d), nx, nd in zip(per, x_sizes, d_sizes):
        per_e2e.append((c, dx[ox:ox + nx].view(x.shape), xq, xs, dd[od:od + nd].view(d.shape)))
        hd_parts.append(hd[od:od + nd].view(d.shape))
        ox, od = ox + nx, od + nd
    per = [per_e2e[j] for j in order]
    hd_parts = [hd_parts[j] for j in order]
    e2e_wsets = wsets
    wsets = lambda i: [e2e_wsets(i)[j] for j in order]   # noqa: E731
    copy_stream = torch.cuda.Stream()
    events = [torch.cuda.Event() for _ in range(len(per) + 1)]
    hx, hd = (hx, dx), (hd_parts, copy_stream, events)
    for i in range(args.warmup):
        _e2e_step(sgq, per, wsets(i), hx, hd, stream)   # e2e warm-up
        stream.synchronize()
    barrier(ws_)
    t0 = time.perf_counter()
    for i in range(steps):
        _e2e_step(sgq, per, wsets(i), hx, hd, stream)
        stream.synchronize()
    t_eager = max_over_ranks((time.perf_counter() - t0) / steps, ws_, device)
    e2e_mode = "graph"
    try:
        e2e_graphs = []
        for r in range(n_rot):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    _e2e_step(sgq, per, wsets(r), hx, hd, torch.cuda.current_stream())
            e2e_graphs.append(g)
    except RuntimeError as e:   # a PyTorch that cannot capture pinned-memory copies
        print(f"e2e graph capture failed ({e}); timing the eager step", file=sys.stderr)
        e2e_mode, e2e_graphs = "eager", None
        torch.cuda.synchronize()
    if e2e_graphs is not None:
        for i in range(args.warmup):
            with torch.cuda.stream(stream):
                e2e_graphs[i % n_rot].replay()
            stream.synchronize()
        barrier(ws_)
        t0 = time.perf_counter()
        for i in range(steps):
            with torch.cuda.stream(stream):
                e2e_graphs[i % n_rot].replay()
            stream.synchronize()   # D is on the host before the next step
        t_e2e = max_over_ranks((time.perf_counter() - t0) / steps, ws_, device)
    else:
        t_e2e = t_eager
    if sgq.sgq_device_status(sptr) != 0:
        raise SystemExit("device status not OK after timing")
    h2d = sum(c.M * c.K * 2 for c in cases)
    d2h = sum(c.M * c.N * 2 for c in cases)

    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]          # measured bf16 burst x nominal fp8:bf16 ratio
    gemm_gbs = gemm_bytes / (ms_gemm * 1e-3) / 1e9
    gemm_tf = step_flops / (ms_gemm * 1e-3) / 1e12
    ridge = fp8_peak * 1e12 / (pk["hbm_gbs"] * 1e9)   # FLOP per byte
    tensor_bound = step_flops / gemm_bytes > ridge
    if tensor_bound:
        unit, scale, to_unit = "TFLOP/s", 1e12, step_flops
        roof = {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(gemm_tf / fp8_peak, 4), "traffic": measured_traffic(args.workload),
                "kernel": "fp8_block_gemm_kernel (128x256 tiles)",
                "peak_source": f"{pk['source']} bf16 burst x 2 (fp8:bf16 nominal)"}
    else:
        unit, scale, to_unit = "GB/s", 1e9, step_bytes
        roof = {"bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(gemm_gbs / pk["hbm_gbs"], 4), "traffic": measured_traffic(args.workload),
                "kernel": "block-scaled GEMM, decode tiles (swap-AB, split-K)", "peak_source": pk["source"]}
    value = ws_ * to_unit / (ms_step * 1e-3) / scale
    per_case = []
    for c, t in zip(cases, ms_case):
        us = t * 1e3
        bound, frac = roofline_frac(c.flops(), c.gemm_bytes(), us)
        per_case.append({"M": c.M, "us": round(us, 3), "gbs": round(c.gemm_bytes() / us / 1e3, 1),
                         "tflops": round(c.flops() / us / 1e6, 2), "bound": bound, "frac": round(frac, 4)})
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": unit,
        "n_gpus": ws_,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8e4m3 x fp8e4m3 -> fp32 accumulate -> bf16",
        "data": "synthetic (seeded; x ~ N(0,1), W ~ N(0,0.02) bf16, quantised on the GPU)",
        "config": {"workload": args.workload, "M": [c.M for c in cases], "N": c0.N, "K": c0.K,
                   "recipe": [1, c0.blk_n, c0.blk_k], "ue8m0": c0.ue8m0,
                   "l2": f"each GEMM of a step streams its own weight copy; copies rotate over {n_rot} "
                         f"({n_rot * wbytes / 2**20:.0f} MiB > 2x L2)",
                   "parallelism": f"replicas x{ws_}"},
        "tflops": round(ws_ * step_flops / (ms_step * 1e-3) / 1e12, 3),
        "gbs": round(ws_ * step_bytes / (ms_step * 1e-3) / 1e9, 2),
        "gemm": {"ms_per_step": round(ms_gemm, 5), "gbs": round(gemm_gbs, 1),
                 "tflops": round(gemm_tf, 3), "per_case": per_case},
        "roofline": roof,
        "e2e": {"value": round(ws_ * to_unit / t_e2e / scale, 2), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(t_e2e * 1e3, 4), "mode": e2e_mode,
                "eager_ms_per_step": round(t_eager * 1e3, 4)},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if ms_fused is not None:
        # algorithmic bytes of the fused layer: x, weights, D (no Aq/As round trip)
        fused_bytes = sum(2 * c.M * c.K + c.N * c.K + 4 * math.ceil(c.N / c.blk_n) * (c.K // c.blk_k)
                          + 2 * c.M * c.N for c in cases)
        result["fused"] = {"entry": "sgq_fp8_block_linear", "ms_per_step": round(ms_fused, 5),
                           "gbs": round(ws_ * fused_bytes / (ms_fused * 1e-3) / 1e9, 2),
                           "launches_per_step": len(cases)}
    if extra:
        result["cases"] = extra
        result["cases_timing"] = (f"each case: a CUDA graph of {reps} calls (weights, or the quantiser's "
                                  "input, rotated over more than twice the L2 size) after one warm-up replay; "
                                  "fractions of min(FP8 peak, AI x HBM peak), FP8 = 2 x measured bf16 burst")
        pre = {r["case"]: r for r in extra if r["path"] == "gemm"}
        big = pre.get("sweep_N24576_K1536_b128_M8192"), pre.get("sweep_N1536_K7168_b128_M8192")
        result["headline"] = {
            "prefill_gemm": [{"case": r["case"], "tflops": r["tflops"], "frac_fp8": r["frac"]}
                             for r in (pre.get("prefill_block128"), pre.get("prefill_block32")) + big if r],
            "decode_gemm": {"M": [c.M for c in cases], "gbs": round(gemm_gbs, 1),
                            "frac_hbm": round(gemm_gbs / pk["hbm_gbs"], 4)},
            "quant": [{"case": r["case"], "gbs": r["gbs"], "frac_hbm": r["frac"]}
                      for r in extra if r["path"] == "quant"],
        }
    return result


def _e2e_step(sgq, per, wsets, hx, hd, stream):
    """One host-to-device copy of the step's activations, then quantisation +
    GEMM for every linear on `stream`, each linear's output copied to the host
    on a copy stream once its GEMM is done; the copy stream joins `stream` at
    the end (the caller waits on `stream`).  hx: (pinned host buffer, device
    buffer), the device views of `per` lie in it; hd: (pinned host views of
    each linear's output, in `per`'s order, copy stream, one event per linear
    and one for the join)."""
    hd_parts, copy_stream, events = hd
    with torch.cuda.stream(stream):
        hx_host, hx_dev = hx
        hx_dev.copy_(hx_host, non_blocking=True)
        for (c, x, xq, xs, d), (wq, ws), h, done in zip(per, wsets, hd_parts, events):
            sgq.sgq_quant_token_group(x, c.M, c.K, c.group, c.ue8m0, xq, xs, stream.cuda_stream)
            sgq.sgq_fp8_block_gemm(xq, xs, wq, ws, d, c.M, c.N, c.K, c.blk_n, c.blk_k, stream.cuda_stream)
            done.record(stream)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                h.copy_(d, non_blocking=True)
        events[-1].record(copy_stream)
        stream.wait_event(events[-1])


# ----------------------------------------------------------------- oracle timing

def oracle_step(cases, data, rows_frac):
    """One pass of the oracle over a sample: quantise x and evaluate the GEMM on
    the first ceil(rows_frac * M) rows of each case."""
    import oracle
    done = {"bytes": 0.0, "flops": 0.0}
    for c, x, wq, ws in data:
        m = max(1, math.ceil(rows_frac * c.M))
        xs_ = x[:m]
        aq, a_s = oracle.quant_token_group(xs_, c.group, c.ue8m0)
        oracle.gemm(aq, a_s, wq, ws, c.blk_n, c.blk_k, with_bound=False)
        cc = synth.Case(c.name, m, c.N, c.K, c.blk_n, c.blk_k, c.ue8m0)
        done["bytes"] += cc.gemm_bytes() + cc.quant_bytes()
        done["flops"] += cc.flops()
    return done


def oracle_data(cases):
    import oracle
    c0 = cases[0]
    wq, ws = oracle.quant_weight_block(c0.w(), c0.blk_n, c0.blk_k, c0.ue8m0)
    return [(c, c.x(), wq, ws) for c in cases]


def _oracle_rate(cases, data, key, budget_s, max_frac):
    """(work per second, passes, row fraction, seconds) of the oracle on a bounded sample."""
    t0 = time.perf_counter()
    first = oracle_step(cases, data, max_frac)
    step_s = time.perf_counter() - t0
    frac = max_frac if step_s < budget_s / 2 else max_frac * budget_s / 2 / step_s
    b = first[key] if frac == max_frac else 0.0
    reps = 1 if frac == max_frac else 0
    t0 = time.perf_counter() if frac != max_frac else t0
    while time.perf_counter() - t0 < budget_s and reps < 20:
        b += oracle_step(cases, data, frac)[key]
        reps += 1
    dt = time.perf_counter() - t0
    return b / dt, reps, frac, dt


def cpu_baseline(cases, budget_s=12.0, max_frac=1.0):
    """The oracle on all host cores, then on one core (a shorter sample)."""
    import oracle
    unit, scale, key = workload_unit(cases)
    data = oracle_data(cases)
    cores = oracle.num_threads()
    rate, reps, frac, dt = _oracle_rate(cases, data, key, budget_s, max_frac)
    oracle.set_num_threads(1)
    try:
        rate1, reps1, frac1, dt1 = _oracle_rate(cases, data, key, budget_s / 2, max_frac)
    finally:
        oracle.set_num_threads(cores)
    return {"value": round(rate / scale, 6), "unit": unit, "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} pass(es) over the first {frac:.3g} of the rows of each GEMM of the "
                      f"workload (quantise + fp64 GEMM), {dt:.1f} s",
            "single_core": {"value": round(rate1 / scale, 6), "cores": 1,
                            "sample": f"{reps1} pass(es) over the first {frac1:.3g} of the rows, {dt1:.1f} s"}}


def run_reference(args, ws_, rank):
    import oracle
    if ws_ > 1:
        dist_init(ws_, "gloo")
        barrier(ws_)
        if rank != 0:
            return None
    cases = synth.WORKLOADS[args.workload]
    unit, scale, key = workload_unit(cases)
    data = oracle_data(cases)
    frac = min(1.0, 16.0 / max(c.M for c in cases))   # probe on a small slice first
    t0 = time.perf_counter()
    oracle_step(cases, data, frac)
    probe = time.perf_counter() - t0
    # bound each step to ~2 s of CPU work
    frac = min(1.0, frac * 2.0 / max(probe, 1e-9))
    for _ in range(args.warmup):
        oracle_step(cases, data, frac)
    t0 = time.perf_counter()
    b = 0.0
    for _ in range(args.steps):
        b += oracle_step(cases, data, frac)[key]
    dt = time.perf_counter() - t0
    v = b / dt / scale
    sample = f"first {frac:.3g} of the rows of each GEMM of the workload per step"
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit, "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same recipe)",
            "config": {"workload": args.workload, "M": [c.M for c in cases], "N": cases[0].N, "K": cases[0].K,
                       "recipe": [1, cases[0].blk_n, cases[0].blk_k], "ue8m0": cases[0].ue8m0},
            "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_block32", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--preheat", type=float, default=1.5,
                    help="seconds of identical load before the timed region (clock sampling)")
    ap.add_argument("--out-dir", default=None, help="directory for clock samples")
    ap.add_argument("--cases", choices=["all", "none"], default="all",
                    help="all: also time the M=1..8192 sweep, the prefill GEMMs and the quantiser alone")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws_, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws_, rank)
        if res is not None and rank == 0:
            print(json.dumps(res))
        return
    res = run_ours(args, ws_, rank, local)
    if rank == 0:
        if ws_ == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(synth.WORKLOADS[args.workload])
        print(json.dumps(res))
    if ws_ > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
