"""Times one library entry point on one shape and prints a JSON line.

    python -m fp8_block_scaled_sgq_gb300.measure PATH M N K [--blk B] [--reps R]

PATH is one of
  quant_per_token   sgq_quant_per_token on x [M, K]            (GB/s: 2 B in + 1 B code per element + 4 B per row)
  quant_per_tensor  sgq_quant_per_tensor, dynamic, on x [M, K] (GB/s: 2 B in + 1 B code per element)
  quant_v2          sgq_quant_token_group_v2, fused SiLU-and-mul, x [1, M, 2K] -> [1, M, K], group --blk, UE8M0
                    (GB/s: 4 B in + 1 B code per output element + 4 B per group)
  scaled_mm         sgq_fp8_scaled_mm, per-row x per-column scales, bias   (TFLOP/s and GB/s)
  block_gemm        sgq_fp8_block_gemm with [B, B] blocks, UE8M0           (TFLOP/s and GB/s)
  linear            sgq_fp8_block_linear with [B, B] blocks, UE8M0         (GB/s of x + W + D)
  pair              sgq_quant_token_group then sgq_fp8_block_gemm, back to back on one stream
                    (programmatic dependent launch), [B, B] blocks, UE8M0  (TFLOP/s; GB/s of the
                    quantiser's and the GEMM's algorithmic bytes)

The metric's own configurations (the M = 1..8192 sweep, the prefill GEMMs and
the quantiser at prefill sizes) are timed by bench.py; this times the other
entry points, one shape at a time.

Timing: CUDA events around one replay of a CUDA graph holding `reps` calls on
one stream, after a warm-up replay; weights (and, for the quantisers, inputs)
rotate over enough copies to exceed twice the L2 size, so they come from HBM.
Inputs are seeded synthetic (x ~ N(0,1), W ~ N(0, 0.02)).
"""
from __future__ import annotations

import argparse
import json
import math

import torch

from . import binding, synth

L2_BYTES = 129 * 2 ** 20


PATHS = ["quant_per_token", "quant_per_tensor", "quant_v2", "scaled_mm", "block_gemm", "linear", "pair"]


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("path", choices=PATHS)
    ap.add_argument("M", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("K", type=int)
    ap.add_argument("--blk", type=int, default=128)
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    print(json.dumps(measure(args.path, args.M, args.N, args.K, args.blk, args.reps)), flush=True)


def measure(path: str, M: int, N: int, K: int, blk: int, reps: int) -> dict:
    args = argparse.Namespace(path=path, reps=reps)
    dev = torch.device("cuda:0")
    st = torch.cuda.Stream()
    s = st.cuda_stream
    quant = args.path.startswith("quant")
    rot_bytes = (M * K * (4 if args.path == "quant_v2" else 2)) if quant else N * K
    n_rot = max(2, math.ceil(2 * L2_BYTES / rot_bytes) + 1)
    calls = []
    if quant:
        W = 2 * K if args.path == "quant_v2" else K
        xr = [synth.activation(M, W, seed=i).to(dev) for i in range(min(n_rot, 4))]
        xr = [xr[i % len(xr)].clone() for i in range(n_rot)]
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sc = torch.empty((max(M, 4),), dtype=torch.float32, device=dev)
        sc2 = torch.empty((M, K // blk), dtype=torch.float32, device=dev)
        for r in range(n_rot):
            if args.path == "quant_per_token":
                calls.append(lambda sp, r=r: binding.sgq_quant_per_token(xr[r], M, K, xq, sc, sp))
            elif args.path == "quant_v2":
                calls.append(lambda sp, r=r: binding.sgq_quant_token_group_v2(xr[r], 1, M, K, blk, 1, 1, None, xq,
                                                                             sc2, sp))
            else:
                calls.append(lambda sp, r=r: binding.sgq_quant_per_tensor(xr[r], M * K, 0, xq, sc, sp))
        moved = {"quant_per_token": M * K * 3 + 4 * M, "quant_per_tensor": M * K * 3 + 4,
                 "quant_v2": M * K * 5 + 4 * M * (K // blk)}[args.path]
        flops = 0
    else:
        x = synth.activation(M, K, seed=1).to(dev)
        w = synth.weight(N, K, seed=2).to(dev)
        d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if args.path == "scaled_mm":
            wq0 = torch.empty((N, K), dtype=torch.uint8, device=dev)
            sb0 = torch.empty((N,), dtype=torch.float32, device=dev)
            binding.sgq_quant_per_token(w, N, K, wq0, sb0, s)
            aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
            sa = torch.empty((M,), dtype=torch.float32, device=dev)
            binding.sgq_quant_per_token(x, M, K, aq, sa, s)
            bias = synth.activation(1, N, seed=3).reshape(N).to(dev)
            wrot = [(wq0, sb0)] + [(wq0.clone(), sb0.clone()) for _ in range(n_rot - 1)]
            for r in range(n_rot):
                calls.append(lambda sp, r=r: binding.sgq_fp8_scaled_mm(aq, sa, M, wrot[r][0], wrot[r][1], N, bias, d,
                                                                      M, N, K, sp))
            moved = M * K + 4 * M + N * K + 4 * N + 2 * N + 2 * M * N
        else:
            nb, kb = -(-N // blk), K // blk
            wq0 = torch.empty((N, K), dtype=torch.uint8, device=dev)
            ws0 = torch.empty((nb, kb), dtype=torch.float32, device=dev)
            binding.sgq_quant_weight_block(w, N, K, blk, blk, 1, wq0, ws0, s)
            wrot = [(wq0, ws0)] + [(wq0.clone(), ws0.clone()) for _ in range(n_rot - 1)]
            if args.path == "block_gemm":
                aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
                as_ = torch.empty((M, K // blk), dtype=torch.float32, device=dev)
                binding.sgq_quant_token_group(x, M, K, blk, 1, aq, as_, s)
                for r in range(n_rot):
                    calls.append(lambda sp, r=r: binding.sgq_fp8_block_gemm(aq, as_, wrot[r][0], wrot[r][1], d, M, N,
                                                                           K, blk, blk, sp))
                moved = M * K + 4 * M * (K // blk) + N * K + 4 * nb * kb + 2 * M * N
            elif args.path == "pair":
                aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
                as_ = torch.empty((M, K // blk), dtype=torch.float32, device=dev)

                def pair_call(sp, r):
                    binding.sgq_quant_token_group(x, M, K, blk, 1, aq, as_, sp)
                    binding.sgq_fp8_block_gemm(aq, as_, wrot[r][0], wrot[r][1], d, M, N, K, blk, blk, sp)
                for r in range(n_rot):
                    calls.append(lambda sp, r=r: pair_call(sp, r))
                moved = (2 * M * K + M * K + 4 * M * (K // blk)) + (M * K + 4 * M * (K // blk) + N * K
                                                                    + 4 * nb * kb + 2 * M * N)
            else:
                for r in range(n_rot):
                    calls.append(lambda sp, r=r: binding.sgq_fp8_block_linear(x, 1, wrot[r][0], wrot[r][1], d, M, N,
                                                                             K, blk, blk, None, None, sp))
                moved = 2 * M * K + N * K + 4 * nb * kb + 2 * M * N
        flops = 2 * M * N * K
    st.synchronize()
    with torch.cuda.stream(st):
        for i in range(n_rot):
            calls[i](s)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            sp = torch.cuda.current_stream().cuda_stream
            for i in range(args.reps):
                calls[i % n_rot](sp)
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        g.replay()
        e1.record(st)
    st.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.reps
    status = binding.sgq_device_status(s)
    if status != 0:
        raise RuntimeError(f"device status {binding.status_string(status)}")
    out = {"path": args.path, "M": M, "N": N, "K": K, "us": round(us, 3), "gbs": round(moved / us / 1e3, 1)}
    if flops:
        out["tflops"] = round(flops / us / 1e6, 2)
        out["blk"] = blk if args.path in ("block_gemm", "linear", "pair") else None
    del calls, g
    torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
