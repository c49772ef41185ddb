"""Runs one quantise + GEMM case of a workload a few times, for profilers.

    python -m fp8_block_scaled_sgq_gb300.profile_case WORKLOAD [INDEX] [--iters N] [--fused | --quant-only]
                                                      [--pow2 | --ue8m0-bytes]
    python -m fp8_block_scaled_sgq_gb300.profile_case --shape M N K BLK [...]

WORKLOAD/INDEX pick a case from ``synth.WORKLOADS`` (e.g. ``decode_block32 2``
is M=16, N=7168, K=2048 with [32,32] blocks); --shape takes any shape with
[BLK, BLK] blocks and UE8M0 scales (x ~ N(0,1), W ~ N(0,0.02)).  Each iteration launches the
activation quantisation kernel, then the block-scaled GEMM, on one stream.
With --fused each iteration is one sgq_fp8_block_linear call instead (one
kernel at decode-sized M); with --quant-only only the quantisation kernel;
--pow2 passes SGQ_GEMM_SCALES_POW2 to the GEMM; --ue8m0-bytes runs the
byte-output quantiser and sgq_fp8_block_gemm_ue8m0 (the weight scales
converted to bytes once up front).  The weight is quantised once up front
(one extra launch; two with --ue8m0-bytes).  The run ends with
the device status word checked and one line of wall-clock timing, which is
not a benchmark number (use bench.py for those).
"""
from __future__ import annotations

import argparse
import json
import time

import torch

from . import binding, synth


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", nargs="?", choices=sorted(synth.WORKLOADS))
    ap.add_argument("index", type=int, nargs="?", default=0)
    ap.add_argument("--shape", type=int, nargs=4, metavar=("M", "N", "K", "BLK"))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--quant-only", action="store_true", help="launch only the activation quantiser")
    ap.add_argument("--pow2", action="store_true", help="GEMM with SGQ_GEMM_SCALES_POW2 (UE8M0 scales)")
    ap.add_argument("--ue8m0-bytes", action="store_true", help="UE8M0 scale bytes (quantiser and GEMM)")
    args = ap.parse_args()
    if args.shape:
        M, N, K, blk = args.shape
        c = synth.Case(f"shape_M{M}_N{N}_K{K}_b{blk}", M, N, K, blk, blk, True)
    elif args.workload:
        c = synth.WORKLOADS[args.workload][args.index]
    else:
        ap.error("give WORKLOAD [INDEX] or --shape M N K BLK")
    dev = torch.device("cuda:0")
    M, N, K = c.M, c.N, c.K
    x = c.x().to(dev)
    w = c.w().to(dev)
    st = torch.cuda.Stream()
    s = st.cuda_stream
    nb, kb = -(-N // c.blk_n), -(-K // c.blk_k)
    wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
    ws = torch.empty((nb, kb), dtype=torch.float32, device=dev)
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty((M, -(-K // c.group)), dtype=torch.float32, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    binding.sgq_quant_weight_block(w, N, K, c.blk_n, c.blk_k, int(c.ue8m0), wq, ws, s)
    if args.ue8m0_bytes:
        we = torch.empty((nb, kb), dtype=torch.uint8, device=dev)
        binding.sgq_scales_to_ue8m0(ws, nb * kb, we, s)
        xe = torch.empty((M, -(-K // c.group)), dtype=torch.uint8, device=dev)
    t0 = time.perf_counter()
    for _ in range(args.iters):
        if args.fused:
            binding.sgq_fp8_block_linear(x, int(c.ue8m0), wq, ws, d, M, N, K, c.blk_n, c.blk_k, None, None, s)
        elif args.ue8m0_bytes:
            binding.sgq_quant_token_group_ue8m0(x, M, K, c.group, xq, xe, s)
            if not args.quant_only:
                binding.sgq_fp8_block_gemm_ue8m0(xq, xe, wq, we, d, M, N, K, c.blk_n, c.blk_k, 0, s)
        else:
            binding.sgq_quant_token_group(x, M, K, c.group, int(c.ue8m0), xq, xs, s)
            if not args.quant_only:
                flags = binding.SGQ_GEMM_SCALES_POW2 if args.pow2 else binding.SGQ_GEMM_DEFAULT
                binding.sgq_fp8_block_gemm_ex(xq, xs, wq, ws, d, M, N, K, c.blk_n, c.blk_k, flags, s)
    st.synchronize()
    wall = time.perf_counter() - t0
    status = binding.sgq_device_status(s)
    if status != 0:
        raise RuntimeError(f"device status {binding.status_string(status)}")
    print(json.dumps({"case": c.name, "fused": args.fused, "quant_only": args.quant_only, "pow2": args.pow2,
                      "ue8m0_bytes": args.ue8m0_bytes,
                      "M": M, "N": N, "K": K, "blk": [c.blk_n, c.blk_k],
                      "iters": args.iters, "wall_ms": round(wall * 1e3, 3)}))


if __name__ == "__main__":
    main()
