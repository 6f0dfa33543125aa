"""Time one stage of the MoE layer through the C ABI on a synthetic shape.

    python -m token_dispatch_grouped_moe_gb300.stage_bench --stage route --T 32768 --H 4096 --E 8 --k 2

Stages:
  route    moe_route (gate logits, top-k, gate weights); work = T*H*2 + H*E*2 + T*k*8 bytes
  permute  moe_permute with x_perm (dispatch indices and the dispatch-ordered copy of x);
           work = 2*T*k*H*2 bytes (x rows read, x_perm written)

Inputs are seeded synthetic bf16 tensors (the package's input recipe). Before
every timed call L2 is emptied of the inputs by writing and then reading a
256 MiB buffer (the read leaves L2 holding clean lines, so the timed kernel
pays no write-back of the flush). Each call is timed with CUDA events on the
current stream; the line printed gives the median over --iters calls.

This is a tuning and profiling aid for single stages at shapes the layer
configurations do not cover (for instance a router input larger than L2).
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import lib
from .inputs import make_inputs

FLUSH_BYTES = 256 << 20


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", choices=["route", "permute"], default="route")
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--E", type=int, default=8)
    ap.add_argument("--k", type=int, default=2)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("stage_bench needs a GPU")
    lib.load()
    dev = torch.device("cuda")
    inp = make_inputs(args.T, args.H, 64, args.E, seed=args.seed, only=("x", "Wg"))
    x, Wg = inp["x"].to(dev), inp["Wg"].to(dev)
    dims = lib.make_dims(args.T, args.H, 64, args.E, args.k)
    idx = torch.empty(args.T, args.k, dtype=torch.int32, device=dev)
    w = torch.empty(args.T, args.k, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ws = None
    if args.stage == "permute":
        ws = lib.workspace(dims, device=dev)
        lib.route(dims, x, Wg, topk_idx=idx, topk_w=w)

    def call():
        if args.stage == "route":
            lib.route(dims, x, Wg, topk_idx=idx, topk_w=w)
        else:
            lib.permute(dims, idx, ws, x=x, want_x_perm=True)

    times = []
    for i in range(args.warmup + args.iters):
        flush.fill_(1)
        flush.view(torch.float32).sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = float(np.median(times))
    T, H, E, k = args.T, args.H, args.E, args.k
    if args.stage == "route":
        work = T * H * 2 + H * E * 2 + T * k * 8
    else:
        work = 2 * T * k * H * 2
    if ws is not None:
        assert lib.check(ws) == lib.MOE_OK
    print(f"{args.stage} T={T} H={H} E={E} k={k}: {t * 1e6:.1f} us, {work / t / 1e9:.0f} GB/s "
          f"({work / 1e6:.1f} MB algorithmic)")


if __name__ == "__main__":
    main()
