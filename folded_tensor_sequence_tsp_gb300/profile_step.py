"""Run one step of the TSP layer forward N times, for a profiler to capture.

    python -m folded_tensor_sequence_tsp_gb300.profile_step --step attention \
        --workload 7b-64k --launches 3

Steps: qkv (Q/K/V projection of shard 0), qkv_gathered (the same with the K/V
all-gather in its epilogue, as the layer runs it), gather (K/V all-gather), attention
(causal attention of shard 0), o_proj (O projection with the fp32 residual copy),
gate_up (SwiGLU gate/up), down (SwiGLU down with the fp32 residual), shard
(zigzag rows), attention_bwd (Delta, key-side and query-side attention backward of
shard 0, after one forward with the log-sum-exp). Inputs are seeded synthetic bf16 values with the workload's shapes;
only the buffers the step touches are allocated, so a 64K-token step fits in a few
GB of device memory. Prints the average CUDA-event time per launch (a number taken
under a profiler is not a measurement).
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import tsp_inputs  # noqa: E402

from . import _binding as B  # noqa: E402


def _bf16(shape, seed, std=1.0):
    bits = tsp_inputs.normal_bf16_bits(shape, std, seed, 77)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--step", required=True,
                    choices=["qkv", "qkv_gathered", "gather", "attention", "o_proj", "gate_up",
                             "down", "shard", "attention_bwd"])
    ap.add_argument("--workload", default="7b-64k", choices=[c.name for c in tsp_inputs.CONFIGS])
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args(argv)

    from . import build
    build.build()
    cfg = tsp_inputs.config_by_name(args.workload)
    plan = B.tsp_plan(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn)
    i = plan.info
    S, H, Hd = i.S, i.hidden, i.shard_hidden
    ws = None
    if args.step not in ("gather", "shard"):  # single steps use only the status word
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    need_w = args.step in ("qkv", "qkv_gathered", "o_proj", "gate_up", "down")
    wpack = _bf16((i.wpack_elems,), 1, 0.02) if need_w else None

    if args.step == "qkv":
        xs, qkv = _bf16((S, H), 2), torch.empty((S, 3 * Hd), dtype=torch.bfloat16, device="cuda")
        run = lambda: B.tsp_qkv_projection(plan, 0, xs, wpack, qkv, ws)
    elif args.step == "qkv_gathered":
        xs = _bf16((S, H), 2)
        q, kn, vn = (torch.empty((S, Hd), dtype=torch.bfloat16, device="cuda") for _ in range(3))
        run = lambda: B.tsp_qkv_projection_gathered(plan, 0, xs, wpack, q, kn, vn, ws)
    elif args.step == "gather":
        qkv = _bf16((S, 3 * Hd), 3)
        kn = torch.empty((S, Hd), dtype=torch.bfloat16, device="cuda")
        vn = torch.empty_like(kn)
        run = lambda: B.tsp_kv_allgather(plan, qkv, kn, vn)
    elif args.step == "attention":
        qkv, kn, vn = _bf16((S, 3 * Hd), 4), _bf16((S, Hd), 5), _bf16((S, Hd), 6)
        o = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
        run = lambda: B.tsp_causal_attention(plan, 0, qkv, kn, vn, o, ws)
    elif args.step == "o_proj":
        o, xs = _bf16((S, H), 7, 0.5), _bf16((S, H), 8)
        h = torch.empty_like(xs)
        h32 = torch.empty((S, H), dtype=torch.float32, device="cuda")
        run = lambda: B.tsp_o_projection(plan, o, wpack, xs, h, ws, out32=h32)
    elif args.step == "gate_up":
        h = _bf16((S, H), 9)
        g = torch.empty((S, i.ffn_padded), dtype=torch.bfloat16, device="cuda")
        run = lambda: B.tsp_swiglu_gate_up(plan, h, wpack, g, ws)
    elif args.step == "down":
        g = _bf16((S, i.ffn_padded), 10, 0.5)
        h32 = torch.randn((S, H), dtype=torch.float32, device="cuda")
        out = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
        run = lambda: B.tsp_swiglu_down(plan, g, wpack, None, out, ws, residual32=h32)
    elif args.step == "attention_bwd":
        q, kn, vn = _bf16((S, Hd), 12), _bf16((S, Hd), 13), _bf16((S, Hd), 14)
        dout = _bf16((S, H), 15)
        o = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
        hpr = i.heads // i.D
        lse = torch.empty(hpr * i.stat_stride, dtype=torch.float32, device="cuda")
        delta = torch.empty_like(lse)
        dqkv = torch.empty((S, 3 * H), dtype=torch.bfloat16, device="cuda")
        B.tsp_causal_attention_lse(plan, 0, q, kn, vn, o, lse, ws)
        run = lambda: B.tsp_causal_attention_bwd(plan, 0, q, kn, vn, o, dout, lse, delta, dqkv, ws)
    else:
        x = _bf16((S, H), 11)
        xs = torch.empty_like(x)
        run = lambda: B.tsp_shard(plan, x, xs)

    run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.launches):
        run()
    b.record()
    torch.cuda.synchronize()
    if ws is not None:
        st = B.tsp_device_status(ws)
        if st != B.TSP_OK:
            raise B.TSPError(st, B.tsp_last_error())
    print(f"{args.step} {cfg.name}: {a.elapsed_time(b) / args.launches:.4f} ms per launch")


if __name__ == "__main__":
    main()
