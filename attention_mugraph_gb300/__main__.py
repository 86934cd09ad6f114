"""Run one named workload through the library and print its time per call.

    python -m attention_mugraph_gb300 --workload long_kv --calls 20 [--n-split S] [--stages K]

A small command-line runner for users and for profilers (a fixed, short sequence of launches on
one set of inputs). It checks nothing against a reference; the tests do that.
"""

from __future__ import annotations

import argparse
import json


def main():
    import torch

    from . import _lib, build, inputs

    ap = argparse.ArgumentParser(prog="python -m attention_mugraph_gb300")
    ap.add_argument("--workload", default="gqa", choices=inputs.CONFIG_ORDER)
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--n-split", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    args = ap.parse_args()

    build.build()
    q, k, v, (B, M, N, d) = inputs.make_config(args.workload)
    plan = _lib.Plan(B, M, N, d, n_split=args.n_split, stages=args.stages)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    O = torch.empty((B, M, d), dtype=torch.float16, device="cuda")
    plan.run(Q, K, V, O)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.calls):
        plan.run(Q, K, V, O)
    e1.record()
    torch.cuda.synchronize()
    status = plan.status()
    print(json.dumps({"workload": args.workload, "B": B, "M": M, "N": N, "d": d, "calls": args.calls,
                      "us_per_call": e0.elapsed_time(e1) * 1e3 / args.calls, "plan": plan.info,
                      "status": status}))
    plan.destroy()
    if status != _lib.MG_OK:
        raise SystemExit(f"device status {status}")


if __name__ == "__main__":
    main()
