"""Run the whole hot path a few times on one workload (for profilers).

    python -m dynamic_block_sparse_projection_gb300.profile_case [workload] [passes]

Draws the workload's seeded inputs on cuda:0, runs predictor -> top-k ->
sparse attention forward -> backward `passes` times (default 3), checks the
device error word and exits 0.  Under ncu, skip the first pass (-s 1) to
capture a warm launch.
"""
import sys

import torch

from dynamic_block_sparse_projection_gb300 import binding as dsv
from dynamic_block_sparse_projection_gb300 import workloads as wl


def main(argv):
    w = wl.WORKLOADS[argv[0] if argv else "latent16k"]
    passes = int(argv[1]) if len(argv) > 1 else 3
    x = wl.make_inputs(w, device="cuda")
    for _ in range(passes):
        S = dsv.predict_scores(x.Q, x.K, x.Wq, x.Wk, w.block)
        lists = dsv.topk_blocks(S, x.k_per_head, w.block, w.N, w.d)
        O, lse = dsv.sparse_attn_fwd(x.Q, x.K, x.V, lists[0], lists[1], w.block)
        dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, *lists, w.block)
    torch.cuda.synchronize()
    st, info = dsv.device_error()
    if st != 0:
        raise SystemExit(f"device error {dsv.status_string(st)} ({info})")
    print("ok", w.name, passes)


if __name__ == "__main__":
    main(sys.argv[1:])
