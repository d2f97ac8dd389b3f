#!/usr/bin/env python3
"""Benchmark of the DSV dynamic sparse 3D attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic video
latents: dsv_predict_scores -> dsv_topk_blocks -> dsv_sparse_attn_fwd ->
the backward (timed as its three public stages dsv_attn_bwd_preprocess,
dsv_attn_bwd_dkdv, dsv_attn_bwd_dq, bitwise equal to dsv_sparse_attn_bwd).  The metric is the effective TFLOP/s of the sparse
attention forward + backward (computed blocks only: 4*block^2*d FLOPs per
selected (group, block) pair forward, 10*block^2*d backward) over the whole
step time, with the inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...    # the fp64 CPU oracle, same metric

Prints ONE JSON line on rank 0.  With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU (the path needs no
exchange between GPUs); the value is the units of all ranks over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "sparse attn fwd+bwd effective TFLOP/s"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# fp32 FMA peak of the CUDA cores (152 SMs x 128 lanes x 2 FLOP at the 2.07 GHz maximum SM clock)
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="latent16k")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mass", type=float, default=0.0, metavar="TAU",
                   help="select per group the smallest top set carrying >= TAU of the predicted mass (instead of top-k)")
    p.add_argument("--scores", choices=["mean", "max"], default="mean",
                   help="block score of the predictor: mean (dsv_predict_scores) or maximum "
                        "(dsv_predict_scores_max) of each group x key-block tile of low-rank logits")
    p.add_argument("--cube", default="", metavar="CT,CY,CX",
                   help="regroup tokens into ct x cy x cx cubes of the latent grid inside the step")
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--traffic-from", metavar="CSV",
                   help="write profiles/traffic.json from an ncu --csv log of dram__bytes_read.sum and "
                        "dram__bytes_write.sum for this bench's kernels, then exit (no GPU needed)")
    p.add_argument("--traffic-command", default="", help="the ncu command line recorded with --traffic-from")
    return p.parse_args(argv)


def load_peaks():
    f = ROOT / "MEASURED_PEAKS.json"
    if f.exists():
        d = json.loads(f.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def pair_flops(block: int, d: int):
    """Algorithmic FLOPs per selected (group, block) pair: forward, backward."""
    return 4 * block * block * d, 10 * block * block * d


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_replicas(values, op: str):
    """Combine one number per rank: 'max' (times) or 'sum' (units).  With one
    rank it is the identity; with torch.distributed initialised it all-reduces."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(values)
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(values)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = Path(tempfile.gettempdir()) / f"dsv_clocks_{os.getpid()}.csv"

    def __enter__(self):
        try:
            self.path.parent.mkdir(exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path.exists():
            return None
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.path.read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our CUDA path
# ---------------------------------------------------------------------------

class _Tensors:
    pass


class HotPath:
    """Preallocated buffers of one step; run() enqueues the four C-ABI calls.

    With cube = (ct, cy, cx) the step also regroups the tokens into 3D cubes
    of the latent grid (dsv_cube_permute on Q, K, V, dO before the path, and
    its inverse on O, dQ, dK, dV after it), so that query groups and key
    blocks are cubes; O and the gradients then come out in raster order."""

    def __init__(self, dsv, x, w, k_per_head, cube=None, mass=None, scores="mean"):
        import torch
        self.dsv, self.x, self.w = dsv, x, w
        self.k = list(k_per_head)
        self.cube = tuple(cube) if cube else None
        self.mass = mass                 # tau of the mass-threshold selection, or None for top-k
        self.scores = scores             # "mean" or "max" block scores
        self.grid = (w.T, w.Hl, w.Wl)
        dev = x.Q.device
        B, H, N, d, G = w.B, w.H, w.N, w.d, w.nb
        # the mass selection's list sizes are known only on the device: room for every block
        self.nnz = B * H * G * G if mass else dsv.nnz_of(B, G, self.k)
        self.S = torch.empty(B, H, G, G, dtype=torch.float32, device=dev)
        self.lists = (torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                      torch.empty(self.nnz, dtype=torch.int32, device=dev),
                      torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                      torch.empty(self.nnz, dtype=torch.int32, device=dev))
        self.O = torch.empty_like(x.Q)
        self.lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
        self.grads = (torch.empty_like(x.Q), torch.empty_like(x.K), torch.empty_like(x.V))
        u8 = torch.uint8
        ws_bytes = dsv.predict_max_workspace_bytes if scores == "max" else dsv.predict_workspace_bytes
        self.ws_p = torch.empty(max(1, ws_bytes(B, H, N, d, w.block, w.r)), dtype=u8, device=dev)
        self.ws_t = torch.empty(max(1, (dsv.topk_mass_workspace_bytes if mass else dsv.topk_workspace_bytes)(
            B, H, N, d, w.block)), dtype=u8, device=dev)
        self.ws_b = torch.empty(max(1, dsv.attn_bwd_workspace_bytes(B, H, N, d, w.block)), dtype=u8, device=dev)
        if self.cube:
            # the path's inputs in cube order, and O / gradients back in raster order
            self.xc = _Tensors()
            self.xc.Q, self.xc.K, self.xc.V, self.xc.dO = (torch.empty_like(t) for t in (x.Q, x.K, x.V, x.dO))
            self.xc.Wq, self.xc.Wk = x.Wq, x.Wk
            self.out_raster = tuple(torch.empty_like(x.Q) for _ in range(4))   # O, dQ, dK, dV

    @property
    def stages(self):
        return (("cube_in",) if self.cube else ()) + STAGES + (("cube_out",) if self.cube else ())

    def run(self, ev=None):
        """The four public calls (six with cube order).  With ev (one CUDA
        event per stage boundary) the backward runs as its three public
        stages with an event between each, so that every kernel of the step
        is timed on its own stream."""
        d, w = self.dsv, self.w
        marks = iter(ev or ())

        def mark():
            if ev:
                next(marks).record()

        mark()
        x = self.x
        if self.cube:
            for src, dst in zip((x.Q, x.K, x.V, x.dO), (self.xc.Q, self.xc.K, self.xc.V, self.xc.dO)):
                d.cube_permute(src, self.grid, self.cube, out=dst)
            mark()
            x = self.xc
        predict = d.predict_scores_max if self.scores == "max" else d.predict_scores
        predict(x.Q, x.K, x.Wq, x.Wk, w.block, out=self.S, workspace=self.ws_p)
        mark()
        if self.mass:
            fp, fc, bp, bc = d.topk_mass_blocks(self.S, self.mass, w.block, w.N, w.d, outs=self.lists,
                                                workspace=self.ws_t, trim=False)
        else:
            fp, fc, bp, bc = d.topk_blocks(self.S, self.k, w.block, w.N, w.d, outs=self.lists, workspace=self.ws_t)
        mark()
        d.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block, out=self.O, lse=self.lse)
        mark()
        if ev:
            d.attn_bwd_preprocess(self.O, x.dO, self.lse, w.block, workspace=self.ws_b)
            mark()
            d.attn_bwd_dkdv(x.Q, x.K, x.V, x.dO, bp, bc, w.block, outs=self.grads[1:], workspace=self.ws_b)
            mark()
            d.attn_bwd_dq(x.Q, x.K, x.V, x.dO, fp, fc, w.block, out=self.grads[0], workspace=self.ws_b)
            mark()
        else:
            d.sparse_attn_bwd(x.Q, x.K, x.V, self.O, x.dO, self.lse, fp, fc, bp, bc, w.block, outs=self.grads,
                              workspace=self.ws_b)
        if self.cube:
            for src, dst in zip((self.O, *self.grads), self.out_raster):
                d.cube_permute(src, self.grid, self.cube, inverse=True, out=dst)
            mark()

    def results(self):
        """O, LSE and the gradients as the step hands them out (raster order;
        LSE stays in the path's token order)."""
        if self.cube:
            return (self.out_raster[0], self.lse, *self.out_raster[1:])
        return (self.O, self.lse, *self.grads)

    def attention_only(self):
        d, x, w = self.dsv, self.x, self.w
        fp, fc, bp, bc = self.lists
        d.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block, out=self.O, lse=self.lse)
        d.sparse_attn_bwd(x.Q, x.K, x.V, self.O, x.dO, self.lse, fp, fc, bp, bc, w.block, outs=self.grads,
                          workspace=self.ws_b)


KERNELS_PER_STEP = {"predict": 2, "topk": 4, "fwd": 1, "bwd_pre": 1, "bwd_kv": 2, "bwd_q": 1, "cube_in": 4,
                    "cube_out": 4}
STAGES = ("predict", "topk", "fwd", "bwd_pre", "bwd_kv", "bwd_q")


def profile_traffic(kernel: str, source_files):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's
    sources still hash to what was profiled; else None."""
    f = ROOT / "profiles" / "traffic.json"
    if not f.exists():
        return None
    data = json.loads(f.read_text())
    ent = data.get(kernel)
    if not ent:
        return None
    h = hashlib.sha256()
    for s in source_files:
        h.update((ROOT / s).read_bytes())
    if ent.get("source_sha256") != h.hexdigest():
        return None
    return ent.get("dram_bytes_per_launch")


def run_ours(args):
    import torch
    from dynamic_block_sparse_projection_gb300 import binding as dsv
    from dynamic_block_sparse_projection_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = wl.WORKLOADS[args.workload]
    x = wl.make_inputs(w, device=dev)
    cube = tuple(int(v) for v in args.cube.split(",")) if args.cube else None
    hp = HotPath(dsv, x, w, x.k_per_head, cube=cube, mass=args.mass or None, scores=args.scores)
    fwd_f, bwd_f = pair_flops(w.block, w.d)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(max(3, args.warmup)):
        hp.run()
    torch.cuda.synchronize()
    if hp.mass:
        hp.nnz = int(hp.lists[0][-1].item())      # the pairs the selection kept (the same every step)
    step_flops = (fwd_f + bwd_f) * hp.nnz
    st, info = dsv.device_error()
    if st != 0:
        raise RuntimeError(f"device error {dsv.status_string(st)} ({info})")

    # timed region: K steps, L2 flushed (untimed) before each step
    stages = hp.stages
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                      if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            hp.run(evs[i])
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    parts = {k: 0.0 for k in stages}
    step_ms = []
    for e in evs:
        t = [e[k].elapsed_time(e[k + 1]) for k in range(len(stages))]
        for name, v in zip(parts, t):
            parts[name] += v
        step_ms.append(e[0].elapsed_time(e[-1]))
    total_ms = sum(step_ms)
    total_ms_max = reduce_replicas(total_ms, "max")
    flops_all = reduce_replicas(step_flops * args.steps, "sum")
    value = flops_all / (total_ms_max * 1e-3) / 1e12
    per_call = {k: v / args.steps for k, v in parts.items()}
    per_call["bwd"] = per_call["bwd_pre"] + per_call["bwd_kv"] + per_call["bwd_q"]
    attn_ms = per_call["fwd"] + per_call["bwd"]
    peaks, peak_src = load_peaks()

    # dense run of the same kernels (k = nb) for the speedup
    dense = None
    if not args.no_dense:
        dense = time_dense(dsv, x, w, hp, flush)

    # roofline of the dominant kernel (the predictor and the top-k are whole calls of 2 and 4 launches)
    dom = max(STAGES, key=lambda k: per_call[k])
    roofline = roofline_entry(dom, per_call, w, hp, peaks, peak_src)

    e2e = None if args.no_e2e else time_e2e(dsv, x, w, hp, args, flops_per_step=step_flops)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "block": w.block, "r": w.r,
                   "k_per_head": None if args.mass else sorted(set(x.k_per_head)), "pairs": hp.nnz,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   **({"cube": list(cube), "token_order": "3D cubes (dsv_cube_permute in and out, timed)"}
                      if cube else {}),
                   **({"selection": f"mass threshold tau={args.mass}, temperature 1/sqrt(d), k in [1, nb]"}
                      if args.mass else {}),
                   **({"block_scores": "tile maximum of the low-rank logits (dsv_predict_scores_max)"}
                      if args.scores == "max" else {}),
                   "l2": "flushed before every step (256 MiB write, outside the step events); "
                         "inputs are also larger than L2"},
        "pct_of_bf16_peak": round(100.0 * value / peaks["bf16_tflops"], 2),
        "attention_only": {"ms": round(attn_ms, 4),
                           "tflops": round(step_flops / (attn_ms * 1e-3) / 1e12, 3),
                           "pct_of_bf16_peak": round(100.0 * step_flops / (attn_ms * 1e-3) / 1e12
                                                     / peaks["bf16_tflops"], 2)},
        "breakdown_ms": {k: round(v, 4) for k, v in per_call.items()},
        "speedup_vs_dense": dense,
        "roofline": roofline,
        "gpu_launches": (sum(KERNELS_PER_STEP[k] for k in stages) + (2 if args.mass else 0)) * args.steps,
        "clocks": clk.summary(),
        "e2e": e2e,
        "peaks_source": peak_src,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, x, cube=cube, mass=args.mass or None, scores=args.scores)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# tcgen05 GEMMs of (block x block x d) each kernel runs per (group, block) pair
MMAS_PER_PAIR = {"fwd": 2, "bwd_kv": 4, "bwd_q": 3}
KERNEL_OF = {"fwd": "attn_fwd_kernel", "bwd_kv": "attn_bwd_kv_kernel", "bwd_q": "attn_bwd_q_kernel",
             "bwd_pre": "bwd_rowdot_kernel"}
KERNEL_SRC = {"fwd": "dynamic_block_sparse_projection_gb300/csrc/attn_fwd.cu",
              "bwd_kv": "dynamic_block_sparse_projection_gb300/csrc/attn_bwd.cu",
              "bwd_q": "dynamic_block_sparse_projection_gb300/csrc/attn_bwd.cu",
              "bwd_pre": "dynamic_block_sparse_projection_gb300/csrc/attn_bwd.cu",
              "predict": "dynamic_block_sparse_projection_gb300/csrc/predict.cu",
              "topk": "dynamic_block_sparse_projection_gb300/csrc/topk.cu"}


def roofline_entry(dom, per_call, w, hp, peaks, peak_src):
    B, H, N, d, G = w.B, w.H, w.N, w.d, w.nb
    srcs = [KERNEL_SRC[dom], "dynamic_block_sparse_projection_gb300/csrc/dsv_device.cuh"]
    if dom in MMAS_PER_PAIR:
        flops = MMAS_PER_PAIR[dom] * 2 * w.block * w.block * d * hp.nnz
        achieved = flops / (per_call[dom] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        return {"kernel": KERNEL_OF[dom], "bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "algorithmic": f"{MMAS_PER_PAIR[dom]} x 2*block^2*d FLOP per (group, block) pair x {hp.nnz} pairs",
                "peak_source": f"{peak_src} bf16 burst (cuBLAS)",
                "traffic": profile_traffic(KERNEL_OF[dom], srcs)}
    if dom == "predict" and hp.scores == "max":
        # every logit of every tile: 2 * r FLOP per (query token, key token) pair, fp32 FMA on the CUDA cores
        flops = 2.0 * B * H * N * N * w.r
        achieved = flops / (per_call[dom] * 1e-3) / 1e12
        peak = FP32_FMA_TFLOPS
        return {"kernel": "dsv_predict_scores_max", "bound": "alu", "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "algorithmic": f"2*r FLOP per (query, key) token pair x {B * H * N * N} pairs",
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz", "traffic": None}
    if dom == "bwd_pre":
        nbytes = 2 * B * H * N * d * 2 + B * H * N * 4 * 3
        kname = KERNEL_OF[dom]
    elif dom == "predict":
        nbytes = 2 * B * H * N * d * 2 + B * H * G * G * 4
        kname = "dsv_predict_scores"
    else:
        nbytes = B * H * G * G * 4 + 2 * hp.nnz * 4 + 2 * (B * H * G + 1) * 4
        kname = "dsv_topk_blocks"
    achieved = nbytes / (per_call[dom] * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} copy",
            "traffic": profile_traffic(kname, srcs)}


def time_dense(dsv, x, w, hp, flush, iters=2):
    """The same attention kernels with every block selected (k = nb)."""
    import torch
    B, H, G = w.B, w.H, w.nb
    dev = x.Q.device
    rows = B * H * G
    fp = torch.arange(0, rows * G + 1, G, dtype=torch.int32, device=dev)
    fc = torch.arange(G, dtype=torch.int32, device=dev).repeat(rows)
    dense_pairs = rows * G
    fwd_f, bwd_f = pair_flops(w.block, w.d)
    O = torch.empty_like(x.Q)
    lse = torch.empty_like(hp.lse)
    grads = tuple(torch.empty_like(t) for t in (x.Q, x.K, x.V))
    # with every block selected the transposed lists have the same form
    dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block, out=O, lse=lse)
    dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, fp, fc, w.block, outs=grads, workspace=hp.ws_b)
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dsv.sparse_attn_fwd(x.Q, x.K, x.V, fp, fc, w.block, out=O, lse=lse)
        dsv.sparse_attn_bwd(x.Q, x.K, x.V, O, x.dO, lse, fp, fc, fp, fc, w.block, outs=grads, workspace=hp.ws_b)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    t_dense = min(ts)
    # sparse attention only, same measurement
    ts = []
    for _ in range(iters):
        flush.fill_(2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        hp.attention_only()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    t_sparse = min(ts)
    dense_tflops = (fwd_f + bwd_f) * dense_pairs / (t_dense * 1e-3) / 1e12
    return {"dense_attn_ms": round(t_dense, 3), "sparse_attn_ms": round(t_sparse, 3),
            "speedup": round(t_dense / t_sparse, 3), "dense_tflops": round(dense_tflops, 3),
            "dense_pairs": dense_pairs}


def time_e2e(dsv, x, w, hp, args, flops_per_step):
    """Same metric through the public API with host buffers.  Every step copies
    its inputs (Q, K, V, dO, W^Q, W^K) from pinned host memory to the device,
    runs the four calls and copies O, LSE and the three gradients back to pinned
    host memory.  Copies run on their own streams, so a step's transfers overlap
    the neighbouring steps' compute (two device buffer sets alternate); the timed
    region runs from the first host-to-device copy to the last device-to-host
    copy."""
    import torch
    host_in = [t.cpu().pin_memory() for t in (x.Q, x.K, x.V, x.dO, x.Wq, x.Wk)]

    class X:
        pass

    sets = []
    for _ in range(2):
        dev_in = [torch.empty_like(t) for t in (x.Q, x.K, x.V, x.dO, x.Wq, x.Wk)]
        xd = X()
        xd.Q, xd.K, xd.V, xd.dO, xd.Wq, xd.Wk = dev_in
        hp2 = HotPath(dsv, xd, w, hp.k, cube=hp.cube, mass=hp.mass, scores=hp.scores)
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in hp2.results()]
        sets.append((dev_in, hp2, host_out))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2])
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        dev_in, hp2, host_out = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(cmp_done[i % 2])          # step i-2 has finished reading this set
            for d_, h_ in zip(dev_in, host_in):
                d_.copy_(h_, non_blocking=True)
            in_ready[i % 2].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(in_ready[i % 2])
            if i >= 2:
                s_cmp.wait_event(out_done[i % 2])         # step i-2's results are out
            hp2.run()
            cmp_done[i % 2].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[i % 2])
            for h_, d_ in zip(host_out, hp2.results()):
                h_.copy_(d_, non_blocking=True)
            out_done[i % 2].record(s_out)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(args.steps):
        step(i)
    b.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    return {"value": round(flops_per_step / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "host-to-device and device-to-host copies on their own streams overlap neighbouring steps' compute (2 buffer sets)"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_head_step(w, x, b, h, cube=None, mass=None, scores="mean"):
    """The fp64 oracle's whole hot path for one (b, h) (with cube, on the
    tokens in cube order, and O and the gradients put back): returns its pair
    count."""
    import numpy as np
    import torch

    import oracle
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    Q, K, V, dO = (f64(t[b:b + 1, h:h + 1]) for t in (x.Q, x.K, x.V, x.dO))
    perm = oracle.cube_order(w.T, w.Hl, w.Wl, *cube) if cube else None
    if cube:
        Q, K, V, dO = (oracle.permute_tokens(t, perm) for t in (Q, K, V, dO))
    Wq, Wk = f64(x.Wq[h:h + 1]), f64(x.Wk[h:h + 1])
    S = (oracle.predict_scores_max if scores == "max" else oracle.predict_scores)(Q, K, Wq, Wk, w.block)
    if mass:
        fp, fc = oracle.mass_lists(S, mass, 1.0 / math.sqrt(w.d), 1, w.nb)
    else:
        fp, fc = oracle.topk_lists(S, [x.k_per_head[h]])
    oracle.transpose_lists(fp, fc, 1, 1, w.nb, w.nb)
    O, _ = oracle.attn_fwd_groups(Q, K, V, fp, fc, w.block)
    grads = oracle.attn_bwd_groups(Q, K, V, dO, fp, fc, w.block)
    if cube:
        for t in (O, *grads):
            oracle.permute_tokens(t, perm, inverse=True)
    return int(fc.shape[0])


def cpu_baseline(w, x, min_s=10.0, max_s=30.0, cube=None, mass=None, scores="mean"):
    fwd_f, bwd_f = pair_flops(w.block, w.d)
    t0 = time.perf_counter()
    pairs, heads = 0, 0
    for h in range(w.H):
        pairs += oracle_head_step(w, x, 0, h, cube, mass, scores)
        heads += 1
        el = time.perf_counter() - t0
        if el >= min_s or el * (heads + 1) / heads > max_s:
            break
    el = time.perf_counter() - t0
    return {"value": round((fwd_f + bwd_f) * pairs / el / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": f"{heads} of {w.B * w.H} (batch, head) slices of {w.name}: predictor, top-k, transpose, "
                      f"attention fwd+bwd in fp64 numpy ({pairs} pairs)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    cube = tuple(int(v) for v in args.cube.split(",")) if args.cube else None
    heads = sorted(set(range(w.H)))
    x = wl.make_inputs(w, device="cpu")
    fwd_f, bwd_f = pair_flops(w.block, w.d)
    slices = [(b, h) for b in range(w.B) for h in heads]
    for i in range(max(3, args.warmup)):
        oracle_head_step(w, x, *slices[i % len(slices)], cube, args.mass or None, args.scores)
    t0 = time.perf_counter()
    pairs = 0
    for i in range(args.steps):
        pairs += oracle_head_step(w, x, *slices[i % len(slices)], cube, args.mass or None, args.scores)
    el = time.perf_counter() - t0
    value = (fwd_f + bwd_f) * pairs / el / 1e12
    sample = (f"each step one (batch, head) slice of {w.name} (1 of {len(slices)}): predictor, top-k, transpose, "
              f"attention fwd+bwd in fp64 numpy on the host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, **({"cube": list(cube)} if cube else {}),
                   **({"selection": f"mass threshold tau={args.mass}, temperature 1/sqrt(d), k in [1, nb]"}
                      if args.mass else {}),
                   **({"block_scores": "tile maximum of the low-rank logits"} if args.scores == "max" else {})},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def write_traffic(csv_path, command, workload):
    """profiles/traffic.json: mean DRAM bytes (read + write) per launch of each
    attention kernel in an ncu CSV, with the sha256 of the sources it was
    built from (bench.py reports null once they change)."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    h = rows[hi]
    ki, mi, vi, ui, idi = (h.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit", "ID"))
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    per_launch = {}
    for r in rows[hi + 1:]:
        if len(r) <= max(ki, mi, vi, ui) or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        name = next((k for k in KERNEL_OF.values() if k in r[ki]), None)
        if name is None:
            continue
        v = float(r[vi].replace(",", "")) * scale.get(r[ui], 1.0)
        key = (name, r[idi])
        per_launch[key] = per_launch.get(key, 0.0) + v
    out = {}
    for stage, name in KERNEL_OF.items():
        vals = [v for (n, _), v in per_launch.items() if n == name]
        if not vals:
            continue
        hsh = hashlib.sha256()
        for src in (KERNEL_SRC[stage], "dynamic_block_sparse_projection_gb300/csrc/dsv_device.cuh"):
            hsh.update((ROOT / src).read_bytes())
        out[name] = {"dram_bytes_per_launch": round(sum(vals) / len(vals)), "launches": len(vals),
                     "workload": workload, "source_sha256": hsh.hexdigest(), "command": command}
    (ROOT / "profiles" / "traffic.json").write_text(json.dumps(out, indent=1) + "\n")
    print(json.dumps(out, indent=1))


def main(argv=None):
    args = parse_args(argv)
    if args.traffic_from:
        write_traffic(args.traffic_from, args.traffic_command, args.workload)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
