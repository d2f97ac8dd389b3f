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


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long518k",
                   help="synthetic workload (default: long518k, the largest one-GPU configuration)")
    p.add_argument("--heads", type=int, default=0, metavar="N",
                   help="keep only the first N heads of the workload (a reduced case of the same per-head "
                        "structure, for profiler captures); 0 = all")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mass", type=float, default=0.0, metavar="TAU",
                   help="select per group the smallest top set carrying >= TAU of the predicted mass (instead of top-k)")
    p.add_argument("--scores", choices=["mean", "max"], default="mean",
                   help="block score of the predictor: mean (dsv_predict_scores) or maximum "
                        "(dsv_predict_scores_max) of each group x key-block tile of low-rank logits")
    p.add_argument("--cube", default="", metavar="CT,CY,CX",
                   help="regroup tokens into ct x cy x cx cubes of the latent grid inside the step")
    p.add_argument("--predict", choices=["fused", "two-call"], default="fused",
                   help="fused: dsv_predict_topk_blocks (scores stay on chip); two-call: dsv_predict_scores "
                        "then dsv_topk_blocks (the score matrix goes through HBM)")
    p.add_argument("--dispatch", action="store_true",
                   help="route each head sparse or dense by the OP dispatcher and the measured profile "
                        "profiles/dispatch_<workload>.json")
    p.add_argument("--dispatch-profile", action="store_true",
                   help="measure the sparse/dense time ratio against the kept fraction on the workload's first "
                        "2 heads, write profiles/dispatch_<workload>.json and exit")
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

    def __init__(self, dsv, x, w, k_per_head, cube=None, mass=None, scores="mean", fused=False):
        import torch
        self.dsv, self.x, self.w = dsv, x, w
        # the fused predictor + top-k serves the mean block scores with a fixed k per head
        self.fused = bool(fused) and not mass and scores == "mean"
        self.k = list(k_per_head)
        self.cube = tuple(cube) if cube else None
        self.mass = mass                 # tau of the mass-threshold selection, or None for top-k
        self.scores = scores             # "mean" or "max" block scores
        self.grid = (w.T, w.Hl, w.Wl)
        dev = x.Q.device
        B, H, N, d, G = w.B, w.H, w.N, w.d, w.nb
        # the mass selection's list sizes are known only on the device: room for every block
        self.nnz = B * H * G * G if mass else dsv.nnz_of(B, G, self.k)
        self.S = None if self.fused else torch.empty(B, H, G, G, dtype=torch.float32, device=dev)
        self.lists = (torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                      torch.empty(self.nnz, dtype=torch.int32, device=dev),
                      torch.empty(B * H * G + 1, dtype=torch.int32, device=dev),
                      torch.empty(self.nnz, dtype=torch.int32, device=dev))
        self.O = torch.empty_like(x.Q)
        self.lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
        self.grads = (torch.empty_like(x.Q), torch.empty_like(x.K), torch.empty_like(x.V))
        u8 = torch.uint8
        if self.fused:
            self.ws_p = torch.empty(max(1, dsv.predict_topk_workspace_bytes(B, H, N, d, w.block, w.r)), dtype=u8,
                                    device=dev)
            self.ws_t = None
        else:
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
        core = FUSED_STAGES if self.fused else STAGES
        return (("cube_in",) if self.cube else ()) + core + (("cube_out",) if self.cube else ())

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
        if self.fused:
            fp, fc, bp, bc = d.predict_topk_blocks(x.Q, x.K, x.Wq, x.Wk, self.k, w.block, outs=self.lists,
                                                   workspace=self.ws_p)
        else:
            predict = d.predict_scores_max if self.scores == "max" else d.predict_scores
            predict(x.Q, x.K, x.Wq, x.Wk, w.block, out=self.S, workspace=self.ws_p)
            mark()
        if self.fused:
            pass
        elif self.mass:
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


KERNELS_PER_STEP = {"predict": 2, "topk": 4, "predict_topk": 7, "fwd": 1, "bwd_pre": 1, "bwd_kv": 2, "bwd_q": 1,
                    "cube_in": 4, "cube_out": 4}


def predict_topk_launches(w) -> int:
    """Kernels of one fused predictor + top-k call: pooling, two statistics
    kernels, the select kernel and three transpose kernels; when the select
    items (128 groups of one head each, one CTA per SM) leave a partly filled
    last wave of at least two full ones, the library launches that wave on its
    own and the transposes in two head ranges (three more launches)."""
    import torch
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    tiles = -(-w.nb // 128)
    items = w.B * w.H * tiles
    tail = items % nsm
    split = tail != 0 and items >= 2 * nsm and (items - tail) // tiles >= 1
    return KERNELS_PER_STEP["predict_topk"] + (3 if split else 0)
STAGES = ("predict", "topk", "fwd", "bwd_pre", "bwd_kv", "bwd_q")
FUSED_STAGES = ("predict_topk", "fwd", "bwd_pre", "bwd_kv", "bwd_q")


def profile_traffic(kernel: str, source_files, w, pairs):
    """DRAM bytes per launch of `kernel` on this workload, from a committed
    ncu summary (profiles/traffic.json): None unless the entry was captured on
    the same workload and the kernel's sources still hash to what was
    profiled.  An entry captured on a head subset of the workload (same
    per-head structure) is scaled to this launch by its pairs; the second
    value says how the figure was obtained."""
    f = ROOT / "profiles" / "traffic.json"
    if not f.exists():
        return None, None
    ent = json.loads(f.read_text()).get(kernel)
    if not ent or ent.get("workload") != w.name:
        return None, None
    h = hashlib.sha256()
    for s in source_files:
        h.update((ROOT / s).read_bytes())
    if ent.get("source_sha256") != h.hexdigest():
        return None, None
    got = float(ent["dram_bytes_per_launch"])
    cap_pairs = ent.get("pairs")
    if cap_pairs and pairs and cap_pairs != pairs:
        return round(got * pairs / cap_pairs), (f"ncu DRAM read+write of a {ent.get('heads')}-head capture of "
                                                f"{w.name} ({cap_pairs} pairs), scaled by pairs to {pairs}")
    return round(got), f"ncu DRAM read+write per launch on {w.name}"


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
    if args.heads and args.heads < w.H:
        w = wl.scaled(w, name=w.name, H=args.heads)
    x = wl.make_inputs(w, device=dev)
    cube = tuple(int(v) for v in args.cube.split(",")) if args.cube else None
    ks, dispatch = list(x.k_per_head), None
    if args.dispatch:
        prof = json.loads((ROOT / "profiles" / f"dispatch_{w.name}.json").read_text())
        ks, dense = dsv.dispatch_heads(ks, w.nb, prof["rho"], prof["ratio"])
        dispatch = {"profile": f"profiles/dispatch_{w.name}.json", "threshold_rho": prof.get("threshold_rho"),
                    "dense_heads": [h for h, d in enumerate(dense) if d]}
    hp = HotPath(dsv, x, w, ks, cube=cube, mass=args.mass or None, scores=args.scores,
                 fused=args.predict == "fused")
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
    # the bf16 denominator: the burst figure for a short timed region, the sustained one
    # (a seconds-long loop under the power cap) once the timed steps run for a second or more
    sustained = total_ms_max >= 1000.0
    bf16_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    bf16_kind = (f"{peak_src} bf16 sustained (cuBLAS, seconds-long loop; the timed region is "
                 f"{total_ms_max / 1e3:.1f} s)" if sustained else f"{peak_src} bf16 burst (cuBLAS)")

    # dense run of the same kernels (k = nb) for the speedup
    dense = None
    if not args.no_dense:
        dense = time_dense(dsv, x, w, hp, flush, attn_ms=attn_ms, pre_ms=pre_ms(per_call))

    # roofline of the dominant kernel (the predictor and the top-k are whole calls of several launches)
    dom = max(hp.stages, key=lambda k: per_call[k])
    roofline = roofline_entry(dom, per_call, w, hp, peaks, peak_src, bf16_peak, bf16_kind)
    bwd_eff = step_flops * bwd_f / (fwd_f + bwd_f) / (per_call["bwd"] * 1e-3) / 1e12

    e2e = None if args.no_e2e else time_e2e(dsv, x, w, hp, args, flops_per_step=step_flops)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "block": w.block, "r": w.r,
                   "k_per_head": None if args.mass else sorted(set(x.k_per_head)), "pairs": hp.nnz,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "predictor_topk": ("fused (dsv_predict_topk_blocks: scores on chip)" if hp.fused else
                                      "two calls (dsv_predict_scores, dsv_topk_blocks)"),
                   **({"heads_kept": w.H, "reduced": "first heads only (profiler case)"} if args.heads else {}),
                   **({"dispatch": dispatch} if dispatch else {}),
                   **({"cube": list(cube), "token_order": "3D cubes (dsv_cube_permute in and out, timed)"}
                      if cube else {}),
                   **({"selection": f"mass threshold tau={args.mass}, temperature 1/sqrt(d), k in [1, nb]"}
                      if args.mass else {}),
                   **({"block_scores": "tile maximum of the low-rank logits (dsv_predict_scores_max)"}
                      if args.scores == "max" else {}),
                   "l2": "flushed before every step (256 MiB write, outside the step events); "
                         "inputs are also larger than L2"},
        "pct_of_bf16_peak": round(100.0 * value / bf16_peak, 2),
        "bf16_peak": {"tflops": bf16_peak, "kind": bf16_kind,
                      "pct_of_burst": round(100.0 * value / peaks["bf16_tflops"], 2)},
        "attention_only": {"ms": round(attn_ms, 4),
                           "tflops": round(step_flops / (attn_ms * 1e-3) / 1e12, 3),
                           "pct_of_bf16_peak": round(100.0 * step_flops / (attn_ms * 1e-3) / 1e12
                                                     / bf16_peak, 2)},
        "breakdown_ms": {k: round(v, 4) for k, v in per_call.items()},
        "backward_effective": {"tflops": round(bwd_eff, 3), "frac": round(bwd_eff / bf16_peak, 4),
                               "algorithmic": "10*block^2*d FLOP per pair (5 GEMMs) over the three backward "
                                              "stages' time; the kernels execute 7 (S and dP twice, no atomics)"},
        "predictor_topk": hbm_fractions(w, hp, per_call, peaks),
        "speedup_vs_dense": dense,
        "roofline": roofline,
        "gpu_launches": (sum(predict_topk_launches(w) if k == "predict_topk" else KERNELS_PER_STEP[k] for k in stages)
                         + (2 if args.mass else 0)) * args.steps,
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
              "topk": "dynamic_block_sparse_projection_gb300/csrc/topk.cu",
              "predict_topk": "dynamic_block_sparse_projection_gb300/csrc/predict_topk.cu"}


def roofline_entry(dom, per_call, w, hp, peaks, peak_src, bf16_peak=None, bf16_kind=None):
    B, H, N, d, G = w.B, w.H, w.N, w.d, w.nb
    srcs = [KERNEL_SRC[dom], "dynamic_block_sparse_projection_gb300/csrc/dsv_device.cuh"]
    traffic, tnote = profile_traffic(KERNEL_OF.get(dom, dom), srcs, w, hp.nnz)
    if dom in MMAS_PER_PAIR:
        flops = MMAS_PER_PAIR[dom] * 2 * w.block * w.block * d * hp.nnz
        achieved = flops / (per_call[dom] * 1e-3) / 1e12
        peak = bf16_peak or peaks["bf16_tflops"]
        return {"kernel": KERNEL_OF[dom], "bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "algorithmic": f"{MMAS_PER_PAIR[dom]} x 2*block^2*d FLOP per (group, block) pair x {hp.nnz} pairs",
                "peak_source": bf16_kind or f"{peak_src} bf16 burst (cuBLAS)",
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic, "traffic_source": tnote}
    if dom == "predict" and hp.scores == "max":
        # every logit of every tile: 2 * r FLOP per (query token, key token) pair; the tensor core runs
        # it as one bf16 contraction of length 3r (hi/lo split of both projections), 3x the FLOPs
        flops = 2.0 * B * H * N * N * w.r
        achieved = flops / (per_call[dom] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        return {"kernel": "dsv_predict_scores_max", "bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "executed_frac": round(3 * achieved / peak, 4),
                "algorithmic": f"2*r FLOP per (query, key) token pair x {B * H * N * N} pairs (executed: 3x, "
                               "the bf16 hi/lo split)",
                "peak_source": f"{peak_src} bf16 burst (cuBLAS)", "traffic": None}
    if dom == "bwd_pre":
        nbytes = 2 * B * H * N * d * 2 + B * H * N * 4 * 3
        kname = KERNEL_OF[dom]
    elif dom == "predict":
        nbytes = 2 * B * H * N * d * 2 + B * H * G * G * 4
        kname = "dsv_predict_scores"
    elif dom == "predict_topk":
        nbytes = 2 * B * H * N * d * 2 + 8 * hp.nnz + 8 * (B * H * G + 1)
        kname = "dsv_predict_topk_blocks"
    else:
        nbytes = B * H * G * G * 4 + 2 * hp.nnz * 4 + 2 * (B * H * G + 1) * 4
        kname = "dsv_topk_blocks"
    achieved = nbytes / (per_call[dom] * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} copy",
            "traffic": profile_traffic(kname, srcs, w, hp.nnz)[0]}


DENSE_MAX_PAIRS = 1 << 25    # a dense run with more pairs is timed on 2 heads and scaled (heads are independent)


def time_dense(dsv, x, w, hp, flush, attn_ms, pre_ms, iters=2):
    """The same attention kernels with every block selected (k = nb).  Heads
    are independent, so a large workload's dense run is timed on its first 2
    heads and scaled by H / 2 (long518k: ~0.5 PFLOP per head, ~10 s for all
    24)."""
    import torch
    B, H, G = w.B, w.H, w.nb
    heads = H if B * H * G * G <= DENSE_MAX_PAIRS else min(2, H)
    dev = x.Q.device
    Q, K, V, dO = ((t if heads == H else t[:, :heads].contiguous()) for t in (x.Q, x.K, x.V, x.dO))
    rows = B * heads * G
    fp = torch.arange(0, rows * G + 1, G, dtype=torch.int32, device=dev)
    fc = torch.arange(G, dtype=torch.int32, device=dev).repeat(rows)
    dense_pairs = rows * G
    fwd_f, bwd_f = pair_flops(w.block, w.d)
    O = torch.empty_like(Q)
    lse = torch.empty(B, heads, w.N, dtype=torch.float32, device=dev)
    grads = tuple(torch.empty_like(t) for t in (Q, K, V))

    def run():
        # with every block selected the transposed lists have the same form as the forward ones
        dsv.sparse_attn_fwd(Q, K, V, fp, fc, w.block, out=O, lse=lse)
        dsv.sparse_attn_bwd(Q, K, V, O, dO, lse, fp, fc, fp, fc, w.block, outs=grads, workspace=hp.ws_b)

    run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    t_meas = min(ts)
    t_dense = t_meas * H / heads
    # sparse attention only, same measurement (the fused backward call)
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
    dense_tflops = (fwd_f + bwd_f) * dense_pairs / (t_meas * 1e-3) / 1e12
    return {"dense_attn_ms": round(t_dense, 3), "sparse_attn_ms": round(t_sparse, 3),
            "speedup": round(t_dense / t_sparse, 3),
            "speedup_with_predictor_topk": round(t_dense / (t_sparse + pre_ms), 3),
            "step_attention_ms": round(attn_ms, 3),
            "dense_tflops": round(dense_tflops, 3), "dense_pairs": dense_pairs * H // heads,
            "dense_heads_timed": heads,
            "method": ("all heads" if heads == H else
                       f"timed on {heads} of {H} heads ({dense_pairs} pairs) and scaled by {H}/{heads}: heads are "
                       f"independent") + "; same kernels with k = nb, L2 flushed, best of %d" % iters}


def pre_ms(per_call):
    """Time of the predictor and the top-k (one fused call or two calls)."""
    return per_call["predict_topk"] if "predict_topk" in per_call else per_call["predict"] + per_call["topk"]


def hbm_fractions(w, hp, per_call, peaks):
    """Algorithmic bytes and HBM fraction of the predictor and of the top-k.
    The fused call's bytes are the Q and K reads and the list writes (its
    score matrix never reaches HBM); the two-call path also writes and reads
    the score matrix."""
    B, H, N, d, G = w.B, w.H, w.N, w.d, w.nb
    lists = 8 * hp.nnz + 4 * (B * H * G + 1) + 4 * (B * H * G + 1)
    if hp.fused:
        fused = 2 * B * H * N * d * 2 + lists
        gbs = fused / (per_call["predict_topk"] * 1e-3) / 1e9
        return {"predict+topk": {"bytes": fused, "ms": round(per_call["predict_topk"], 4), "gbs": round(gbs, 1),
                                 "frac": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8tbs": round(gbs / 8000.0, 4)},
                "bytes_rule": "fused call: read Q and K + write both column arrays and both row-pointer arrays"}
    pred = 2 * B * H * N * d * 2 + 4 * B * H * G * G
    topk = 4 * B * H * G * G + lists
    out = {}
    for nm, nbytes, ms in (("predict", pred, per_call["predict"]), ("topk", topk, per_call["topk"]),
                           ("predict+topk", pred + topk, per_call["predict"] + per_call["topk"])):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[nm] = {"bytes": nbytes, "ms": round(ms, 4), "gbs": round(gbs, 1),
                   "frac": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8tbs": round(gbs / 8000.0, 4)}
    out["bytes_rule"] = ("predict: read Q and K + write S; top-k: read S + write both column arrays and "
                         "both row-pointer arrays")
    return out


def time_e2e(dsv, x, w, hp, args, flops_per_step):
    """Same metric through the public API with host buffers.  Every step copies
    its inputs (Q, K, V, dO, W^Q, W^K) from pinned host memory to the device,
    runs the four calls and copies O, LSE and the three gradients back to pinned
    host memory.  Copies run on their own streams, so a step's transfers overlap
    the neighbouring steps' compute (two device buffer sets alternate); the timed
    region runs from the first host-to-device copy to the last device-to-host
    copy."""
    import torch
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in (x.Q, x.K, x.V, x.dO, x.Wq, x.Wk)]
    host_out = None     # one set of pinned result buffers: the device-to-host copies run in order on one stream

    class X:
        pass

    sets = []
    for _ in range(2):
        dev_in = [torch.empty_like(t) for t in (x.Q, x.K, x.V, x.dO, x.Wq, x.Wk)]
        xd = X()
        xd.Q, xd.K, xd.V, xd.dO, xd.Wq, xd.Wk = dev_in
        hp2 = HotPath(dsv, xd, w, hp.k, cube=hp.cube, mass=hp.mass, scores=hp.scores, fused=hp.fused)
        if host_out is None:
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
    del sets, host_in, host_out
    torch.cuda.empty_cache()
    if hasattr(torch._C, "_host_emptyCache"):
        torch._C._host_emptyCache()          # hand the pinned buffers back before the oracle leg
    return {"value": round(flops_per_step / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "pinned_host_bytes": h2d + d2h,
            "overlap": "host-to-device and device-to-host copies on their own streams overlap neighbouring steps' compute (2 buffer sets)"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

ORACLE_HEADS, ORACLE_GROUPS_PER_HEAD = 4, 16       # 64 seeded query groups in 4 seeded (batch, head) slices
BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def oracle_sample(w):
    """The seeded sample the oracle legs time: ORACLE_HEADS (batch, head)
    slices and ORACLE_GROUPS_PER_HEAD query groups in each, as
    [((b, h), [g, ...]), ...]."""
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    bhs = wl.sample_indices(w.B * w.H, ORACLE_HEADS, w.seed)
    out = []
    for i, bh in enumerate(bhs):
        groups = wl.sample_indices(w.nb, ORACLE_GROUPS_PER_HEAD, w.seed, gid=100 + i)
        out.append(((bh // w.H, bh % w.H), groups))
    return out


class _Bf16Head:
    """A [1, 1, N, d] stand-in for one (batch, head) slice of a bf16 tensor
    kept as raw 16-bit patterns (a memory-mapped file): indexing widens just
    the rows it selects to fp32, exactly.  Lets the oracle functions index a
    518k-token head without every worker holding it in floating point."""

    def __init__(self, bits):
        self.bits = bits
        self.shape = (1, 1) + tuple(bits.shape)

    def __getitem__(self, idx):
        import numpy as np
        rest = idx[2:] if isinstance(idx, tuple) else ()
        sel = self.bits[rest] if rest else self.bits
        return (np.asarray(sel).astype(np.uint32) << 16).view(np.float32)

    def full(self):
        return self[(0, 0)][None, None]


def _oracle_worker(conn, path, meta):
    """One host core: loads its (batch, head) slice from `path` once (input
    staging, untimed), then on each request runs the fp64 oracle's whole hot
    path for one of its query groups -- predictor row, top-k (or the mass
    count), attention forward and the group's backward (dQ and the group's
    dK/dV contributions, every pair of its list) -- and answers the pairs and
    the seconds it took."""
    import numpy as np

    import oracle
    X = {nm: _Bf16Head(np.load(os.path.join(path, nm + ".npy"), mmap_mode="r")) for nm in ("Q", "K", "V", "dO")}
    Wq = np.load(os.path.join(path, "Wq.npy"))[None]
    Wk = np.load(os.path.join(path, "Wk.npy"))[None]
    block, d, k, nb = meta["block"], meta["d"], meta["k"], meta["nb"]
    if meta["cube"]:
        perm = oracle.cube_order(*meta["grid"], *meta["cube"])
        X = {nm: oracle.permute_tokens(t.full(), perm) for nm, t in X.items()}
    Q, K, V, dO = X["Q"], X["K"], X["V"], X["dO"]
    conn.send("ready")
    while True:
        g = conn.recv()
        if g is None:
            break
        t0 = time.perf_counter()
        rows = [(0, 0, g)]
        pred = oracle.predict_scores_max_rows if meta["scores"] == "max" else oracle.predict_scores_rows
        s = pred(Q, K, Wq, Wk, block, rows)[0]
        m = (oracle.mass_count_row(s, meta["mass"], 1.0 / math.sqrt(d), 1, nb) if meta["mass"] else k)
        cols = oracle.topk_row(s, m)
        ptr = np.zeros(nb + 1, dtype=np.int64)
        ptr[g + 1:] = len(cols)
        oracle.attn_fwd_groups(Q, K, V, ptr, cols, block, rows=rows)
        oracle.attn_bwd_dq_rows(Q, K, V, dO, ptr, cols, block, rows)
        conn.send((len(cols), time.perf_counter() - t0))
    conn.close()


class OraclePool:
    """The fp64 oracle on the host cores: one spawned process per core, each
    owning a few of the seeded query groups of one sampled (batch, head)
    slice (ORACLE_GROUPS_PER_HEAD per head, split over the cores).  A round
    asks every process for one of its groups; a round's wall time is the
    slowest process.  BLAS runs single-threaded in each process, so the
    cores used are the processes."""

    def __init__(self, w, x_heads, cube=None, mass=None, scores="mean", cores=None):
        import multiprocessing as mp

        import numpy as np
        self.w = w
        sample = oracle_sample(w)
        cores = cores or os.cpu_count() or 1
        per_head = max(1, cores // len(sample))
        self.tmp = tempfile.mkdtemp(prefix="dsv_oracle_", dir=_scratch_dir(w, len(sample)))
        self.slots = []                                  # (process, conn, [groups])
        ctx = mp.get_context("spawn")
        saved = {v: os.environ.get(v) for v in BLAS_THREAD_VARS}
        os.environ.update({v: "1" for v in BLAS_THREAD_VARS})
        try:
            for i, ((b, h), groups) in enumerate(sample):
                path = os.path.join(self.tmp, f"bh{i}")
                os.mkdir(path)
                for nm in ("Q", "K", "V", "dO"):
                    t = getattr(x_heads, nm)[b, x_heads.head_index[h]]
                    np.save(os.path.join(path, nm + ".npy"), t.cpu().view(__import__("torch").int16).numpy())
                hi = x_heads.head_index[h]
                np.save(os.path.join(path, "Wq.npy"), x_heads.Wq[hi].double().cpu().numpy())
                np.save(os.path.join(path, "Wk.npy"), x_heads.Wk[hi].double().cpu().numpy())
                meta = {"block": w.block, "d": w.d, "k": int(x_heads.k_per_head[hi]), "nb": w.nb, "cube": cube,
                        "grid": (w.T, w.Hl, w.Wl), "mass": mass, "scores": scores}
                for part in range(min(per_head, len(groups))):
                    mine = groups[part::per_head]
                    a, bconn = ctx.Pipe()
                    p = ctx.Process(target=_oracle_worker, args=(bconn, path, meta), daemon=True)
                    p.start()
                    self.slots.append((p, a, mine))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
        for _, a, _ in self.slots:
            if a.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")
        self.groups = sum(len(s[2]) for s in self.slots)
        self.max_groups = max(len(s[2]) for s in self.slots)     # rounds until every group has run once
        self.rounds = 0

    @property
    def cores(self):
        return len(self.slots)

    def round(self):
        """Every process runs one of its groups (in turn); returns (pairs, wall seconds)."""
        t0 = time.perf_counter()
        for _, a, mine in self.slots:
            a.send(mine[self.rounds % len(mine)])
        pairs = sum(a.recv()[0] for _, a, _ in self.slots)
        self.rounds += 1
        return pairs, time.perf_counter() - t0

    def close(self):
        import shutil
        for p, a, _ in self.slots:
            try:
                a.send(None)
            except OSError:
                pass
        for p, _, _ in self.slots:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
        shutil.rmtree(self.tmp, ignore_errors=True)

    def describe(self):
        sample = oracle_sample(self.w)
        return (f"{self.groups} seeded query groups of {self.w.name} ({len(sample[0][1])} in each of "
                f"{len(sample)} seeded (batch, head) slices {[bh for bh, _ in sample]}); per group the fp64 numpy "
                f"oracle's predictor row, top-k, attention forward and the group's backward (dQ and its dK/dV "
                f"contributions) over every pair of its list; {self.cores} processes, one per host core, BLAS "
                f"single-threaded")


def _scratch_dir(w, heads):
    """A directory with room for the sampled slices' raw bf16 tensors."""
    import shutil
    need = 2 * heads * 4 * w.N * w.d * 2
    for cand in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(cand) and shutil.disk_usage(cand).free > need:
                return cand
        except OSError:
            continue
    return tempfile.gettempdir()


def oracle_inputs(w, device):
    """The workload's tensors for the sampled (batch, head) slices only (drawn
    on `device` from the same seeded generators, so they are the values the
    GPU arm sees), with head_index mapping a head to its position."""
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    heads = sorted({h for (_, h), _ in oracle_sample(w)})
    x = wl.make_inputs(w, device=device, heads=heads)
    x.head_index = {h: i for i, h in enumerate(heads)}
    return x


def cpu_baseline(w, x, min_s=10.0, max_s=30.0, cube=None, mass=None, scores="mean"):
    """The oracle on the host cores over the seeded sample, in the metric's
    unit: effective FLOPs of the pairs it processed over its wall time.
    Rounds repeat (cycling through the sample) until min_s has passed."""
    xs = _Tensors()
    for nm in ("Q", "K", "V", "dO", "Wq", "Wk", "k_per_head"):
        setattr(xs, nm, getattr(x, nm))
    xs.head_index = {h: h for h in range(w.H)}
    pool = OraclePool(w, xs, cube=cube, mass=mass, scores=scores)
    try:
        fwd_f, bwd_f = pair_flops(w.block, w.d)
        pairs, el = 0, 0.0
        while True:
            p, t = pool.round()
            pairs, el = pairs + p, el + t
            per = el / pool.rounds
            if (el >= min_s and pool.rounds >= pool.max_groups) or el + per > max_s:
                break
        return {"value": round((fwd_f + bwd_f) * pairs / el / 1e12, 6), "unit": UNIT, "cores": pool.cores,
                "host_cpus": os.cpu_count(), "kind": "oracle", "seconds": round(el, 2), "pairs": pairs,
                "rounds": pool.rounds,
                "sample": f"sampled: {pool.describe()}; {pool.rounds} rounds of one group per process"}
    finally:
        pool.close()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    cube = tuple(int(v) for v in args.cube.split(",")) if args.cube else None
    # the inputs come from the seeded generators on the GPU when there is one (the values the GPU arm sees)
    x = oracle_inputs(w, "cuda" if torch.cuda.is_available() else "cpu")
    pool = OraclePool(w, x, cube=cube, mass=args.mass or None, scores=args.scores)
    try:
        fwd_f, bwd_f = pair_flops(w.block, w.d)
        for _ in range(max(3, args.warmup)):
            pool.round()
        pairs, el = 0, 0.0
        for _ in range(args.steps):
            p, t = pool.round()
            pairs, el = pairs + p, el + t
        sample = f"sampled: each step one group per process; {pool.describe()}"
        cores = pool.cores
    finally:
        pool.close()
    value = (fwd_f + bwd_f) * pairs / el / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "pairs": pairs,
                   **({"cube": list(cube)} if cube else {}),
                   **({"selection": f"mass threshold tau={args.mass}, temperature 1/sqrt(d), k in [1, nb]"}
                      if args.mass else {}),
                   **({"block_scores": "tile maximum of the low-rank logits"} if args.scores == "max" else {})},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "host_cpus": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


TRAFFIC_KERNELS = {name: KERNEL_SRC[stage] for stage, name in KERNEL_OF.items()}


def write_traffic(csv_path, command, workload, heads):
    """Merge into profiles/traffic.json the mean DRAM bytes (read + write) per
    launch of each attention kernel found in an ncu CSV, with the workload and
    head count it was captured on, the pairs one launch processed, and the
    sha256 of the sources it was built from (bench.py reports null once they
    change, or on another workload)."""
    import csv

    from dynamic_block_sparse_projection_gb300 import workloads as wl
    w = wl.WORKLOADS[workload]
    if heads and heads < w.H:
        w = wl.scaled(w, name=w.name, H=heads)
    ks = wl.head_params(w)[0]
    pairs = w.B * w.nb * sum(ks)
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    h = rows[hi]
    ki, mi, vi, ui, idi = (h.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit", "ID"))
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    per_launch = {}
    for r in rows[hi + 1:]:
        if len(r) <= max(ki, mi, vi, ui) or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        name = next((k for k in TRAFFIC_KERNELS if k in r[ki]), None)
        if name is None:
            continue
        v = float(r[vi].replace(",", "")) * scale.get(r[ui], 1.0)
        key = (name, r[idi])
        per_launch[key] = per_launch.get(key, 0.0) + v
    f = ROOT / "profiles" / "traffic.json"
    out = json.loads(f.read_text()) if f.exists() else {}
    for name, src in TRAFFIC_KERNELS.items():
        vals = [v for (n, _), v in per_launch.items() if n == name]
        if not vals:
            continue
        hsh = hashlib.sha256()
        for s in (src, "dynamic_block_sparse_projection_gb300/csrc/dsv_device.cuh"):
            hsh.update((ROOT / s).read_bytes())
        out[name] = {"dram_bytes_per_launch": round(sum(vals) / len(vals)), "launches": len(vals),
                     "workload": workload, "heads": w.H, "pairs": pairs, "source_sha256": hsh.hexdigest(),
                     "command": command}
    f.write_text(json.dumps(out, indent=1) + "\n")
    print(json.dumps(out, indent=1))


DISPATCH_RHO = (0.05, 0.1, 0.2, 0.35, 0.5, 0.65, 0.8, 0.9, 0.95, 1.0)


def dispatch_profile(args):
    """The OP dispatcher's profile: on the workload's first 2 heads, the time
    of the sparse path (fused predictor + top-k, attention forward and
    backward) at kept fractions rho over the dense path (the same attention
    kernels with every block, no predictor), best of 2 after a warm-up, L2
    flushed before each run.  Written to profiles/dispatch_<workload>.json."""
    import torch
    from dynamic_block_sparse_projection_gb300 import binding as dsv
    from dynamic_block_sparse_projection_gb300 import workloads as wl
    torch.cuda.set_device(0)
    w0 = wl.WORKLOADS[args.workload]
    w = wl.scaled(w0, name=w0.name, H=min(w0.H, args.heads or 2))
    x = wl.make_inputs(w, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def timed(fn, reps=2):
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            flush.fill_(3)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    dense_hp = HotPath(dsv, x, w, [w.nb] * w.H, fused=True)
    dense_hp.run()                                     # the all-block lists (select-all path)
    torch.cuda.synchronize()
    t_dense = timed(dense_hp.attention_only)
    with ClockSampler(0) as clk:
        t_sparse = []
        for rho in DISPATCH_RHO:
            k = max(1, min(w.nb, math.ceil(rho * w.nb)))
            hp = HotPath(dsv, x, w, [k] * w.H, fused=True)
            t_sparse.append(timed(hp.run))
            del hp
    ratio = [t / t_dense for t in t_sparse]
    thr = None
    for i, r in enumerate(ratio):
        if r >= 1.0:
            if i == 0:
                thr = DISPATCH_RHO[0]
            else:
                r0, r1, x0, x1 = ratio[i - 1], r, DISPATCH_RHO[i - 1], DISPATCH_RHO[i]
                thr = x0 + (1.0 - r0) * (x1 - x0) / (r1 - r0)
            break
    out = {"workload": w.name, "heads_timed": w.H, "rho": list(DISPATCH_RHO), "ratio": [round(v, 4) for v in ratio],
           "t_sparse_ms": [round(v, 3) for v in t_sparse], "t_dense_ms": round(t_dense, 3),
           "threshold_rho": None if thr is None else round(thr, 4),
           "rule": "dense when t_sparse(rho) / t_dense >= 1 at the head's kept fraction (linear between points)",
           "sparse_path": "dsv_predict_topk_blocks + dsv_sparse_attn_fwd + the three backward stages",
           "dense_path": "dsv_sparse_attn_fwd + dsv_sparse_attn_bwd with every block (k = nb), no predictor",
           "clocks": clk.summary(),
           "command": "python bench.py --dispatch-profile --workload " + w.name}
    (ROOT / "profiles" / f"dispatch_{w.name}.json").write_text(json.dumps(out, indent=1) + "\n")
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.dispatch_profile:
        dispatch_profile(args)
        return
    if args.traffic_from:
        write_traffic(args.traffic_from, args.traffic_command, args.workload, args.heads)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
