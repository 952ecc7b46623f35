#!/usr/bin/env python
"""Benchmark of the chunked gated delta rule (forward + backward) on GB300.

One step = gdr_fwd followed by gdr_bwd over one batch of the named workload
(default: bf16, B=2, T=4096, H=16, DK=DV=128, "KV" states, S0 and dS_T given), with
the inputs already resident in HBM.  An L2 flush (a 512 MB write, > 2x the 129 MB
L2) runs between timed steps, outside the timed intervals.  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
(weak scaling, no collective on the data path); the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle (the baseline arm) on a bounded
sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDR fwd+bwd tokens/s & % of roofline at B=2 T=4096 H=16 DK=DV=128 bf16"
UNIT = "tokens/s"
FLUSH_BYTES = 512 << 20
CHUNK = 64

# Which of the operator's own tensors each kernel stage reads (r) or writes (w): its
# algorithmic bytes are the compulsory bytes of those tensors (workspace traffic is
# not algorithmic and shows up only in the ncu "traffic" figure).
STAGE_IO = {
    "index": ("", ""),
    "fwd_prep": ("q k v g beta", ""),
    "fwd_state": ("q k S0", "o h_saved S_T"),
    "fwd_fused": ("q k v g beta S0", "o h_saved S_T"),
    "fwd_out": ("q", "o"),
    "bwd_prep": ("q k v g beta", ""),
    "bwd_vn": ("h_saved", ""),
    "bwd_walk": ("dO dS_T", "dS0"),
    "bwd_grad": ("q k v dO beta h_saved", "dq dk dv dg dbeta"),

    "bwd_group_reduce": ("", "dq dk"),
    "bwd_walkgrad": ("q k v dO beta h_saved dS_T", "dq dk dv dg dbeta dS0"),
    "prologue": ("q k g beta", ""),
    # context-parallel passes: the outputs are written by both passes; the second is counted
    "fwd_cp_maps": ("q k S0", ""),
    "fwd_cp_scan": ("", ""),
    "fwd_cp_state": ("q k", "o h_saved S_T"),
    "bwd_cp_maps": ("dO dS_T", ""),
    "bwd_cp_scan": ("", ""),
    "bwd_cp_walk": ("dO", "dS0"),
    "prologue_bwd": ("", "dq dk dg dbeta"),
}


def rank_info():
    r = int(os.environ.get("RANK", "0"))
    w = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return r, w, lr


# ----------------------------------------------------------------------------- work model
def chunk_lengths(seqlens):
    out = []
    for L in seqlens:
        out += [min(CHUNK, L - s) for s in range(0, L, CHUNK)]
    return out


def tensor_bytes(inp, w, h_el=4):
    """Bytes of every operator-level tensor of one fwd+bwd call (h_el: bytes per saved-state
    element, 4 for fp32 h_saved and 2 for the bf16 option)."""
    el = 2 if w.dtype.itemsize == 2 else 4
    tok = sum(inp["seqlens"])
    N = inp["num_seqs"]
    nch = len(chunk_lengths(inp["seqlens"]))
    st = N * w.Hv * w.DK * w.DV * 4
    qk = tok * w.Hk * w.DK * el
    vv = tok * w.Hv * w.DV * el
    return {
        "q": qk, "k": qk, "dq": qk, "dk": qk, "v": vv, "o": vv, "dO": vv, "dv": vv,
        "g": tok * w.Hv * 4, "dg": tok * w.Hv * 4, "beta": tok * w.Hv * el, "dbeta": tok * w.Hv * el,
        "S0": st if inp["S0"] is not None else 0, "S_T": st, "dS_T": st if inp["dS_T"] is not None else 0,
        "dS0": st, "h_saved": nch * w.Hv * w.DK * w.DV * h_el,
    }


def work_model(inp, w, h_el=4, save_wy=False):
    """Algorithmic FLOPs (the chunked method's GEMMs, C x C products dense, the T inverse
    as C^3/3) and compulsory HBM bytes of the forward and the backward.  With save_wy the
    backward reads the chunk factors the forward kept instead of recomputing them, so its
    flops leave out W = T' K (2 c^2 DK), U = T'' V (2 c^2 DV) and the inverse (c^3 / 3)."""
    G = w.Hv // w.Hk
    DK, DV = w.DK, w.DV
    ff = fb = 0.0
    for c in chunk_lengths(inp["seqlens"]):
        ff += 4 * c * c * DK / G + 2 * c * c * DK + 4 * c * c * DV + 6 * c * DK * DV + c ** 3 / 3
        fb += 14 * c * DK * DV + 2 * c * c * DK * (7 + 2 / G) + 10 * c * c * DV + 4 * c ** 3 + c ** 3 / 3
        if save_wy:
            fb -= 2 * c * c * DK + 2 * c * c * DV + c ** 3 / 3
    ff *= w.Hv
    fb *= w.Hv
    tb = tensor_bytes(inp, w, h_el)
    bf = sum(tb[k] for k in ["q", "k", "v", "g", "beta", "o", "h_saved", "S0", "S_T"])
    bb = sum(tb[k] for k in ["q", "k", "v", "dO", "g", "beta", "h_saved", "dq", "dk", "dv", "dg", "dbeta",
                             "dS_T", "dS0"])
    return {"flops_fwd": ff, "flops_bwd": fb, "bytes_fwd": bf, "bytes_bwd": bb, "tensor_bytes": tb}


def stage_alg_bytes(stage, tb):
    r, wr = STAGE_IO.get(stage, ("", ""))
    return sum(tb[k] for k in (r + " " + wr).split() if k)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def ncu_traffic(stage):
    """dram bytes per launch of a stage from profiles/ncu_traffic.txt, or None when the
    kernel's source has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == stage:
            src = os.path.join(ROOT, "chunked_gated_delta_04_gb300", "csrc", parts[3])
            if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != parts[2]:
                return None
            return float(parts[1])
    return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # raw samples go to BENCH_CLOCKS_DIR (default: the system temp directory)
        self.path = os.path.join(os.environ.get("BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for nm, val in zip(names[1:], p[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle arms
def _head_slice(inp, qk_heads):
    Hk = inp["q"].shape[2]
    Hv = inp["v"].shape[2]
    G = Hv // Hk
    vh = [i * G + jj for i in qk_heads for jj in range(G)]
    out = dict(inp)
    out["q"] = inp["q"][:, :, qk_heads]
    out["k"] = inp["k"][:, :, qk_heads]
    for key in ["v", "dO", "g", "beta"]:
        out[key] = inp[key][:, :, vh]
    for key in ["S0", "dS_T"]:
        if inp[key] is not None:
            out[key] = inp[key][:, vh]
    return out


def time_oracle(inp, w, n_qk_heads, nthreads, prologue=0):
    """Times the fp64 oracle (fwd + bwd, with the fused input prologue when asked) on the
    first n_qk_heads q/k heads of every sequence; returns (seconds, tokens-equivalent of the
    full workload processed)."""
    import oracle
    from oracle import prologue as oracle_prologue

    sub = _head_slice(inp, list(range(n_qk_heads)))
    t0 = time.perf_counter()
    if prologue:
        oracle_prologue.reference_with_prologue(sub, inp["layout"], prologue, backward=True, nthreads=nthreads)
    else:
        oracle.reference(sub, inp["layout"], backward=True, nthreads=nthreads)
    dt = time.perf_counter() - t0
    tokens = sum(inp["seqlens"]) * n_qk_heads / w.Hk
    return dt, tokens


def reference_arm(args, w, inp):
    r, world, _ = rank_info()
    if r != 0:
        return 0
    nthreads = os.cpu_count() or 1
    # per step: as many q/k heads (with their v-heads) of every sequence as there are host cores
    n_heads = max(1, min(w.Hk, nthreads // max(1, inp["num_seqs"])))
    for _ in range(args.warmup):
        time_oracle(inp, w, n_heads, nthreads, 7 if args.prologue else 0)
    total_t, total_tok = 0.0, 0.0
    for _ in range(args.steps):
        dt, tok = time_oracle(inp, w, n_heads, nthreads, 7 if args.prologue else 0)
        total_t += dt
        total_tok += tok
    value = total_tok / total_t
    units = inp["num_seqs"] * n_heads
    sample = (f"per step: fp64 oracle fwd+bwd on {n_heads} of {w.Hk} q/k heads (each with its {w.Hv // w.Hk} v-head{'s' if w.Hv // w.Hk > 1 else ''}) "
              f"of all {inp['num_seqs']} sequences ({sum(inp['seqlens'])} tokens); tokens scaled by {n_heads}/{w.Hk}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, inp, args.h_dtype, args.prologue, args.recompute_wy,
                              (args.cp_fwd, args.cp_bwd)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(nthreads, units), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, inp, h_dtype="f32", prologue=False, recompute_wy=False, cp=(1, 1)):
    extra = {"context_parallel_segments": {"fwd": cp[0], "bwd": cp[1]}} if max(cp) > 1 else {}
    return {**extra, "workload": w.name, "B": w.B if inp["cu_seqlens"] is None else 1, "T": int(sum(inp["seqlens"])) if
            inp["cu_seqlens"] is not None else w.T, "Hk": w.Hk, "Hv": w.Hv, "DK": w.DK, "DV": w.DV,
            "layout": w.layout, "num_seqs": inp["num_seqs"], "chunk": CHUNK,
            "varlen": inp["cu_seqlens"] is not None, "S0": inp["S0"] is not None,
            "dS_T": inp["dS_T"] is not None, "h_saved": h_dtype,
            "prologue": "qk_l2norm+g_logsigmoid+beta_sigmoid (raw inputs)" if prologue else "none",
            "wy_factors": "recomputed by the backward" if recompute_wy else "saved by the forward (save_wy)",
            "l2": "flushed (512 MB write) between timed steps", "parallelism": "replicas"}


def aggregate_throughput(local_ms, local_tokens, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: every rank processed local_tokens
    in local_ms; the job time is the max over ranks.  Returns (tokens/s, max ms)."""
    import torch

    total_ms = float(local_ms)
    world = 1
    if dist is not None:
        world = dist.get_world_size()
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return world * local_tokens / (total_ms / 1e3), total_ms


# ----------------------------------------------------------------------------- our arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="b2_t4096")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--h-dtype", default="f32", choices=["f32", "bf16"],
                    help="dtype of the saved chunk-start states (bf16 halves the largest tensor)")
    ap.add_argument("--prologue", action="store_true",
                    help="raw q, k, gate and beta logits; the operator applies the L2 norm, logsigmoid, sigmoid")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct C-ABI calls instead of a CUDA-graph replay of the same calls")
    ap.add_argument("--cp-fwd", type=int, default=1,
                    help="intra-card context parallelism: segments per sequence in the forward (1: off, -1: the "
                         "library chooses)")
    ap.add_argument("--cp-bwd", type=int, default=1,
                    help="intra-card context parallelism: segments per sequence in the backward (1: off, -1: the "
                         "library chooses)")
    ap.add_argument("--recompute-wy", action="store_true",
                    help="the backward recomputes the chunk factors (gamma, W, U, P, T) instead of reading the "
                         "ones the forward saved")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch

    from chunked_gated_delta_04_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    inp = make_inputs(w, raw=args.prologue)
    prologue_bits = 7 if args.prologue else 0
    if args.impl == "reference":
        return reference_arm(args, w, inp)

    import chunked_gated_delta_04_gb300 as gdr

    rank, world, local_rank = rank_info()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    dev = torch.device("cuda", local_rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, Hk, DK = d["q"].shape
    Hv, DV = d["v"].shape[2], d["v"].shape[3]
    h_dtype = torch.bfloat16 if args.h_dtype == "bf16" else torch.float32
    p = gdr.make_problem(B, T, Hk, Hv, DK, DV, d["q"].dtype, w.layout, d["cu_seqlens"], h_dtype=h_dtype,
                         prologue=prologue_bits, save_wy=not args.recompute_wy, cp_fwd=args.cp_fwd,
                         cp_bwd=args.cp_bwd)
    stream = torch.cuda.current_stream()
    N = p.num_seqs
    sshape = (N, Hv, DK, DV) if w.layout == "KV" else (N, Hv, DV, DK)
    o = torch.empty_like(d["v"])
    S_T = torch.empty(sshape, dtype=torch.float32, device=dev)
    h_saved = gdr.alloc_saved(p, h_dtype, dev)
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    dg, dbeta = torch.empty_like(d["g"]), torch.empty_like(d["beta"])
    dS0 = torch.empty(sshape, dtype=torch.float32, device=dev)
    ws_bytes = max(gdr.gdr_fwd_workspace_bytes(p), gdr.gdr_bwd_workspace_bytes(p))
    ws = gdr.alloc_workspace(ws_bytes, dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    outs0 = [o, S_T, dq, dk, dv, dg, dbeta, dS0]

    def fwd(src=d, outs=None, strm=None):
        oo, sT = (outs or outs0)[:2]
        st = gdr.gdr_fwd(p, src["q"], src["k"], src["v"], src["g"], src["beta"], src["S0"], oo, sT, h_saved, ws,
                         ws_bytes, strm or stream)
        if st != 0:
            raise RuntimeError(f"gdr_fwd: {gdr.gdr_status_string(st)}")

    def bwd(src=d, outs=None, strm=None):
        _, _, gq, gk, gv, gg, gb, gs0 = outs or outs0
        st = gdr.gdr_bwd(p, src["q"], src["k"], src["v"], src["g"], src["beta"], h_saved, src["dO"], src["dS_T"],
                         gq, gk, gv, gg, gb, gs0, ws, ws_bytes, strm or stream)
        if st != 0:
            raise RuntimeError(f"gdr_bwd: {gdr.gdr_status_string(st)}")

    def step(strm=None):
        fwd(strm=strm)
        bwd(strm=strm)

    def capture(fn):
        """A CUDA graph of fn's launches (the same C-ABI calls, recorded once on a capture
        stream); None when capture is not possible."""
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        try:
            with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
                fn(strm=torch.cuda.current_stream())
        except Exception as exc:  # e.g. a launch kind the driver cannot capture
            print(f"graph capture failed, timing direct calls: {exc}", file=sys.stderr)
            torch.cuda.synchronize()
            return None
        torch.cuda.synchronize()
        return g

    def flush():
        flush_buf.fill_(1)

    def timed(fn, n):
        """Device time (ms) of n calls of fn, each after an L2 flush, via CUDA events."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, flags = gdr.gdr_workspace_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {gdr.gdr_status_string(st)} (flags {flags:#x})")

    # Kernel launches of one step (counted by the library on a direct call).
    launches0 = gdr.gdr_debug_launch_count()
    flush()
    step()
    torch.cuda.synchronize()
    launches_per_step = gdr.gdr_debug_launch_count() - launches0
    # The timed steps replay a CUDA graph of the step's C-ABI calls: the same kernels with the
    # same arguments, without the host's per-launch gaps (small workloads are launch-bound).
    graphs = {}
    if not args.no_graph:
        for name, fn in (("step", step), ("fwd", fwd), ("bwd", bwd)):
            graphs[name] = capture(fn)
            if graphs[name] is None:
                graphs = {}
                break
    run = {name: (g.replay if g is not None else None) for name, g in graphs.items()}
    run_step = run.get("step") or step
    launch_mode = "cuda_graph" if graphs else "direct"

    # ---- main timed region: exactly K steps
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        step_ms = timed(run_step, args.steps)
        torch.cuda.synchronize()
        barrier()
    launches = launches_per_step * args.steps
    tokens = float(sum(inp["seqlens"]))
    value, total_ms = aggregate_throughput(sum(step_ms), tokens * args.steps, dist, dev)
    ms_per_step = total_ms / args.steps

    # ---- fwd / bwd separately (informational)
    fwd_ms = statistics.median(timed(run.get("fwd") or fwd, max(5, args.steps // 2)))
    bwd_ms = statistics.median(timed(run.get("bwd") or bwd, max(5, args.steps // 2)))

    # ---- per-kernel times with stage events (separate pass; the main loop has no hooks)
    nev = 16
    events = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    stage_tot = {}
    reps = max(5, args.steps // 2)
    stage_runs = []
    for fn in (fwd, bwd):  # each direction with its stage events (recorded inside the graph)
        gdr.gdr_debug_set_stage_events(events)
        g = capture(fn) if graphs else None
        if g is None:
            stage_runs.append((fn, None))
        else:
            stage_runs.append((g.replay, gdr.gdr_debug_stage_names()))
        gdr.gdr_debug_set_stage_events(None)
    for _ in range(reps):
        for fn, names_at_capture in stage_runs:
            if names_at_capture is None:
                gdr.gdr_debug_set_stage_events(events)
            flush()
            fn()
            torch.cuda.synchronize()
            names = names_at_capture if names_at_capture is not None else gdr.gdr_debug_stage_names()
            if names_at_capture is None:
                gdr.gdr_debug_set_stage_events(None)
            per_call = {}
            for i, nm in enumerate(names):  # a stage may launch several kernels: sum them per call
                per_call[nm] = per_call.get(nm, 0.0) + events[i].elapsed_time(events[i + 1])
            for nm, t in per_call.items():
                stage_tot.setdefault(nm, []).append(t)
    stage_ms = {k: statistics.mean(v) for k, v in stage_tot.items()}

    wm = work_model(inp, w, 2 if args.h_dtype == "bf16" else 4, save_wy=not args.recompute_wy)
    hbm, bf16_burst, bf16_sus, peak_src = load_peaks()
    dom = max(stage_ms, key=stage_ms.get)
    alg = stage_alg_bytes(dom, wm["tensor_bytes"])
    achieved = alg / (stage_ms[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": ncu_traffic(dom), "alg_bytes": alg,
                "avg_launch_ms": stage_ms[dom], "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    t_hbm_step = (wm["bytes_fwd"] + wm["bytes_bwd"]) / (hbm * 1e9) * 1e3
    t_flop_step = (wm["flops_fwd"] + wm["flops_bwd"]) / (bf16_sus * 1e12) * 1e3
    step_roof = max(t_hbm_step, t_flop_step)

    def dir_obj(ms, flops, nbytes):
        t_roof = max(nbytes / (hbm * 1e9), flops / (bf16_sus * 1e12)) * 1e3
        return {"ms": ms, "tokens_per_s": tokens / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
                "gbs": nbytes / (ms / 1e3) / 1e9, "roofline_ms": t_roof, "roofline_frac": t_roof / ms}

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region.
    # Every step uploads its own inputs and downloads all its outputs; with two buffer sets and
    # separate upload / download streams, step k+1's upload and step k-1's download run while
    # step k computes (the inputs come from the host each step, larger than L2: no flush here).
    in_keys = ["q", "k", "v", "g", "beta", "S0", "dO", "dS_T"]
    host_in = {k: inp[k].pin_memory() for k in in_keys if inp[k] is not None}
    sets = []
    for b in range(2):
        din = {k: torch.empty_like(d[k]) for k in host_in}
        din["cu_seqlens"] = d["cu_seqlens"]
        for k in in_keys:
            din.setdefault(k, None)
        douts = outs0 if b == 0 else [torch.empty_like(t) for t in outs0]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
        ev = {n: torch.cuda.Event() for n in ("in", "done", "out")}
        sets.append((din, douts, hout, ev))
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in outs0)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n_steps):
        for kstep in range(n_steps):
            din, douts, hout, ev = sets[kstep % 2]
            with torch.cuda.stream(up):  # inputs of this step (after step k-2 has read this set)
                up.wait_event(ev["done"])
                for k, t in host_in.items():
                    din[k].copy_(t, non_blocking=True)
                ev["in"].record(up)
            stream.wait_event(ev["in"])
            stream.wait_event(ev["out"])  # step k-2's results have left this set's outputs
            fwd(din, douts, stream)
            bwd(din, douts, stream)
            ev["done"].record(stream)
            with torch.cuda.stream(down):  # all outputs of this step to the host
                down.wait_event(ev["done"])
                for h, t in zip(hout, douts):
                    h.copy_(t, non_blocking=True)
                ev["out"].record(down)

    for b in range(2):  # events start recorded (nothing pending)
        for e in sets[b][3].values():
            e.record(stream)
    e2e_run(2)
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    e2e_run(args.steps)
    stream.wait_stream(up)
    stream.wait_stream(down)
    t_b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = [t_a.elapsed_time(t_b)]
    e2e_value, _ = aggregate_throughput(sum(e2e_ms), tokens * args.steps, dist, dev)

    # ---- oracle on host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # about 10 s of host time: repeat the oracle on a head sample until 10 s have passed
        nthreads = os.cpu_count() or 1
        n_heads = max(1, min(w.Hk, nthreads // max(1, inp["num_seqs"])))
        tot_t = tot_tok = 0.0
        reps = 0
        while tot_t < 10.0 and reps < 50:
            dt, tok = time_oracle(inp, w, n_heads, nthreads, 7 if args.prologue else 0)
            tot_t += dt
            tot_tok += tok
            reps += 1
        cpu = {"value": tot_tok / tot_t, "unit": UNIT, "cores": min(nthreads, inp["num_seqs"] * n_heads),
               "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd, {reps} run(s) over {n_heads} of {w.Hk} q/k heads of all "
                         f"{inp['num_seqs']} sequences ({tot_t:.1f} s); tokens scaled by {n_heads}/{w.Hk}"}

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded; see chunked_gated_delta_04_gb300/inputs.py)",
            "config": config_dict(w, inp, args.h_dtype, args.prologue, args.recompute_wy,
                                  gdr.gdr_debug_cp_segments(p)),
            "roofline": roofline,
            "step_roofline": {"ms": step_roof, "frac": step_roof / ms_per_step, "bound": "hbm" if
                              t_hbm_step >= t_flop_step else "tensor", "bytes": wm["bytes_fwd"] + wm["bytes_bwd"],
                              "flops": wm["flops_fwd"] + wm["flops_bwd"]},
            "fwd": dir_obj(fwd_ms, wm["flops_fwd"], wm["bytes_fwd"]),
            "bwd": {**dir_obj(bwd_ms, wm["flops_bwd"], wm["bytes_bwd"]),
                    "flops_counted": "with the chunk-factor recompute" if args.recompute_wy else
                    "without the chunk-factor recompute (W, U, T read from the forward's saved buffer)"},
            "stages_ms": stage_ms,
            "path": "tcgen05" if gdr.gdr_path(p) == 1 else "simt",
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "2 buffer sets; upload, compute, download on 3 streams"},
            "gpu_launches": launches,
            "launch": launch_mode,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
