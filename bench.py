"""Benchmark of the SwiGLU-FFN backward (M=220000, K=512, N=1024, bf16) and SwishGrad.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one whole backward over the seeded synthetic workload: one call of
the public C-ABI entry point swiglu_bwd (dg, dfc not returned), with CUDA
events around every call. The default (--path fused) is the fused chain
(SWG_FUSED): the x and w stages with the b-stage math inside both GEMMs'
operand producers; when the w stage leaves SMs free, the call runs the x
stage's last tiles beside it. The kernels' own times ("stages", "roofline")
come from a second timed pass of the same chain as stage calls
(swiglu_bwd_x_fused, then swiglu_bwd_w_fused) with events between them. The
other chain -- the b stage (dg, dfc, db), the w stage and the x stage as three
calls -- is timed beside it as stage calls and reported under "other_path". Inputs (dy, g, fc: 450 MB each) are larger than the
129 MB L2, so no flush is needed between steps; SwishGrad (100 MB of bf16 I/O
per launch) is timed over back-to-back launches that rotate through six
input/output sets (576 MB), so that every launch reads its inputs from HBM.
The sibling activation gradients (GELU, HardSwish) are timed the same way;
the GroupNorm backward on ResNet-50 stage-1 activations at batch 32
([32, 256, 56, 56], 32 groups, fp16) over three rotating sets (462 MB), with
PyTorch's own GroupNorm backward on the same inputs beside it.

Prints ONE JSON line (rank 0). `value` is milliseconds per backward (lower is
better); `pct_roofline` is the roofline time max(8MKN / tensor peak,
(6MN + 4MK + 8KN + 4N) / HBM peak) over the measured time. `--impl reference`
times the fp64 CPU oracle on a row sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, K, N = 220000, 512, 1024
METRIC = "SwiGLU-bwd ms & % roofline (M220000 K512 N1024 bf16); SwishGrad GB/s"
WORKLOAD = "swiglu_bwd M=220000 K=512 N=1024 bf16 (pages' test shape), seed 0"
SWISH_N = 1 << 24


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def _roofline_ms(pk, sustained=False):
    flop = 8.0 * M * K * N
    byts = 6.0 * M * N + 4.0 * M * K + 8.0 * K * N + 4.0 * N  # every input read once, outputs written once
    tf = pk["bf16_sustained"] if sustained else pk["bf16"]
    return max(flop / (tf * 1e12), byts / (pk["hbm"] * 1e9)) * 1e3


# ---------------------------------------------------------------- distributed plumbing
def _dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("SWG_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- traffic from the committed ncu summary
def _src_sha(name):
    p = os.path.join(ROOT, "swiglu_ffn_backward_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _traffic(kernel):
    """Per-launch DRAM bytes from profiles/dram_traffic.json, or None when the
    kernel's source changed since those counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            t = json.load(f)[kernel]
        if t["source_sha"] != _src_sha(t["source"]):
            return None
        return float(t["bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch

    import swiglu_ffn_backward_gb300 as swg
    from synth import SWIGLU_CONFIGS, swiglu_inputs, swish_inputs

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")
    pk = _peaks()
    shape = SWIGLU_CONFIGS["pages"][0]
    if M != shape.M:
        from synth import SwigluShape
        shape = SwigluShape(f"pages_M{M}", M, K, N, shape.seed, shape.dist)
    inp = swiglu_inputs(shape, device=dev)
    # the e2e leg's pinned host buffers, allocated before any other host memory comes and goes
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
    for k, v in inp.items():
        host_in[k].copy_(v)
    host_out = {k: torch.empty(shp, dtype=torch.bfloat16, pin_memory=True)
                for k, shp in (("dx", (M, K)), ("dw_g", (K, N)), ("dw_fc", (K, N)), ("db_g", (1, N)), ("db_fc", (1, N)))}
    bf = dict(dtype=torch.bfloat16, device=dev)
    dg = torch.empty((M, N), **bf)
    dfc = torch.empty((M, N), **bf)
    db_g = torch.empty((1, N), **bf)
    db_fc = torch.empty((1, N), **bf)
    dw_g = torch.empty((K, N), **bf)
    dw_fc = torch.empty((K, N), **bf)
    dx = torch.empty((M, K), **bf)
    ws_b = torch.empty(max(swg.swiglu_bwd_b_workspace_size(M, N), 16), dtype=torch.uint8, device=dev)
    ws_w_bytes = swg.swiglu_bwd_w_workspace_size(M, K, N)
    ws_w = torch.empty(max(ws_w_bytes, 16), dtype=torch.uint8, device=dev)
    ws_fw_bytes = swg.swiglu_bwd_w_fused_workspace_size(M, K, N)
    ws_fw = torch.empty(max(ws_fw_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # each path: a list of (kernel name, launch) issued in order; CUDA events
    # go between them so every kernel is timed inside the timed region
    unfused = [
        ("b_stage", lambda: swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"], dg, dfc, db_g, db_fc, workspace=ws_b)),
        ("w_gemm", lambda: swg.swiglu_bwd_w(inp["x"], dg, dfc, dw_g, dw_fc, workspace=ws_w)),
        ("x_gemm", lambda: swg.swiglu_bwd_x(dg, dfc, inp["w_g"], inp["w_fc"], dx)),
    ]
    fused = [
        ("x_fused", lambda: swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"], dx)),
        ("w_fused", lambda: swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"], dw_g, dw_fc,
                                                   db_g, db_fc, workspace=ws_fw)),
    ]
    paths = {"unfused": unfused, "fused": fused}
    # the timed step: the public whole-backward call of the chain (dg, dfc not returned)
    call_outs = dict(dx=dx, dw_g=dw_g, dw_fc=dw_fc, db_g=db_g, db_fc=db_fc)
    flag_of = {"fused": swg.SWG_FUSED, "unfused": swg.SWG_UNFUSED}
    call_ws = torch.empty(max(swg.swiglu_bwd_workspace_size(M, K, N, flag_of[args.path]), 16), dtype=torch.uint8,
                          device=dev)
    whole = [("swiglu_bwd", lambda: swg.swiglu_bwd(**inp, fused=args.path == "fused", return_dg=False,
                                                   out=call_outs, workspace=call_ws))]
    launches = {p: swg.swiglu_bwd_kernel_count(M, K, N, f) for p, f in flag_of.items()}

    def step(seq, ev=None):
        for j, (_, fn) in enumerate(seq):
            if ev is not None:
                ev[j].record(stream)
            fn()
        if ev is not None:
            ev[len(seq)].record(stream)

    main_path = paths[args.path]
    for seq in [whole] + list(paths.values()):
        for _ in range(args.warmup):
            step(seq)
    swg.swg_check()
    if args.profile_only:
        # a plain launch sequence for ncu captures: no timing is reported
        for _ in range(args.steps):
            step(main_path)
        swg.swg_check()
        if rank == 0:
            print(json.dumps({"profile_only": True, "path": args.path, "M": M, "K": K, "N": N,
                              "steps": args.steps}), flush=True)
        return

    def timed(seq, steps, with_clocks):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(seq) + 1)] for _ in range(steps)]
        clocks = Clocks(torch.cuda.current_device()) if with_clocks else None
        _barrier(world)
        torch.cuda.synchronize()
        if clocks:
            clocks.start()
            time.sleep(0.3)  # let the sampler start before the timed region
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            step(seq, evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks else None
        _barrier(world)
        swg.swg_check()
        ms_ = _max_over_ranks(t0.elapsed_time(t1) / steps, world)
        per = {}
        for j, (name, _) in enumerate(seq):
            per[name] = sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps
        return ms_, per, clk

    # algorithmic work per launch (bytes for HBM-bound, flops for tensor-bound)
    gemm_flop = 4.0 * M * K * N
    kernels = {
        "b_stage": dict(bound="hbm", work=10.0 * M * N + 4.0 * N, peak=pk["hbm"], unit="GB/s", src="b_stage.cu"),
        "w_gemm": dict(bound="tensor", work=gemm_flop, peak=pk["bf16"], unit="TFLOP/s", src="gemm_tc.cu"),
        "x_gemm": dict(bound="tensor", work=gemm_flop, peak=pk["bf16"], unit="TFLOP/s", src="xgemm_tc.cu"),
        "x_fused": dict(bound="tensor", work=gemm_flop, peak=pk["bf16"], unit="TFLOP/s", src="fused_tc.cu"),
        "w_fused": dict(bound="tensor", work=gemm_flop, peak=pk["bf16"], unit="TFLOP/s", src="fused_tc.cu"),
    }

    def describe(per):
        out = {}
        for k, t in per.items():
            kd = kernels[k]
            sc = 1e-9 if kd["unit"] == "GB/s" else 1e-12
            a = kd["work"] * sc / (t * 1e-3)
            out[k] = {"ms": round(t, 4), "achieved": round(a, 1), "unit": kd["unit"], "frac": round(a / kd["peak"], 4)}
            if kd["unit"] == "TFLOP/s":
                out[k]["frac_sustained"] = round(a / pk["bf16_sustained"], 4)
        return out

    ms, _, clk = timed(whole, args.steps, True)
    # the same chain as stage calls, events between them: each kernel's own time. The GPU idles
    # for two seconds first, so that this pass does not start where the previous one left the
    # power-capped clocks.
    time.sleep(2.0)
    ms_stages, per_main, _ = timed(main_path, args.steps, False)
    other = "unfused" if args.path == "fused" else "fused"
    ms_other, per_other, _ = timed(paths[other], max(args.steps // 4, 10), False)
    dom = max(per_main, key=per_main.get)
    kd = kernels[dom]
    scale = 1e-9 if kd["unit"] == "GB/s" else 1e-12
    achieved = kd["work"] * scale / (per_main[dom] * 1e-3)
    roof = {"kernel": dom, "bound": kd["bound"], "achieved": round(achieved, 1), "peak": kd["peak"],
            "unit": kd["unit"], "frac": round(achieved / kd["peak"], 4), "traffic": _traffic(dom),
            "peak_source": pk["source"] + (" burst" if kd["unit"] == "TFLOP/s" else "")}
    if kd["unit"] == "TFLOP/s":
        # the timed passes are ~0.8 s loops under the power cap: the sustained peak is the like-for-like one
        roof["frac_sustained"] = round(achieved / pk["bf16_sustained"], 4)
    stages = describe(per_main)

    # SwishGrad GB/s, bf16, n = 2^24, beta = 1.702. One launch moves 100 MB, less
    # than the 129 MB L2, so launches rotate over 6 input/output sets (576 MB):
    # each launch's inputs come from HBM and the previous launches' outputs are
    # written back during the timed launches, as in a steady stream. (An L2
    # flush by a memset would instead leave the flush's dirty lines to be
    # written back inside the timed launch.)
    sets = []
    for j in range(6):
        grad, xs = swish_inputs(SWISH_N, torch.bfloat16, device=dev, seed=1 + j)
        sets.append((grad, xs, torch.empty_like(grad)))
    sw_warm = max(3, args.warmup)
    sw_n = 60

    def stream_time(fn):
        """(stream average, per-launch median) in ms of fn over sw_n rotating launches: the
        average comes from one event pair around all launches (back-to-back calls, as in a
        stream of work), the median from events between every two launches."""
        for i in range(sw_warm):
            fn(*sets[i % 6])
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(sw_n):
            fn(*sets[(sw_warm + i) % 6])
        e1.record(stream)
        torch.cuda.synchronize()
        avg = e0.elapsed_time(e1) / sw_n
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(sw_n + 1)]
        for i in range(sw_n):
            ev[i].record(stream)
            fn(*sets[(sw_warm + i) % 6])
        ev[sw_n].record(stream)
        torch.cuda.synchronize()
        return avg, statistics.median([ev[i].elapsed_time(ev[i + 1]) for i in range(sw_n)])

    sw_bytes = 3.0 * SWISH_N * 2
    gbs = lambda ms_: sw_bytes / (ms_ * 1e-3) / 1e9  # noqa: E731
    sw_ms, sw_med = stream_time(lambda g_, x_, o_: swg.swish_grad(g_, x_, 1.702, grad_x=o_))
    sw_gbs = gbs(sw_ms)
    # the same bytes (two reads, one write of 2^24 bf16) through PyTorch's own
    # elementwise kernel, same rotation and timing
    add_ms, add_med = stream_time(lambda g_, x_, o_: torch.add(g_, x_, out=o_))
    add_gbs = gbs(add_ms)
    # the sibling activation gradients through the same streaming kernels, same timing
    act = {}
    for name in ("gelu", "hardswish"):
        a_ms, a_med = stream_time(lambda g_, x_, o_, nm=name: swg.act_grad(g_, x_, nm, grad_x=o_))
        act[name] = {"ms": round(a_ms, 5), "gbs": round(gbs(a_ms), 1), "frac_hbm": round(gbs(a_ms) / pk["hbm"], 4),
                     "per_launch_median_ms": round(a_med, 5)}
    swg.swg_check()
    del sets

    # GroupNorm backward (dx, dgamma, dbeta): ResNet-50 stage-1 activations at batch 32,
    # [32, 256, 56, 56], 32 groups, fp16; three rotating input/output sets (462 MB, over L2).
    # PyTorch's own CUDA GroupNorm backward on the same inputs is timed beside it (its
    # forward's mean and rstd computed outside the timing).
    from synth import GROUP_NORM_CONFIGS, GROUP_NORM_EPS, group_norm_inputs
    gN, gC, gHW, gG = GROUP_NORM_CONFIGS["resnet50_stage1_b32"]
    gsets = []
    for j in range(3):
        g_dy, g_x, g_gam = group_norm_inputs(gN, gC, gHW, gG, torch.float16, device=dev, seed=20 + j)
        gsets.append(dict(dy=g_dy, x=g_x, g=g_gam, dx=torch.empty_like(g_x), dg=torch.empty_like(g_gam),
                          db=torch.empty_like(g_gam),
                          ws=torch.empty(swg.group_norm_bwd_workspace_size(gN, gC, gHW, gG), dtype=torch.uint8,
                                         device=dev)))

    def gn_ours(s_):
        swg.group_norm_bwd(s_["dy"], s_["x"], gG, gamma=s_["g"], eps=GROUP_NORM_EPS, dx=s_["dx"],
                           dgamma=s_["dg"], dbeta=s_["db"], workspace=s_["ws"])

    def gn_torch(s_):
        torch.ops.aten.native_group_norm_backward(s_["dy"], s_["x"], s_["mean"], s_["rstd"], s_["g"], gN, gC,
                                                  gHW, gG, [True, True, True])

    for s_ in gsets:
        _, s_["mean"], s_["rstd"] = torch.ops.aten.native_group_norm(s_["x"], s_["g"], None, gN, gC, gHW, gG,
                                                                      GROUP_NORM_EPS)

    def time_rot(fn, n=60):
        for i in range(max(3, args.warmup)):
            fn(gsets[i % 3])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        for i in range(n):
            ev[i].record(stream)
            fn(gsets[i % 3])
        ev[n].record(stream)
        torch.cuda.synchronize()
        return statistics.median([ev[i].elapsed_time(ev[i + 1]) for i in range(n)])

    gn_ms = time_rot(gn_ours)
    swg.swg_check()
    gn_torch_ms = time_rot(gn_torch)

    def time_graph(fn, reps=20):
        # the same calls replayed from a CUDA graph: no host launch overhead between them
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for s_ in gsets:
                fn(s_)
        for _ in range(3):
            graph.replay()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        return g0.elapsed_time(g1) / (reps * len(gsets))

    gn_graph_ms = time_graph(gn_ours)
    swg.swg_check()
    gn_bytes = 3.0 * gN * gC * gHW * 2 + 3.0 * gC * 2
    gn = {"workload": "resnet50 stage-1 activations, batch 32", "shape": [gN, gC, 56, 56], "groups": gG,
          "dtype": "f16", "ms": round(gn_ms, 5), "gbs": round(gn_bytes / (gn_ms * 1e-3) / 1e9, 1),
          "frac_hbm": round(gn_bytes / (gn_ms * 1e-3) / 1e9 / pk["hbm"], 4),
          "graph_ms": round(gn_graph_ms, 5), "torch_native_ms": round(gn_torch_ms, 5)}
    del gsets

    # accumulate mode: the public whole-backward call (fused chain, dg/dfc not
    # returned) with and without SWG_ACCUMULATE, device-resident inputs
    acc_outs = dict(dx=dx, dw_g=dw_g, dw_fc=dw_fc, db_g=db_g, db_fc=db_fc)
    acc_ws = torch.empty(max(swg.swiglu_bwd_workspace_size(M, K, N, 1), 16), dtype=torch.uint8, device=dev)

    def acc_call(acc):
        swg.swiglu_bwd(**inp, fused=True, return_dg=False, out=acc_outs, workspace=acc_ws, accumulate=acc)

    acc_ms = {}
    for acc in (False, True):
        for _ in range(3):
            acc_call(acc)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(20):
            acc_call(acc)
        a1.record(stream)
        torch.cuda.synchronize()
        acc_ms["accumulate" if acc else "overwrite"] = round(a0.elapsed_time(a1) / 20, 4)
    swg.swg_check()

    # forward (g, fc, y from x, W, b) at the same shape: one launch
    from synth import swiglu_fwd_biases
    fb_g, fb_fc = swiglu_fwd_biases(shape, device=dev)
    fout = {k: torch.empty((M, N), **bf) for k in ("g", "fc", "y")}

    def fwd_call():
        swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], fb_g, fb_fc, out=fout)

    for _ in range(3):
        fwd_call()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(30):
        fwd_call()
    f1.record(stream)
    torch.cuda.synchronize()
    swg.swg_check()
    fwd_ms = f0.elapsed_time(f1) / 30
    fwd_flop = 4.0 * M * K * N
    fwd_bytes = 2.0 * M * K + 4.0 * K * N + 4.0 * N + 6.0 * M * N
    fwd_roof = max(fwd_flop / (pk["bf16"] * 1e12), fwd_bytes / (pk["hbm"] * 1e9)) * 1e3
    fwd = {"ms": round(fwd_ms, 4), "tflops": round(fwd_flop / (fwd_ms * 1e-3) / 1e12, 1),
           "gbs": round(fwd_bytes / (fwd_ms * 1e-3) / 1e9, 1), "roofline_ms": round(fwd_roof, 4),
           "pct_roofline": round(fwd_roof / fwd_ms, 4)}
    del fout

    # e2e: every input and output in pinned host memory, all host<->device copies
    # inside the timed region. The public call is swiglu_bwd_host (the fused
    # backward from host buffers: chunked over M, copies overlapped with the
    # compute); beside it, the same work as PyTorch copies around the
    # device-resident swiglu_bwd call (copies, then compute, then copies).
    outs = dict(dx=dx, dw_g=dw_g, dw_fc=dw_fc, db_g=db_g, db_fc=db_fc)
    ws_host = torch.empty(swg.swiglu_bwd_host_workspace_size(M, K, N), dtype=torch.uint8, device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def e2e_step():
        swg.swiglu_bwd_host(**host_in, out=host_out, workspace=ws_host)

    dev_in = {k: torch.empty_like(v) for k, v in inp.items()}
    use_fused = args.path == "fused"
    ws_full = torch.empty(max(swg.swiglu_bwd_workspace_size(M, K, N, 1 if use_fused else 0), 16),
                          dtype=torch.uint8, device=dev)

    def e2e_serial_step():
        for k in dev_in:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        swg.swiglu_bwd(**dev_in, fused=use_fused, return_dg=False, out=outs, workspace=ws_full)
        for k in host_out:
            host_out[k].copy_(outs[k], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))

    def time_e2e(step):
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        _barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        swg.swg_check()
        return _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    e2e_ms = time_e2e(e2e_step)
    e2e_serial_ms = time_e2e(e2e_serial_step)
    del ws_host, dev_in, ws_full

    llm = None if args.no_llm else llm_leg(swg, pk, stream)
    tail = tail_leg(swg, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp)

    roof_ms = _roofline_ms(pk)
    line = {
        "metric": METRIC, "value": round(ms, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded randn, bf16)",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N,
                   "path": (f"{args.path}: swiglu_bwd whole call; kernel times from a second timed pass of "
                            "the stage calls " + ", ".join(n for n, _ in main_path)),
                   "l2": "inputs larger than L2 (dy, g, fc 450 MB each); SwishGrad: 6 rotating sets, 576 MB",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_roofline": round(roof_ms / ms, 4), "roofline_ms": round(roof_ms, 4),
        "pct_roofline_sustained": round(_roofline_ms(pk, sustained=True) / ms, 4),
        "tflops": round(8.0 * M * K * N / (ms * 1e-3) / 1e12, 1),
        "roofline": roof, "stages": stages, "stage_calls_ms": round(ms_stages, 4),
        "other_path": {"path": other, "ms": round(ms_other, 4), "pct_roofline": round(roof_ms / ms_other, 4),
                       "stages": describe(per_other)},
        "swish_grad": {"n": SWISH_N, "dtype": "bf16", "scale": 1.702, "ms": round(sw_ms, 5),
                       "gbs": round(sw_gbs, 1), "frac_hbm": round(sw_gbs / pk["hbm"], 4),
                       "timing": "60 back-to-back launches over 6 rotating input/output sets (576 MB), "
                                 "one event pair around them; per_launch_median_ms has events between launches",
                       "per_launch_median_ms": round(sw_med, 5),
                       "same_bytes_torch_add": {"ms": round(add_ms, 5), "gbs": round(add_gbs, 1),
                                                "frac_hbm": round(add_gbs / pk["hbm"], 4),
                                                "per_launch_median_ms": round(add_med, 5)},
                       "vs_torch_add": round(add_ms / sw_ms, 4)},
        "act_grad": {"n": SWISH_N, "dtype": "bf16", **act},
        "group_norm_bwd": gn,
        "swiglu_bwd_call": {"unit": "ms", "fused": True, **acc_ms},
        "swiglu_fwd": fwd,
        "llm": llm,
        "tail": tail,
        "e2e": {"value": round(e2e_ms, 3), "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "call": "swiglu_bwd_host (fused; pinned host buffers, copies overlapped)",
                "serial_ms": round(e2e_serial_ms, 3),
                "serial_call": f"torch copies + swiglu_bwd ({args.path}, dg/dfc not returned)"},
        "gpu_launches": launches[args.path] * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "peaks": pk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- other workloads
def _chain_timer(seq, steps, stream):
    """Per-launch CUDA-event times (ms, mean over steps) of a list of (name, fn), and the
    whole sequence's time per step."""
    import torch

    for _ in range(3):
        for _, fn in seq:
            fn()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(seq) + 1)] for _ in range(steps)]
    for i in range(steps):
        for j, (_, fn) in enumerate(seq):
            evs[i][j].record(stream)
            fn()
        evs[i][len(seq)].record(stream)
    torch.cuda.synchronize()
    per = {name: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps for j, (name, _) in enumerate(seq)}
    total = sum(e[0].elapsed_time(e[len(seq)]) for e in evs) / steps
    return total, per


def llm_leg(swg, pk, stream, steps=10):
    """The whole backward at LLM-FFN scale (M=16384 tokens, K=4096 hidden, N=14336
    intermediate, bf16): both chains, per-kernel time and fraction of the measured
    bf16 peak (burst and sustained), and which chain is faster at this shape."""
    import torch

    from synth import SWIGLU_CONFIGS, swiglu_inputs

    sh = SWIGLU_CONFIGS["llm"][0]
    Ml, Kl, Nl = sh.M, sh.K, sh.N
    dev = torch.device("cuda")
    inp = swiglu_inputs(sh, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    dg, dfc = torch.empty((Ml, Nl), **bf), torch.empty((Ml, Nl), **bf)
    db_g, db_fc = torch.empty((1, Nl), **bf), torch.empty((1, Nl), **bf)
    dw_g, dw_fc = torch.empty((Kl, Nl), **bf), torch.empty((Kl, Nl), **bf)
    dx = torch.empty((Ml, Kl), **bf)
    ws_b = torch.empty(max(swg.swiglu_bwd_b_workspace_size(Ml, Nl), 16), dtype=torch.uint8, device=dev)
    ws_w = torch.empty(max(swg.swiglu_bwd_w_workspace_size(Ml, Kl, Nl), 16), dtype=torch.uint8, device=dev)
    ws_fw = torch.empty(max(swg.swiglu_bwd_w_fused_workspace_size(Ml, Kl, Nl), 16), dtype=torch.uint8, device=dev)
    chains = {
        "unfused": [
            ("b_stage", lambda: swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"], dg, dfc, db_g, db_fc,
                                                 workspace=ws_b)),
            ("w_gemm", lambda: swg.swiglu_bwd_w(inp["x"], dg, dfc, dw_g, dw_fc, workspace=ws_w)),
            ("x_gemm", lambda: swg.swiglu_bwd_x(dg, dfc, inp["w_g"], inp["w_fc"], dx)),
        ],
        "fused": [
            ("x_fused", lambda: swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"], dx)),
            ("w_fused", lambda: swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"], dw_g, dw_fc,
                                                       db_g, db_fc, workspace=ws_fw)),
        ],
    }
    flop_gemm = 4.0 * Ml * Kl * Nl
    flop = 2 * flop_gemm
    byts = 6.0 * Ml * Nl + 4.0 * Ml * Kl + 8.0 * Kl * Nl + 4.0 * Nl
    roof_ms = max(flop / (pk["bf16"] * 1e12), byts / (pk["hbm"] * 1e9)) * 1e3
    out = {"workload": "swiglu_bwd LLM FFN M=16384 K=4096 N=14336 bf16, seed 3", "M": Ml, "K": Kl, "N": Nl,
           "roofline_ms": round(roof_ms, 4), "steps": steps}
    for name, seq in chains.items():
        total, per = _chain_timer(seq, steps, stream)
        kern = {}
        for k, t in per.items():
            if k == "b_stage":
                gbs = (10.0 * Ml * Nl + 4.0 * Nl) / (t * 1e-3) / 1e9
                kern[k] = {"ms": round(t, 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm"], 4)}
            else:
                tf = flop_gemm / (t * 1e-3) / 1e12
                kern[k] = {"ms": round(t, 4), "tflops": round(tf, 1), "frac_burst": round(tf / pk["bf16"], 4),
                           "frac_sustained": round(tf / pk["bf16_sustained"], 4)}
        out[name] = {"ms": round(total, 4), "tflops": round(flop / (total * 1e-3) / 1e12, 1),
                     "pct_roofline": round(roof_ms / total, 4), "kernels": kern}
    swg.swg_check()
    out["faster_path"] = min(chains, key=lambda n: out[n]["ms"])
    del inp, dg, dfc, ws_b, ws_w, ws_fw
    torch.cuda.empty_cache()
    return out


def tail_leg(swg, stream, reps=20):
    """The dynamic-M tail sweep (K=512, N=1024, M in 1, 127, 1025, 4097, 65537): the
    public whole-backward call per chain, microseconds per call. L2 is flushed
    (a 512 MB write) before each timed call, outside its events."""
    import torch

    from synth import SWIGLU_CONFIGS, swiglu_inputs

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rows = []
    for sh in SWIGLU_CONFIGS["tail"]:
        inp = swiglu_inputs(sh, device="cuda")
        r = {"M": sh.M}
        bf = dict(dtype=torch.bfloat16, device="cuda")
        out = dict(dx=torch.empty((sh.M, sh.K), **bf), dw_g=torch.empty((sh.K, sh.N), **bf),
                   dw_fc=torch.empty((sh.K, sh.N), **bf), db_g=torch.empty((1, sh.N), **bf),
                   db_fc=torch.empty((1, sh.N), **bf))
        for fused in (False, True):
            ws = torch.empty(max(swg.swiglu_bwd_workspace_size(sh.M, sh.K, sh.N, 1 if fused else 0), 16),
                             dtype=torch.uint8, device="cuda")

            def call():
                swg.swiglu_bwd(**inp, fused=fused, return_dg=False, out=out, workspace=ws)

            for _ in range(3):
                call()
            ts = []
            for _ in range(reps):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            r["fused_us" if fused else "unfused_us"] = round(statistics.median(ts) * 1e3, 2)
        rows.append(r)
    swg.swg_check()
    del flush
    return {"K": 512, "N": 1024, "call": "swiglu_bwd (dg, dfc not returned), L2 flushed before each call",
            "rows": rows}


# ---------------------------------------------------------------- CPU oracle
def _oracle_inputs(inp, rows):
    """The first `rows` rows of the workload widened exactly to fp64 (outside any timing)."""
    import numpy as np

    h = {}
    for k, v in inp.items():
        t = v[:rows] if k in ("x", "dy", "g", "fc") else v
        h[k] = t.detach().float().cpu().numpy().astype(np.float64)
    return h


def _time_oracle(h):
    import oracle

    t0 = time.perf_counter()
    oracle.swiglu_bwd(h["x"], h["w_g"], h["w_fc"], h["dy"], h["g"], h["fc"], stage_dtype="bf16")
    return time.perf_counter() - t0


def _cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(inp=None):
    """Time the fp64 oracle, as it stands, on the whole workload (all M rows) once."""
    from synth import SWIGLU_CONFIGS, swiglu_inputs

    if inp is None:
        inp = swiglu_inputs(SWIGLU_CONFIGS["pages"][0], device="cpu")
    h = _oracle_inputs(inp, M)
    t = _time_oracle(h)
    del h
    return {"value": round(t * 1e3, 1), "unit": "ms", "cores": _cpu_threads(), "kind": "oracle",
            "sample": f"the whole workload (M={M}, K={K}, N={N}), one run of the fp64 numpy oracle; "
                      f"BLAS threads = library default"}


def run_reference(args, rank, world):
    """The fp64 CPU oracle on the same workload, metric and unit. Each step runs
    the oracle on a sample of the first `rows` rows (sized so that warm-up and
    steps end within about two minutes); ms_per_step is the measured time of
    such a step and value is that time scaled to all M rows (the oracle's work
    is linear in M), labelled as an extrapolation in config."""
    if rank != 0:
        return
    from synth import SWIGLU_CONFIGS, swiglu_inputs

    inp = swiglu_inputs(SWIGLU_CONFIGS["pages"][0], device="cpu")
    probe_rows = 2048
    sec_per_row = _time_oracle(_oracle_inputs(inp, probe_rows)) / probe_rows
    budget = 120.0 / (args.steps + args.warmup + 1)
    rows = int(min(args.ref_rows, M, max(256, budget / max(sec_per_row, 1e-12))))
    h = _oracle_inputs(inp, rows)
    for _ in range(args.warmup):
        _time_oracle(h)
    t_steps = [_time_oracle(h) for _ in range(args.steps)]
    step_ms = statistics.median(t_steps) * 1e3
    v = round(step_ms * M / rows, 1)
    cb = {"value": v, "unit": "ms", "cores": _cpu_threads(), "kind": "oracle",
          "sample": f"first {rows} of {M} rows per step (K={K}, N={N}), fp64 numpy; value = step time x M/{rows}"}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "ms", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 2), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn, bf16 inputs widened to fp64)",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "sample_rows": rows,
                   "path": "fp64 CPU oracle (numpy) on the first sample_rows rows per step",
                   "value_kind": f"extrapolated: measured step time x M/sample_rows = x {M / rows:.2f}"},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["fused", "unfused"], default="fused",
                    help="which chain the timed step runs (the other is timed too and reported beside it)")
    ap.add_argument("--ref-rows", type=int, default=8192)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-llm", action="store_true", help="skip the LLM-FFN-shape leg")
    ap.add_argument("--m", type=int, default=None,
                    help="rows M of a smaller case of the same kernels (profiling only; the metric is M=220000)")
    ap.add_argument("--profile-only", action="store_true",
                    help="run warmup + steps of the timed step without timing or the other legs (for ncu)")
    args = ap.parse_args()
    if args.m is not None:
        global M
        M = args.m
    if args.warmup < 3:
        args.warmup = 3
    rank, world = _dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
