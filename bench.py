"""Benchmark of the block-FP8 MoE layer forward on GB300 (decode shape).

Workload: the decode configuration -- M tokens (default 32) of hidden size 7168, local
intermediate size 256 (gate/up width 512), E = 256 experts, top-k 8, uniform random routing,
E4M3 weights with 128x128 fp32 block scales, BF16 activations ~N(0, 1), fp32 dynamic
activation scales.  Inputs are seeded and synthetic; weights are random (no checkpoint).

One step = one whole layer forward (route preparation, input quantisation, gate/up GEMM,
fused SiLU*mul + quantisation, down GEMM, moe_reduce) through moe_blockfp8_forward on the path
the library picks for the shape (the fused persistent kernel, or the staged launches), replayed
from a CUDA graph; both paths are also timed and reported side by side.  Eight routing batches rotate between steps and a 256 MiB buffer is written
and then read back between timed steps (outside the events), so no step starts with its
weights in L2 and no dirty line of the flush is written back inside the timed region.

Beside the headline, "configs" holds the other measured rows: every stage of the decode layer
alone through its own entry point (device time, algorithmic bytes, fraction of the HBM peak),
the fused SiLU*mul + quantisation against the two-kernel arm (clamped UE8M0 sweep and the decode
shape), route preparation on both paths, and whole layers at the expert-parallel shape (T=1024
tokens, 32 of 256 experts local) and at the prefill shape (M=512, Zipf routing), the latter with
its FP8 MMA rate against the FP8 peak.  --no-configs skips them.

Prints one JSON line.  --impl reference times the CPU oracle instead (a bounded token sample
per step, scaled to the layer latency).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer latency (us) & HBM GB/s (fraction of roofline) at decode M=1..256"
DECODE = dict(H=7168, N=256, E=256, k=8)
NROT = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--M", type=int, default=32)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--layer", choices=["prefill", "ep"], default=None,
                    help="only run this configuration's layer forward --steps times (no timing line): "
                         "the command a profiler wraps")
    ap.add_argument("--experts", type=int, default=0,
                    help="with --layer: number of experts (0 = the configuration's), for a small profiling case")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-stage, act-quant, route-preparation, expert-parallel and prefill arms")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--weights", default="tiled", choices=["tiled", "row"],
                    help="expert weight layout: 128x128 tiles contiguous (packed once) or row-major")
    return ap.parse_args()


def workload_config(M, seed):
    """The workload both arms (the library and the CPU oracle) report, as the same dict."""
    H, N, E, k = DECODE["H"], DECODE["N"], DECODE["E"], DECODE["k"]
    return {"workload": f"decode MoE layer M={M} H={H} N={N} E={E} top-k={k}, block-FP8 128x128",
            "M": M, "H": H, "N": N, "E": E, "topk": k, "routing": "uniform (softmax top-k of N(0,1) logits)",
            "weights": "E4M3, fp32 scale per 128x128 block, ~N(0, 0.02)", "activations": "BF16 ~N(0,1)",
            "seed": seed, "routing_batches": NROT}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if smax and s >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------------------------
def active_bytes(ids_list, H, N, E):
    """Algorithmic HBM bytes of one layer forward per routing batch: the active experts'
    E4M3 weights and fp32 block scales, read once."""
    per_expert_gu = 2 * N * H + (2 * N // 128) * (H // 128) * 4
    per_expert_d = H * N + (H // 128) * (N // 128) * 4
    out = []
    for ids in ids_list:
        a = len(np.unique(ids[(ids >= 0) & (ids < E)]))
        out.append((a, a * per_expert_gu, a * per_expert_d))
    return out


def make_inputs(M, seed, dev):
    """The layer inputs of each routing batch: x [M, H] bf16, topk_ids [M, k] i32 and topk_w
    [M, k] f32, laid out back to back (256-byte aligned) in one device buffer, so that one copy
    moves a step's inputs from the host."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    H, k = DECODE["H"], DECODE["k"]
    al = lambda n: (n + 255) // 256 * 256
    o_ids = al(M * H * 2)
    o_w = o_ids + al(M * k * 4)
    xs, ids, ws = [], [], []
    for r in range(NROT):
        i, w = wl.routing_topk(M, DECODE["E"], k, seed=seed * 1000 + r, kind="uniform")
        x = wl.bf16_normal((M, H), 1.0, seed * 1000 + 500 + r)
        buf = torch.zeros(o_w + M * k * 4, dtype=torch.uint8, device=dev)
        xv = buf[:M * H * 2].view(torch.bfloat16).view(M, H)
        iv = buf[o_ids:o_ids + M * k * 4].view(torch.int32).view(M, k)
        wv = buf[o_w:o_w + M * k * 4].view(torch.float32).view(M, k)
        xv.copy_(x.to(dev))
        iv.copy_(torch.from_numpy(i).to(dev))
        wv.copy_(torch.from_numpy(w).to(dev))
        xs.append(xv)
        ids.append(iv)
        ws.append(wv)
    return xs, ids, ws


def packed_buffer(t):
    """The whole device buffer a make_inputs view lives in."""
    import torch
    return torch.empty(0, dtype=torch.uint8, device=t.device).set_(t.untyped_storage())


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def make_event(external=False):
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=external)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def flush_l2(flush):
    """Evicts the previous step's data from L2 (129 MB): writes a 256 MiB buffer, then reads it
    back, so the dirty lines of the write are written back here, outside the timed region, and
    the next step starts with a clean L2 that holds none of its weights."""
    import torch
    flush.zero_()
    flush.view(torch.float32).sum()


def time_graph_steps(graphs, steps, warmup, flush, stream):
    """Per-step device time (ms) of graph replays, L2 flushed between steps (outside events)."""
    import torch
    times = []
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush_l2(flush)
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        evs = [(make_event(), make_event()) for _ in range(steps)]
        for i in range(steps):
            flush_l2(flush)
            evs[i][0].record(stream)
            graphs[i % len(graphs)].replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        times = [a.elapsed_time(b) for a, b in evs]
    return times


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from block_fp8_mixture_moe_gb300 import ops, workloads as wl

    H, N, E, k = DECODE["H"], DECODE["N"], DECODE["E"], DECODE["k"]
    M = args.M
    wgu_q, wgu_s = wl.quantized_weights(E, 2 * N, H, seed=args.seed * 7919 + 5, device=dev)
    wd_q, wd_s = wl.quantized_weights(E, H, N, seed=args.seed * 7919 + 6, device=dev)
    if args.weights == "tiled":  # one-time regrouping when the weights are loaded (not timed)
        wgu_use, wd_use = ops.moe_blockfp8_pack_weights(wgu_q), ops.moe_blockfp8_pack_weights(wd_q)
    else:
        wgu_use, wd_use = wgu_q, wd_q
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def layer_graphs(M_, path):
        xs, ids, ws = make_inputs(M_, args.seed, dev)
        need = ops.moe_blockfp8_workspace_bytes(M_, k, E, E, H, N)
        work = torch.empty(need, dtype=torch.uint8, device=dev)
        outs = [torch.empty((M_, H), dtype=torch.bfloat16, device=dev) for _ in range(NROT)]
        graphs = []
        for r in range(NROT):
            fn = (lambda r=r: ops.moe_blockfp8_forward(xs[r], ids[r], ws[r], E, None, wgu_use, wgu_s,
                                                       wd_use, wd_s, out=outs[r], workspace=work,
                                                       stream=stream, path=path))
            graphs.append(capture(fn, stream))
        return xs, ids, ws, outs, work, graphs

    path = ops.moe_forward_path_for(M, k, E, E, H, N)
    path_name = {ops.FORWARD_FUSED: "fused", ops.FORWARD_STAGED: "staged"}[path]
    xs, ids, ws, outs, work, graphs = layer_graphs(M, path)
    ids_host = [t.cpu().numpy() for t in ids]
    act = active_bytes(ids_host, H, N, E)
    bm, B_cap, splits = ops.moe_blockfp8_plan(M, k, E, E, H, N)

    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    step_ms = time_graph_steps(graphs, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    layer_bytes = [a[1] + a[2] for a in act]
    mean_bytes = sum(layer_bytes[i % NROT] for i in range(args.steps)) / args.steps

    # ---- both paths of the same layer, for comparison ----------------------------------------
    path_ms = {}
    for pth, nm in ((ops.FORWARD_FUSED, "fused"), (ops.FORWARD_STAGED, "staged")):
        arm = layer_graphs(M, pth)  # the graphs write into these tensors: kept alive while replayed
        path_ms[nm] = time_graph_steps(arm[-1], min(args.steps, 200), args.warmup, flush, stream)
        del arm

    # ---- the gate/up GEMM of the staged path alone, events on its stream --------------------
    gemm_ms = time_gate_up_kernel(ops, dev, stream, flush, xs, ids, ws, wgu_use, wgu_s,
                                  M, H, N, E, k, min(args.steps, 200), args.warmup)
    padded_ms = time_gate_up_kernel(ops, dev, stream, flush, xs, ids, ws, wgu_use, wgu_s,
                                    M, H, N, E, k, min(args.steps, 100), args.warmup, padded=True)
    gu_bytes = []
    for i, (a, gub, _) in enumerate(act):
        kept = M * k
        gu_bytes.append(gub + kept * (H + (H // 128) * 4) + kept * 2 * N * 2)
    gu_mean_bytes = sum(gu_bytes) / len(gu_bytes)

    # ---- end to end through the public API with host buffers --------------------------------
    # (a) the kernels read and write pinned host memory themselves; (b) copy-engine copies in and
    # out around the device-buffer graph
    def fwd_host(x_, i_, w_, o_):
        return ops.moe_blockfp8_forward(x_, i_, w_, E, None, wgu_use, wgu_s, wd_use, wd_s, out=o_,
                                        workspace=work, stream=stream, path=path)
    e2e_ms, h2d, d2h, e2e_wall = time_e2e_zero_copy(ops, dev, stream, flush, xs, ids, ws, outs, fwd_host,
                                                    args.steps, args.warmup, dev_graphs=graphs)
    e2e_copy_ms, _, _ = time_e2e(ops, dev, stream, flush, xs, ids, ws, outs, graphs, args.steps, args.warmup)
    clocks = sampler.stop()

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    # FP8 dense peak: the measured bf16 GEMM peak times the nominal fp8 / bf16 ratio (2)
    fp8_peak = 2.0 * peaks.get("bf16_tflops", 1900.0)
    configs = None
    if not args.no_configs:
        from block_fp8_mixture_moe_gb300 import workloads as wl
        configs = {
            "stages_decode": dict(M=M, **stage_times(ops, dev, stream, flush, xs, ids, ws, wgu_use, wgu_s, wd_use,
                                                     wd_s, M, H, N, E, k, act, hbm_peak)),
            "act_quant": act_quant_arms(ops, dev, stream, flush),
            "act_quant_expert_filtered": act_quant_ep_arms(ops, dev, stream, flush),
            "route_prepare_us": route_prep_arms(ops, dev, stream, flush),
            "tiny": layer_arm(ops, dev, stream, flush, wl.CONFIGS["tiny"], 0, hbm_peak, fp8_peak, steps=50,
                              warmup=5, clamp=7.0, fmt=1),
            "expert_parallel": layer_arm(ops, dev, stream, flush, dict(wl.CONFIGS["ep"], M=1024), 2, hbm_peak,
                                         fp8_peak, clamp=7.0, fmt=1),
            "expert_parallel_tokens": {str(T): layer_arm(ops, dev, stream, flush, dict(wl.CONFIGS["ep"], M=T), 2,
                                                         hbm_peak, fp8_peak, steps=50, warmup=5, clamp=7.0, fmt=1)
                                       for T in wl.EP_TOKENS},
            "prefill": layer_arm(ops, dev, stream, flush, wl.CONFIGS["prefill"], 3, hbm_peak, fp8_peak),
            "fp8_peak_source": "measured bf16 GEMM peak x 2 (nominal fp8/bf16 ratio)" if "bf16_tflops" in peaks
                              else "fallback bf16 1.9 PFLOP/s x 2",
        }

    sweep = None
    if not args.no_sweep:
        sweep = {}
        for Ms in (1, 4, 16, 32, 64, 128, 256):
            row = {}
            for pth, nm in ((ops.FORWARD_FUSED, "fused"), (ops.FORWARD_STAGED, "staged")):
                arm = layer_graphs(Ms, pth)  # kept alive while its graphs are replayed
                ids_s = arm[1]
                t = time_graph_steps(arm[-1], 50, 5, flush, stream)
                del arm
                row[nm + "_us"] = round(statistics.mean(t) * 1e3, 2)
            a_s = active_bytes([t.cpu().numpy() for t in ids_s], H, N, E)
            by = sum(a_s[i % NROT][1] + a_s[i % NROT][2] for i in range(50)) / 50
            auto = "fused" if ops.moe_forward_path_for(Ms, k, E, E, H, N) == ops.FORWARD_FUSED else "staged"
            us = row[auto + "_us"]
            row.update({"us": us, "path": auto, "active_experts": round(sum(a[0] for a in a_s) / NROT, 1),
                        "GBps": round(by / (us * 1e-6) / 1e9, 1)})
            sweep[str(Ms)] = row

    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    layer_us = ms_per_step * 1e3
    achieved = mean_bytes / (layer_us * 1e-6) / 1e9
    gemm_achieved = gu_mean_bytes / (statistics.mean(gemm_ms) * 1e-3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = oracle_layer(M, ids_host[0], ws[0].cpu().numpy(), xs[0], wgu_q, wgu_s, wd_q, wd_s, H, N, E, k)
        cpu = cpu_baseline(host, M)

    route_launches = 1 if M * k <= 2048 else 2
    launches_per_step = route_launches + (1 if path == ops.FORWARD_FUSED else 5)
    if path == ops.FORWARD_FUSED:
        # the dominant kernel is the persistent kernel; timed with its route preparation
        roofline = {"bound": "hbm", "kernel": f"k_moe_fused<{bm}> with its route preparation (one forward call)",
                    "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), "traffic": recorded_traffic("fused"),
                    "algorithmic_bytes": int(mean_bytes), "kernel_us": round(layer_us, 2),
                    "weights": args.weights, "peak_source": peak_src}
    else:
        # the dominant kernel of the staged layer: the gate/up grouped GEMM, timed alone
        roofline = {"bound": "hbm",
                    "kernel": f"k_grouped_gemm<{bm}> (gate/up, split-K {splits}; timed alone through "
                              f"moe_blockfp8_grouped_gemm, static unit split)",
                    "achieved": round(gemm_achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(gemm_achieved / hbm_peak, 4), "traffic": recorded_traffic("staged"),
                    "algorithmic_bytes": int(gu_mean_bytes),
                    "kernel_us": round(statistics.mean(gemm_ms) * 1e3, 2),
                    "weights": args.weights, "peak_source": peak_src}
    line = {
        "metric": METRIC, "value": round(layer_us, 3), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded; random weights, uniform random routing)",
        "config": workload_config(M, args.seed),
        "setup": {"block_m": bm, "path": path_name, "weight_layout": args.weights,
                  "l2": "256 MiB buffer written then read back between timed steps (outside the events); 8 rotating routing batches",
                  "timing": "CUDA graph replay per step, CUDA events per step", "parallelism": f"replicas x{world}"},
        "layer_hbm": {"GBps": round(achieved, 1), "frac": round(achieved / hbm_peak, 4),
                      "active_bytes": int(mean_bytes), "peak": hbm_peak, "peak_source": peak_src,
                      "us_median": round(statistics.median(step_ms) * 1e3, 2),
                      "us_p10": round(float(np.percentile(step_ms, 10)) * 1e3, 2),
                      "us_p90": round(float(np.percentile(step_ms, 90)) * 1e3, 2)},
        "roofline": roofline,
        "paths_us": {nm: round(statistics.mean(t) * 1e3, 2) for nm, t in path_ms.items()},
        "staged_gate_up": {"splits": splits, "us": round(statistics.mean(gemm_ms) * 1e3, 2),
                           "GBps": round(gemm_achieved, 1), "frac": round(gemm_achieved / hbm_peak, 4),
                           "padded_grid_us": round(statistics.mean(padded_ms) * 1e3, 2)},
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "transfer": "zero-copy: inputs and output in pinned host memory, read and written by "
                            "the layer's kernels across NVLink-C2C inside the timed graph",
                "copy_engine_us": round(e2e_copy_ms * 1e3, 3),
                "host_wall_launch_to_sync_us": e2e_wall},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "sweep_M": sweep,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_events(fn, steps, warmup, flush, stream):
    """Device time (ms) of fn() per call: L2 flushed before each call, the device kept busy while
    the host enqueues (so the events time the GPU work, not the host), events on the stream."""
    import torch
    times = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            flush_l2(flush)
            torch.cuda._sleep(2_000_000)
            e0, e1 = make_event(), make_event()
            e0.record(stream)
            fn(i)
            e1.record(stream)
            if i >= warmup:
                times.append((e0, e1))
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def stage_times(ops, dev, stream, flush, xs, ids, ws, wgu_q, wgu_s, wd_q, wd_s, M, H, N, E, k,
                act, hbm_peak, steps=50, warmup=5):
    """Each stage of the staged layer through its own C-ABI entry point, on the decode inputs,
    L2 flushed before each call: device time, algorithmic bytes, GB/s and fraction of the HBM
    peak.  The input quantisation goes through the public per-route entry (silu_mul_quant_fp8,
    identity, one gathered row per route); inside the layer forward the same codes come from a
    per-token kernel that scatters each token's row to its routes' slots."""
    import torch
    bm, B_cap, splits = ops.moe_blockfp8_plan(M, k, E, E, H, N)
    slots, R = B_cap * bm, M * k
    with torch.cuda.stream(stream):
        routes = [ops.moe_route_prepare(ids[r], E, None, E, bm, stream=stream) for r in range(NROT)]
        xq = torch.zeros((slots, H), dtype=torch.uint8, device=dev)
        xsc = torch.ones((slots, H // 128), dtype=torch.float32, device=dev)
        gu = torch.zeros((splits, slots, 2 * N), dtype=torch.float32, device=dev)
        aq = torch.zeros((slots, N), dtype=torch.uint8, device=dev)
        asc = torch.ones((slots, N // 128), dtype=torch.float32, device=dev)
        z = torch.zeros((R, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        for r in range(NROT):  # one pass so every stage reads well-formed inputs
            rt = routes[r]
            ops.silu_mul_quant_fp8(0, xs[r], H, rows=R, row_map=rt["route_slot"], row_div=k,
                                   out_rows=slots, out_q=xq, out_s=xsc, stream=stream)
        torch.cuda.synchronize()
    n_act = [a[0] for a in act]
    mean_act = sum(n_act) / len(n_act)
    gu_w = 2 * N * H + (2 * N // 128) * (H // 128) * 4
    d_w = H * N + (H // 128) * (N // 128) * 4
    stages = [
        ("route_prepare", lambda i: ops.moe_route_prepare(ids[i % NROT], E, None, E, bm, stream=stream),
         R * 4 + slots * 4 + R * 4),
        ("input_quant", lambda i: ops.silu_mul_quant_fp8(0, xs[i % NROT], H, rows=R,
                                                          row_map=routes[i % NROT]["route_slot"], row_div=k,
                                                          out_rows=slots, out_q=xq, out_s=xsc, stream=stream),
         M * 2 * H + R * (H + 4 * H // 128)),
        ("gate_up_gemm", lambda i: ops.moe_blockfp8_grouped_gemm(0, xq, xsc, wgu_q, wgu_s, routes[i % NROT], bm,
                                                                 out_dtype=ops.DTYPE_F32, out_rows=slots,
                                                                 splits=splits, out=gu, stream=stream),
         mean_act * gu_w + R * (H + 4 * H // 128) + R * 2 * N * 4 * splits),
        ("act_quant", lambda i: ops.silu_mul_quant_fp8(1, gu, N, rows=R, row_map=routes[i % NROT]["route_slot"],
                                                        out_rows=slots, out_q=aq, out_s=asc, in_splits=splits,
                                                        strategy=2, stream=stream),
         R * splits * 2 * N * 4 + R * (N + 4 * N // 128)),
        ("down_gemm", lambda i: ops.moe_blockfp8_grouped_gemm(1, aq, asc, wd_q, wd_s, routes[i % NROT], bm,
                                                              out_dtype=ops.DTYPE_BF16, out_rows=R, out=z,
                                                              stream=stream),
         mean_act * d_w + R * (N + 4 * N // 128) + R * 2 * H),
        ("moe_reduce", lambda i: ops.moe_reduce(z, ws[i % NROT], ids[i % NROT], None, E, H, out=out, stream=stream),
         R * 2 * H + M * 2 * H),
    ]
    res = {}
    for name, fn, nbytes in stages:
        t = time_events(fn, steps, warmup, flush, stream)
        us = statistics.mean(t) * 1e3
        gbps = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 2), "algorithmic_bytes": int(nbytes), "GBps": round(gbps, 1),
                     "frac": round(gbps / hbm_peak, 4)}
    res["sum_us"] = round(sum(v["us"] for v in res.values()), 2)
    # the same protocol around a one-element fill: what a kernel costs here before it does work
    one = torch.zeros(1, device=dev)
    res["event_floor_us"] = round(statistics.mean(time_events(lambda i: one.fill_(1.0), steps, warmup,
                                                              flush, stream)) * 1e3, 2)
    res["note"] = ("each stage alone, L2 flushed before it; event_floor_us is the same protocol around a "
                   "trivial kernel; the layer overlaps a stage's start with the previous stage's tail "
                   "(programmatic dependent launch), so the layer is below the sum")
    return res


def act_quant_arms(ops, dev, stream, flush, steps=50, warmup=5):
    """Fused SiLU*mul + quantisation against the two-kernel arm (BF16 SiLU*mul written to memory,
    then quantised).  (1) the clamped UE8M0 sweep: rows 8*T, gate/up width 1024, activation width
    512, clamp +-7; (2) the decode shape of the fused-vs-separate comparison: 8 routed rows
    (M=1, top-8), activation width 256, fp32 scales."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    per_row = lambda n: 2 * (2 * n) + n + 4 * (n // 128)  # bf16 in, e4m3 + fp32 scales out
    out = {"clamped_ue8m0_width512": {}, "decode_width256_f32": {}}
    cases = [("clamped_ue8m0_width512", T, 8 * T, 512, 7.0, ops.SCALE_UE8M0) for T in wl.ACT_SWEEP_TOKENS]
    cases.append(("decode_width256_f32", 1, 8, 256, float("inf"), ops.SCALE_F32))
    for key, T, rows, n, clamp, fmt in cases:
        bits = wl.act_rows(rows, 2 * n, 2.0 if clamp < 1e9 else 1.0, 31 + T)
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        q = torch.empty((rows, n), dtype=torch.uint8, device=dev)
        sc = torch.empty((rows, n // 128), dtype=torch.float32, device=dev)
        fused = lambda i: ops.silu_mul_quant_fp8(1, x, n, clamp_limit=clamp, fmt=fmt, out_q=q, out_s=sc,
                                                stream=stream)

        def separate(i):
            a = ops.silu_and_mul_bf16(1, x, n, clamp_limit=clamp, stream=stream)
            ops.silu_mul_quant_fp8(0, a, n, fmt=fmt, out_q=q, out_s=sc, stream=stream)
        tf = statistics.mean(time_events(fused, steps, warmup, flush, stream)) * 1e3
        ts = statistics.mean(time_events(separate, steps, warmup, flush, stream)) * 1e3
        out[key][str(rows)] = {"fused_us": round(tf, 2), "separate_us": round(ts, 2),
                               "fused_GBps": round(rows * per_row(n) / (tf * 1e-6) / 1e9, 1)}
    return out


def act_quant_ep_arms(ops, dev, stream, flush, steps=50, warmup=5):
    """The expert-filtered act-quant sweep (vLLM PR #53875, "Kernel microbenchmarks": top-k 6,
    width 2048, 32 of 256 experts local, the filter in both arms): routed rows 6T for T in
    {1, 10, 100, 1024}, clamp +-7, UE8M0 scales.  Fused: one silu_mul_quant_fp8 that skips the
    non-local rows.  Two kernels: silu_and_mul_bf16 (same filter, BF16 written) then the
    identity quantisation (same filter)."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    E, k, El, n = 256, 6, 32, 2048
    emap = torch.from_numpy(wl.expert_map_random(E, El, 4242)).to(dev)
    out = {}
    for T in wl.EP_TOKENS:
        rows = k * T
        ids, _ = wl.routing_topk(T, E, k, seed=51 + T, kind="uniform")
        re = torch.from_numpy(ids.reshape(-1)).to(dev)
        x = torch.from_numpy(wl.act_rows(rows, 2 * n, 1.0, 61 + T).view(np.int16)).view(torch.bfloat16).to(dev)
        q = torch.zeros((rows, n), dtype=torch.uint8, device=dev)
        sc = torch.zeros((rows, n // 128), dtype=torch.float32, device=dev)
        mid = torch.zeros((rows, n), dtype=torch.bfloat16, device=dev)
        kept = int((emap[re.long()] >= 0).sum().item())
        fused = lambda i: ops.silu_mul_quant_fp8(1, x, n, clamp_limit=7.0, fmt=ops.SCALE_UE8M0, row_expert=re,
                                                expert_map=emap, E=E, out_q=q, out_s=sc, stream=stream)

        def separate(i):
            ops.silu_and_mul_bf16(1, x, n, clamp_limit=7.0, row_expert=re, expert_map=emap, E=E, out=mid,
                                  stream=stream)
            ops.silu_mul_quant_fp8(0, mid, n, fmt=ops.SCALE_UE8M0, row_expert=re, expert_map=emap, E=E,
                                   out_q=q, out_s=sc, stream=stream)
        tf = statistics.mean(time_events(fused, steps, warmup, flush, stream)) * 1e3
        ts = statistics.mean(time_events(separate, steps, warmup, flush, stream)) * 1e3
        out[str(rows)] = {"tokens": T, "kept_rows": kept, "fused_us": round(tf, 2), "separate_us": round(ts, 2),
                          "speedup": round(ts / tf, 2)}
    return out


def route_prep_arms(ops, dev, stream, flush, steps=50, warmup=5):
    """Route preparation alone: 512 routes over 256 experts (single CTA), and 2048 and 4096 (the
    prefill's) routes over 512 experts on both paths."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    res = {}
    for M, E, path, name in ((64, 256, 1, "512_routes_256_experts_single"),
                             (256, 512, 1, "2048_routes_512_experts_single"),
                             (256, 512, 2, "2048_routes_512_experts_multi"),
                             (512, 512, 1, "4096_routes_512_experts_single"),
                             (512, 512, 2, "4096_routes_512_experts_multi")):
        i, _ = wl.routing_topk(M, E, 8, seed=97 + M, kind="uniform")
        ids = torch.from_numpy(i).to(dev)
        fn = lambda it: ops.moe_route_prepare(ids, E, None, E, 16, path=path, stream=stream)
        res[name] = round(statistics.mean(time_events(fn, steps, warmup, flush, stream)) * 1e3, 2)
    return res


def layer_only(args):
    """--layer: the prefill or expert-parallel layer forward, run --steps times back to back, for
    a profiler to wrap.  --experts shrinks the expert count (the expert-parallel shape keeps its
    1/8 local fraction)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from block_fp8_mixture_moe_gb300 import ops, workloads as wl
    dev = torch.device("cuda", 0)
    cfg = dict(wl.CONFIGS["prefill"]) if args.layer == "prefill" else dict(wl.CONFIGS["ep"], M=1024)
    if args.experts > 0:
        cfg["E_local"] = max(1, cfg["E_local"] * args.experts // cfg["E"])
        cfg["E"] = args.experts
    seed = 3 if args.layer == "prefill" else 2
    clamp, fmt = (float("inf"), 0) if args.layer == "prefill" else (7.0, 1)
    M, H, N, E, k, El = cfg["M"], cfg["H"], cfg["N"], cfg["E"], cfg["k"], cfg["E_local"]
    wgu_q, wgu_s = wl.quantized_weights(El, 2 * N, H, seed=seed * 7919 + 5, device=dev)
    wd_q, wd_s = wl.quantized_weights(El, H, N, seed=seed * 7919 + 6, device=dev)
    wgu_t, wd_t = ops.moe_blockfp8_pack_weights(wgu_q), ops.moe_blockfp8_pack_weights(wd_q)
    del wgu_q, wd_q
    i, w = wl.routing_topk(M, E, k, seed=seed * 7919 + 1, kind=cfg["routing"])
    emap = None if El == E else torch.from_numpy(wl.expert_map_random(E, El, seed * 7919 + 3)).to(dev)
    x = wl.bf16_normal((M, H), 1.0, seed * 7919 + 4).to(dev)
    ids, ws = torch.from_numpy(i).to(dev), torch.from_numpy(w).to(dev)
    work = torch.empty(ops.moe_blockfp8_workspace_bytes(M, k, E, El, H, N), dtype=torch.uint8, device=dev)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    for _ in range(max(1, args.steps)):
        ops.moe_blockfp8_forward(x, ids, ws, E, emap, wgu_t, wgu_s, wd_t, wd_s, clamp_limit=clamp,
                                 act_fmt=fmt, out=out, workspace=work)
    torch.cuda.synchronize()
    print(json.dumps({"layer": args.layer, "M": M, "H": H, "N": N, "E": E, "E_local": El, "k": k,
                      "block_m": ops.moe_forward_block_m(M, k, El, H, N), "forwards": max(1, args.steps),
                      "device_status": ops.device_status()}))


def layer_arm(ops, dev, stream, flush, cfg, seed, hbm_peak, fp8_peak_tflops, steps=20, warmup=3,
              clamp=float("inf"), fmt=0):
    """One forward of a whole layer at a non-decode configuration (graph-replayed, L2 flushed
    between steps): latency, active-expert weight bytes against HBM, and FP8 MMA flops against
    the FP8 peak."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    M, H, N, E, k, El = cfg["M"], cfg["H"], cfg["N"], cfg["E"], cfg["k"], cfg["E_local"]
    wgu_q, wgu_s = wl.quantized_weights(El, 2 * N, H, seed=seed * 7919 + 5, device=dev)
    wd_q, wd_s = wl.quantized_weights(El, H, N, seed=seed * 7919 + 6, device=dev)
    wgu_t, wd_t = ops.moe_blockfp8_pack_weights(wgu_q), ops.moe_blockfp8_pack_weights(wd_q)
    del wgu_q, wd_q
    i, w = wl.routing_topk(M, E, k, seed=seed * 7919 + 1, kind=cfg["routing"])
    emap = None if El == E else wl.expert_map_random(E, El, seed * 7919 + 3)
    x = wl.bf16_normal((M, H), 1.0, seed * 7919 + 4).to(dev)
    ids, ws = torch.from_numpy(i).to(dev), torch.from_numpy(w).to(dev)
    em = None if emap is None else torch.from_numpy(emap).to(dev)
    work = torch.empty(ops.moe_blockfp8_workspace_bytes(M, k, E, El, H, N), dtype=torch.uint8, device=dev)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    fn = lambda: ops.moe_blockfp8_forward(x, ids, ws, E, em, wgu_t, wgu_s, wd_t, wd_s, clamp_limit=clamp,
                                          act_fmt=fmt, out=out, workspace=work, stream=stream)
    g = capture(fn, stream)
    t = time_graph_steps([g], steps, warmup, flush, stream)
    us = statistics.mean(t) * 1e3
    loc = i[(i >= 0) & (i < E)]
    if emap is not None:
        loc = emap[loc]
        loc = loc[loc >= 0]
    counts = np.bincount(loc, minlength=El)
    active = int((counts > 0).sum())
    wbytes = active * (3 * H * N + ((2 * N // 128) * (H // 128) + (H // 128) * (N // 128)) * 4)
    flops = 2.0 * 3 * H * N * int(counts.sum())
    bm = ops.moe_forward_block_m(M, k, El, H, N)
    return {"workload": f"M={M} H={H} N={N} E={E} E_local={El} top-k={k} {cfg['routing']} routing",
            "block_m": bm, "us": round(us, 2), "active_experts": active, "routes_kept": int(counts.sum()),
            "max_routes_per_expert": int(counts.max()),
            "hbm": {"bytes": int(wbytes), "GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
                    "frac": round(wbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)},
            "fp8_mma": {"flops": flops, "TFLOPs": round(flops / (us * 1e-6) / 1e12, 1),
                        "frac": round(flops / (us * 1e-6) / 1e12 / fp8_peak_tflops, 4),
                        "peak_TFLOPs": round(fp8_peak_tflops, 1)}}


def padded_grid_route(route, E, bm, dev):
    """The schedule before active-expert dispatch: every expert owns a block, so every expert's
    weights are streamed whether or not it received routes (lmdeploy PR #4956, "Motivation");
    the route table comes from workloads.padded_grid_route, the builder the GEMM parity tests
    check, at setup time."""
    import torch
    from block_fp8_mixture_moe_gb300 import workloads as wl
    pg = wl.padded_grid_route(route["sorted_idx"].cpu().numpy(), route["block_expert"].cpu().numpy(),
                              int(route["num_blocks"].item()), E, bm)
    return dict(sorted_idx=torch.from_numpy(pg["sorted_idx"]).to(dev),
                block_expert=torch.from_numpy(pg["block_expert"]).to(dev),
                num_blocks=torch.tensor([pg["num_blocks"]], dtype=torch.int32, device=dev), B_cap=pg["B_cap"])


def time_gate_up_kernel(ops, dev, stream, flush, xs, ids, ws, wgu_q, wgu_s, M, H, N,
                        E, k, steps, warmup, padded=False):
    """The layer's stages launched one by one through the per-stage entry points, with events
    around the gate/up GEMM only; returns its per-launch device times (ms).  padded=True times
    the padded-grid schedule (every expert's weights) on the same activations."""
    import torch
    bm, B_cap, splits = ops.moe_blockfp8_plan(M, k, E, E, H, N)
    slots = B_cap * bm
    gu = torch.empty((splits, slots, 2 * N), dtype=torch.float32, device=dev)
    xq = torch.empty((slots, H), dtype=torch.uint8, device=dev)
    xsc = torch.empty((slots, H // 128), dtype=torch.float32, device=dev)
    routes = []
    with torch.cuda.stream(stream):
        for r in range(NROT):
            route = ops.moe_route_prepare(ids[r], E, None, E, bm, stream=stream)
            routes.append(route)
        torch.cuda.synchronize()
    if padded:
        # the padded grid reads activations from its own slots (the values do not change the
        # time: the same bytes are read)
        proutes = [padded_grid_route(rt, E, bm, dev) for rt in routes]
        slots_p = max(pr["B_cap"] for pr in proutes) * bm
        xq_p = torch.zeros((max(slots, slots_p), H), dtype=torch.uint8, device=dev)
        xs_p = torch.ones((max(slots, slots_p), H // 128), dtype=torch.float32, device=dev)
        gu_p = torch.empty((splits, max(slots, slots_p), 2 * N), dtype=torch.float32, device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            r = i % NROT
            route = routes[r]
            ops.silu_mul_quant_fp8(0, xs[r], H, rows=M * k, row_map=route["route_slot"], row_div=k,
                                   out_rows=slots, out_q=xq, out_s=xsc, stream=stream)
            flush_l2(flush)
            torch.cuda._sleep(2_000_000)  # keep the device busy while the host enqueues
            e0, e1 = make_event(), make_event()
            e0.record(stream)
            if padded:
                ops.moe_blockfp8_grouped_gemm(0, xq_p, xs_p, wgu_q, wgu_s, proutes[r], bm,
                                              out_dtype=ops.DTYPE_F32, out_rows=xq_p.shape[0],
                                              splits=splits, out=gu_p, stream=stream)
            else:
                ops.moe_blockfp8_grouped_gemm(0, xq, xsc, wgu_q, wgu_s, route, bm, out_dtype=ops.DTYPE_F32,
                                              out_rows=slots, splits=splits, out=gu, stream=stream)
            e1.record(stream)
            if i >= warmup:
                times.append((e0, e1))
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def time_e2e(ops, dev, stream, flush, xs, ids, ws, outs, graphs, steps, warmup):
    """Per step: one host->device copy of the step's inputs (x, topk_ids and topk_w, packed in
    one pinned host buffer that mirrors the device buffer the layer reads), the layer (graph of
    moe_blockfp8_forward), the device->host copy of the output; events around all of it."""
    import torch
    dbuf = [packed_buffer(x) for x in xs]
    hbuf = [b.cpu().pin_memory() for b in dbuf]
    ho = [o.cpu().pin_memory() for o in outs]
    h2d = hbuf[0].numel()
    d2h = ho[0].numel() * 2
    evs = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            r = i % NROT
            flush_l2(flush)
            e0, e1 = make_event(), make_event()
            e0.record(stream)
            dbuf[r].copy_(hbuf[r], non_blocking=True)
            graphs[r].replay()
            ho[r].copy_(outs[r], non_blocking=True)
            e1.record(stream)
            if i >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize()
    t = [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(t), h2d, d2h


def wall_steps(graphs, steps, flush, stream):
    """Median host wall time (us) from a graph's launch to the end of a stream sync, when its
    result is visible to the host; L2 flushed and the stream idle before each step."""
    import time
    import torch
    t = []
    with torch.cuda.stream(stream):
        for i in range(steps + 3):
            flush_l2(flush)
            stream.synchronize()
            t0 = time.perf_counter()
            graphs[i % len(graphs)].replay()
            stream.synchronize()
            if i >= 3:
                t.append((time.perf_counter() - t0) * 1e6)
    return statistics.median(t)


def time_e2e_zero_copy(ops, dev, stream, flush, xs, ids, ws, outs, fwd, steps, warmup, dev_graphs=None):
    """Per step: the layer (graph of moe_blockfp8_forward) called on pinned HOST buffers: its
    kernels read x, topk_ids and topk_w from host memory and the reduce writes the output to
    host memory across the host link, so the step starts with the inputs on the host and ends
    with the result there; events around it.  Each graph's host output is first checked to be
    bitwise the device-buffer output of the same inputs."""
    import torch
    hx = [x.cpu().pin_memory() for x in xs]
    hi = [t.cpu().pin_memory() for t in ids]
    hw = [t.cpu().pin_memory() for t in ws]
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    graphs = [capture(lambda r=r: fwd(hx[r], hi[r], hw[r], ho[r]), stream) for r in range(NROT)]
    with torch.cuda.stream(stream):
        for r in range(NROT):
            ho[r].zero_()
            graphs[r].replay()
        torch.cuda.synchronize()
    for r in range(NROT):
        if not torch.equal(ho[r], outs[r].cpu()):
            raise RuntimeError("zero-copy forward differs from the device-buffer forward")
    evs = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            flush_l2(flush)
            e0, e1 = make_event(), make_event()
            e0.record(stream)
            graphs[i % NROT].replay()
            e1.record(stream)
            if i >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize()
    t = [a.elapsed_time(b) for a, b in evs]
    h2d = hx[0].numel() * 2 + hi[0].numel() * 4 + hw[0].numel() * 4
    d2h = ho[0].numel() * 2
    # the same steps on the host's clock: launch to sync, zero-copy and device-buffer graphs
    wall = {"zero_copy": round(wall_steps(graphs, 40, flush, stream), 1)}
    if dev_graphs is not None:
        wall["device_buffers"] = round(wall_steps(dev_graphs, 40, flush, stream), 1)
    del graphs
    return statistics.mean(t), h2d, d2h, wall


def recorded_traffic(path):
    """DRAM bytes (read + write) per launch of the dominant kernel, scaled to this workload, from
    the committed ncu summary -- only if that summary was taken on the current kernel source
    (its sha256 is recorded there); otherwise null."""
    import re
    name, src = {"staged": ("gate_up_gemm_decode_m32_traffic.md", "grouped_gemm.cu"),
                 "fused": ("fused_layer_decode_m32_traffic.md", "fused_layer.cu")}[path]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        want = re.search(re.escape(src) + r" sha256: `([0-9a-f]{64})`", text).group(1)
        data = open(os.path.join(ROOT, "block_fp8_mixture_moe_gb300", "csrc", src), "rb").read()
        if want != hashlib.sha256(data).hexdigest():
            return None
        return int(re.search(r"dram_bytes_per_launch: (\d+)", text).group(1))
    except Exception:
        return None


def oracle_layer(M, ids0, w0, x0, wgu_q, wgu_s, wd_q, wd_s, H, N, E, k):
    """Host (numpy) copy of routing batch 0's whole layer for the oracle: the batch's routing,
    weights and activations, and the weights of its active experts (the same bytes the library
    reads; the other experts are zero, and no route reaches them)."""
    from block_fp8_mixture_moe_gb300 import workloads as wl
    import torch
    layer = dict(x=x0.view(torch.int16).cpu().numpy().view(np.uint16), topk_ids=ids0, topk_w=w0,
                 expert_map=None, wgu_q=wgu_q, wgu_s=wgu_s, wd_q=wd_q, wd_s=wd_s, E=E, M=M, H=H, N=N, k=k)
    return wl.layer_numpy(layer, experts=np.unique(ids0))


def time_oracle(host, threads, min_runs, budget_s):
    """Median wall time (us) of the oracle's whole layer with `threads` OpenMP threads (0 = all
    host cores), at least min_runs runs and at most about budget_s seconds; returns (us, runs,
    threads used)."""
    import oracle
    used = oracle.set_threads(threads)
    runs = []
    t_end = time.time() + budget_s
    while len(runs) < min_runs or (time.time() < t_end and len(runs) < 20):
        t0 = time.perf_counter()
        oracle.moe_forward(host)
        runs.append(time.perf_counter() - t0)
    oracle.set_threads(0)
    return statistics.median(runs) * 1e6, len(runs), used


def cpu_baseline(host, M):
    """The oracle's whole layer (all M tokens of routing batch 0, the bench's own inputs) on the
    host cores: all cores, and one thread."""
    import oracle
    oracle.build()
    oracle.moe_forward(host)  # warm (page-in)
    us_all, n_all, threads = time_oracle(host, 0, 3, 8.0)
    us_one, n_one, _ = time_oracle(host, 1, 1, 4.0)
    return {"value": round(us_all, 1), "unit": "us", "cores": threads, "kind": "oracle",
            "sample": f"the whole layer (all {M} tokens of routing batch 0, the timed inputs), median of {n_all} runs on {threads} threads",
            "single_thread": {"value": round(us_one, 1), "unit": "us", "cores": 1, "runs": n_one}}


# ---------------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle on the library arm's own workload: the same seeds give the same routing,
    activations and weights (generated with torch's CUDA generator when a GPU is present, as the
    library arm does; only input generation touches the GPU), and each step is one whole layer
    of routing batch 0 on all host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import oracle
    from block_fp8_mixture_moe_gb300 import workloads as wl
    oracle.build()
    H, N, E, k = DECODE["H"], DECODE["N"], DECODE["E"], DECODE["k"]
    M = args.M
    gen_dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    wgu_q, wgu_s = wl.quantized_weights(E, 2 * N, H, seed=args.seed * 7919 + 5, device=gen_dev)
    wd_q, wd_s = wl.quantized_weights(E, H, N, seed=args.seed * 7919 + 6, device=gen_dev)
    ids0, w0 = wl.routing_topk(M, E, k, seed=args.seed * 1000, kind="uniform")
    x0 = wl.bf16_normal((M, H), 1.0, args.seed * 1000 + 500)
    host = oracle_layer(M, ids0, w0, x0, wgu_q, wgu_s, wd_q, wd_s, H, N, E, k)
    del wgu_q, wgu_s, wd_q, wd_s
    threads = oracle.set_threads(0)
    for _ in range(args.warmup):
        oracle.moe_forward(host)
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.moe_forward(host)
        t.append(time.perf_counter() - t0)
    per_layer_us = statistics.mean(t) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(per_layer_us, 1), "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(t) * 1e3, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded; random weights, uniform random routing)",
        "config": workload_config(M, args.seed),
        "cpu_baseline": {"value": round(per_layer_us, 1), "unit": "us", "kind": "oracle", "cores": threads,
                         "sample": f"the whole layer (all {M} tokens of routing batch 0) per step, "
                                   f"inputs generated on {gen_dev.type}"},
        "e2e": {"value": round(per_layer_us, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    a = parse()
    if a.layer:
        layer_only(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
