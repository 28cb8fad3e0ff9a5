"""Benchmark of the routed-expert MoE layer on GB300 (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode-6] [--impl reference]

A step is one whole layer call (route -> MXFP8 quant -> W13+SwiGLU+requant -> W2 -> combine) over
one batch of the workload, inputs resident in HBM. L2 is flushed between timed steps (a 256 MiB
write, then a 256 MiB read of a second buffer so that the write's dirty lines are drained before
the step rather than written back inside it); each step is timed with CUDA events on the launching stream and the per-step times summed.
`value` is tokens/s over all ranks (rows are independent: every rank runs its own replica of the
batch, weak scaling). `e2e` repeats the measurement through the public API with the batch
copied host->device (pinned) and the output copied back inside the timed region. `roofline`
times the dominant kernel alone (W13 grouped GEMM for decode, by algorithmic bytes against HBM;
the W13 + W2 MMA FLOPs against the FP8 tensor peak for prefill). `cpu_baseline` times the CPU
oracle on a bounded sample of the same workload in a child process.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0          # profiling recipe fallback (one earlier GB300 measurement)
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0                # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode-6")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=1)
    ap.add_argument("--tokens", type=int, default=0, help="override T of the workload (profiling aid)")
    ap.add_argument("--experts", type=int, default=0, help="override E of the workload (profiling aid)")
    ap.add_argument("--shared-inter", type=int, default=0,
                    help="add a dense MXFP8 shared expert of this intermediate size on a side stream")
    ap.add_argument("--record-traffic", default="", metavar="RAW_CSV",
                    help="store DRAM bytes per launch of the grouped GEMMs from `ncu -i REP --page raw --csv` "
                         "output into profiles/traffic.json for --config (stamped with the GEMM source hash)")
    ap.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def reduce_max(value: float, device) -> float:
    """Max over ranks of a per-rank float (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tokens_per_s(world: int, rows_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processes its own batch of rows each step."""
    return world * rows_per_rank * steps / (max_ms / 1e3)


GEMM_SOURCES = ("gemm.cu", "ptx.cuh", "mx.cuh", "common.cuh")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def gemm_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "block_scaled_fp8_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def record_traffic(raw_csv: str, workload: str) -> dict:
    """Average dram__bytes_read.sum + dram__bytes_write.sum per launch of each grouped GEMM."""
    import csv
    rows = list(csv.reader(open(raw_csv)))
    hdr = rows[0]
    unit = dict(zip(hdr, rows[1]))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    acc: dict = {}
    for r in rows[2:]:
        d = dict(zip(hdr, r))
        name = d.get("Kernel Name", "")
        if "grouped_gemm_kernel" not in name:
            continue
        key = "w13" if name.rstrip().endswith("1>(CUtensorMap_st, CUtensorMap_st, GemmParams)") else "w2"
        b = sum(float(d[m]) * scale[unit[m]] for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"))
        acc.setdefault(key, []).append(b)
    entry = {k: sum(v) / len(v) for k, v in acc.items()}
    entry["source_hash"] = gemm_source_hash()
    data = json.load(open(TRAFFIC_JSON)) if os.path.exists(TRAFFIC_JSON) else {}
    data[workload] = entry
    with open(TRAFFIC_JSON, "w") as fh:
        json.dump(data, fh, indent=1, sort_keys=True)
    return entry


def measured_traffic(workload: str, keys) -> float | None:
    """Bytes per launch from profiles/traffic.json, or None if absent or taken on other sources."""
    try:
        entry = json.load(open(TRAFFIC_JSON))[workload]
    except Exception:
        return None
    if entry.get("source_hash") != gemm_source_hash() or any(k not in entry for k in keys):
        return None
    return float(sum(entry[k] for k in keys))


def workload_name(cfg):
    return f"{cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} k={cfg.k} I={cfg.I}"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs")
            bf16 = d.get("bf16_tflops")
            if hbm and bf16:
                return float(hbm), float(bf16), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ----------------------------------------------------------------------------------------------
# CPU oracle timing (child process, single-threaded BLAS so `cores` is exact)
# ----------------------------------------------------------------------------------------------
def oracle_sample_timing(cfg_name: str, n_tokens: int, steps: int, warmup: int) -> dict:
    import numpy as np
    import torch

    from block_scaled_fp8_moe_gb300 import synth
    from oracle import moe as M

    cfg = synth.CONFIGS[cfg_name]
    rng = np.random.default_rng(cfg.seed)
    x = torch.from_numpy(rng.standard_normal((n_tokens, cfg.H), dtype=np.float32)).to(torch.bfloat16)
    wr = torch.from_numpy(rng.standard_normal((cfg.E, cfg.H), dtype=np.float32) * np.float32(0.02)).to(torch.bfloat16)
    if cfg.bias == "zipf":
        bias = synth.zipf_bias(cfg.E, cfg.zipf_s, cfg.zipf_gamma, rng.permutation(cfg.E))
    elif cfg.bias == "zero":
        bias = np.zeros(cfg.E, np.float32)
    else:
        bias = (rng.standard_normal(cfg.E) * 0.1).astype(np.float32)
    xf, wrf = x.float().numpy(), wr.float().numpy()
    used = sorted(set(M.route(xf, wrf, bias, cfg.k).topk_idx.reshape(-1).tolist()))
    # oracle-quantised MXFP4 weights of the experts the sample reaches (set-up, not timed)
    q13 = np.zeros((cfg.E, 2 * cfg.I, cfg.H // 2), np.uint8)
    s13 = np.zeros((cfg.E, 2 * cfg.I, cfg.H // 32), np.uint8)
    q2 = np.zeros((cfg.E, cfg.H, cfg.I // 2), np.uint8)
    s2 = np.zeros((cfg.E, cfg.H, cfg.I // 32), np.uint8)
    for e in used:
        er = np.random.default_rng([cfg.seed, e])
        q13[e], s13[e] = M.quant_mxfp4((er.standard_normal((2 * cfg.I, cfg.H), dtype=np.float32) * np.float32(0.02)))
        q2[e], s2[e] = M.quant_mxfp4((er.standard_normal((cfg.H, cfg.I), dtype=np.float32) * np.float32(0.02)))
    times = []
    for i in range(warmup + steps):
        w13 = M.ExpertWeights(q13, s13, cache=len(used) + 1)   # fresh: every step decodes its experts
        w2 = M.ExpertWeights(q2, s2, cache=len(used) + 1)
        t0 = time.perf_counter()
        M.forward(xf, wrf, bias, cfg.k, w13, w2, cfg.I)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    total = sum(times)
    return {"value": n_tokens * len(times) / total, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_tokens} of the {cfg.T} rows of {cfg_name} per step ({len(used)} experts reached), "
                      f"{len(times)} steps, numpy float64 oracle with 1 BLAS thread",
            "ms_per_step": 1e3 * total / len(times)}


def run_oracle_child(cfg_name: str, n_tokens: int, steps: int, warmup: int) -> dict:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", "--config", cfg_name,
           "--cpu-tokens", str(n_tokens), "--steps", str(steps), "--warmup", str(warmup)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


# ----------------------------------------------------------------------------------------------
# clocks sampling during the timed region
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------
def launches_per_step(cfg) -> int:
    """Kernels one moe_forward launches for this shape (mirrors the library's dispatch)."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    nc = H // 64
    decode_router = T <= 64 and 2 * nc <= 256 and (min(T, 16) * nc * 144 + 2 * T * nc * 4) <= 210 * 1024
    if decode_router:
        n = 1                                         # logits (+ fused MXFP8 quantisation)
    elif T > 16 and E <= 256 and H % 64 == 0 and H <= 4096:
        n = 3                                         # norms, tensor-core screen, exact recompute
    else:
        n = 1                                         # small-T or tiled logits
    n += 1 if T <= 256 else 4                         # top-k + plan (+ grid-wide select, scan, scatter)
    if not decode_router:
        n += 1                                        # MXFP8 quantisation (straight into plan order when wide)
    return n + 3                                      # W13, W2, combine


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    from block_scaled_fp8_moe_gb300 import binding as B
    from block_scaled_fp8_moe_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    cfg = synth.CONFIGS[args.config]
    if args.tokens or args.experts:
        import dataclasses
        cfg = dataclasses.replace(cfg, name=cfg.name + "-reduced", T=args.tokens or cfg.T, E=args.experts or cfg.E)

    inp = synth.make_inputs_cuda(cfg, device=dev)
    layer = B.MoeLayer.from_fp32(inp.w_router, inp.bias, inp.w13, inp.w2, cfg.k)
    del inp.w13, inp.w2
    inp.w13 = inp.w2 = None
    torch.cuda.empty_cache()
    x = inp.x
    dead = inp.dead if cfg.dead_frac > 0 else None
    shp = layer.shape(cfg.T)
    ws = layer.workspace(cfg.T)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_clean = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2(v: float) -> None:
        """Write a buffer larger than L2, then read another one: L2 then holds none of the previous
        step's data and no dirty lines whose write-back would land in the next timed region."""
        flush.fill_(v)
        torch.sum(flush_clean, dim=0, out=flush_sink)

    stream = torch.cuda.current_stream()
    shared = side_s = None
    if args.shared_inter:
        # synthetic shared expert: N(0, 0.02) weights -> bf16 -> MXFP8 by the library's quantiser
        n_s = args.shared_inter
        g = torch.Generator(device=dev)
        g.manual_seed(cfg.seed + 1000)
        q = []
        for rows, cols in ((2 * n_s, cfg.H), (cfg.H, n_s)):
            w = (torch.randn((rows, cols), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            q.extend(B.moe_quant_mxfp8(w))
        shared = B.SharedExpert(cfg.H, n_s, *q)
        side_s = torch.cuda.Stream()

    def fwd(xx, dd):
        return layer.forward(xx, dead=dd, out=out, shared=shared, side_stream=side_s)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- warm-up ----
    for _ in range(args.warmup):
        fwd(x, dead)
    B.moe_check_device_status(ws)
    torch.cuda.synchronize()

    # ---- timed: whole layer, inputs resident ----
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(float(i))
        evs[i][0].record(stream)
        fwd(x, dead)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = reduce_max(sum(step_ms), dev)
    B.moe_check_device_status(ws)
    ms_per_step = total_ms / args.steps
    value = tokens_per_s(world, cfg.T, args.steps, total_ms)

    # ---- the same step replayed from a CUDA graph (launch overhead removed) ----
    graph_ms = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fwd(x, dead)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fwd(x, dead)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(float(i))
            gev[i][0].record(stream)
            g.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        graph_ms = sum(a.elapsed_time(b) for a, b in gev) / args.steps
        B.moe_check_device_status(ws)
    except Exception as exc:  # graph capture is a reported variant, not the headline
        graph_ms = f"unavailable: {type(exc).__name__}: {exc}"

    # ---- dominant kernel alone: the four step entry points, events around W13 and W2 ----
    plan = B.Plan(shp, dev)
    xq = torch.empty(cfg.T, cfg.H, dtype=torch.uint8, device=dev)
    xs = torch.empty(cfg.T, cfg.H // 32, dtype=torch.uint8, device=dev)
    hq = torch.empty(cfg.T * cfg.k, cfg.I, dtype=torch.uint8, device=dev)
    hs = torch.empty(cfg.T * cfg.k, B.hs_pitch(cfg.I), dtype=torch.uint8, device=dev)
    k13 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    k2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2(float(i))
        B.moe_route_topk(shp, x, layer.w_router, layer.bias, dead, ws, plan=plan)
        B.moe_quant_mxfp8(x, xq, xs)
        k13[i][0].record(stream)
        B.moe_w13_swiglu_grouped(shp, xq, xs, layer.w13p, layer.w13sp, plan, ws, hq=hq, hs=hs)
        k13[i][1].record(stream)
        flush_l2(float(i) + 0.5)
        k2[i][0].record(stream)
        B.moe_w2_combine_grouped(shp, hq, hs, layer.w2p, layer.w2sp, plan, ws, out=out)
        k2[i][1].record(stream)
    torch.cuda.synchronize()
    B.moe_check_device_status(ws)
    w13_ms = statistics.mean(a.elapsed_time(b) for a, b in k13)
    w2_ms = statistics.mean(a.elapsed_time(b) for a, b in k2)
    counts = plan.expert_counts.cpu()
    touched = int((counts > 0).sum())
    live_slots = int(counts.sum())
    hbm_gbs, bf16_tflops, peak_src = peaks()
    w13_bytes_per_expert = 2 * cfg.I * cfg.H // 2 + 2 * cfg.I * cfg.H // 32
    w2_bytes_per_expert = cfg.H * cfg.I // 2 + cfg.H * cfg.I // 32
    act_bytes_w13 = cfg.T * (cfg.H + cfg.H // 32) + live_slots * (cfg.I + cfg.I // 32)
    decode_like = live_slots <= 2 * cfg.E
    if decode_like:
        alg_bytes = touched * w13_bytes_per_expert + act_bytes_w13
        achieved = alg_bytes / (w13_ms * 1e-3) / 1e9
        roofline = {"kernel": "w13_swiglu_grouped (grouped_gemm_kernel<W13>)", "bound": "hbm",
                    "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                    "frac": round(achieved / hbm_gbs, 4), "traffic": measured_traffic(cfg.name, ("w13",)),
                    "peak_source": f"{peak_src} HBM copy bandwidth",
                    "alg_bytes_per_launch": alg_bytes, "touched_experts": touched,
                    "launch_ms": round(w13_ms, 5)}
    else:
        flops = 2.0 * live_slots * (2 * cfg.I * cfg.H + cfg.H * cfg.I)
        achieved = flops / ((w13_ms + w2_ms) * 1e-3) / 1e12
        peak = FP8_OVER_BF16 * bf16_tflops
        roofline = {"kernel": "w13 + w2 grouped GEMMs", "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": measured_traffic(cfg.name, ("w13", "w2")),
                    "peak_source": f"{peak_src} bf16 x {FP8_OVER_BF16} (nominal fp8/bf16 ratio)",
                    "alg_flops_per_step": flops, "launch_ms": round(w13_ms + w2_ms, 5)}

    # ---- end to end through the public API, host buffers ----
    x_host = x.cpu().pin_memory()
    dead_host = dead.cpu().pin_memory() if dead is not None else None
    out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    dead_dev = torch.empty_like(dead) if dead is not None else None
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for i in range(args.steps):
        flush_l2(float(i))
        e0.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        if dead_dev is not None:
            dead_dev.copy_(dead_host, non_blocking=True)
        fwd(x_dev, dead_dev)
        out_host.copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    barrier()
    e2e_ms = reduce_max(e2e_ms, dev)
    h2d = x_host.numel() * 2 + (dead_host.numel() if dead_host is not None else 0)
    e2e = {"value": tokens_per_s(world, cfg.T, args.steps, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_host.numel() * 2}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_oracle_child(args.config, args.cpu_tokens, steps=3, warmup=0)

    if rank == 0:
        line = {
            "metric": "MoE layer tokens/s", "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 x mxfp4 -> f32",
            "data": "synthetic (seeded; weights N(0,0.02) quantised to MXFP4 by the library)",
            "config": {"workload": workload_name(cfg), "l2": "flushed between timed steps (256 MiB write, then 256 MiB read of another buffer)",
                       "parallelism": f"replica per GPU x{world}", "touched_experts": touched,
                       "live_slots": live_slots,
                       **({"shared_expert_inter": args.shared_inter, "shared_expert": "MXFP8, side stream"}
                          if args.shared_inter else {})},
            "e2e": e2e, "gpu_launches": (launches_per_step(cfg) + (3 if args.shared_inter else 0)) * args.steps,
            "clocks": clk,
            "roofline": roofline,
            "kernels_ms": {"w13": round(w13_ms, 5), "w2_combine": round(w2_ms, 5)},
            "graph_replay": ({"ms_per_step": round(graph_ms, 5),
                              "value": round(world * cfg.T / (graph_ms / 1e3), 2)}
                             if isinstance(graph_ms, float) else graph_ms),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from block_scaled_fp8_moe_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    r = run_oracle_child(args.config, 1, steps=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": "MoE layer tokens/s", "value": r["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": workload_name(cfg)},
        "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.config)))
        return
    if args.oracle_child:
        print(json.dumps(oracle_sample_timing(args.config, args.cpu_tokens, args.steps, args.warmup)))
        return
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
