"""Benchmark of the routed-expert MoE layer on GB300 (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode-6] [--impl reference]

A step is one whole layer call (route -> MXFP8 quant -> W13+SwiGLU+requant -> W2 -> combine) over
one batch of the workload, inputs resident in HBM. L2 is flushed between timed steps (a 256 MiB
write, then a 256 MiB read of a second buffer so that the write's dirty lines are drained before
the step rather than written back inside it); each step is timed with CUDA events on the launching
stream. `value` is tokens/s over all ranks (rows are independent: every rank runs its own replica
of the batch, weak scaling), from the summed step times; the median and a 95 % interval of the
per-step times are reported beside it.

The headline workload (decode-6 unless --config says otherwise) also gets:
  e2e           the same metric through the public API with the batch copied host->device
                (pinned) and the output copied back inside the timed region;
  roofline      the dominant kernel alone (decode: W13 grouped GEMM by algorithmic bytes against
                the measured HBM copy bandwidth), plus the whole layer's bytes per step;
  cpu_baseline  the CPU oracle on the same rows, on one core and on every core of the host;
  prefill       (decode headline only) prefill-32k: tokens/s, and W13 / W2 GEMMs timed alone by
                MMA FLOPs against the block-scaled tensor peak (the larger of the library's
                kind::mxf8f6f4 rate probe and 2 x the measured bf16 peak);
  decode48      (decode headline only) decode-48 with 14 dead rows: tokens/s of all rows and of
                the live rows.
--gpus N without a torchrun environment re-launches this script under torch.distributed.run with
N ranks (one GPU each).
"""
from __future__ import annotations

import argparse
import json
import os
import re
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
NOMINAL_HBM_GBS = 8000.0           # the decode target's HBM figure (about 8 TB/s)
METRIC = "MoE layer tokens/s; decode HBM GB/s and prefill tensor util vs GB300 roofline"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode-6")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="only the --config workload (no prefill / decode-48)")
    ap.add_argument("--tokens", type=int, default=0, help="override T of the workload (profiling aid)")
    ap.add_argument("--experts", type=int, default=0, help="override E of the workload (profiling aid)")
    ap.add_argument("--shared-inter", type=int, default=0,
                    help="add a dense MXFP8 shared expert of this intermediate size on a side stream")
    ap.add_argument("--record-traffic", default="", metavar="RAW_CSV",
                    help="store DRAM bytes per launch of the grouped GEMMs from `ncu -i REP --page raw --csv` "
                         "output into profiles/traffic.json for --config (stamped with the GEMM source hash)")
    ap.add_argument("--launch-check", action="store_true",
                    help="check the multi-rank launch only: every rank reports itself, no GPU work, no bench line")
    ap.add_argument("--oracle-child", default="", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


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


def median_ci(values, level=0.95, resamples=2000, seed=0):
    """Median of per-step times and a bootstrap interval for it (fixed seed: reproducible)."""
    import numpy as np
    v = np.asarray(values, dtype=np.float64)
    if v.size == 0:
        return None
    rng = np.random.default_rng(seed)
    meds = np.median(v[rng.integers(0, v.size, size=(resamples, v.size))], axis=1)
    lo, hi = np.quantile(meds, [(1 - level) / 2, 1 - (1 - level) / 2])
    return {"median": round(float(np.median(v)), 5), "ci95": [round(float(lo), 5), round(float(hi), 5)],
            "mean": round(float(v.mean()), 5), "n": int(v.size)}


GEMM_SOURCES = ("gemm.cu", "gemm.cuh", "gemm2sm.cu", "gemm_ws.cu", "combine.cuh", "topk.cuh", "ptx.cuh", "mx.cuh",
                "common.cuh")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def gemm_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "block_scaled_fp8_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_kind(name: str):
    """Which step a grouped-GEMM launch is, from its demangled name: the MODE template argument of
    grouped_gemm_kernel (0 down, 1 gate/up, 2 both in one launch, 3 the same launch routing a small
    batch itself), the weight-stationary and the CTA-pair kernels; None for every other kernel."""
    if name.startswith("grouped_gemm_ws_kernel"):
        return "w2"
    m = re.search(r"grouped_gemm_pair_kernel<(true|false)", name)
    if m:
        return "w13" if m.group(1) == "true" else "w2"
    m = re.search(r"grouped_gemm_kernel<\d+, (\d)>", name)
    if m:
        return {"0": "w2", "1": "w13", "2": "experts", "3": "experts_selfroute"}[m.group(1)]
    return None


def record_traffic(raw_csv: str, workload: str) -> dict:
    """Average dram__bytes_read.sum + dram__bytes_write.sum per launch of each grouped GEMM."""
    import csv
    # ncu writes its own log lines ahead of the table: the table starts at the "ID" header
    lines = open(raw_csv).read().splitlines()
    start = next(i for i, ln in enumerate(lines) if ln.startswith('"ID"'))
    rows = list(csv.reader(lines[start:]))
    hdr = rows[0]
    unit = dict(zip(hdr, rows[1]))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    acc: dict = {}
    for r in rows[2:]:
        d = dict(zip(hdr, r))
        key = gemm_kind(d.get("Kernel Name", ""))
        if key is None:
            continue
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


def cpu_identity() -> dict:
    """The host's CPU model, logical CPU count and the CPUs this process may run on."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    try:
        affinity = len(os.sched_getaffinity(0))
    except Exception:
        affinity = os.cpu_count()
    import platform
    return {"model": model or platform.processor() or "unknown", "arch": platform.machine(),
            "nproc": os.cpu_count(), "affinity": affinity}


# ----------------------------------------------------------------------------------------------
# CPU oracle timing (child process with one BLAS thread per process; rows split over a pool of
# spawned worker processes for the all-core figure: rows are independent, results identical)
# ----------------------------------------------------------------------------------------------
_ORACLE_STATE: dict = {}


def _oracle_quant_expert(job):
    """Seeded fp32 weights of one expert, quantised by the oracle (set-up, not timed)."""
    import numpy as np
    from oracle import moe as M
    seed, e, H, I = job
    er = np.random.default_rng([seed, e])
    q13, s13 = M.quant_mxfp4(er.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02))
    q2, s2 = M.quant_mxfp4(er.standard_normal((H, I), dtype=np.float32) * np.float32(0.02))
    return e, q13, s13, q2, s2


def _oracle_init(state_dir):
    """Worker set-up: load the sample's inputs and the quantised weights of the experts it reaches."""
    import numpy as np
    from oracle import moe as M
    meta = json.load(open(os.path.join(state_dir, "meta.json")))
    E, H, I = meta["E"], meta["H"], meta["I"]
    q13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.zeros((E, 2 * I, H // 32), np.uint8)
    q2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.zeros((E, H, I // 32), np.uint8)
    for e in meta["used"]:
        for name, arr in (("q13", q13), ("s13", s13), ("q2", q2), ("s2", s2)):
            arr[e] = np.load(os.path.join(state_dir, f"{name}_{e}.npy"))
    _ORACLE_STATE.update(meta=meta, M=M, x=np.load(os.path.join(state_dir, "x.npy")),
                         wr=np.load(os.path.join(state_dir, "wr.npy")), bias=np.load(os.path.join(state_dir, "bias.npy")),
                         w=(q13, s13, q2, s2))


def _oracle_rows(rows):
    """One timed piece of a step: the oracle's whole layer for `rows` (weights decoded afresh)."""
    st = _ORACLE_STATE
    M, meta = st["M"], st["meta"]
    q13, s13, q2, s2 = st["w"]
    n = len(meta["used"]) + 1
    t0 = time.perf_counter()
    M.forward(st["x"][rows], st["wr"], st["bias"], meta["k"], M.ExpertWeights(q13, s13, cache=n),
              M.ExpertWeights(q2, s2, cache=n), meta["I"])
    return time.perf_counter() - t0


def oracle_timing(cfg_name: str, n_rows: int, steps: int, warmup: int, one_core_steps: int) -> dict:
    """Times the oracle's layer over n_rows rows of the workload (numpy-seeded rows of the same
    shape and distribution): `one_core_steps` steps in this process (one core), then, when the host
    has more than one core, warmup + steps steps with the rows split over one process per core."""
    import multiprocessing as mp
    import tempfile

    import numpy as np
    import torch

    from block_scaled_fp8_moe_gb300 import synth
    from oracle import moe as M

    cfg = synth.CONFIGS[cfg_name]
    rng = np.random.default_rng(cfg.seed)
    x = torch.from_numpy(rng.standard_normal((n_rows, cfg.H), dtype=np.float32)).to(torch.bfloat16).float().numpy()
    wr = torch.from_numpy(rng.standard_normal((cfg.E, cfg.H), dtype=np.float32) * np.float32(0.02)
                          ).to(torch.bfloat16).float().numpy()
    if cfg.bias == "zipf":
        bias = synth.zipf_bias(cfg.E, cfg.zipf_s, cfg.zipf_gamma, rng.permutation(cfg.E))
    elif cfg.bias == "zero":
        bias = np.zeros(cfg.E, np.float32)
    else:
        bias = (rng.standard_normal(cfg.E) * 0.1).astype(np.float32)
    used = sorted(set(M.route(x, wr, bias, cfg.k).topk_idx.reshape(-1).tolist()))
    ident = cpu_identity()
    workers = max(1, min(ident["affinity"] or 1, 64))
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory(prefix="moe_oracle_") as d:
        t_setup = time.perf_counter()
        with ctx.Pool(workers) as pool:
            for e, q13, s13, q2, s2 in pool.imap_unordered(_oracle_quant_expert,
                                                           [(cfg.seed, e, cfg.H, cfg.I) for e in used]):
                for name, arr in (("q13", q13), ("s13", s13), ("q2", q2), ("s2", s2)):
                    np.save(os.path.join(d, f"{name}_{e}.npy"), arr)
        np.save(os.path.join(d, "x.npy"), x)
        np.save(os.path.join(d, "wr.npy"), wr)
        np.save(os.path.join(d, "bias.npy"), bias)
        json.dump({"E": cfg.E, "H": cfg.H, "I": cfg.I, "k": cfg.k, "used": used}, open(os.path.join(d, "meta.json"), "w"))
        setup_s = time.perf_counter() - t_setup
        res = {"kind": "oracle", "unit": "tokens/s", "cpu": ident, "rows": n_rows, "experts_reached": len(used),
               "setup_s": round(setup_s, 2)}
        # one core: this process, every row in one call
        _oracle_init(d)
        one = [_oracle_rows(np.arange(n_rows)) for _ in range(max(1, one_core_steps))]
        res["one_core"] = {"value": n_rows * len(one) / sum(one), "ms_per_step": 1e3 * sum(one) / len(one),
                           "cores": 1, "steps": len(one)}
        if steps > 0 and workers > 1:
            groups = [g for g in np.array_split(np.arange(n_rows), min(workers, n_rows)) if len(g)]
            with ctx.Pool(len(groups), initializer=_oracle_init, initargs=(d,)) as pool:
                pool.map(_oracle_rows, groups)                    # workers warm (imports, first decode)
                times = []
                for i in range(warmup + steps):
                    t0 = time.perf_counter()
                    pool.map(_oracle_rows, groups, chunksize=1)
                    if i >= warmup:
                        times.append(time.perf_counter() - t0)
            res["all_cores"] = {"value": n_rows * len(times) / sum(times), "ms_per_step": 1e3 * sum(times) / len(times),
                                "cores": len(groups), "steps": len(times)}
    return res


def run_oracle_child(cfg_name: str, n_rows: int, steps: int, warmup: int, one_core_steps: int = 1) -> dict:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    job = json.dumps({"config": cfg_name, "rows": n_rows, "steps": steps, "warmup": warmup,
                      "one_core_steps": one_core_steps})
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", job]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_line(r: dict, cfg_name: str, cfg_T: int, extrapolated: bool) -> dict:
    """The `cpu_baseline` object: the all-core figure when there is one, the one-core one beside it."""
    best = max((v for v in (r.get("all_cores"), r["one_core"]) if v), key=lambda v: v["value"])
    what = (f"{r['rows']} of the {cfg_T} rows of {cfg_name} per step ({r['experts_reached']} experts reached; "
            f"numpy float64 oracle, weights decoded every step, one BLAS thread per process)")
    if extrapolated:
        what += "; rows are independent, so tokens/s of the sample stands for the whole batch (extrapolated)"
    return {"value": round(best["value"], 4), "unit": "tokens/s", "cores": best["cores"], "kind": "oracle",
            "sample": what, "one_core": {k: round(v, 4) if isinstance(v, float) else v for k, v in r["one_core"].items()},
            "all_cores": ({k: round(v, 4) if isinstance(v, float) else v for k, v in r["all_cores"].items()}
                          if "all_cores" in r else None),
            "cpu": r["cpu"], "setup_s": r["setup_s"]}


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
def decode_router_fits(T: int, H: int, E: int) -> bool:
    """Whether moe_forward routes T rows with the decode router (mirrors decode_router_cfg in the
    library: experts per CTA and per thread, rows per token block, threads and shared memory)."""
    nc = H // 64
    small = T <= 16
    ept, epc = (1, 2) if small else (2, 8)
    epc = min(epc, E)
    tpc = min(T, 2) if small else 8
    threads = -(-epc // ept) * nc

    def smem(tp):
        return tp * nc * 144 + epc * tp * (nc + 1) * 4

    while tpc > 1 and smem(tpc) > 210 * 1024:
        tpc -= 1
    return T <= 64 and threads <= 512 and smem(tpc) <= 210 * 1024


def launches_per_step(cfg, shared: bool = False) -> int:
    """Kernels one moe_forward launches for this shape (mirrors the library's dispatch); `shared`:
    with a shared expert (its identity plan and two GEMMs on the side stream)."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    decode_router = decode_router_fits(T, H, E)
    if decode_router and self_routed_gemms(cfg) and not shared:
        return 2                                      # router (+ quantisation), then GEMMs routing themselves
    if decode_router:
        n = 1                                         # logits (+ fused MXFP8 quantisation)
    elif T > 16 and E <= 256 and H % 64 == 0 and H <= 4096:
        n = 3                                         # norms, tensor-core screen, exact recompute
    else:
        n = 1                                         # small-T or tiled logits
    if T <= 256:
        # top-k + plan in one CTA; more than 24 rows (16 above 256 experts) take a grid-wide top-k
        # launch first
        n += 2 if T > (24 if E <= 256 else 16) else 1
    else:
        n += 4                                        # grid-wide top-k, plan blocks, scan, scatter
    if not decode_router:
        n += 1                                        # MXFP8 quantisation (straight into plan order when wide)
    if fused_gemms(cfg):
        # W13 + W2 (+ the combine, unless a shared expert's row is added in a separate combine)
        return n + (1 + 3 + 1 if shared else 1)
    return n + 3 + (3 if shared else 0)               # W13, W2, combine (+ the shared expert's three)


def wide_w13(cfg) -> bool:
    """True when W13 runs the wide (prefill) token tiles, which read plan-order activation rows."""
    return cfg.T * cfg.k / cfg.E > 64


def self_routed_gemms(cfg) -> bool:
    """True when the one-launch GEMMs also select the experts and build the plan (at most 12 rows,
    256 experts; the library's self_plan_supported, given the decode router and no shared expert)."""
    return 1 <= cfg.T <= 12 and cfg.E <= 256 and fused_gemms(cfg)


def fused_gemms(cfg) -> bool:
    """True when the layer runs W13 and W2 as one launch (decode-sized tiles: at most 32 plan rows
    per expert on average)."""
    return cfg.T * cfg.k / cfg.E <= 32


class Gpu:
    """Device-side state shared by the workloads: the L2 flush and event helpers."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.dev = dev
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_clean = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_sink = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2(self, v: float) -> None:
        """Write a buffer larger than L2, then read another one: L2 then holds none of the previous
        step's data and no dirty lines whose write-back would land in the next timed region."""
        self.flush_buf.fill_(v)
        self.torch.sum(self.flush_clean, dim=0, out=self.flush_sink)

    def events(self, n):
        E = self.torch.cuda.Event
        return [(E(enable_timing=True), E(enable_timing=True)) for _ in range(n)]

    def timed(self, fn, steps, stream, flush=True):
        """Per-step milliseconds of fn() with CUDA events on `stream`, L2 flushed before each."""
        evs = self.events(steps)
        for i in range(steps):
            if flush:
                self.flush_l2(float(i))
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        self.torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]


def build_workload(cfg, dev):
    import torch

    from block_scaled_fp8_moe_gb300 import binding as B
    from block_scaled_fp8_moe_gb300 import synth
    inp = synth.make_inputs_cuda(cfg, device=dev)
    layer = B.MoeLayer.from_fp32(inp.w_router, inp.bias, inp.w13, inp.w2, cfg.k)
    inp.w13 = inp.w2 = None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return inp, layer


def mma_peak(gpu, stream, ws, bf16_tflops, peak_src) -> dict:
    """Block-scaled tensor peak: the larger of the library's kind::mxf8f6f4 rate probe (best of 5
    launches) and 2 x the measured bf16 peak."""
    from block_scaled_fp8_moe_gb300 import binding as B
    iters = 16384
    def rate(mode):
        B.moe_probe_mma_rate(256, ws, mode)                    # warm-up launch
        best = 0.0
        ctas = 0
        for _ in range(5):
            e0, e1 = gpu.events(1)[0]
            e0.record(stream)
            ctas, flops = B.moe_probe_mma_rate(iters, ws, mode)
            e1.record(stream)
            e1.synchronize()
            best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        return best, ctas
    best, ctas = rate(0)
    # the same instruction stream as the grouped GEMMs' wide tiles issue it (context, not the peak):
    # 4 rotating operand buffers, scale copies before each K-chunk, N = 224
    gemm_like, _ = rate(7)
    B.moe_check_device_status(ws)
    doubled = FP8_OVER_BF16 * bf16_tflops
    use_probe = best >= doubled
    return {"tflops": round(max(best, doubled), 1),
            "source": ("tcgen05 kind::mxf8f6f4 rate probe (M=128 N=256 K=32, operands resident, "
                       f"{ctas} CTAs, best of 5)") if use_probe else
                      f"{peak_src} bf16 x {FP8_OVER_BF16} (nominal fp8/bf16 ratio)",
            "probe_tflops": round(best, 1), "bf16_x2_tflops": round(doubled, 1),
            "gemm_sequence_tflops": round(gemm_like, 1)}


def measure(cfg, args, gpu, world, headline: bool, peak_info=None):
    """Time one workload: the whole layer (eager and CUDA-graph replay), then its kernels alone."""
    import torch

    from block_scaled_fp8_moe_gb300 import binding as B
    dev = gpu.dev
    inp, layer = build_workload(cfg, dev)
    x = inp.x
    dead = inp.dead if cfg.dead_frac > 0 else None
    shp = layer.shape(cfg.T)
    ws = layer.workspace(cfg.T)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    shared = side_s = None
    if headline and args.shared_inter:
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

    def fwd(xx=x, dd=dead):
        return layer.forward(xx, dead=dd, out=out, shared=shared, side_stream=side_s)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        fwd()
    B.moe_check_device_status(ws)
    torch.cuda.synchronize()

    # ---- timed: whole layer, inputs resident ----
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    # the pause idles the GPU: a few untimed steps bring its clocks back up before the timed ones
    for i in range(3):
        gpu.flush_l2(float(i))
        fwd()
    barrier()
    torch.cuda.synchronize()
    step_ms = gpu.timed(fwd, args.steps, stream)
    barrier()
    clk = clocks.stop()
    total_ms = reduce_max(sum(step_ms), dev)
    B.moe_check_device_status(ws)
    ms_per_step = total_ms / args.steps
    rec = {"workload": workload_name(cfg), "ms_per_step": round(ms_per_step, 5),
           "value": round(tokens_per_s(world, cfg.T, args.steps, total_ms), 2), "unit": "tokens/s",
           "step_ms": median_ci(step_ms), "clocks": clk}

    # ---- the same step replayed from a CUDA graph (launch overhead removed) ----
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fwd()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fwd()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        gms = gpu.timed(graph.replay, args.steps, stream)
        B.moe_check_device_status(ws)
        gmean = sum(gms) / len(gms)
        rec["graph_replay"] = {"ms_per_step": round(gmean, 5), "value": round(world * cfg.T / (gmean / 1e3), 2),
                               "step_ms": median_ci(gms)}
        del graph
    except Exception as exc:  # graph capture is a reported variant, not the headline
        rec["graph_replay"] = f"unavailable: {type(exc).__name__}: {exc}"

    # ---- the kernels alone, through the step entry points (the same kernels moe_forward runs) ----
    plan = B.Plan(shp, dev)
    S = cfg.T * cfg.k
    xq = torch.empty(cfg.T, cfg.H, dtype=torch.uint8, device=dev)
    xs = torch.empty(cfg.T, cfg.H // 32, dtype=torch.uint8, device=dev)
    hq = torch.empty(S, cfg.I, dtype=torch.uint8, device=dev)
    hs = torch.empty(S, B.hs_pitch(cfg.I), dtype=torch.uint8, device=dev)
    y = torch.empty(S, cfg.H, dtype=torch.float32, device=dev)
    wide = wide_w13(cfg)
    if wide:
        xqp = torch.empty(S, cfg.H, dtype=torch.uint8, device=dev)
        xsp = torch.empty(S, cfg.H // 32, dtype=torch.uint8, device=dev)
        shp_w13 = layer.shape(cfg.T, B.MOE_FLAG_X_PLAN_ORDER)
    else:
        shp_w13 = shp
    ev = {n: gpu.events(args.steps) for n in ("w13", "w2", "combine", "experts")}
    for i in range(args.steps):
        gpu.flush_l2(float(i))
        B.moe_route_topk(shp, x, layer.w_router, layer.bias, dead, ws, plan=plan)
        if wide:
            B.moe_quant_mxfp8_plan(shp, x, plan, xqp, xsp)
            a_q, a_s = xqp, xsp
        else:
            B.moe_quant_mxfp8(x, xq, xs)
            a_q, a_s = xq, xs
        gpu.flush_l2(float(i) + 0.25)
        ev["w13"][i][0].record(stream)
        B.moe_w13_swiglu_grouped(shp_w13, a_q, a_s, layer.w13p, layer.w13sp, plan, ws, hq=hq, hs=hs)
        ev["w13"][i][1].record(stream)
        gpu.flush_l2(float(i) + 0.5)
        ev["w2"][i][0].record(stream)
        B.moe_w2_grouped(shp, hq, hs, layer.w2p, layer.w2sp, plan, ws, y=y)
        ev["w2"][i][1].record(stream)
        gpu.flush_l2(float(i) + 0.75)
        ev["combine"][i][0].record(stream)
        B.moe_combine(shp, y, plan, ws, dead=dead, out=out)
        ev["combine"][i][1].record(stream)
        # both expert GEMMs as the layer runs them (one launch for decode-sized batches)
        gpu.flush_l2(float(i) + 0.875)
        ev["experts"][i][0].record(stream)
        B.moe_experts_grouped(shp_w13, a_q, a_s, layer.w13p, layer.w13sp, layer.w2p, layer.w2sp, plan, ws,
                              hq=hq, hs=hs, y=y)
        ev["experts"][i][1].record(stream)
    torch.cuda.synchronize()
    B.moe_check_device_status(ws)
    kms = {n: statistics.mean(a.elapsed_time(b) for a, b in v) for n, v in ev.items()}
    rec["kernels_ms"] = {n: round(v, 5) for n, v in kms.items()}
    counts = plan.expert_counts.cpu()
    touched = int((counts > 0).sum())
    live_slots = int(counts.sum())
    rec["touched_experts"] = touched
    rec["live_slots"] = live_slots
    rec["expert_histogram"] = counts.tolist()
    live_rows = cfg.T - (int(dead.sum().item()) if dead is not None else 0)
    if dead is not None:
        rec["live_rows"] = live_rows
        rec["value_live_rows"] = round(tokens_per_s(world, live_rows, args.steps, total_ms), 2)

    hbm_gbs, bf16_tflops, peak_src = peaks()
    w13_bytes_per_expert = 2 * cfg.I * cfg.H // 2 + 2 * cfg.I * cfg.H // 32
    w2_bytes_per_expert = cfg.H * cfg.I // 2 + cfg.H * cfg.I // 32
    act_w13 = cfg.T * (cfg.H + cfg.H // 32) + live_slots * (cfg.I + cfg.I // 32)
    act_w2 = live_slots * (cfg.I + cfg.I // 32) + 4 * live_slots * cfg.H
    decode_like = not wide
    if decode_like:
        alg13 = touched * w13_bytes_per_expert + act_w13
        alg2 = touched * w2_bytes_per_expert + act_w2
        ach13 = alg13 / (kms["w13"] * 1e-3) / 1e9
        ach2 = alg2 / (kms["w2"] * 1e-3) / 1e9
        w13_line = {"kernel": "w13_swiglu_grouped (grouped_gemm_kernel, gate/up)", "bound": "hbm",
                    "achieved": round(ach13, 1), "peak": hbm_gbs, "unit": "GB/s", "frac": round(ach13 / hbm_gbs, 4),
                    "alg_bytes_per_launch": alg13, "launch_ms": round(kms["w13"], 5)}
        w2_line = {"kernel": "w2_grouped (grouped_gemm_kernel, down)", "bound": "hbm", "achieved": round(ach2, 1),
                   "peak": hbm_gbs, "unit": "GB/s", "frac": round(ach2 / hbm_gbs, 4), "alg_bytes_per_launch": alg2,
                   "launch_ms": round(kms["w2"], 5)}
        if fused_gemms(cfg):
            # the layer runs both GEMMs as one persistent launch: that launch is the dominant kernel
            achf = (alg13 + alg2) / (kms["experts"] * 1e-3) / 1e9
            # DRAM bytes per launch: of this launch if captured, else of the layer's own launch of
            # the same GEMMs (the self-routing variant, which also reads the router's scores from L2)
            traffic, traffic_kernel = measured_traffic(cfg.name, ("experts",)), "grouped_gemm_kernel<BN, 2>"
            if traffic is None:
                traffic, traffic_kernel = measured_traffic(cfg.name, ("experts_selfroute",)), "grouped_gemm_kernel<BN, 3>"
            rec["roofline"] = {"kernel": "experts_grouped (grouped_gemm_kernel, gate/up then down in one launch)",
                               "bound": "hbm", "achieved": round(achf, 1), "peak": hbm_gbs, "unit": "GB/s",
                               "frac": round(achf / hbm_gbs, 4), "traffic": traffic,
                               "traffic_kernel": traffic_kernel if traffic is not None else None,
                               "peak_source": f"{peak_src} HBM copy bandwidth (burst)",
                               "alg_bytes_per_launch": alg13 + alg2, "touched_experts": touched,
                               "launch_ms": round(kms["experts"], 5)}
            rec["w13_alone"] = w13_line
            rec["w2_roofline"] = w2_line
        else:
            rec["roofline"] = dict(w13_line, traffic=measured_traffic(cfg.name, ("w13",)),
                                   peak_source=f"{peak_src} HBM copy bandwidth (burst)", touched_experts=touched)
            rec["w2_roofline"] = w2_line
        # the whole layer: every touched expert's W13 + W2 codes and scales, the router weight,
        # and the activations, over the step time
        layer_bytes = (touched * (w13_bytes_per_expert + w2_bytes_per_expert) + cfg.E * cfg.H * 2
                       + cfg.T * cfg.H * 2 + act_w13 + act_w2 + 4 * live_slots * cfg.H + cfg.T * cfg.H * 2)
        lr = {"bytes_per_step": layer_bytes}
        for key, ms in (("eager", ms_per_step),
                        ("graph", rec["graph_replay"]["ms_per_step"] if isinstance(rec["graph_replay"], dict) else None)):
            if ms:
                gbs = layer_bytes / (ms * 1e-3) / 1e9
                lr[key] = {"achieved_gbs": round(gbs, 1), "frac_of_measured": round(gbs / hbm_gbs, 4),
                           "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
        rec["layer_roofline"] = lr
    else:
        pk = peak_info
        f13 = 2.0 * live_slots * 2 * cfg.I * cfg.H
        f2 = 2.0 * live_slots * cfg.H * cfg.I
        a13 = f13 / (kms["w13"] * 1e-3) / 1e12
        a2 = f2 / (kms["w2"] * 1e-3) / 1e12
        rec["roofline"] = {"kernel": "w13_swiglu_grouped (grouped_gemm_kernel<W13>)", "bound": "tensor",
                           "achieved": round(a13, 1), "peak": pk["tflops"], "unit": "TFLOP/s",
                           "frac": round(a13 / pk["tflops"], 4), "traffic": measured_traffic(cfg.name, ("w13",)),
                           "peak_source": pk["source"], "alg_flops_per_launch": f13,
                           "launch_ms": round(kms["w13"], 5)}
        rec["w2_roofline"] = {"bound": "tensor", "achieved": round(a2, 1), "peak": pk["tflops"], "unit": "TFLOP/s",
                              "frac": round(a2 / pk["tflops"], 4), "alg_flops_per_launch": f2,
                              "launch_ms": round(kms["w2"], 5)}
        ystep = 4 * live_slots * cfg.H + 2 * cfg.T * cfg.H + 8 * live_slots
        rec["combine_hbm"] = {"bytes_per_launch": ystep,
                              "achieved_gbs": round(ystep / (kms["combine"] * 1e-3) / 1e9, 1)}
        lf = (f13 + f2) / (ms_per_step * 1e-3) / 1e12
        rec["layer_roofline"] = {"flops_per_step": f13 + f2, "achieved_tflops": round(lf, 1),
                                 "frac": round(lf / pk["tflops"], 4)}
    rec["_state"] = (layer, inp, fwd, out, ws, dead)
    return rec


def e2e_measure(cfg, args, gpu, world, state) -> dict:
    """The same metric through the public API with the batch copied in from pinned host memory and
    the output copied back, inside the timed region."""
    import torch
    layer, inp, fwd, out, ws, dead = state
    x = inp.x
    stream = torch.cuda.current_stream()
    x_host = x.cpu().pin_memory()
    dead_host = dead.cpu().pin_memory() if dead is not None else None
    out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    dead_dev = torch.empty_like(dead) if dead is not None else None
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = gpu.events(1)[0]
    e2e_ms = 0.0
    for i in range(args.steps):
        gpu.flush_l2(float(i))
        e0.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        if dead_dev is not None:
            dead_dev.copy_(dead_host, non_blocking=True)
        fwd(x_dev, dead_dev)
        out_host.copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    if world > 1:
        torch.distributed.barrier()
    e2e_ms = reduce_max(e2e_ms, gpu.dev)
    h2d = x_host.numel() * 2 + (dead_host.numel() if dead_host is not None else 0)
    return {"value": round(tokens_per_s(world, cfg.T, args.steps, e2e_ms), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_host.numel() * 2}


def gpu_arm(args):
    import dataclasses

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
    gpu = Gpu(dev)
    stream = torch.cuda.current_stream()
    cfg = synth.CONFIGS[args.config]
    if args.tokens or args.experts:
        cfg = dataclasses.replace(cfg, name=cfg.name + "-reduced", T=args.tokens or cfg.T, E=args.experts or cfg.E)

    hbm_gbs, bf16_tflops, peak_src = peaks()
    status_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    pk = mma_peak(gpu, stream, status_ws, bf16_tflops, peak_src)

    head = measure(cfg, args, gpu, world, headline=True, peak_info=pk)
    e2e = e2e_measure(cfg, args, gpu, world, head.pop("_state"))
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra and cfg.name == "decode-6":
        for key, name in (("decode48", "decode-48"), ("prefill", "prefill-32k")):
            r = measure(synth.CONFIGS[name], args, gpu, world, headline=False, peak_info=pk)
            r.pop("_state")
            torch.cuda.empty_cache()
            if key == "decode48":
                r["launches_per_step"] = launches_per_step(synth.CONFIGS[name])
            extra[key] = r

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the headline's rows: all of them for a decode batch (C1: 6 rows); a few rows of a
        # prefill batch, extrapolated (rows are independent)
        n = cfg.T if cfg.T <= 8 else 8
        cpu = cpu_baseline_line(run_oracle_child(cfg.name.replace("-reduced", ""), n, steps=3, warmup=0,
                                                 one_core_steps=1), cfg.name, cfg.T, extrapolated=n < cfg.T)
        if "prefill" in extra:
            extra["prefill"]["cpu_baseline"] = cpu_baseline_line(
                run_oracle_child("prefill-32k", 8, steps=2, warmup=0, one_core_steps=1), "prefill-32k", 32768,
                extrapolated=True)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 x mxfp4 -> f32",
            "data": "synthetic (seeded; weights N(0,0.02) quantised to MXFP4 by the library)",
            "config": {"workload": head["workload"],
                       "l2": "flushed between timed steps (256 MiB write, then 256 MiB read of another buffer)",
                       "parallelism": f"replica per GPU x{world}", "touched_experts": head["touched_experts"],
                       "live_slots": head["live_slots"], "expert_histogram": head["expert_histogram"],
                       **({"shared_expert_inter": args.shared_inter, "shared_expert": "MXFP8, side stream"}
                          if args.shared_inter else {})},
            "step_ms": head["step_ms"],
            "e2e": e2e, "gpu_launches": launches_per_step(cfg, bool(args.shared_inter)) * args.steps,
            "clocks": head["clocks"],
            "roofline": head["roofline"],
            "w2_roofline": head["w2_roofline"],
            "layer_roofline": head["layer_roofline"],
            "kernels_ms": head["kernels_ms"],
            "graph_replay": head["graph_replay"],
            "tensor_peak": pk,
            **extra,
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
    n = cfg.T if cfg.T <= 8 else 8
    # the oracle has nothing to warm up beyond its first step: one warm-up step at most keeps the
    # whole arm within a few minutes
    r = run_oracle_child(args.config, n, steps=args.steps, warmup=min(args.warmup, 1), one_core_steps=1)
    best = max((v for v in (r.get("all_cores"), r["one_core"]) if v), key=lambda v: v["value"])
    cb = cpu_baseline_line(r, cfg.name, cfg.T, extrapolated=n < cfg.T)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(best["value"], 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(best["ms_per_step"], 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": workload_name(cfg)},
        "cpu_baseline": cb,
        "e2e": {"value": round(best["value"], 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def relaunch_under_torchrun(args, argv) -> int:
    """`--gpus N` outside a torchrun environment: run this script as N ranks on this node."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def launch_check(args):
    """Every rank reports (rank, world) and a rank-dependent time; rank 0 prints the max over ranks
    and the throughput the bench would derive from it (gloo without GPUs, NCCL with them)."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dev = "cpu"
    if world > 1:
        if backend == "nccl":
            local = int(os.environ.get("LOCAL_RANK", "0"))
            torch.cuda.set_device(local)
            dev = torch.device("cuda", local)
        dist.init_process_group(backend)
    local_ms = 10.0 + 5.0 * rank
    ranks = [None] * world
    if world > 1:
        dist.all_gather_object(ranks, rank)
    else:
        ranks = [0]
    m = reduce_max(local_ms, dev)
    if rank == 0:
        print(json.dumps({"launch_check": True, "world": world, "ranks": sorted(ranks), "max_ms": m,
                          "tokens_per_s": tokens_per_s(world, 6, args.steps, m), "backend": backend}))
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse(argv)
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.config)))
        return 0
    if args.oracle_child:
        job = json.loads(args.oracle_child)
        print(json.dumps(oracle_timing(job["config"], job["rows"], job["steps"], job["warmup"], job["one_core_steps"])))
        return 0
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch_under_torchrun(args, argv)
    if args.launch_check:
        launch_check(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
