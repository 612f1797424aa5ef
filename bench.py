"""Benchmark of the MoE dispatch/combine hot path on GB300.

One step = one pass of the whole path over one batch of the DeepSeek-V3-shaped
workload (8192 tokens, hidden 7168, 256 experts in 8 groups, top-4 groups then
top-8 experts, 32 logical ranks x 8 experts): group-limited gating and layout
(one call, ep_gate_layout) -> FP8 e4m3 1x128 dispatch -> weighted BF16
combine of the expert outputs (identity experts: the BF16-dispatched rows,
made once before timing).

Prints ONE JSON line (rank 0): whole-job tokens/s, per-op times and HBM
GB/s, the roofline of the dominant kernel, an end-to-end figure through the
public API with host buffers, the CPU oracle as a baseline, and SM clocks
sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) each rank runs an independent replica on its own
batch (weak scaling, no collective on the data path); the time is the max
over ranks.
"""
import argparse
import hashlib
import json
import os
import random
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of peak), 1×GB300"
WORKLOAD = "dsv3"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20          # twice the 129 MB L2
QUEUE_AHEAD_CYCLES = 200_000        # ~0.1 ms of GPU spin before each timed step (host launches get ahead)
# The CUDA event clock ticks in steps of about 2 us on this GPU, and a fixed
# spin before each timed call starts it at the same phase of a tick every
# time, so every repetition rounds the same way.  A random extra spin of up
# to ~4 us (two ticks) spreads the phase: the mean over repetitions then
# resolves below a tick.
DITHER_CYCLES = 8192
_dither = random.Random(20261203)


def queue_ahead():
    """The spin before a timed call (outside the events): queue-ahead plus
    a random phase."""
    import torch
    torch.cuda._sleep(QUEUE_AHEAD_CYCLES + _dither.randrange(DITHER_CYCLES))
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def workload_desc(cfg):
    return ("DeepSeek-V3-shaped MoE layer: T=%d H=%d E=%d in %d groups, top-%d groups then top-%d experts, "
            "%d logical ranks x %d experts; FP8 e4m3 1x128 dispatch, BF16 combine"
            % (cfg["T"], cfg["H"], cfg["E"], cfg["n_groups"], cfg["topk_group"], cfg["k"],
               cfg["E"] // cfg["experts_per_rank"], cfg["experts_per_rank"]))


def algorithmic_bytes(cfg):
    """Bytes each op must move at least (per launch over the whole batch)."""
    T, H, E, k = cfg["T"], cfg["H"], cfg["E"], cfg["k"]
    return {
        "gate": T * (4 * E + 8 * k) + (4 * E if cfg["bias"] else 0),
        "layout": T * k * 4 * 3,                                        # idx in, pos + src out
        "dispatch_fp8": T * (2 * H + k * (H + 4 * (H // 128)) + 4 * k),
        "dispatch_bf16": T * (2 * H + 2 * H * k + 4 * k),
        "combine": T * (2 * H * k + 8 * k + 2 * H),
    }


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# The source files each timed kernel is compiled from.
KERNEL_SOURCES = {
    "combine_kernel": ("combine.cu", "coop.cuh", "ep_internal.cuh"),
    "dispatch_bulk_kernel": ("dispatch.cu", "dispatch_impl.cuh", "ep_internal.cuh"),
    "route_kernel": ("route.cu", "coop.cuh", "gate_fast.cuh", "gate_impl.cuh", "ep_internal.cuh"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_group_limited_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(op):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel as it is now (the same hash of its sources); else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get("kernels", {}).get(op)
    if op not in KERNEL_SOURCES or not rec or rec.get("source_hash") != kernel_source_hash(op):
        return None
    return int(rec["bytes_per_launch"])


class Replicas:
    """One process per GPU, each an independent replica of the path on its
    own seeded batch: the tokens are data-parallel, so there is no collective
    on the data path.  The only collectives are the barriers around the timed
    region and the max over ranks of the measured times.  `value` is the
    tokens of all ranks over that max time (weak scaling)."""

    SEED_STRIDE = 1000

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self._dist = None
        self._device = None

    def init(self, backend, device):
        """Join the process group (only when there is more than one rank)."""
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                dist.init_process_group(backend, device_id=device)
            else:
                dist.init_process_group(backend)
            self._dist = dist
        self._device = device
        return self

    def seed_offset(self):
        return self.SEED_STRIDE * self.rank

    def is_printer(self):
        return self.rank == 0

    def barrier(self):
        if self._dist is not None:
            self._dist.barrier()

    def max(self, x):
        """The maximum of a float over all ranks (x itself for one rank)."""
        if self._dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self._device)
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX)
        return float(t.item())

    def tokens_per_s(self, tokens_per_rank, ms):
        return self.world * tokens_per_rank / (ms * 1e-3)

    def close(self):
        if self._dist is not None:
            self._dist.destroy_process_group()
            self._dist = None


class ClockSampler:
    """SM clocks and throttle reasons sampled while the GPU works.

    A thread polls NVML (libnvidia-ml through ctypes, read-only queries)
    every millisecond, so that even a timed region of a few milliseconds
    holds samples; where NVML cannot be loaded, `nvidia-smi -lms` is read
    instead.  Only the samples taken between mark_start() and mark_end()
    count."""

    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    # NVML clocks-event reason bits of those four names
    NVML_BITS = [0x8, 0x40, 0x20, 0x4]
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=1.0, uuid=None):
        self.index, self.period_ms, self.uuid = index, period_ms, uuid
        self.samples, self.t0, self.t1 = [], None, None
        self.proc, self.thread, self.source = None, None, None
        self._stop = False

    # --- NVML
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-%s" % self.uuid).encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _nvml_loop(self, lib, h, reasons):
        import ctypes
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            t = time.monotonic()
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons(h, ctypes.byref(rs)) == 0):
                self.samples.append((t, float(clk.value), float(mx.value),
                                     [bool(rs.value & b) for b in self.NVML_BITS]))
            time.sleep(self.period_ms / 1000.0)

    # --- nvidia-smi fallback
    def _smi_loop(self):
        for ln in self.proc.stdout:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                self.samples.append((time.monotonic(), float(f[0]), float(f[1]),
                                     [v.lower() == "active" for v in f[3:7]]))
            except ValueError:
                continue

    def __enter__(self):
        import threading
        try:
            lib, h, reasons = self._nvml_open()
            self.thread = threading.Thread(target=self._nvml_loop, args=(lib, h, reasons), daemon=True)
            self.source = "nvml"
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                              "--format=csv,noheader,nounits", "-lms", "20"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.thread = threading.Thread(target=self._smi_loop, daemon=True)
                self.source = "nvidia-smi"
            except OSError:
                self.thread = None
        if self.thread is not None:
            self.thread.start()
        time.sleep(0.1)
        return self

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *a):
        self._stop = True
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        rows = [(c, m, r) for ts, c, m, r in list(self.samples)
                if self.t0 is not None and self.t0 <= ts <= (self.t1 or ts)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source,
                    "note": "no sample fell inside the timed region"}
        reasons = sorted({self.NAMES[i] for _, _, r in rows for i, a in enumerate(r) if a})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": self.source}


class PathRunner:
    """Device buffers and launches of one step of the hot path (rank-local)."""

    def __init__(self, cfg, seed_offset=0, device="cuda"):
        import torch

        import combine_group_limited_gb300 as ep
        self.torch, self.ep, self.cfg = torch, ep, dict(cfg)
        self.cfg["seed"] = cfg["seed"] + seed_offset
        c = self.cfg
        T, H, E, k, epr = c["T"], c["H"], c["E"], c["k"], c["experts_per_rank"]
        inp = synth.make_inputs(c)
        self.host = inp
        self.scores = torch.from_numpy(inp["scores"]).to(device)
        self.bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(device)
        self.x = torch.from_numpy(inp["x"].view(np.int16)).to(device).view(torch.bfloat16)
        self.gcfg = ep.gate_cfg(E, k, c["n_groups"], c["topk_group"], c["topk_in_group"], c["score_fn"],
                                c["normalize"])
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=device)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.lay = ep.alloc_layout(T, k, E, epr, device)
        self.ws = ep.alloc_layout_workspace(T, k, E, epr, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.recv_q = torch.empty((T * k, H), dtype=torch.uint8, device=device)
        self.recv_s = torch.empty((T * k, H // 128), dtype=torch.float32, device=device)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        # expert outputs for the combine: identity experts = the BF16 rows
        self.gate()
        self.layout()
        self.y = ep.ep_dispatch(self.x, self.lay.pos, "bf16")
        torch.cuda.synchronize()

    # the launches of a step (gpu_launches counts them): gating and layout in
    # one cooperative launch, then dispatch, then combine
    LAUNCHES_PER_STEP = 3

    def gate(self):
        self.ep.ep_gate(self.scores, self.bias, self.gcfg, self.topk_idx, self.topk_w)

    def layout(self):
        c = self.cfg
        self.ep.ep_get_layout(self.topk_idx, c["E"], c["experts_per_rank"], out=self.lay, workspace=self.ws,
                              err_flag=self.err)

    def route(self):
        """Gating and layout in one call (one cooperative launch above 4096
        entries, as on the bench's workload)."""
        c = self.cfg
        self.ep.ep_gate_layout(self.scores, self.bias, self.gcfg, c["experts_per_rank"], topk_idx=self.topk_idx,
                               topk_w=self.topk_w, out=self.lay, workspace=self.ws, err_flag=self.err)

    def dispatch(self):
        self.ep.ep_dispatch(self.x, self.lay.pos, "fp8", recv=self.recv_q, recv_scales=self.recv_s,
                            err_flag=self.err)

    def dispatch_bf16(self):
        if not hasattr(self, "recv_b"):
            self.recv_b = self.torch.empty_like(self.y)
        self.ep.ep_dispatch(self.x, self.lay.pos, "bf16", recv=self.recv_b, err_flag=self.err)

    def combine(self):
        self.ep.ep_combine(self.y, self.lay.pos, self.topk_w, out=self.out, err_flag=self.err)

    def step(self):
        self.route()
        self.dispatch()
        self.combine()


def pct(xs, q):
    """The q-th percentile (0..100) of xs, by linear interpolation."""
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


# Every workload of the benchmark's configuration list, with the dispatch
# payloads it is quoted with (the first one is the step's); each gets its
# routing, dispatch and combine timed in the bench line's "configs".
CONFIG_RUNS = {
    "tiny": ("bf16",),
    "mixtral": ("bf16",),
    "dsv3": ("fp8", "bf16"),
    "skewed": ("fp8", "bf16"),
    "qwen3": ("bf16",),
    "decode": ("fp8", "bf16"),
}


def trimmed_mean(ts, cut=0.05):
    """Mean of the values between the `cut` and 1 - `cut` quantiles."""
    v = sorted(ts)
    n = int(len(v) * cut)
    return statistics.mean(v[n:len(v) - n] if len(v) > 2 * n else v)


def time_configs(reps, peak, flush_l2):
    """Per workload: mean (of the central 90 %), median, p10 and p90 event
    times of each op over `reps` L2-flushed calls, GB/s and fraction of the
    HBM peak from its algorithmic bytes and the mean time, and the tokens/s
    of one routing + dispatch + combine step (means)."""
    import torch
    stream = torch.cuda.current_stream()
    out = {}
    for name, payloads in CONFIG_RUNS.items():
        cfg = synth.config(name)
        r = PathRunner(cfg)
        nb = op_bytes(cfg)
        ops = [("route", r.route, nb["gate_layout"])]
        for p in payloads:
            fn = r.dispatch if p == "fp8" else r.dispatch_bf16
            ops.append(("dispatch_" + p, fn, nb["dispatch_" + p]))
        ops.append(("combine", r.combine, nb["combine"]))
        if cfg["H"] % 128 == 0:
            # the FP8 paths on every workload whose rows take 1x128 blocks:
            # the dispatches, and the combines from the FP8 / MXFP8 rows they
            # wrote (identity experts)
            T, H, k = cfg["T"], cfg["H"], cfg["k"]
            mq = torch.empty((T * k, H), dtype=torch.uint8, device="cuda")
            me = torch.empty((T * k, H // 32), dtype=torch.uint8, device="cuda")
            fp8_out = torch.empty_like(r.out)
            if "fp8" not in payloads:
                ops.append(("dispatch_fp8", r.dispatch, nb["dispatch_fp8"]))
            ops.append(("dispatch_mxfp8", lambda: r.ep.ep_dispatch(r.x, r.lay.pos, "mxfp8", recv=mq, recv_scales=me,
                                                                   err_flag=r.err), nb["dispatch_mxfp8"]))
            ops.append(("combine_fp8", lambda: r.ep.ep_combine_fp8(r.recv_q, r.recv_s, r.lay.pos, r.topk_w,
                                                                   out=fp8_out, err_flag=r.err), nb["combine_fp8"]))
            ops.append(("combine_mxfp8", lambda: r.ep.ep_combine_fp8(mq, me, r.lay.pos, r.topk_w, out=fp8_out,
                                                                     err_flag=r.err), nb["combine_mxfp8"]))
        res = {}
        for op, fn, nbytes in ops:
            fn()
            ts = []
            for i in range(reps + 2):
                flush_l2(i)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                if i >= 2:
                    ts.append(a.elapsed_time(b) * 1e3)
            # The event clock ticks in steps of about 2 us on this GPU: the
            # mean over the repetitions (random phase, queue_ahead) resolves
            # below a tick and gives the rates; the percentiles show the
            # spread.
            mean = trimmed_mean(ts)
            gbs = nbytes / (mean * 1e-6) / 1e9
            res[op] = {"us": round(mean, 2), "us_median": round(pct(ts, 50), 2), "us_p10": round(pct(ts, 10), 2),
                       "us_p90": round(pct(ts, 90), 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                       "bytes": nbytes}
        if int(r.err.item()) != 0:
            raise RuntimeError("device error flag set on %s: %d" % (name, int(r.err.item())))
        step_us = res["route"]["us"] + res["dispatch_" + payloads[0]]["us"] + res["combine"]["us"]
        out[name] = {"T": cfg["T"], "H": cfg["H"], "E": cfg["E"], "k": cfg["k"],
                     "step_dispatch": payloads[0], "step_us": round(step_us, 2),
                     "step_tokens_per_s": round(cfg["T"] / (step_us * 1e-6), 1), "ops": res}
        ops = None  # the FP8 buffers the timed calls hold
        del r
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    rep = Replicas()
    world, local = rep.world, rep.local
    torch.cuda.set_device(local)
    rep.init("nccl", torch.device("cuda", local))

    from combine_group_limited_gb300 import build as epbuild
    epbuild.build()

    cfg = synth.config(WORKLOAD)
    r = PathRunner(cfg, seed_offset=rep.seed_offset())
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")  # summed in fp32: no cast kernel

    def flush_l2(s):
        # Evict the step's data from L2: write a buffer twice the L2 size,
        # then read another one so that the written lines are back in HBM
        # before the timed events (L2 is write-back; otherwise the next
        # step would pay for writing the flush buffer).  Then keep the GPU
        # busy for a while (a spin kernel, outside the events), so that the
        # host has enqueued the step's launches before the GPU reaches the
        # first event: the events then time the kernels, not the host's
        # launch calls.
        flush.fill_(s & 0xFF)
        flush_rd.sum()
        queue_ahead()

    ops = ("route", "dispatch", "combine")

    for w in range(args.warmup):
        flush_l2(w)
        r.step()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(args.steps)]
    rep.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        for s in range(args.steps):
            flush_l2(s)                                 # evict L2 between steps (outside the events)
            ev[s][0].record(stream)
            for i, op in enumerate(ops):
                getattr(r, op)()
                ev[s][i + 1].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    rep.barrier()
    if int(r.err.item()) != 0:
        raise RuntimeError("device error flag set: %d" % int(r.err.item()))

    per_op = {op: [ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)] for i, op in enumerate(ops)}
    step_ms = [ev[s][0].elapsed_time(ev[s][-1]) for s in range(args.steps)]
    ms_per_step = rep.max(sum(step_ms) / args.steps)

    # end to end through the public API: pinned host inputs -> device -> path -> host output
    e2e = run_e2e(r, args, chunks=args.e2e_chunks, graph=not args.e2e_no_graph, nsets=args.e2e_sets)
    e2e["ms"] = rep.max(e2e["ms"])

    configs = None
    if rep.is_printer() and not args.no_configs:
        configs = time_configs(args.config_reps, measured_hbm_peak()[0], flush_l2)

    if rep.is_printer():
        T = cfg["T"]
        peak, peak_kind = measured_hbm_peak()
        ab = algorithmic_bytes(cfg)
        bytes_of = {"route": ab["gate"] + ab["layout"], "dispatch": ab["dispatch_fp8"], "combine": ab["combine"]}
        kname = {"route": "route_kernel", "dispatch": "dispatch_bulk_kernel", "combine": "combine_kernel"}
        op_summary = {}
        for op in ops:
            us = 1e3 * statistics.mean(per_op[op])
            gbs = bytes_of[op] / (us * 1e-6) / 1e9
            op_summary[op] = {"us": round(us, 2), "us_median": round(1e3 * pct(per_op[op], 50), 2),
                              "us_p10": round(1e3 * pct(per_op[op], 10), 2),
                              "us_p90": round(1e3 * pct(per_op[op], 90), 2), "GB/s": round(gbs, 1),
                              "frac": round(gbs / peak, 4), "bytes": bytes_of[op], "kernel": kname[op]}
        dom = max(("dispatch", "combine"), key=lambda o: op_summary[o]["us"])
        traffic = recorded_traffic(kname[dom])
        cpu = cpu_baseline(cfg, args)
        line = {
            "metric": METRIC,
            "value": round(rep.tokens_per_s(T, ms_per_step), 1),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4),
            "ms_per_step_median": round(pct(step_ms, 50), 4),
            "ms_per_step_p10": round(pct(step_ms, 10), 4),
            "ms_per_step_p90": round(pct(step_ms, 90), 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp32",
            "data": "synthetic (seeded splitmix64: U(0,1) scores, N(0,0.01) bias, N(0,1) bf16 hidden rows)",
            "config": {"workload": workload_desc(cfg), "T": T, "H": cfg["H"], "E": cfg["E"], "k": cfg["k"],
                       "n_groups": cfg["n_groups"], "topk_group": cfg["topk_group"],
                       "logical_ranks": cfg["E"] // cfg["experts_per_rank"],
                       "payload": "bf16 rows in, e4m3+fp32 1x128 scales dispatched, bf16 expert outputs combined",
                       "l2": "flushed between steps outside the timed events: 256 MB write, then 256 MB read",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "ops": op_summary,
            "roofline": {"bound": "hbm", "kernel": kname[dom], "achieved": op_summary[dom]["GB/s"],
                         "peak": peak, "peak_source": "%s (MEASURED_PEAKS.json hbm)" % peak_kind
                         if peak_kind == "measured" else "fallback 6.8 TB/s", "unit": "GB/s",
                         "frac": op_summary[dom]["frac"], "traffic": traffic,
                         "algorithmic_bytes": bytes_of[dom]},
            "e2e": {"value": round(rep.tokens_per_s(T, e2e["ms"]), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": round(e2e["ms"], 4),
                    "method": "public API, pinned host buffers; per step H2D of scores then x in %d token "
                              "chunks, dispatch+combine per chunk, D2H per chunk, on three streams, %d device "
                              "buffer sets so that a step's uploads overlap the previous step; %d consecutive "
                              "steps timed together%s; the last step's output checked against the "
                              "device-resident path"
                              % (e2e["chunks"], e2e["sets"], e2e["steps"],
                                 ", captured once as a CUDA graph and replayed" if e2e["graph"] else "")},
            "cpu_baseline": cpu,
            "configs": configs,
            "clocks": clk.summary(),
            "gpu_launches": PathRunner.LAUNCHES_PER_STEP * args.steps,
        }
        print(json.dumps(line), flush=True)
    rep.close()


def run_e2e(r, args, chunks=16, graph=True, steps=10, nsets=2):
    """The same path through the public API with host buffers: every step's
    inputs (scores, bias, hidden rows) are copied in from pinned host memory
    and its output copied back, inside the timed region.  The copies overlap
    the kernels the way a caller streaming batches through this API would
    arrange it, on three streams:
      - the scores go first, so that gating and layout run while the hidden
        rows stream in by token chunks; each chunk is dispatched and combined
        as soon as it has landed, and its output rows go back on a third
        stream;
      - `nsets` sets of device buffers rotate between steps, so step i+1's
        uploads run while step i computes and downloads (a set is refilled
        once the step nsets back has read its inputs and downloaded its
        output).
    The kernels run in order on one stream.  `steps` consecutive steps are
    timed together (one CUDA graph when `graph`); the result is per step,
    and the last step's downloaded output is checked against the same path
    run on device-resident inputs."""
    import torch
    ep = r.ep
    c = r.cfg
    T, H, k, E, epr = c["T"], c["H"], c["k"], c["E"], c["experts_per_rank"]
    hs = torch.from_numpy(r.host["scores"]).pin_memory()
    hb = None if r.host["bias"] is None else torch.from_numpy(r.host["bias"]).pin_memory()
    hx = torch.from_numpy(r.host["x"].view(np.int16)).pin_memory()
    ho = torch.empty(r.out.shape, dtype=torch.int16).pin_memory()
    sets = []
    for p in range(nsets):
        sets.append(dict(
            scores=torch.empty_like(r.scores), bias=None if r.bias is None else torch.empty_like(r.bias),
            x=torch.empty_like(r.x), idx=torch.empty_like(r.topk_idx), w=torch.empty_like(r.topk_w),
            lay=ep.alloc_layout(T, k, E, epr, r.x.device), out=torch.empty_like(r.out)))
    comp = torch.cuda.Stream()  # a side stream: graphs are captured off the default stream
    comp.wait_stream(torch.cuda.current_stream())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    bounds = [T * i // chunks for i in range(chunks + 1)]

    def run_steps():
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        done = []  # (compute done, download done) events per step
        for i in range(steps):
            S = sets[i % nsets]
            xi, oi = S["x"].view(torch.int16), S["out"].view(torch.int16)
            if i >= nsets:
                s_in.wait_event(done[i - nsets][0])     # the set's inputs were read
            with torch.cuda.stream(s_in):
                S["scores"].copy_(hs, non_blocking=True)
                if hb is not None:
                    S["bias"].copy_(hb, non_blocking=True)
                ev_scores = torch.cuda.Event()
                ev_scores.record(s_in)
                ev_x = []
                for ci in range(chunks):
                    a, b = bounds[ci], bounds[ci + 1]
                    xi[a:b].copy_(hx[a:b], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    ev_x.append(ev)
            comp.wait_event(ev_scores)
            if i >= nsets:
                comp.wait_event(done[i - nsets][1])    # the set's output was downloaded
            with torch.cuda.stream(comp):
                ep.ep_gate_layout(S["scores"], S["bias"], r.gcfg, epr, topk_idx=S["idx"], topk_w=S["w"],
                                  out=S["lay"], workspace=r.ws, err_flag=r.err)
                for ci in range(chunks):
                    a, b = bounds[ci], bounds[ci + 1]
                    comp.wait_event(ev_x[ci])
                    ep.ep_dispatch(S["x"][a:b], S["lay"].pos[a:b], "fp8", recv=r.recv_q, recv_scales=r.recv_s,
                                   err_flag=r.err)
                    ep.ep_combine(r.y, S["lay"].pos[a:b], S["w"][a:b], out=S["out"][a:b], err_flag=r.err)
                    ev = torch.cuda.Event()
                    ev.record(comp)
                    s_out.wait_event(ev)
                    with torch.cuda.stream(s_out):
                        ho[a:b].copy_(oi[a:b], non_blocking=True)
                ev_c = torch.cuda.Event()
                ev_c.record(comp)
            ev_o = torch.cuda.Event()
            ev_o.record(s_out)
            done.append((ev_c, ev_o))
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    with torch.cuda.stream(comp):
        res = _time_e2e(run_steps, comp, steps, graph, hs, hb, hx, ho, chunks)
    res["sets"] = nsets
    # the downloaded output equals the same path on device-resident inputs
    r.route()
    r.dispatch()
    r.combine()
    torch.cuda.synchronize()
    if not torch.equal(ho, r.out.view(torch.int16).cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident path")
    return res


def _time_e2e(run_steps, comp, steps, graph, hs, hb, hx, ho, chunks):
    import torch
    run_steps()
    torch.cuda.synchronize()
    run = run_steps
    if graph:
        # The steps' calls (copies, the C-ABI launches, the stream joins)
        # recorded once as a CUDA graph and replayed: per-chunk host work
        # (Python, argument checks, launch calls) then stays off the timed
        # path, as in a caller that captures its steady-state loop.
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=comp):
            run_steps()
        g.replay()
        torch.cuda.synchronize()
        run = g.replay
    reps = 3
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(reps):
        run()
    b.record(comp)
    b.synchronize()
    h2d = hs.numel() * 4 + (0 if hb is None else hb.numel() * 4) + hx.numel() * 2
    return {"ms": a.elapsed_time(b) / (reps * steps), "h2d": h2d, "d2h": ho.numel() * 2, "chunks": chunks,
            "graph": graph, "steps": steps}


def _oracle_path(cfg, inp, y_bits):
    import oracle
    idx, w = oracle.gate(inp["scores"], inp["bias"], cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    lay = oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])
    oracle.dispatch_fp8(inp["x"], lay["pos"])
    oracle.combine(y_bits, lay["pos"], w.astype(np.float32))


def _oracle_inputs(cfg):
    import oracle
    inp = synth.make_inputs(cfg)
    idx, _ = oracle.gate(inp["scores"], inp["bias"], cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    lay = oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])
    y = oracle.dispatch_bf16(inp["x"], lay["pos"])     # identity experts, made outside the timing
    return inp, y


def cpu_baseline(cfg, args, tokens=None, reps=3):
    """The CPU oracle (single-threaded C, as it stands) on the same workload."""
    tokens = tokens or cfg["T"]
    c = synth.config(WORKLOAD, T=tokens)
    inp, y = _oracle_inputs(c)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        _oracle_path(c, inp, y)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": round(tokens / t, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "host_cores": os.cpu_count(),
            "sample": "%d tokens of the same workload through gate+layout+FP8 dispatch+combine, median of %d runs"
                      % (tokens, reps)}


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on this workload."""
    if not Replicas().is_printer():
        return                       # the other ranks exit 0 without work
    cfg = synth.config(WORKLOAD)
    per_token_s = 0.45e-3
    n_steps = args.steps + args.warmup
    tokens = int(120.0 / max(n_steps, 1) / per_token_s) // 64 * 64
    tokens = max(64, min(cfg["T"], tokens))
    c = synth.config(WORKLOAD, T=tokens)
    inp, y = _oracle_inputs(c)
    for _ in range(args.warmup):
        _oracle_path(c, inp, y)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_path(c, inp, y)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = round(tokens / (ms * 1e-3), 1)
    sample = "%d of the workload's %d tokens per step through gate+layout+FP8 dispatch+combine" % (tokens, cfg["T"])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "T": cfg["T"], "sample_tokens": tokens},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": 1,
                         "host_cores": os.cpu_count(), "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def op_bytes(cfg):
    """Algorithmic bytes of every op over the whole batch (bench sweep)."""
    T, H, E, k = cfg["T"], cfg["H"], cfg["E"], cfg["k"]
    fp8_row = H + H // 32                          # e4m3 codes + scales (1x128 fp32 or 1x32 E8M0)
    b = algorithmic_bytes(cfg)
    return {
        "gate": b["gate"], "layout": b["layout"], "gate_layout": b["gate"] + b["layout"], "layout_capacity": b["layout"],
        "dispatch_bf16": b["dispatch_bf16"], "dispatch_fp8": b["dispatch_fp8"],
        "dispatch_mxfp8": T * (2 * H + k * fp8_row + 4 * k),
        "combine": b["combine"], "combine_fp8": T * (k * fp8_row + 8 * k + 2 * H),
        "combine_mxfp8": T * (k * fp8_row + 8 * k + 2 * H),
        "dispatch_backward": T * (2 * H * k + 4 * k + 2 * H),
        "combine_backward": T * (2 * H + 4 * H * k + 12 * k),
        "decode_fused": b["gate"] + b["layout"] + b["dispatch_fp8"],
    }


def run_sweep(args):
    """--sweep: every op on every workload, one JSON line per workload."""
    import torch

    import combine_group_limited_gb300 as ep
    from combine_group_limited_gb300 import build as epbuild
    epbuild.build()
    torch.cuda.set_device(0)
    peak, peak_kind = measured_hbm_peak()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")  # summed in fp32: no cast kernel
    stream = torch.cuda.current_stream()

    def timed(fn, reps):
        ts = []
        for i in range(reps + 3):
            flush.fill_(i & 0xFF)
            flush_rd.sum()
            queue_ahead()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b) * 1e3)
        # the event clock ticks in steps of about 2 us here: the mean over
        # many repetitions (random phase) resolves below a tick, a median
        # does not; the slowest and fastest 5 % are left out (a host stall
        # can hold one repetition for milliseconds)
        return trimmed_mean(ts)

    def hot(fn, per_graph=20, replays=20):
        """Back-to-back calls replayed from a CUDA graph, no flush between
        them: the per-call device time of a latency-bound op with its
        inputs L2-resident (as in a decode loop).  None if capture fails."""
        try:
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for _ in range(per_graph):
                        fn()
            stream.wait_stream(side)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(replays):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3 / (replays * per_graph)
        except RuntimeError:
            torch.cuda.synchronize()
            return None

    names = args.configs.split(",") if args.configs else list(synth.CONFIGS)
    for name in names:
        cfg = synth.config(name)
        T, H, E, k, epr = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["experts_per_rank"]
        r = PathRunner(cfg)
        gc = r.gcfg
        cap = -(-T * k // E)
        recv_b = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
        recv_mq = torch.empty((T * k, H), dtype=torch.uint8, device="cuda")
        recv_me = torch.empty((T * k, H // 32), dtype=torch.uint8, device="cuda")
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        gy = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
        gw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        ws = r.ws
        ops = {
            "gate": lambda: r.gate(),
            "layout": lambda: r.layout(),
            "gate_layout": lambda: ep.ep_gate_layout(r.scores, r.bias, gc, epr, topk_idx=r.topk_idx, topk_w=r.topk_w,
                                                     out=r.lay, workspace=ws),
            "layout_capacity": lambda: ep.ep_get_layout_capacity(r.topk_idx, E, epr, cap, workspace=ws),
            "dispatch_bf16": lambda: ep.ep_dispatch(r.x, r.lay.pos, "bf16", recv=recv_b),
            "dispatch_mxfp8": lambda: ep.ep_dispatch(r.x, r.lay.pos, "mxfp8", recv=recv_mq, recv_scales=recv_me),
            "combine": lambda: r.combine(),
            "combine_mxfp8": lambda: ep.ep_combine_fp8(recv_mq, recv_me, r.lay.pos, r.topk_w, out=out),
            "dispatch_backward": lambda: ep.ep_dispatch_backward(r.y, r.lay.pos, out=out),
            "combine_backward": lambda: ep.ep_combine_backward(r.x, r.y, r.lay.pos, r.topk_w, grad_y=gy, grad_w=gw),
        }
        if H % 128 == 0:
            ops["dispatch_fp8"] = lambda: r.dispatch()
            ops["combine_fp8"] = lambda: ep.ep_combine_fp8(r.recv_q, r.recv_s, r.lay.pos, r.topk_w, out=out)
        if T * k <= 4096 and H % 128 == 0:
            dws = torch.zeros(64, dtype=torch.uint8, device="cuda")
            ops["decode_fused"] = lambda: ep.ep_decode_dispatch(
                r.scores, r.bias, gc, epr, r.x, "fp8", topk_idx=r.topk_idx, topk_w=r.topk_w, out=r.lay,
                recv=r.recv_q, recv_scales=r.recv_s, workspace=dws)
        if args.ops:  # a subset (e.g. one kernel under a profiler), in the same order
            keep = set(args.ops.split(","))
            ops = {n: f for n, f in ops.items() if n in keep}
        # run every op once so that its inputs exist (mxfp8 codes for its combine)
        for fn in ops.values():
            fn()
        torch.cuda.synchronize()
        nb = op_bytes(cfg)
        res = {}
        for op, fn in ops.items():
            us = timed(fn, args.reps)
            gbs = nb[op] / (us * 1e-6) / 1e9
            res[op] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nb[op]}
            if T * k <= 8192 and not args.no_hot:       # small enough to be latency-bound
                h = hot(fn)
                res[op]["hot_us"] = None if h is None else round(h, 3)
        dsp = "dispatch_fp8" if H % 128 == 0 else "dispatch_bf16"
        step_us = float("nan")
        if dsp in ops:
            step = lambda: (r.route(), ops[dsp](), r.combine())  # noqa: E731
            step_us = timed(step, args.reps)
        if "decode_fused" in ops and not args.ops:
            sep = lambda: (r.gate(), r.layout(), r.dispatch())  # noqa: E731
            h = hot(sep)
            res["decode_separate"] = {"us": round(timed(sep, args.reps), 2),
                                      "hot_us": None if h is None else round(h, 3)}
        line = {"sweep": name, "T": T, "H": H, "E": E, "k": k, "peak_GBs": peak, "peak_source": peak_kind,
                "step_us": round(step_us, 2), "step_tokens_per_s": round(T / (step_us * 1e-6), 1),
                "step_dispatch": dsp, "ops": res}
        print(json.dumps(line), flush=True)
        del r, recv_b, recv_mq, recv_me, out, gy, gw, ops
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--sweep", action="store_true", help="time every op on every workload (one line each)")
    ap.add_argument("--configs", default="", help="comma-separated workloads for --sweep")
    ap.add_argument("--ops", default="", help="comma-separated ops for --sweep (default: all)")
    ap.add_argument("--no-hot", action="store_true", help="--sweep: skip the graph-replayed back-to-back timing")
    # 4 chunks of 2048 tokens: with the next step's uploads overlapping, fewer
    # and larger copies use the host link best (GB300: 16 chunks 0.88 ms a
    # step, 8 0.82, 4 0.80, 2 0.80)
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="token chunks the end-to-end leg pipelines its copies and kernels over")
    ap.add_argument("--e2e-sets", type=int, default=2,
                    help="device buffer sets the end-to-end leg rotates between steps")
    ap.add_argument("--e2e-no-graph", action="store_true",
                    help="issue the end-to-end leg's calls from Python every step instead of replaying a CUDA graph")
    ap.add_argument("--reps", type=int, default=20, help="timed repetitions per op in --sweep")
    ap.add_argument("--config-reps", type=int, default=20,
                    help="L2-flushed repetitions per op of every workload in the line's 'configs'")
    ap.add_argument("--no-configs", action="store_true", help="leave the per-workload 'configs' out of the line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
