#!/usr/bin/env python
"""Benchmark of the speculate-and-verify step on GB300.

One step = retrieval (gate + kappa-gram + continuations) || row pass, then the
finish kernel || verification attention, for one batch of the chosen workload (default: the Llama-3.1-8B-shaped verify, batch 1,
prefix 4096, W=4 D=20, V=128256). Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: each step is a CUDA-graph replay; R input copies rotate so that their
total exceeds twice the L2 (each step reads data last touched R steps ago).
K steps are bracketed by a barrier + synchronize and CUDA events; the maximum
over ranks is taken. Every library kernel is bracketed by event nodes inside
the graphs, which gives per-kernel durations over the timed region.
`--impl reference` times the CPU oracle (the reference arm) instead.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify steps/s and candidate tokens/s on 1 GB300; % of HBM roofline"
UNIT = "verify steps/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0          # the "about 8 TB/s" the step's roofline is also quoted against
FALLBACK_TFLOPS_BURST = 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--e2e-steps", type=int, default=100, help="0 leaves out the end-to-end measurement")
    ap.add_argument("--copies", type=int, default=0,
                    help="input copies that rotate through the timed graphs (0: enough for more than twice "
                         "the L2, at least 3); 1 keeps a small device footprint for profiler captures of "
                         "workloads far larger than the L2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the measurements of the rows after the step (commit, paged cache, tax, head) "
                         "and the burst curve")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the step measurements of the other workload shapes")
    ap.add_argument("--two-streams", action="store_true",
                    help="run attention on a second stream beside the acceptance chain (default: one stream, "
                         "acceptance first, attention overlapping the finish kernel)")
    ap.add_argument("--order", choices=["rows_first", "attn_first", "split"], default="rows_first",
                    help="kernel order: rows_first = retrieval, row pass, finish, attention (one stream); "
                         "attn_first = retrieval, attention, row pass (early mode) beside it, finish (one "
                         "stream); split = the attention (every row) on a second stream on --attn-ctas SMs "
                         "beside retrieval, row pass (--rows-ctas SMs) and finish")
    ap.add_argument("--attn-ctas", type=int, default=0, help="split order: SMs for the attention (0: all)")
    ap.add_argument("--rows-ctas", type=int, default=0, help="split order: SMs for the row pass (0: all)")
    ap.add_argument("--early-rows", choices=["auto", "on", "off"], default="auto",
                    help="row pass in its early mode (it streams every row while the retrieval runs and "
                         "lets the finish kernel launch once the retrieval is done); auto: on unless the "
                         "gate can send sequences to the chain draft, whose unused copy-block rows the "
                         "early mode would read too")
    ap.add_argument("--section", choices=["head", "burst"], default=None,
                    help="run one extra measurement alone and print its JSON (head: the low-rank draft head; "
                         "burst: read bandwidth against burst size)")
    ap.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-seconds", type=float, default=20.0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-warmup", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-procs", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-sample-seqs", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# shared helpers
# ---------------------------------------------------------------------------
def workload_config(wl, tokens_per_step, extra=None):
    cfg = {"workload": f"{wl.name}: {wl.description}, {wl.mode} mode",
           "batch": wl.B, "prefix": list(wl.ctx_len), "W": wl.W, "D": wl.D, "K_chain": wl.K,
           "heads": f"{wl.Hq}q/{wl.Hkv}kv dh{wl.dh}", "vocab": wl.V,
           "candidate_tokens_per_step": tokens_per_step}
    if extra:
        cfg.update(extra)
    return cfg


def measured_tensor_peak():
    """Burst dense bf16 TFLOP/s measured on this machine (a cuBLAS GEMM timed alone): the
    kernels here run in sub-millisecond regions, not under a seconds-long power cap.
    Else the recipe's fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured"
    return FALLBACK_TFLOPS_BURST, "fallback"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


_ORACLE = {}          # inputs and workload of the oracle worker's parallel step (inherited by forked workers)


def _oracle_attn_chunk(task):
    """One worker's share of the oracle attention: its slots of the batch (the inputs are
    inherited from the parent at the fork; the block lengths come with the task)."""
    from oracle import ssd_oracle as O
    slots, bl = task
    inp, wl = _ORACLE["inp"], _ORACLE["wl"]
    return O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"], inp["v_cand"],
                              inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype, slots)


def oracle_parallel_step(inp, wl, pool, procs):
    """One oracle step with the attention's present slots dealt round-robin to `procs`
    worker processes while the parent runs gate, retrieval and acceptance (the oracle's
    own functions, unchanged; only the slots are split)."""
    from oracle import ssd_oracle as O
    r = O.verify_step(inp, wl, attention_slots=None)
    bl = r["blk_len"]
    slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(int(bl[b, k]))]
    parts = pool.map(_oracle_attn_chunk, [(slots[i::procs], bl) for i in range(procs)])
    r["attn"] = {k: v for part in parts for k, v in part.items()}
    return r


def oracle_worker(args):
    """Time the CPU oracle on full steps of the workload (runs in a child process that
    never touches the GPU). One process: one BLAS thread. --oracle-procs N > 1: the
    attention is split over N forked worker processes (one BLAS thread each).
    --oracle-sample-seqs S > 0: a batch of S sequences drawn with the workload's recipe
    stands in for the full batch (the step rate is scaled by S / B). Prints a JSON dict."""
    import numpy as np  # noqa: F401
    from oracle import ssd_oracle as O
    from speculative_decoding_copy_gb300 import workloads as WL
    wl_full = WL.WORKLOADS[args.workload]
    S = args.oracle_sample_seqs
    wl = wl_full.replace(B=S) if 0 < S < wl_full.B else wl_full
    inp = WL.make_inputs(wl, WL.default_seed(wl_full.name))
    procs = max(1, args.oracle_procs)
    pool = None
    if procs > 1:
        import multiprocessing as mp
        _ORACLE["inp"], _ORACLE["wl"] = inp, wl
        pool = mp.get_context("fork").Pool(procs)    # this process has no CUDA context
    step = (lambda: oracle_parallel_step(inp, wl, pool, procs)) if pool else (lambda: O.verify_step(inp, wl))
    for _ in range(args.oracle_warmup):          # untimed
        step()
    budget = args.oracle_seconds
    n, t0 = 0, time.perf_counter()
    while True:
        r = step()
        n += 1
        if time.perf_counter() - t0 >= budget or n >= 1000:
            break
    dt = time.perf_counter() - t0
    if pool:
        pool.close()
        pool.join()
    tokens = int(r["blk_len"].sum())
    print(json.dumps({"steps": n, "seconds": dt, "tokens_per_step": tokens, "procs": procs, "sample_seqs": wl.B,
                      "batch": wl_full.B}))


def run_oracle_subprocess(workload, seconds, warmup=0, procs=1, sample_seqs=0, timeout=900):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-worker", "--workload", workload,
           "--oracle-seconds", str(seconds), "--oracle-warmup", str(warmup), "--oracle-procs", str(procs),
           "--oracle-sample-seqs", str(sample_seqs)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_baseline(workload, seconds, procs=1, sample_seqs=0):
    """The cpu_baseline record of one oracle run (steps/s of the full batch; a sample of
    sequences is scaled to it)."""
    try:
        res = run_oracle_subprocess(workload, seconds, 0, procs, sample_seqs)
    except Exception as e:  # report, do not hide
        return {"value": None, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": f"failed: {e}"}
    scale = res["sample_seqs"] / res["batch"]
    value = res["steps"] / res["seconds"] * scale
    how = "one BLAS thread" if procs == 1 else f"attention split over {procs} processes, one BLAS thread each"
    part = ("full batches" if res["sample_seqs"] == res["batch"] else
            f"batches of {res['sample_seqs']} of the {res['batch']} sequences (same recipe), rate scaled by "
            f"{res['sample_seqs']}/{res['batch']}")
    return {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"{res['steps']} oracle steps on {part} in {res['seconds']:.1f} s ({how})",
            "cpu": cpu_model(), "nproc": os.cpu_count()}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from speculative_decoding_copy_gb300 import workloads as WL
    wl = WL.WORKLOADS[args.workload]
    seconds = max(10.0, min(60.0, 0.002 * args.steps))
    warm = max(0, min(args.warmup, 5))          # full oracle steps take seconds each: at most 5
    res = run_oracle_subprocess(args.workload, seconds, warm)
    value = res["steps"] / res["seconds"]
    sample = (f"{res['steps']} full oracle steps of the {wl.name} workload in {res['seconds']:.1f} s "
              f"after {warm} untimed ones (one BLAS thread)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": res["steps"],
            "warmup": warm, "ms_per_step": 1000.0 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, res["tokens_per_step"]), "impl": "reference",
            "candidate_tokens_per_s": value * res["tokens_per_step"],
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, power = [], None, set(), []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"], f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
KERNELS = ["gate_match", "verify_attn", "vocab_stats", "accept_finish"]


def rank_seed(rank):
    """Each rank verifies its own batch: independent synthetic inputs per rank."""
    from speculative_decoding_copy_gb300 import workloads as WL
    return WL.SEED_BASE + 1 + 1000 * rank


def max_over_ranks(ms, device):
    """The slowest rank's time (all ranks end the timed region behind a barrier)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, steps, ms):
    """Steps of all ranks per second of the slowest rank (weak scaling: a batch per rank)."""
    return world * steps / (ms / 1000.0)


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "speculative_decoding_copy_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {"vocab_stats": ("ssd_accept.cu", "ssd_accept.cuh", "ssd_common.cuh"),
                  "verify_attn": ("ssd_attn.cu", "ssd_attn_tc.cu", "ssd_attn.cuh", "ssd_tc.cuh", "ssd_common.cuh")}


def dram_traffic(kernel, workload, alg_bytes=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source; else None. Where the capture's inputs differ from this
    launch's (same shapes, other draws), its bytes are scaled by the ratio of the two
    launches' algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kernel not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{workload}")
    if not e or e.get("source_sha") != source_sha(*KERNEL_SOURCES[kernel]):
        return None
    b = e.get("dram_bytes_per_launch")
    a = e.get("algorithmic_bytes_per_launch")
    if b is not None and a and alg_bytes and alg_bytes != a:
        return round(b * alg_bytes / a)
    return b


REPEATS = 7          # timed repeats of the K-step region; the reported step time is their median


class StepTimer:
    """CUDA graphs of consecutive steps over R input copies (one step per copy, in order)
    and timed replays of exactly K steps."""

    def __init__(self, steps, main, aux, world=1, dev=None):
        self.steps, self.main, self.aux, self.world, self.dev = steps, main, aux, world, dev
        self.R = len(steps)

    def capture(self, idx, hooked):
        """One graph running the steps of copies `idx` in order; `hooked` kernels are
        bracketed by event nodes (one pair per step and kernel)."""
        import torch
        from speculative_decoding_copy_gb300 import _binding as ssd
        main = self.main
        evs = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in hooked}
               for _ in idx]
        for d in evs:
            for a, b2 in d.values():
                a.record(main)
                b2.record(main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for j, i in enumerate(idx):
                for k in hooked:
                    ssd.ssd_profile_kernel(k, *evs[j][k])
                self.steps[i].run(main, self.aux)
                ssd.ssd_profile_kernel(None)
        torch.cuda.synchronize()
        return g, evs

    def plan(self, K, hooked):
        """Graphs that run exactly K steps: K // R replays of the R-step graph and one
        replay of a graph of the first K % R steps."""
        R = self.R
        full, ev_full = self.capture(list(range(R)), hooked)
        tail, ev_tail = (self.capture(list(range(K % R)), hooked) if K % R else (None, []))
        seq = [full] * (K // R) + ([tail] if tail is not None else [])
        return full, seq, ev_full + ev_tail

    def warm(self, n):
        import torch
        with torch.cuda.stream(self.main):
            for i in range(n):
                self.steps[i % self.R].run(self.main, self.aux)
        torch.cuda.synchronize()

    @staticmethod
    def mean_us(evs, k):
        v = [d[k][0].elapsed_time(d[k][1]) * 1000.0 for d in evs]
        v = [x for x in v if x > 0]
        return statistics.mean(v) if v else None

    def kernel_us(self, kernels, replays):
        """Per-kernel durations (µs, mean) with every kernel of `kernels` bracketed (untimed pass)."""
        import torch
        g, ev = self.capture(list(range(self.R)), kernels)
        with torch.cuda.stream(self.main):
            for _ in range(replays):
                g.replay()
        torch.cuda.synchronize()
        out = {k: self.mean_us(ev, k) for k in kernels}
        del g
        return {k: v for k, v in out.items() if v is not None}

    def timed(self, seq, repeats):
        """Replay `seq` (exactly K steps) `repeats` times, each bracketed by a barrier, a
        synchronize and CUDA events on the launching stream; ms per repeat (max over ranks)."""
        import torch
        import torch.distributed as dist
        out = []
        for _ in range(repeats):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if self.world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            with torch.cuda.stream(self.main):
                t0.record(self.main)
                for g in seq:
                    g.replay()
                t1.record(self.main)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1)
            out.append(max_over_ranks(ms, self.dev) if self.world > 1 else ms)
        return out


def kernel_roofline(dom, dom_us, wl, ab, blk_len, prefix, hbm, peak_kind, tf_burst, tf_kind):
    """The dominant kernel against its bound: the attention against the burst bf16 tensor
    rate when its flops take longer there than its bytes at the copy bandwidth, else
    against HBM; the row pass against HBM."""
    kb = {"vocab_stats": ab["logits"], "verify_attn": ab["kv"] + (ab["q_o"] // 2)}
    kf = {"vocab_stats": 0.0,
          "verify_attn": float(sum(4.0 * int(blk_len[b].sum()) * wl.Hq * wl.dh * int(prefix[b])
                                   for b in range(wl.B)))}
    t_hbm = kb[dom] / (hbm * 1e9)
    t_tc = kf[dom] / (tf_burst * 1e12) if kf[dom] else 0.0
    hbm_view = {"bound": "hbm", "achieved": kb[dom] / (dom_us * 1e-6) / 1e9 if dom_us else None, "peak": hbm,
                "unit": "GB/s", "algorithmic_bytes_per_launch": kb[dom],
                "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth, burst)"}
    hbm_view["frac"] = hbm_view["achieved"] / hbm if hbm_view["achieved"] else None
    timing = ("CUDA events around the kernel inside the graphs of a second timed region of the same "
              "K steps (event nodes break the kernel chaining, so the step time is taken without them)")
    if t_tc > t_hbm:
        ach = kf[dom] / (dom_us * 1e-6) / 1e12 if dom_us else None
        return {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": (ach / tf_burst) if ach else None, "traffic": dram_traffic(dom, wl.name, kb[dom]),
                "algorithmic_flops_per_launch": kf[dom], "algorithmic_bytes_per_launch": kb[dom],
                "launch_us": dom_us, "timing": timing,
                "peak_source": f"{tf_kind} bf16_tflops (cuBLAS bf16 GEMM, burst: the kernel runs in "
                               f"sub-millisecond regions)",
                "hbm_view": hbm_view}
    return dict(hbm_view, kernel=dom, traffic=dram_traffic(dom, wl.name, kb[dom]), launch_us=dom_us, timing=timing)


def step_record(wl, ab, ms_list, K, world, hbm):
    ms_per_step = statistics.median(ms_list) / K
    step_bytes = ab["total"]
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    return ms_per_step, {"algorithmic_bytes_per_step": step_bytes, "achieved_gbs": step_gbs,
                         "frac_of_measured_hbm": step_gbs / hbm, "frac_of_nominal_hbm": step_gbs / NOMINAL_HBM_GBS}


def run_ours(args):
    import numpy as np  # noqa: F401
    import torch
    import torch.distributed as dist

    from speculative_decoding_copy_gb300 import _binding as ssd
    from speculative_decoding_copy_gb300 import workloads as WL
    from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = WL.WORKLOADS[args.workload]
    inp = WL.make_inputs(wl, rank_seed(rank))
    ssd.lib()
    early = args.early_rows == "on" or (args.early_rows == "auto" and default_early_rows(wl))

    # rotating copies: total bytes above twice the L2
    kw = dict(order=args.order, early_rows=early, attn_ctas=args.attn_ctas, rows_ctas=args.rows_ctas)
    probe = VerifyStep(wl, inp, device=dev, **kw)
    main = torch.cuda.Stream(dev)
    aux = torch.cuda.Stream(dev) if (args.two_streams or args.order == "split") else None
    with torch.cuda.stream(main):
        probe.run(main, aux)
    torch.cuda.synchronize()
    blk_len = probe.ret_out["blk_len"].cpu().numpy()
    prefix = inp["prefix_len"]
    ab = WL.algorithmic_bytes(wl, prefix, blk_len)
    R = args.copies or max(3, min(16, math.ceil(2 * L2_BYTES / max(ab["total"], 1)) + 1))
    steps = [probe] + [VerifyStep(wl, inp, device=dev, **kw) for _ in range(R - 1)]
    tokens = ab["tokens"]
    K = args.steps
    timer = StepTimer(steps, main, aux, world, dev)
    timer.warm(max(3, args.warmup // 10))

    # diagnostic pass (untimed): every kernel hooked, per-kernel durations
    kern_us = timer.kernel_us(KERNELS, max(3, 60 // R))
    streaming = [k for k in ("vocab_stats", "verify_attn") if k in kern_us]
    dom = max(streaming, key=lambda k: kern_us[k])

    # timed region 1: the step, no event nodes inside the graphs
    n0 = ssd.launch_count()
    full, seq, _ = timer.plan(K, [])
    launches_per_step = (ssd.launch_count() - n0) // (R + K % R)
    # timed region 2: the same K steps with the dominant kernel bracketed by event nodes
    full_h, seq_h, ev_h = timer.plan(K, [dom])

    with torch.cuda.stream(main):
        for _ in range(max(1, -(-args.warmup // R))):
            full.replay()
            full_h.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms_list = timer.timed(seq, REPEATS)
    with torch.cuda.stream(main):
        for g in seq_h:
            g.replay()
    torch.cuda.synchronize()
    time.sleep(0.2)
    clk = clocks.stop()
    hbm, peak_kind = measured_peaks()
    tf_burst, tf_kind = measured_tensor_peak()
    ms_per_step, step_roof = step_record(wl, ab, ms_list, K, world, hbm)
    value = whole_job_value(world, K, ms_per_step * K)
    dom_us = StepTimer.mean_us(ev_h, dom)
    roofline = kernel_roofline(dom, dom_us, wl, ab, blk_len, prefix, hbm, peak_kind, tf_burst, tf_kind)
    del full, seq, full_h, seq_h

    # end to end through the public API with host buffers
    e2e = run_e2e(args, wl, inp, steps[0], main, aux, dev, world) if args.e2e_steps > 0 else None
    nxt = None if args.no_next else {
           "commit_kv": measure_commit(wl, main, dev), "paged_attn": measure_paged(wl, steps[0], main, dev),
           "spec_tax": measure_tax(main, dev), "slimspec_head": measure_head(main, dev)}
    del steps, probe, timer
    torch.cuda.empty_cache()
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    others = None if args.no_workloads else measure_workloads(args, main, dev, world, rank, do_cpu)
    burst = None if args.no_next else measure_burst_curve(main, dev)

    cpu = cpu_par = None
    if do_cpu:
        cpu = oracle_baseline(args.workload, args.oracle_seconds, 1)
        cpu_par = oracle_baseline(args.workload, min(args.oracle_seconds, 15.0), os.cpu_count() or 1)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
                "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16/f32", "data": "synthetic",
                "config": workload_config(wl, tokens, {
                    "l2": f"{R} rotating input copies ({R * ab['total'] / 2**20:.0f} MiB"
                          f"{' > 2x L2' if R * ab['total'] > 2 * L2_BYTES else ', NOT above 2x L2'}); no flush",
                    "timing": f"median of {REPEATS} timed repeats of the K-step region (each bracketed by a "
                              f"barrier, a synchronize and CUDA events); value and ms_per_step from the median",
                    "parallelism": f"replicas x{world} (independent batches per GPU)",
                    "step_order": "two streams" if args.two_streams else args.order,
                    "attn_ctas": args.attn_ctas, "rows_ctas": args.rows_ctas,
                    "early_rows": early}),
                "ms_per_step_repeats": [m / K for m in ms_list],
                "ms_per_step_spread": [min(ms_list) / K, max(ms_list) / K],
                "candidate_tokens_per_s": value * tokens,
                "hbm_roofline_step": step_roof,
                "roofline": roofline,
                "kernels_us_diagnostic": kern_us,
                "e2e": e2e,
                "workloads": others,
                "next": nxt,
                "burst_curve": burst,
                "gpu_launches": launches_per_step * K,
                "clocks": clk,
                "cpu_baseline": cpu,
                "cpu_baseline_parallel": cpu_par}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


OTHER_WORKLOADS = ["batched", "llama70b", "qwen8b_mixed", "qwen8b_mixed_act086"]


def measure_workloads(args, main, dev, world, rank, do_cpu, steps=10):
    """The other workload shapes: per workload its step time (median of REPEATS timed
    repeats of `steps` graph-replayed steps), steps/s, candidate tokens/s, the step's
    fraction of the HBM roofline and the dominant kernel against its bound. Inputs are
    drawn on the device (workloads.make_inputs_device): one copy of 0.7-5 GB per workload,
    far above the L2, so every step reads HBM. With do_cpu, the oracle on a sample of
    sequences with the attention split over the host's cores (cpu_baseline)."""
    import torch
    from speculative_decoding_copy_gb300 import workloads as WL
    from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows
    hbm, peak_kind = measured_peaks()
    tf_burst, tf_kind = measured_tensor_peak()
    out = {}
    for name in OTHER_WORKLOADS:
        wl = WL.WORKLOADS[name]
        inp = WL.make_inputs_device(wl, WL.default_seed(name) + 1000 * rank, dev)
        early = default_early_rows(wl)
        st = VerifyStep(wl, inp, device=dev, early_rows=early)
        with torch.cuda.stream(main):
            st.run(main)
        torch.cuda.synchronize()
        blk_len = st.ret_out["blk_len"].cpu().numpy()
        prefix = inp["prefix_len"]
        ab = WL.algorithmic_bytes(wl, prefix, blk_len)
        timer = StepTimer([st], main, None, world, dev)
        timer.warm(3)
        kern_us = timer.kernel_us(KERNELS, 3)
        dom = max([k for k in ("vocab_stats", "verify_attn") if k in kern_us], key=lambda k: kern_us[k])
        full, seq, _ = timer.plan(steps, [])
        _, seq_h, ev_h = timer.plan(steps, [dom])
        with torch.cuda.stream(main):
            full.replay()
        torch.cuda.synchronize()
        ms_list = timer.timed(seq, REPEATS)
        with torch.cuda.stream(main):
            for g in seq_h:
                g.replay()
        torch.cuda.synchronize()
        ms_per_step, step_roof = step_record(wl, ab, ms_list, steps, world, hbm)
        dom_us = StepTimer.mean_us(ev_h, dom)
        value = whole_job_value(world, steps, ms_per_step * steps)
        rec = {"workload": f"{wl.name}: {wl.description}, {wl.mode} mode", "batch": wl.B,
               "steps": steps, "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1000.0,
               "ms_per_step_spread": [min(ms_list) / steps, max(ms_list) / steps],
               "steps_per_s": value, "candidate_tokens_per_step": ab["tokens"],
               "candidate_tokens_per_s": value * ab["tokens"], "early_rows": early, "skip_absent": st.skip_absent,
               "hbm_roofline_step": step_roof, "kernels_us_diagnostic": kern_us,
               "roofline": kernel_roofline(dom, dom_us, wl, ab, blk_len, prefix, hbm, peak_kind, tf_burst, tf_kind),
               "inputs": "drawn on the device (seeded torch generator), one copy above the L2; no flush"}
        del full, seq, seq_h, timer, st, inp
        torch.cuda.empty_cache()
        if do_cpu:
            rec["cpu_baseline"] = oracle_baseline(name, 8.0, os.cpu_count() or 1, sample_seqs=2 if wl.B > 4 else 1)
        out[name] = rec
    return out


def measure_commit(wl, main, dev, calls=200):
    """The commit of accepted keys/values (the step after the hot path) on the workload's
    shapes with every token of a full block accepted: mean time per call over `calls`
    graph-replayed calls, each preceded by a reset of prefix_len (a 4-byte copy per
    sequence, included in the time)."""
    import torch
    from speculative_decoding_copy_gb300 import _binding as ssd
    B, Hkv, dh, NT, D = wl.B, wl.Hkv, wl.dh, wl.NB * wl.Dmax, wl.D
    P = 4096
    es = 4 if wl.kv_dtype == "f32" else 2
    dt = torch.float32 if es == 4 else torch.int16
    kc = torch.zeros((B, Hkv, P + NT, dh), dtype=dt, device=dev)
    vc = torch.zeros_like(kc)
    kd = torch.ones((B, NT, Hkv, dh), dtype=dt, device=dev)
    vd = torch.ones_like(kd)
    p0 = torch.full((B,), P, dtype=torch.int32, device=dev)
    pl = p0.clone()
    best = torch.zeros(B, dtype=torch.int32, device=dev)
    n_out = torch.full((B,), D + 1, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(main):
        for _ in range(3):
            pl.copy_(p0)
            ssd.ssd_commit_kv(kc, vc, kd, vd, pl, best, n_out, wl.Dmax, ws=ws, stream=main)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        for _ in range(calls):
            pl.copy_(p0)
            ssd.ssd_commit_kv(kc, vc, kd, vd, pl, best, n_out, wl.Dmax, ws=ws, stream=main)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(main):
        g.replay()
        a.record(main)
        g.replay()
        b.record(main)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1000.0 / calls
    nbytes = 2 * 2 * B * D * Hkv * dh * es            # K and V rows, read once and written once
    return {"us_per_call": us, "bytes_per_call": nbytes, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
            "bound": "latency (one CTA per sequence copying a few rows)",
            "case": f"B={B}, {D} accepted tokens of block 0, {Hkv} kv heads, dh {dh}, prefix {P}",
            "device_error": ssd.ssd_read_device_error(ws, main)}


def measure_paged(wl, st, main, dev, calls=100):
    """The verification attention alone on the workload's tensors, contiguous cache against
    the same cache scattered into 128-token pages in reverse order (block table), each the
    mean over `calls` graph-replayed launches."""
    import torch
    from speculative_decoding_copy_gb300 import _binding as ssd
    x = st.x
    B, Hkv, P_max, dh = x["k_cache"].shape
    pps = -(-P_max // 128)
    n = B * pps
    kp = torch.zeros((n, Hkv, 128, dh), dtype=x["k_cache"].dtype, device=dev)
    vp = torch.zeros_like(kp)
    table = torch.arange(n - 1, -1, -1, dtype=torch.int32, device=dev).view(B, pps)
    for b in range(B):
        for j in range(pps):
            r0, r1 = j * 128, min(P_max, (j + 1) * 128)
            kp[int(table[b, j]), :, :r1 - r0] = x["k_cache"][b, :, r0:r1]
            vp[int(table[b, j]), :, :r1 - r0] = x["v_cache"][b, :, r0:r1]
    out = torch.empty_like(x["q"])
    res = {}
    for name, kc, vc, bt in (("contiguous", x["k_cache"], x["v_cache"], None), ("paged", kp, vp, table)):
        a = ssd.attn_args(x["q"], kc, vc, x["k_cand"], x["v_cand"], x["prefix_len"], st.ret_out["blk_len"], wl.Dmax,
                          out, block_table=bt)
        ws = torch.zeros(max(256, ssd.ssd_verify_attn_workspace_size(a)), dtype=torch.uint8, device=dev)
        run = lambda: ssd.ssd_verify_attn(x["q"], kc, vc, x["k_cand"], x["v_cand"], x["prefix_len"],
                                          st.ret_out["blk_len"], wl.Dmax, out=out, ws=ws, stream=main, block_table=bt)
        with torch.cuda.stream(main):
            for _ in range(3):
                run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for _ in range(calls):
                run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(main):
            g.replay()
            e0.record(main)
            g.replay()
            e1.record(main)
        torch.cuda.synchronize()
        res[name + "_us"] = e0.elapsed_time(e1) * 1000.0 / calls
        res[name + "_device_error"] = ssd.ssd_read_device_error(ws, main)
    res["case"] = f"{wl.name} attention alone, back to back (L2 holds the {P_max}-key cache between launches)"
    return res


def measure_tax(main, dev, steps=50):
    """The speculation-tax experiment: a batch in which every sequence ends in a repeated
    5-gram, half copy-intended (probe high, the target follows the copy), half accidental
    (probe low). For the surface gate (tau = 0) and the probe gate (tau = 0.4): copy
    attempts, taxed attempts, mean accepted copy run per attempt (ssd_copy_stats), and the
    step time (graphs of `steps` steps)."""
    import dataclasses
    import numpy as np
    import torch
    from speculative_decoding_copy_gb300 import _binding as ssd
    from speculative_decoding_copy_gb300 import workloads as WL
    from speculative_decoding_copy_gb300.step import VerifyStep
    wl0 = WL.TAX_WORKLOAD
    B = wl0.B
    intended = np.zeros(B, bool)
    intended[::2] = True
    inp = WL.make_inputs(wl0, WL.SEED_BASE + 77, with_attention=False, gate_on=np.ones(B, bool), probe_on=intended)
    # the candidates the surface gate retrieves (on the GPU), so that the target can follow
    # the copy of the intended sequences
    probe = VerifyStep(dataclasses.replace(wl0, tau=0.0), inp, device=dev, with_attention=False)
    probe.gate_retrieve(main)
    torch.cuda.synchronize()
    bt, bl = probe.ret_out["blk_tok"].cpu().numpy(), probe.ret_out["blk_len"].cpu().numpy()
    rows = {}
    for b in np.flatnonzero(intended):
        for k in range(wl0.NB):
            for d in range(int(bl[b, k])):
                rows[(int(b), 0 if d == 0 else 1 + k * wl0.Dmax + d - 1)] = int(bt[b, k, d])
    inp["tgt"] = WL.boost_accepts(inp["tgt"], wl0.logit_dtype, rows)
    res = {"case": wl0.description}
    for tau in (0.0, 0.4):
        wl = dataclasses.replace(wl0, tau=tau)
        st = VerifyStep(wl, inp, device=dev, with_attention=False)
        counts = torch.zeros(4, dtype=torch.int64, device=dev)
        with torch.cuda.stream(main):
            st.run(main)
            ssd.ssd_copy_stats(st.gate_out["gate"], st.ret_out["n_cand"], st.acc_out["acc_len"], wl.W, counts,
                               stream=main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for _ in range(steps):
                st.run(main)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(main):
            g.replay()
            e0.record(main)
            g.replay()
            e1.record(main)
        torch.cuda.synchronize()
        a, t, tok, n = (int(v) for v in counts.cpu().numpy())
        res[f"tau_{tau}"] = {"copy_attempts": a, "taxed_attempts": t, "taxed_fraction": t / a if a else None,
                             "mean_accepted_copy_run": tok / a if a else None, "sequences": n,
                             "step_us": e0.elapsed_time(e1) * 1000.0 / steps}
    return res


def measure_head(main, dev, iters=20):
    """The SlimSpec low-rank draft head on Llama-3.1-8B sizes (d 4096, r 512, V 128256) at
    batch 64 and batch 1. Each call is timed alone with CUDA events after a 256 MiB write
    that flushes L2, mean over `iters` calls after 3 warm-up calls:
      ours_logits   ssd_lowrank_head writing fp32 logits and the statistics
      ours_stats    ssd_lowrank_head, statistics only (max, log-sum-exp, argmax)
      cublas_lowrank  the same product by cuBLAS (u = h W_down^T, z = u W_up^T) with torch
                    logsumexp / max / argmax
      cublas_fullrank the full-rank head the method replaces, z = h W_full^T, W_full [V][d]
    k_head_up's own time comes from the profiling hook in a separate pass. Inputs are the
    seeded synthetic weights of the head workloads; W_full is random bf16 on the device."""
    import numpy as np
    import torch
    from speculative_decoding_copy_gb300 import _binding as ssd
    from speculative_decoding_copy_gb300 import workloads as WL
    hbm, peak_kind = measured_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(WL.SEED_BASE + 0xF0)

    def timed(fn):
        with torch.cuda.stream(main):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(iters):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(main)
                fn()
                e1.record(main)
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) * 1000.0 for a, b in ts]))

    res = {"peak_gbs": hbm, "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth, burst)",
           "l2": "256 MiB write before every timed call"}
    w_full = None
    for name in ("head_llama8b_b64", "head_llama8b_b1"):
        hw = WL.HEAD_WORKLOADS[name]
        x = WL.make_head_inputs(hw)
        dv = lambda b: torch.from_numpy(b.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        h, wd, wu = dv(x["h"]), dv(x["w_down"]), dv(x["w_up"])
        M, V, d, r = hw.M, hw.V, hw.d, hw.r
        rm = torch.empty(M, dtype=torch.float32, device=dev)
        ls = torch.empty(M, dtype=torch.float32, device=dev)
        am = torch.empty(M, dtype=torch.int32, device=dev)
        lg = torch.empty(M, V, dtype=torch.float32, device=dev)
        ws = torch.zeros(ssd.ssd_lowrank_head_workspace_size(ssd.head_args(h, wd, wu, rm, ls, am, lg)),
                         dtype=torch.uint8, device=dev)
        ours_l = lambda: ssd.ssd_lowrank_head(h, wd, wu, out=(rm, ls, am, lg), ws=ws, stream=main)
        ours_s = lambda: ssd.ssd_lowrank_head(h, wd, wu, out=(rm, ls, am), ws=ws, stream=main)

        def cublas_low():
            z = (h @ wd.t()) @ wu.t()
            zf = z.float()
            return torch.logsumexp(zf, dim=1), zf.max(dim=1)

        if w_full is None:
            w_full = torch.randn(V, d, generator=gen, device=dev, dtype=torch.float32).mul_(
                hw.z_std / d ** 0.5).to(torch.bfloat16)

        def cublas_full():
            zf = (h @ w_full.t()).float()
            return torch.logsumexp(zf, dim=1), zf.max(dim=1)

        t = {"ours_logits_us": timed(ours_l), "ours_stats_us": timed(ours_s),
             "cublas_lowrank_us": timed(cublas_low), "cublas_fullrank_us": timed(cublas_full)}
        # k_head_up alone (the hook's event nodes sit between the three kernels)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ssd.ssd_profile_kernel("head_up", e0, e1)
        up = []
        with torch.cuda.stream(main):
            for _ in range(iters):
                flush.zero_()
                ours_s()
                torch.cuda.synchronize()
                up.append(e0.elapsed_time(e1) * 1000.0)
        ssd.ssd_profile_kernel(None)
        t["head_up_us"] = float(np.mean(up))
        w_bytes = V * r * 2 + r * d * 2
        io = M * d * 2 + 2 * M * r * 2
        b_stats = w_bytes + io
        b_logits = b_stats + M * V * 4
        t["bytes_stats"] = b_stats
        t["bytes_logits"] = b_logits
        t["achieved_gbs_stats"] = b_stats / (t["ours_stats_us"] * 1e-6) / 1e9
        t["achieved_gbs_logits"] = b_logits / (t["ours_logits_us"] * 1e-6) / 1e9
        t["frac_stats"] = t["achieved_gbs_stats"] / hbm
        t["frac_logits"] = t["achieved_gbs_logits"] / hbm
        t["head_up_bytes"] = V * r * 2 + M * r * 2
        t["head_up_frac"] = t["head_up_bytes"] / (t["head_up_us"] * 1e-6) / 1e9 / hbm
        t["speedup_vs_fullrank"] = t["cublas_fullrank_us"] / t["ours_stats_us"]
        t["speedup_vs_cublas_lowrank"] = t["cublas_lowrank_us"] / t["ours_stats_us"]
        torch.cuda.synchronize()
        t["device_error"] = ssd.ssd_read_device_error(ws, main)
        res[name] = t
    del w_full, flush
    torch.cuda.empty_cache()
    return res


def measure_burst_curve(main, dev, sizes_mb=(8, 16, 32, 42, 64, 128, 256, 1024), reps=24, pool_mb=2048):
    """Read bandwidth against burst size: ssd_read_probe (plain 16-byte loads, 8 in flight per
    thread) reads X MB once per launch. Rotating buffers whose total is at least `pool_mb`
    (> 15x L2), so every launch reads from DRAM. For each size and grid (2 or 4 CTAs of 256
    threads per SM): `single` = median of the per-launch times between event pairs placed
    around each of `reps` launches issued back to back (first 4 dropped); `stream` = the same
    launches between one pair of events, mean per launch."""
    import torch
    from speculative_decoding_copy_gb300 import _binding as ssd
    hbm, peak_kind = measured_peaks()
    sink = torch.zeros(16, dtype=torch.uint8, device=dev)
    pool = torch.empty(pool_mb << 20, dtype=torch.uint8, device=dev)
    pool.fill_(1)
    rows = []
    for mb in sizes_mb:
        nb = mb << 20
        R = (pool_mb << 20) // nb        # >= 2: the pool holds at least two buffers of the largest size
        bufs = [pool[i * nb:(i + 1) * nb] for i in range(R)]
        for cps in (2, 4):
            with torch.cuda.stream(main):
                for j in range(3):
                    ssd.ssd_read_probe(bufs[j % R], nb, sink, cps, stream=main)
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
                for j in range(reps):
                    evs[j].record(main)
                    ssd.ssd_read_probe(bufs[j % R], nb, sink, cps, stream=main)
                evs[reps].record(main)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(main)
                for j in range(reps):
                    ssd.ssd_read_probe(bufs[(j + 1) % R], nb, sink, cps, stream=main)
                b.record(main)
            torch.cuda.synchronize()
            per = sorted(evs[j].elapsed_time(evs[j + 1]) * 1000.0 for j in range(4, reps))
            single = statistics.median(per)
            stream_us = a.elapsed_time(b) * 1000.0 / reps
            rows.append({"mb": mb, "ctas_per_sm": cps, "buffers": R, "single_us": single,
                         "single_gbs": nb / (single * 1e-6) / 1e9, "single_us_min": per[0], "single_us_max": per[-1],
                         "stream_us": stream_us, "stream_gbs": nb / (stream_us * 1e-6) / 1e9})
    del pool
    torch.cuda.empty_cache()
    for r in rows:
        r["single_frac"] = r["single_gbs"] / hbm
    return {"peak_gbs": hbm, "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth, burst)",
            "kernel": "ssd_read_probe: grid-stride 16-byte loads, 8 in flight per thread, 256-thread CTAs",
            "l2": f"rotating buffers over {pool_mb} MiB: each launch reads data last touched at least one buffer "
                  f"pool's worth of reads earlier (>= 1 GiB)",
            "rows": rows}


def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


def gpu_local_cpus(dev):
    """(NUMA node, CPUs of that node this process may run on) for the host node the GPU
    hangs off, read from sysfs; (None, None) when the topology cannot be read."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        addr = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        base = os.path.join("/sys/bus/pci/devices", addr)
        node = int(open(os.path.join(base, "numa_node")).read())
        cpus = _cpulist(open(os.path.join(base, "local_cpulist")).read()) & os.sched_getaffinity(0)
        return (node, cpus) if node >= 0 and cpus else (None, None)
    except (AttributeError, OSError, ValueError):
        return None, None


def pinned_like(tensors, dev):
    """Pinned host copies of `tensors`, allocated while this thread runs on the GPU's own
    host node, so that the pages (placed by first touch) sit next to the GPU and the copy
    engines do not cross the CPU-to-CPU link. Returns (copies, node used or None)."""
    import torch
    node, cpus = gpu_local_cpus(dev)
    before = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        out = {}
        for k, t in tensors.items():
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t.cpu())
            out[k] = h
    finally:
        if cpus:
            os.sched_setaffinity(0, before)
    return out, node


def run_e2e(args, wl, inp, st, main, aux, dev, world=1):
    """Same step through the public API with host inputs. Every step copies all of its
    inputs host->device from one pinned buffer (one copy into the step's input arena)
    and reads the emitted tokens back. Two input arenas alternate: the copy of step i+1
    runs on a copy stream while step i computes, and a copy into an arena waits until
    the step that last read it has finished."""
    import torch
    from speculative_decoding_copy_gb300.step import VerifyStep, arena_bytes

    nbytes = arena_bytes(inp, True)
    slots = [VerifyStep(wl, inp, device=dev, order=st.order, early_rows=st.early_rows, attn_ctas=st.attn_ctas,
                        rows_ctas=st.rows_ctas, arena=torch.empty(nbytes, dtype=torch.uint8, device=dev))
             for _ in range(2)]
    bufs = {"arena": slots[0].arena}
    for j, s in enumerate(slots):
        bufs[f"out_tok{j}"] = s.acc_out["out_tok"]
        bufs[f"n_out{j}"] = s.acc_out["n_out"]
    host, node = pinned_like(bufs, dev)
    h2d = host["arena"].numel()
    d2h = host["out_tok0"].numel() * 4 + host["n_out0"].numel() * 4
    copy = torch.cuda.Stream(dev)
    E = args.e2e_steps

    def run(n, t0=None, t1=None):
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        if t0 is not None:
            t0.record(main)
        for j in range(2):
            freed[j].record(main)
        for i in range(n):
            j = i % 2
            s = slots[j]
            copy.wait_event(freed[j])
            with torch.cuda.stream(copy):
                s.arena.copy_(host["arena"], non_blocking=True)
            copied[j].record(copy)
            main.wait_event(copied[j])
            with torch.cuda.stream(main):
                s.run(main, aux)
                host[f"out_tok{j}"].copy_(s.acc_out["out_tok"], non_blocking=True)
                host[f"n_out{j}"].copy_(s.acc_out["n_out"], non_blocking=True)
            freed[j].record(main)
        if t1 is not None:
            t1.record(main)

    run(4)
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    run(E, s0, s1)
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1)
    if world > 1:
        ms = max_over_ranks(ms, dev)
    # whole job, like `value`: every rank's steps over the slowest rank's time
    return {"value": whole_job_value(world, E, ms), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": E, "host_buffers_numa_node": node,
            "copies": "one host-to-device copy of a pinned input arena per step; two arenas alternate so "
                      "that step i+1's copy overlaps step i"}


def free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def relaunch_ranks(n):
    """`--gpus N` outside torchrun: start N ranks of this same command under
    torch.distributed.run (one per GPU, rendezvous on 127.0.0.1); rank 0 prints the line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def main():
    args = parse_args()
    if args.oracle_worker:
        oracle_worker(args)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_ranks(args.gpus))
    if args.impl == "reference":
        run_reference(args)
        return
    if args.section is not None:
        import torch
        from speculative_decoding_copy_gb300 import _binding as ssd
        ssd.lib()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        if args.section == "head":
            print(json.dumps({"slimspec_head": measure_head(torch.cuda.Stream(dev), dev)}), flush=True)
        else:
            print(json.dumps({"burst_curve": measure_burst_curve(torch.cuda.Stream(dev), dev)}), flush=True)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
