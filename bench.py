"""Benchmark of the persistent serial Markov draft walk.

A step is one round: the whole gamma-step walk of one batch, one launch of
the persistent kernel, on seeded synthetic inputs already resident in HBM.
The default workload is the long-block fully resident walk (V = 151,936,
r = 256, gamma = 16, B = 1, greedy), the configuration whose on-chip-read
roofline fraction is the figure of merit.  Between timed steps L2 is flushed
by writing a 256 MiB buffer, so every step starts with a cold L2 (as the
pages time the walk: CUDA-graph replay, cold L2).  Each step's kernel is
timed with CUDA events on the stream it is launched on.

`roofline` is the on-chip-read roofline of the resident tiers: W2 is read
from HBM once per process, and every step reads the whole table (gamma V r 2
bytes per walk) out of tensor memory, registers and shared memory at the
tier rates `--unit-rates` measures.  `effective_w2` reports the same bytes
against the HBM copy peak.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded sample per step, and prints the same metric.

Multi-GPU (torchrun, one rank per GPU): the walk does not shard across GPUs
on this path; every rank runs independent replicas of the workload (weak
scaling) and the slowest rank's time is reported.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("µs per γ-step draft walk at B=1..128; effective W2 GB/s vs "
          "on-chip/HBM roofline")
# context only (another GPU, int8 weights): the pages' H100 resident walk at
# V = 151,936, bs = 1 took 37 us per call at gamma = 7 and 62 us at gamma = 16
PAGES_US = {("qwen3_resident", 1): 37.0, ("long_block", 1): 62.0}
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="long_block", choices=sorted(synth.CONFIGS))
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--sampler", default="gumbel", choices=["gumbel", "group"],
                   help="sampling of T > 0 requests: per-token Gumbel-max (the configs') or the "
                        "group inverse-CDF sampler")
    p.add_argument("--cell", default="markov", choices=["markov", "gated", "rnn", "gru"],
                   help="serial head: DSpark's Markov head (the configs') or a recurrent "
                        "head (gated / RNN / GRU state update, synthetic recurrent weights)")
    p.add_argument("--kernel", default="planned", choices=["planned", "resident", "batched", "stream"],
                   help="force a kernel (dspark_walk_set_kernel); default: the handle's plan")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--sweep", action="store_true",
                   help="also time every workload and batch size (fewer steps) into 'sweep'")
    p.add_argument("--gamma-fit", action="store_true",
                   help="also time the V=151,936 B=1 walk at gamma in {1,4,7,16} and fit "
                        "us = entry + gamma * per-step into 'gamma_fit'")
    p.add_argument("--trace", action="store_true",
                   help="after timing, run traced rounds and report the per-phase breakdown")
    p.add_argument("--ncu-csv", default=None,
                   help="an ncu --csv --page raw export (dram__bytes_read.sum, "
                        "dram__bytes_write.sum) of the walk kernel of this build and workload: "
                        "reported as roofline.traffic (DRAM bytes per launch); else null")
    p.add_argument("--unit-rates", action="store_true",
                   help="measure the tier rates the on-chip roofline uses (tensor-memory "
                        "tcgen05.mma and mma.sync cycles per SM) and print them as one JSON line")
    p.add_argument("--trace-skew", action="store_true",
                   help="after timing, run rounds with global-timer stamps and report how far "
                        "apart the CTAs post and see each step's keys")
    p.add_argument("--only-timed", action="store_true",
                   help="warm-up and timed steps only (for profiler runs): no warm-L2 pass, "
                        "no end-to-end pass, no CPU baseline")
    return p.parse_args()


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, dist
    if torch.cuda.is_available():
        torch.cuda.set_device(0)
    return 0, 1, None


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms, with timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [s for t, s in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not inside:                       # timed region shorter than a sample
            mid = (t0 + t1) / 2
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_tflops():
    """Sustained dense bf16 (the walk is a long step): measured, else fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback (sustained)"


def load_inputs(cfg, B, n_rounds):
    W1, W2, _ = synth.make_weights(cfg.V, cfg.r, cfg.seed)
    rounds = [synth.make_inputs(cfg, B=B, round_index=i, weights=(W1, W2))
              for i in range(n_rounds)]
    return W1, W2, rounds


# stamps 1..7 of a step (see dspark_walk_set_trace): the time between stamp
# i - 1 and stamp i is phase i - 1
PHASES = ["projection k loop", "epilogue (keys or logits)", "key pass", "CTA barrier",
          "post key", "wait for all keys", "gather next u"]
ENTRY = ["load tensor-memory + register tiers", "shared tier, first u"]


def phase_breakdown(walk, w, B, cfg, launch, stream, n_rounds, clocks, rounds=20):
    """Median per-phase time (us) of CTA thread 0 over traced rounds (warm L2).

    Stamps are SM clock64() values, converted with the SM clock sampled
    during the timed region.
    """
    plan = w.plan()
    n = plan["n_cta"] if (plan["kernel"] == walk.KERNEL_RESIDENT and B <= 16) else \
        -(-cfg.V // (-(-(-(-cfg.V // plan["sm_count"])) // 128) * 128))
    g = cfg.gamma
    buf = torch.zeros(n * (g + 1) * 8, dtype=torch.int64, device="cuda")
    walk.dspark_walk_set_trace(w.h, buf, buf.numel() * 8)
    mhz = clocks.get("sm_mhz") or 1965.0
    steps, entry = [], []
    for i in range(rounds):
        buf.zero_()
        with torch.cuda.stream(stream):
            launch(i)
        torch.cuda.synchronize()
        t = buf.view(n, g + 1, 8).cpu().numpy().astype(np.float64) / mhz   # us
        if not t[:, :g, 0].all():
            break                       # this kernel writes no stamps
        steps.append(np.diff(t[:, :g, :], axis=2))       # [n, g, 7]
        entry.append(np.diff(t[:, g, :3], axis=1))       # [n, 2]
        step_total = t[:, 1:g, 0] - t[:, :g - 1, 0] if g > 1 else None
        if step_total is not None:
            steps[-1] = np.concatenate([steps[-1][:, :g - 1, :], step_total[..., None]], axis=2)
    walk.dspark_walk_set_trace(w.h, None, 0)
    if not steps:
        return None
    st = np.stack(steps)
    en = np.stack(entry)
    names = PHASES + ["whole step"]
    out = {"unit": "us (median over CTAs, steps and %d rounds; warm L2)" % len(steps),
           "sm_mhz": mhz}
    for j, name in enumerate(names[:st.shape[-1]]):
        out[name] = float(np.median(st[..., j]))
    for j, name in enumerate(ENTRY):
        out["entry: " + name] = float(np.median(en[..., j]))
    return out


def skew_report(walk, w, B, cfg, launch, stream, rounds=10):
    """Cross-CTA timing of the rendezvous from global-timer stamps (warm L2):
    how far apart the CTAs start a step and post their keys, and how long
    after the last post the CTAs see the winner.  The global timer ticks in
    coarse steps (256 ns on GB300), so the figures are medians over steps."""
    plan = w.plan()
    if plan["kernel"] != walk.KERNEL_RESIDENT or B > 16:
        return None
    n, g = plan["n_cta"], cfg.gamma
    buf = torch.zeros(n * (g + 1) * 8, dtype=torch.int64, device="cuda")
    walk.dspark_walk_set_trace(w.h, buf, buf.numel() * 8)
    walk.dspark_walk_set_trace_clock(w.h, walk.TRACE_GLOBAL_TIMER)
    steps = []
    for i in range(rounds):
        buf.zero_()
        with torch.cuda.stream(stream):
            launch(i)
        torch.cuda.synchronize()
        t = buf.view(n, g + 1, 8).cpu().numpy().astype(np.float64)
        if not t[:, :g, 0].all():
            break
        steps.append(t[:, 1:g, :])                       # steps 1.. (step 0 follows the entry)
    walk.dspark_walk_set_trace_clock(w.h, walk.TRACE_SM_CLOCK)
    walk.dspark_walk_set_trace(w.h, None, 0)
    if not steps:
        return None
    t = np.concatenate(steps, axis=1) / 1000.0          # [n, S, 8] us
    start, post, seen = t[:, :, 0], t[:, :, 5], t[:, :, 6]
    med = lambda x: float(np.median(x))                 # noqa: E731
    last_post = post.max(axis=0)
    resolution = np.diff(np.unique(t[:, :, 0]))
    return {
        "unit": "us, median over %d steps of %d rounds (global timer, warm L2)" % (
            t.shape[1], len(steps)),
        "timer_step_ns": float(resolution[resolution > 0].min() * 1000) if resolution.size else None,
        "step_start_spread": med(start.max(0) - start.min(0)),
        "post_spread": med(post.max(0) - post.min(0)),
        "post_p90_to_last": med(last_post - np.percentile(post, 90, axis=0)),
        "last_post_to_first_seen": med(seen.min(0) - last_post),
        "last_post_to_median_seen": med(np.median(seen, 0) - last_post),
        "last_post_to_last_seen": med(seen.max(0) - last_post),
        "step_start_to_post": med(np.median(post - start, 0)),
    }


def kernel_label(walk, plan, B):
    """Which kernel a run of B requests takes on a handle with this plan."""
    if plan["kernel"] == walk.KERNEL_RESIDENT and B <= min(plan["max_B"], 16):
        return "resident+streamed tier" if plan["rows_stream"] > 0 else "resident"
    return "batched"


# Tier rates of the on-chip roofline, in SM cycles (dspark_walk_unit_rates
# re-measures them at the start of every run; these are the values a GB300
# gave, used only if that probe fails): an mma.sync m16n8k16 from registers
# holds the tensor pipe 2.0 cycles per SM, one fed by ldmatrix from shared
# memory 4.0 (the shared-memory port: 128 B per cycle), a tcgen05.mma M=128
# N=16 K=16 with A in tensor memory 13.5; bulk copies bring ~142 GB/s per SM
# from L2.
FALLBACK_RATES = {"hmma_rf_cycles": 2.0, "hmma_smem_cycles": 4.0, "tc_tmem_a_cycles": 13.5}
STREAM_GBS_PER_SM = 142.0


def unit_rates(walk):
    """The tier rates measured on this device now, or the fallback values."""
    try:
        r = walk.dspark_walk_unit_rates()
        if all(r.get(k, 0) > 0 for k in FALLBACK_RATES):
            return r, "measured in this run (dspark_walk_unit_rates)"
    except Exception as e:             # noqa: BLE001 -- reported, not hidden
        return dict(FALLBACK_RATES), "fallback constants (probe failed: %s)" % e
    return dict(FALLBACK_RATES), "fallback constants"


def onchip_step_us(plan, rates, mhz):
    """Lower bound of one walk step from on-chip reads, per SM (the slowest
    CTA's shard): every resident row is read once per step, each tier by its
    fastest consumer -- tensor-memory rows at the tcgen05.mma rate (4 KB per
    M=128 K=16 MMA), register and shared rows at the mma.sync rate (512 B per
    m16n8k16); the tensor pipe is shared, so the times add; the shared-memory
    port (512 B per ldmatrix-fed MMA) is a parallel bound, and so are streamed
    rows at the L2 streaming rate.  W2 is read once from HBM per process, so
    the round's entry load is not counted."""
    if plan["kernel"] != 1 or not plan["rows_per_cta"]:      # 1: a resident kernel
        return None
    tc = plan["rows_tmem"] / 128 * 16 * rates["tc_tmem_a_cycles"]
    hmma = (plan["rows_rf"] + plan["rows_smem"] + plan["rows_stream"]) / 16 * 16 * \
        rates["hmma_rf_cycles"]
    port = (plan["rows_smem"] + plan["rows_stream"]) / 16 * 16 * rates["hmma_smem_cycles"]
    t_cyc = max(tc + hmma, port)
    t_stream = plan["rows_stream"] * 512 / (STREAM_GBS_PER_SM * 1e3)
    return max(t_cyc / mhz, t_stream)


def read_ncu_traffic(path, pattern="walk_"):
    """Mean DRAM bytes (read + write) per launch of the kernels whose name
    contains `pattern`, from an `ncu --csv --page raw` export; None if absent."""
    import csv
    scale = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "b": 1, "kb": 1e3,
             "mb": 1e6, "gb": 1e9}
    try:
        with open(path, newline="") as f:
            rows = [r for r in csv.reader(f) if r]
    except OSError:
        return None
    hdr = next((i for i, r in enumerate(rows) if "dram__bytes_read.sum" in r), None)
    if hdr is None:
        return None
    names = rows[hdr]
    ir, iw = names.index("dram__bytes_read.sum"), names.index("dram__bytes_write.sum")
    ik = next((i for i, n in enumerate(names) if n in ("Kernel Name", "kernel_name")), None)
    units = rows[hdr + 1] if len(rows) > hdr + 1 else []
    per = []
    for r in rows[hdr + 1:]:
        if ik is None or len(r) <= max(ir, iw) or pattern not in r[ik]:
            continue
        try:
            ur = scale.get(units[ir].strip().lower(), 1) if units else 1
            uw = scale.get(units[iw].strip().lower(), 1) if units else 1
            per.append(float(r[ir].replace(",", "")) * ur + float(r[iw].replace(",", "")) * uw)
        except (ValueError, IndexError):
            continue
    return statistics.mean(per) if per else None


def gamma_fit(walk, gammas=(1, 4, 7, 16), steps=100, warmup=5):
    """Warm- and cold-L2 us per walk of the long-block vocabulary at B=1 for
    several walk lengths, and the least-squares line us = entry + gamma x step."""
    cfg = synth.CONFIGS["long_block"]
    dev = torch.device("cuda", torch.cuda.current_device())
    W1, W2, _ = synth.make_weights(cfg.V, cfg.r, cfg.seed)
    x = synth.make_inputs(cfg, B=1, round_index=0, weights=(W1, W2))
    w = walk.Walk(W1.to(dev), W2.to(dev), 1, max(gammas))
    anchor, temp = x.anchor.to(dev), x.temperature.to(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    rows = []
    for g in gammas:
        base = x.base[:, :g].contiguous().to(dev)
        tok = torch.empty(1, g, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                w.run(base, anchor, temp, x.seed, tok, stream=stream)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for i in range(steps):
                flush.fill_(i)
                ev[i][0].record(stream)
                w.run(base, anchor, temp, x.seed, tok, stream=stream)
                ev[i][1].record(stream)
            ws, we = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ws.record(stream)
            for _ in range(steps):
                w.run(base, anchor, temp, x.seed, tok, stream=stream)
            we.record(stream)
        torch.cuda.synchronize()
        cold = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1000.0
        warm = ws.elapsed_time(we) / steps * 1000.0
        rows.append({"gamma": g, "us_cold_l2": cold, "us_warm_l2": warm})
    w.close()
    out = {"workload": "V=151,936, B=1, greedy", "points": rows}
    gs = np.array([r["gamma"] for r in rows], dtype=np.float64)
    for key in ("us_cold_l2", "us_warm_l2"):
        ys = np.array([r[key] for r in rows])
        slope, icpt = np.polyfit(gs, ys, 1)
        out[key.replace("us_", "fit_")] = {"us_per_step": float(slope), "entry_us": float(icpt)}
    return out


CELLS = {"markov": 0, "gated": 1, "rnn": 2, "gru": 3}


def cell_weights(cfg, cell):
    """A recurrent head's synthetic weights for a workload: M (bf16 [256, 256];
    [768, 256] for the GRU) and the GRU's token tables X ([3, V, 256]; else None)."""
    if cell == "gru":
        return (synth.make_cell_matrix(cfg.seed + 500, rows=768),
                synth.make_cell_tables(cfg.V, cfg.seed + 501))
    return synth.make_cell_matrix(cfg.seed + 500), None


def measure_config(walk, cfg, B, steps=50, warmup=5, sampler="gumbel", cell="markov",
                   rates=None, mhz=2070.0):
    """Cold- and warm-L2 us per walk of one workload at batch B (sweep mode)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    W1, W2, _ = synth.make_weights(cfg.V, cfg.r, cfg.seed)
    x = synth.make_inputs(cfg, B=B, round_index=0, weights=(W1, W2))
    w = walk.Walk(W1.to(dev), W2.to(dev), B, cfg.gamma)
    if sampler == "group":
        w.set_sampler(walk.SAMPLER_GROUP)
    if cell != "markov":
        M, X = cell_weights(cfg, cell)
        w.set_cell(CELLS[cell], M.to(dev), None if X is None else X.to(dev))
    plan = w.plan()
    base, anchor, temp = x.base.to(dev), x.anchor.to(dev), x.temperature.to(dev)
    tok = torch.empty(B, cfg.gamma, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            w.run(base, anchor, temp, x.seed, tok, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i)
            ev[i][0].record(stream)
            w.run(base, anchor, temp, x.seed, tok, stream=stream)
            ev[i][1].record(stream)
        ws, we = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ws.record(stream)
        for i in range(steps):
            w.run(base, anchor, temp, x.seed, tok, stream=stream)
        we.record(stream)
    torch.cuda.synchronize()
    st = w.status(stream)
    cold = statistics.mean(s.elapsed_time(e) for s, e in ev) * 1000.0
    warm = ws.elapsed_time(we) / steps * 1000.0
    res = {"workload": cfg.name, "V": cfg.V, "gamma": cfg.gamma, "B": B,
           "temperatures": list(cfg.temperatures), "sampler": sampler, "cell": cell,
           "status": st,
           "kernel": kernel_label(walk, plan, B),
           "us_cold_l2": cold, "us_warm_l2": warm,
           "eff_w2_GBs_cold": cfg.gamma * cfg.V * cfg.r * 2 * B / (cold * 1e-6) / 1e9}
    if res["kernel"] != "batched" and rates is not None:
        step = onchip_step_us(plan, rates, mhz)
        if step is not None:
            res["onchip_roofline_us"] = cfg.gamma * step
            res["onchip_frac_cold_l2"] = cfg.gamma * step / cold
            res["onchip_frac_warm_l2"] = cfg.gamma * step / warm
    w.close()
    del flush, base
    torch.cuda.empty_cache()
    return res


def oracle_walk(O, cell, MX, W1, W2, base, anchor, temperature, seed, nthreads=0):
    """One oracle walk of the bench's head (tokens only); MX = (M, X) bits."""
    if cell == "markov":
        return O.walk(W1, W2, base, anchor, temperature, seed, want_logits=False,
                      nthreads=nthreads)
    return O.walk_cell(W1, W2, base, anchor, temperature, seed, CELLS[cell], M=MX[0], X=MX[1],
                       want_logits=False, nthreads=nthreads)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "processor name")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cell_bits(cfg, cell):
    M, X = cell_weights(cfg, cell)
    return synth.bits(M), (None if X is None else synth.bits(X))


def cpu_baseline(cfg, B, rounds, seconds, cell="markov"):
    """The oracle, as it stands, on all host cores: full walks for ~`seconds`."""
    import oracle
    from oracle import cpu_threads
    O = oracle.default()
    W1 = synth.bits(rounds[0].W1)
    W2 = synth.bits(rounds[0].W2)
    MX = cell_bits(cfg, cell)
    n = 0
    t0 = time.perf_counter()
    while True:
        x = rounds[n % len(rounds)]
        oracle_walk(O, cell, MX, W1, W2, synth.bits(x.base), x.anchor.numpy(),
                    x.temperature.numpy(), x.seed)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    # the same oracle on one thread, a third of the time budget
    n1 = 0
    t1 = time.perf_counter()
    while True:
        x = rounds[n1 % len(rounds)]
        oracle_walk(O, cell, MX, W1, W2, synth.bits(x.base), x.anchor.numpy(),
                    x.temperature.numpy(), x.seed, nthreads=1)
        n1 += 1
        if time.perf_counter() - t1 >= seconds / 3:
            break
    dt1 = time.perf_counter() - t1
    return {"value": dt / n * 1e6, "unit": "us", "cores": cpu_threads(0), "kind": "oracle",
            "sample": "%d full walks (rounds 0..%d of the workload), fp64 oracle on all "
                      "host cores" % (n, min(n, len(rounds)) - 1),
            "single_thread_us": dt1 / n1 * 1e6, "single_thread_walks": n1,
            "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def run_reference(args, cfg, B, rank, world):
    """--impl reference: the CPU oracle on this arm's workload and metric."""
    if rank != 0:
        return
    import oracle
    from oracle import cpu_threads
    O = oracle.default()
    n_rounds = min(cfg.rounds, 8)
    W1t, W2t, rounds = load_inputs(cfg, B, n_rounds)
    W1, W2 = synth.bits(W1t), synth.bits(W2t)
    MX = cell_bits(cfg, args.cell)

    def one_step(i):
        # bounded sample: the work of ONE of the gamma steps of round i (all V
        # tokens, all B requests, started from the round's anchor), scaled by
        # gamma to a whole walk
        x = rounds[i % n_rounds]
        k = i % cfg.gamma
        anchor = x.anchor.numpy()
        base = synth.bits(x.base)[:, k:k + 1]
        t0 = time.perf_counter()
        oracle_walk(O, args.cell, MX, W1, W2, np.ascontiguousarray(base), anchor,
                    x.temperature.numpy(), x.seed)
        return time.perf_counter() - t0

    for i in range(args.warmup):
        one_step(i)
    times = [one_step(args.warmup + i) for i in range(args.steps)]
    us = statistics.mean(times) * cfg.gamma * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1000.0, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.note, "cell": args.cell, "V": cfg.V, "gamma": cfg.gamma,
                   "B": B, "r": cfg.r},
        "cpu_baseline": {"value": us, "unit": "us", "cores": cpu_threads(0), "kind": "oracle",
                         "sample": "per step: the work of one of the gamma walk steps (all V "
                                   "tokens, all B requests, from the round's anchor), x gamma"},
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    cfg = synth.CONFIGS[args.workload]
    B = args.batch or cfg.batches[0]
    rank, world, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, cfg, B, rank, world)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    from serial_draft_head_gb300 import walk
    walk.load(build_if_missing=True)
    if args.unit_rates:
        rates, kind = unit_rates(walk)
        if rank == 0:
            print(json.dumps({"unit_rates": rates, "kind": kind}), flush=True)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return
    dev = torch.device("cuda", torch.cuda.current_device())
    n_rounds = min(cfg.rounds, 100)
    W1c, W2c, rounds = load_inputs(cfg, B, n_rounds)
    W1 = W1c.to(dev)
    W2 = W2c.to(dev)
    w = walk.Walk(W1, W2, B, cfg.gamma)
    if args.sampler == "group":
        w.set_sampler(walk.SAMPLER_GROUP)
    cell_dev = None
    if args.cell != "markov":
        M, X = cell_weights(cfg, args.cell)
        cell_dev = (M.to(dev), None if X is None else X.to(dev))   # referenced by the handle
        w.set_cell(CELLS[args.cell], *cell_dev)
    if args.kernel != "planned":
        w.set_kernel({"resident": walk.KERNEL_RESIDENT, "batched": walk.KERNEL_BATCHED,
                      "stream": walk.KERNEL_STREAM}[args.kernel])
    plan = w.plan()
    del W2
    base = torch.stack([r.base for r in rounds]).to(dev)          # [R, B, gamma, V]
    anchor = torch.stack([r.anchor for r in rounds]).to(dev)
    temp = torch.stack([r.temperature for r in rounds]).to(dev)
    seed = rounds[0].seed
    tokens = torch.empty(n_rounds, B, cfg.gamma, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def launch(i):
        j = i % n_rounds
        walk.dspark_walk_run(w.h, base[j], anchor[j], temp[j], seed + i, tokens[j], B,
                             cfg.gamma, None, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush.fill_(i)
            launch(i)
    torch.cuda.synchronize()
    st = w.status(stream)
    if st != 0:
        raise RuntimeError("walk status %d during warm-up" % st)
    rates, rates_kind = unit_rates(walk)         # the roofline's tier rates, this device

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.fill_(i)                     # cold L2: 256 MiB written between steps
            starts[i].record(stream)
            launch(i)
            ends[i].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t1 = time.time()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]        # ms
    st = w.status(stream)
    if st != 0:
        raise RuntimeError("walk status %d in the timed region" % st)

    sampler.stop()
    clocks = sampler.summary(t0, t1)
    warm_ms = e2e_us = graph_warm_ms = None
    e2e_n = 0
    if not args.only_timed:
        # warm L2 (back-to-back, no flush): W2 stays in L2 across rounds
        ws, we = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ws.record(stream)
            for i in range(args.steps):
                launch(i)
            we.record(stream)
        torch.cuda.synchronize()
        warm_ms = ws.elapsed_time(we) / args.steps

        # warm L2 through a CUDA graph of back-to-back rounds (how a serving
        # loop replays the walk): no per-launch host overhead
        n_graph = min(args.steps, 50)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_graph):
                launch(i)
        g.replay()
        torch.cuda.synchronize()
        gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gs.record()
        g.replay()
        ge.record()
        torch.cuda.synchronize()
        graph_warm_ms = gs.elapsed_time(ge) / n_graph
        del g

        # end to end through the C ABI with host buffers (pinned), copies included
        hb = [r.base.pin_memory() for r in rounds[:8]]
        ha = [r.anchor.pin_memory() for r in rounds[:8]]
        ht = [r.temperature.pin_memory() for r in rounds[:8]]
        nh = len(hb)
        hout = torch.empty(B, cfg.gamma, dtype=torch.int32).pin_memory()
        e2e_n = min(args.steps, 200)
        for i in range(5):
            walk.dspark_walk_run_host(w.h, hb[i % nh], ha[i % nh], ht[i % nh], seed, hout, B,
                                      cfg.gamma, None, stream)
        te0 = time.perf_counter()
        for i in range(e2e_n):
            rc = walk.dspark_walk_run_host(w.h, hb[i % nh], ha[i % nh], ht[i % nh], seed + i,
                                           hout, B, cfg.gamma, None, stream)
            if rc != 0:
                raise RuntimeError("run_host status %d" % rc)
        e2e_us = (time.perf_counter() - te0) / e2e_n * 1e6
    h2d = B * cfg.gamma * cfg.V * 2 + B * 4 + B * 4
    d2h = B * cfg.gamma * 4 + 4                             # tokens + the status word

    trace = phase_breakdown(walk, w, B, cfg, launch, stream, n_rounds, clocks) if args.trace else None
    skew = skew_report(walk, w, B, cfg, launch, stream) if args.trace_skew else None

    mean_ms = statistics.mean(per)
    local = torch.tensor([mean_ms, (t1 - t0)], dtype=torch.float64, device=dev)
    if dist:
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
    mean_ms = float(local[0])
    us = mean_ms * 1000.0

    w2_bytes = cfg.gamma * cfg.V * cfg.r * 2 * B           # effective W2 bytes per walk
    eff_gbs = w2_bytes / (mean_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    label = kernel_label(walk, plan, B) if args.kernel == "planned" else args.kernel
    mhz = clocks.get("sm_mhz") or 2070.0
    traffic = read_ncu_traffic(args.ncu_csv) if args.ncu_csv else None
    step = onchip_step_us(plan, rates, mhz) if label != "batched" else None
    if step is not None:
        onchip_bytes = cfg.gamma * cfg.V * cfg.r * 2          # every step reads all of W2
        achieved = onchip_bytes / (mean_ms * 1e-3) / 1e9
        roof_peak = cfg.V * cfg.r * 2 / (step * 1e-6) / 1e9
        roof = {"bound": "onchip", "achieved": achieved, "peak": roof_peak, "unit": "GB/s",
                "frac": achieved / roof_peak, "traffic": traffic,
                "roofline_us": cfg.gamma * step, "per_step_us": step,
                "frac_warm_l2": cfg.gamma * step / (warm_ms * 1000.0) if warm_ms else None,
                "peak_kind": "on-chip tier rates " + rates_kind,
                "sm_mhz": mhz,
                "rates": {k: rates[k] for k in rates},
                "how": "achieved = W2 bytes read from on-chip tiers per walk (gamma*V*r*2, "
                       "W2 read from HBM once per process) / mean launch time; peak = the "
                       "same bytes per step / the step's on-chip roofline (per SM: tensor-"
                       "memory rows at the tcgen05.mma rate plus register and shared rows "
                       "at the mma.sync rate, or the shared-memory port if slower); frac = "
                       "roofline time / measured time; traffic = DRAM bytes per launch from "
                       "an ncu capture of this build (--ncu-csv), else null"}
    else:
        hbm_bytes = B * cfg.gamma * cfg.V * 2                  # base logits, read once
        flops = 2.0 * cfg.V * cfg.r * B * cfg.gamma
        tflops_peak, tkind = measured_tflops()
        hbm_frac = hbm_bytes / (mean_ms * 1e-3) / 1e9 / peak
        tc_frac = flops / (mean_ms * 1e-3) / 1e12 / tflops_peak
        if tc_frac >= hbm_frac:
            roof = {"bound": "tensor", "achieved": flops / (mean_ms * 1e-3) / 1e12,
                    "peak": tflops_peak, "unit": "TFLOP/s", "frac": tc_frac,
                    "peak_kind": tkind}
        else:
            roof = {"bound": "hbm", "achieved": hbm_bytes / (mean_ms * 1e-3) / 1e9,
                    "peak": peak, "unit": "GB/s", "frac": hbm_frac, "peak_kind": peak_kind}
        roof.update({"traffic": traffic, "hbm_frac": hbm_frac, "tensor_frac": tc_frac,
                     "how": "hbm: base logits B*gamma*V*2 bytes per walk against the HBM "
                            "copy peak; tensor: 2*V*r*B*gamma flops against the sustained "
                            "bf16 GEMM peak; bound = the larger fraction"})
    effective = {"achieved": eff_gbs, "unit": "GB/s", "hbm_peak": peak, "ratio": eff_gbs / peak,
                 "peak_kind": peak_kind,
                 "how": "gamma*V*r*2*B bytes per walk / mean launch time, against the HBM "
                        "copy peak (above 1: W2 is served from on-chip memory)"}
    line = {
        "metric": METRIC, "value": us, "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": (us / PAGES_US[(cfg.name, B)]) if (cfg.name, B) in PAGES_US else None,
        "vs_baseline_note": "value / the pages' %.0f us (H100, int8 W2): context on other "
                            "hardware and precision" % PAGES_US[(cfg.name, B)]
                            if (cfg.name, B) in PAGES_US else None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.note, "sampler": args.sampler, "cell": args.cell, "V": cfg.V, "r": cfg.r, "gamma": cfg.gamma, "B": B,
                   "rounds": n_rounds, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "kernel": label, "n_cta": plan["n_cta"] if label != "batched" else None,
                   "threads": plan["threads"] if label != "batched" else None},
        "median_us": statistics.median(per) * 1000.0,
        "p10_us": float(np.percentile(per, 10)) * 1000.0,
        "p90_us": float(np.percentile(per, 90)) * 1000.0,
        "warm_l2_us": warm_ms * 1000.0 if warm_ms is not None else None,
        "graph_warm_l2_us": graph_warm_ms * 1000.0 if graph_warm_ms is not None else None,
        "roofline": roof,
        "effective_w2": effective,
        "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "dspark_walk_run_host on pinned host buffers: base/anchor/temperature "
                       "cross the host link (read in place by the kernel up to 16 MiB of base, "
                       "copied above), tokens written to host memory, status copied back, one "
                       "stream sync; wall clock, mean of %d" % e2e_n},
        "gpu_launches": args.steps,
        "phases": trace,
        "rendezvous_skew": skew,
        "clocks": clocks,
        "plan": plan,
    }
    if args.ncu_csv:
        line["traffic_source"] = os.path.basename(args.ncu_csv)
    if args.sweep or args.gamma_fit:
        w.close()
    if args.sweep:
        line["sweep"] = [measure_config(walk, c, b, rates=rates, mhz=mhz)
                         for c in synth.CONFIGS.values() for b in c.batches]
        # the group inverse-CDF sampler on the sampled workload (not the configs' sampler)
        line["sweep"] += [measure_config(walk, synth.CONFIGS["sampled"], b, sampler="group",
                                         rates=rates, mhz=mhz)
                          for b in synth.CONFIGS["sampled"].batches]
        # the metric's batch range up to 128 on the long block: above 16 requests
        # the batched kernel
        line["sweep"] += [measure_config(walk, synth.CONFIGS["long_block"], b, rates=rates, mhz=mhz)
                          for b in (32, 64, 128)]
        # the recurrent heads on the fully resident long block (B = 1 as the pages
        # time them, and the largest resident batch)
        line["sweep"] += [measure_config(walk, synth.CONFIGS["long_block"], b, cell=c,
                                         rates=rates, mhz=mhz)
                          for c in ("gated", "rnn", "gru") for b in (1, 16)]
    if args.gamma_fit:
        line["gamma_fit"] = gamma_fit(walk)
    if rank == 0 and not args.no_cpu_baseline and not args.only_timed:
        line["cpu_baseline"] = cpu_baseline(cfg, B, rounds, args.cpu_seconds, args.cell)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if not (args.sweep or args.gamma_fit):
        w.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
