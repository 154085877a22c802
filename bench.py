"""Benchmark of the fused adaLN norm+modulate hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input, four
launches through the C ABI:
  ln_modulate           x [1,4216,4096] (1% outlier channels x20), scale/shift ~ N(0,0.2)
  rms_modulate          x [1,4216,4096] ~ N(0,1), scale/shift ~ N(0,0.1)
  gated_rms_modulate    r, h [1,4216,4096] ~ N(0,1), gate/scale/shift ~ N(0,0.1)
  qk_norm_rope_epilogue packed QKV, 256 text + 4096 image tokens, 24 heads x 128
Metric: algorithmic GB/s (read x [, r, h] + write y [, r'] + broadcast vectors
once) and its fraction of the measured HBM peak, plus rows/s.

Timed region: K steps replayed from CUDA graphs, inputs rotating over four
buffer sets (about 1.8 GB; between two uses of a buffer at least 200 MB of
other traffic passes, above the 129 MB L2) so every kernel reads cold data;
CUDA events on the launching stream, barrier + synchronize on both sides,
max over ranks.  Per-kernel launch durations come from separate graph
loops of each kernel alone.  e2e: the same step with pinned host inputs
copied in and every output copied back inside the timed region (one copy
each way per step: a buffer set's tensors are views into one flat buffer).

--impl reference times the CPU oracle (test infrastructure, the reference arm
of this comparison) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
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

EPS = 1e-6
T_ROWS, D = 4216, 4096
T_TXT, T_IMG, HEADS = 256, 4096, 24
WORKLOAD = ("adaLN hot path step: ln_modulate + rms_modulate + gated_rms_modulate at "
            "[1,4216,4096] bf16, qk_norm_rope_epilogue at 256+4096 tokens x 24 heads x 128")


# ----------------------------------------------------------- byte accounting

def kernel_bytes():
    """Algorithmic bytes per launch and rows per launch of each kernel."""
    row = T_ROWS * D * 2
    vec = D * 2
    qkv = (T_TXT + T_IMG) * 3 * HEADS * 128 * 2
    return {
        "ln_modulate": (2 * row + 2 * vec, T_ROWS),
        "rms_modulate": (2 * row + 2 * vec, T_ROWS),
        "gated_rms_modulate": (4 * row + 3 * vec, T_ROWS),
        "qk_norm_rope_epilogue": (2 * qkv + 4 * 128 * 2 + (T_TXT + T_IMG) * 128 * 4,
                                  T_TXT + T_IMG),
    }


def step_bytes():
    kb = kernel_bytes()
    return sum(b for b, _ in kb.values()), sum(r for _, r in kb.values())


def aggregate(elapsed_max_s: float, steps: int, world: int):
    """Whole-job throughput from the max-over-ranks elapsed time (weak
    scaling: every rank processes its own full step)."""
    b, r = step_bytes()
    return {"gbs": world * b * steps / elapsed_max_s / 1e9,
            "rows_per_s": world * r * steps / elapsed_max_s,
            "ms_per_step": elapsed_max_s * 1e3 / steps}


def max_over_ranks(v: float, dist=None, device="cpu") -> float:
    """The largest of the ranks' values (the slowest rank's elapsed time);
    `dist` is torch.distributed (NCCL on GPUs, gloo on CPU) or None."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def hbm_peak():
    p = peaks()
    if p and p.get("hbm_gbs"):
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------- workloads

class HostInputs:
    """Seeded synthetic inputs as numpy bf16 bit patterns."""

    def __init__(self):
        from dit_adaln_norm_gb300 import synth
        self.ln_x = synth.outlier_rows_bf16((1, T_ROWS, D), synth.SEED_X, synth.SEED_OUTLIER)
        self.ln_emb = synth.normal_bf16((1, 6 * D), synth.SEED_VEC, 0.2)
        self.rms_x = synth.normal_bf16((1, T_ROWS, D), synth.SEED_X + 10)
        self.rms_emb = synth.normal_bf16((1, 6 * D), synth.SEED_VEC + 10, 0.1)
        self.g_r = synth.normal_bf16((1, T_ROWS, D), synth.SEED_X + 20)
        self.g_h = synth.normal_bf16((1, T_ROWS, D), synth.SEED_X + 21)
        self.g_emb = synth.normal_bf16((1, 6 * D), synth.SEED_VEC + 20, 0.1)
        self.qk_txt = synth.packed_qkv(T_TXT, HEADS, synth.SEED_X + 30)
        self.qk_img = synth.packed_qkv(T_IMG, HEADS, synth.SEED_X + 31)
        self.qk_w = np.stack(synth.head_weights(4, synth.SEED_VEC + 30))
        self.rope_txt = synth.rope_table(T_TXT)
        self.rope_img = synth.rope_table(T_IMG, pos0=T_TXT)


class DeviceSet:
    """One set of device buffers for a full step.  The inputs are views into
    one flat device buffer and the outputs into another (each view 256-byte
    aligned), so the e2e step moves each direction with a single copy."""

    ALIGN = 256

    def __init__(self, h: HostInputs, dev):
        import torch
        bf16 = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        srcs = [("ln_x", bf16(h.ln_x)), ("ln_emb", bf16(h.ln_emb)), ("rms_x", bf16(h.rms_x)),
                ("rms_emb", bf16(h.rms_emb)), ("g_r", bf16(h.g_r)), ("g_h", bf16(h.g_h)),
                ("g_emb", bf16(h.g_emb)), ("qk_txt", bf16(h.qk_txt)), ("qk_img", bf16(h.qk_img)),
                ("qk_w", bf16(h.qk_w)), ("rope_txt", torch.from_numpy(h.rope_txt)),
                ("rope_img", torch.from_numpy(h.rope_img))]
        self.in_buf, views = self._pack([(n, t.shape, t.dtype) for n, t in srcs], dev)
        for (n, t), v in zip(srcs, views):
            v.copy_(t)
            setattr(self, n, v)
        T = T_TXT + T_IMG
        row = (1, T_ROWS, D)
        outs = [("ln_y", row, torch.bfloat16), ("rms_y", row, torch.bfloat16),
                ("g_rout", row, torch.bfloat16), ("g_y", row, torch.bfloat16)] + \
               [(n, (T, HEADS, 128), torch.bfloat16) for n in ("q_out", "k_out", "v_out")]
        self.out_buf, views = self._pack(outs, dev)
        for (n, _, _), v in zip(outs, views):
            setattr(self, n, v)

    @classmethod
    def _pack(cls, specs, dev):
        """A flat byte buffer on `dev` and one view per (name, shape, dtype)."""
        import torch
        offs, total = [], 0
        for _, shape, dtype in specs:
            offs.append(total)
            nb = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            total += (nb + cls.ALIGN - 1) // cls.ALIGN * cls.ALIGN
        buf = torch.empty(total, dtype=torch.uint8, device=dev)
        views = []
        for (_, shape, dtype), off in zip(specs, offs):
            nb = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            views.append(buf[off:off + nb].view(dtype).view(shape))
        return buf, views

    def vec(self, emb, i):
        return emb[:, i * D:(i + 1) * D]

    def launch(self, name):
        from dit_adaln_norm_gb300 import ops
        from dit_adaln_norm_gb300.synth import split_qkv
        if name == "ln_modulate":
            ops.ln_modulate(self.ln_x, self.vec(self.ln_emb, 0), self.vec(self.ln_emb, 1), EPS,
                            out=self.ln_y)
        elif name == "rms_modulate":
            ops.rms_modulate(self.rms_x, self.vec(self.rms_emb, 0), self.vec(self.rms_emb, 1), EPS,
                             out=self.rms_y)
        elif name == "gated_rms_modulate":
            ops.gated_rms_modulate(self.g_r, self.g_h, self.vec(self.g_emb, 0),
                                   self.vec(self.g_emb, 1), self.vec(self.g_emb, 2), EPS,
                                   r_out=self.g_rout, out=self.g_y)
        else:
            w = self.qk_w
            ops.qk_norm_rope_epilogue(split_qkv(self.qk_txt, HEADS), split_qkv(self.qk_img, HEADS),
                                      w[0], w[1], w[2], w[3], self.rope_txt, self.rope_img, EPS,
                                      EPS, HEADS, out=(self.q_out, self.k_out, self.v_out))

    def step(self):
        for name in KERNELS:
            self.launch(name)


NSETS = 4
KERNELS = ["ln_modulate", "rms_modulate", "gated_rms_modulate", "qk_norm_rope_epilogue"]
E2E_SETS = 2        # device buffer sets the e2e steps rotate through
E2E_MAX_STEPS = 64  # e2e steps timed (at most; fewer for short runs)
KERNEL_WORKLOADS = {"ln_modulate": "[1,4216,4096] bf16", "rms_modulate": "[1,4216,4096] bf16",
                    "gated_rms_modulate": "[1,4216,4096] bf16",
                    "qk_norm_rope_epilogue": "256+4096 tokens x 24 heads x 128 bf16"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while running; kept with timestamps."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu  # nvidia-smi -i selector: "GPU-<uuid>" or an index
        self.windows = []

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if any(a - 0.3 <= r[0] <= b + 0.3 for a, b in self.windows)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for n, v in zip(names, r[3][6:10]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_windows": len(inside)}


# ------------------------------------------------------------ oracle timing

def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def host_cpu() -> str:
    """The host CPU's model as /proc/cpuinfo names it (best effort)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    arm_parts = {"0xd40": "Arm Neoverse V1", "0xd4f": "Arm Neoverse V2", "0xd0c": "Arm Neoverse N1",
                 "0xd49": "Arm Neoverse N2"}
    for key in ("model name", "Model name", "CPU part"):
        for line in info:
            if line.startswith(key):
                v = line.split(":", 1)[1].strip()
                return v if key != "CPU part" else f"{arm_parts.get(v, 'Arm')} (CPU part {v})"
    return "unknown"


def _oracle_slice(h: HostInputs, a: int, b: int, ta: int, tb: int):
    """The oracle on rows [a, b) of each row workload and tokens [ta, tb) of
    the QKV epilogue (text tokens first, then image tokens)."""
    import oracle
    from dit_adaln_norm_gb300.synth import split_qkv
    vec = lambda emb, i: emb[:, i * D:(i + 1) * D]
    if b > a:
        oracle.ln_modulate(h.ln_x[:, a:b], vec(h.ln_emb, 0), vec(h.ln_emb, 1), EPS)
        oracle.rms_modulate(h.rms_x[:, a:b], vec(h.rms_emb, 0), vec(h.rms_emb, 1), EPS)
        oracle.gated_rms_modulate(h.g_r[:, a:b], h.g_h[:, a:b], vec(h.g_emb, 0),
                                  vec(h.g_emb, 1), vec(h.g_emb, 2), EPS)
    t0, t1 = min(ta, T_TXT), min(tb, T_TXT)
    i0, i1 = max(ta, T_TXT) - T_TXT, max(tb, T_TXT) - T_TXT
    if tb > ta:
        oracle.qk_norm_rope_epilogue(split_qkv(h.qk_txt[t0:t1], HEADS),
                                     split_qkv(h.qk_img[i0:i1], HEADS), HEADS, list(h.qk_w),
                                     h.rope_txt[t0:t1], h.rope_img[i0:i1], EPS, EPS)


def oracle_sample(h: HostInputs, rows: int, threads: int = 1):
    """Run the CPU oracle on the first `rows` rows of each of the three row
    workloads and on `rows` tokens of the QKV epilogue (a proportional mix
    of text and image tokens), split over `threads` host threads (the C
    oracle runs without the interpreter lock).  Returns (seconds, algorithmic
    bytes covered, rows + tokens covered)."""
    rows = max(1, min(rows, T_ROWS))
    tt = min(rows * T_TXT // T_ROWS + 1, T_TXT)
    ti = max(1, rows - tt)
    t_idx = list(range(tt)) + [T_TXT + i for i in range(ti)]
    threads = max(1, min(threads, rows))
    cut = lambda n, k: (n * k) // threads
    t0 = time.perf_counter()
    if threads == 1:
        _oracle_slice(h, 0, rows, 0, tt)
        _oracle_slice(h, rows, rows, T_TXT, T_TXT + ti)
    else:
        from concurrent.futures import ThreadPoolExecutor
        jobs = []
        with ThreadPoolExecutor(threads) as ex:
            for k in range(threads):
                a, b = cut(rows, k), cut(rows, k + 1)
                ta, tb = cut(len(t_idx), k), cut(len(t_idx), k + 1)
                # token slices never straddle the text/image boundary
                mid = min(max(ta, tt), tb)
                jobs.append(ex.submit(_oracle_slice, h, a, b, t_idx[ta] if ta < mid else 0,
                                      t_idx[mid - 1] + 1 if ta < mid else 0))
                if mid < tb:
                    jobs.append(ex.submit(_oracle_slice, h, 0, 0, t_idx[mid], t_idx[tb - 1] + 1))
            for j in jobs:
                j.result()
    dt = time.perf_counter() - t0
    kb = kernel_bytes()
    frac_rows = rows / T_ROWS
    frac_tok = (tt + ti) / (T_TXT + T_IMG)
    b = (kb["ln_modulate"][0] + kb["rms_modulate"][0] + kb["gated_rms_modulate"][0]) * frac_rows \
        + kb["qk_norm_rope_epilogue"][0] * frac_tok
    return dt, b, 3 * rows + tt + ti


def _oracle_rate(h: HostInputs, threads: int, budget_s: float):
    """GB/s, rows/s and the sample of the oracle on `threads` threads for
    about `budget_s` seconds."""
    dt1, _, _ = oracle_sample(h, 16 * threads, threads)  # calibrate
    rows = int(max(16, min(T_ROWS, 16 * threads * budget_s / max(dt1, 1e-6) / 3)))
    total_t, total_b, total_r, reps = 0.0, 0.0, 0, 0
    while total_t < budget_s / 3 and reps < 50:
        dt, b, r = oracle_sample(h, rows, threads)
        total_t += dt
        total_b += b
        total_r += r
        reps += 1
    sample = (f"{reps} passes over the first {rows} rows of each row workload and {rows} "
              f"QKV tokens, {threads} threads")
    return total_b / total_t / 1e9, total_r / total_t, sample


def cpu_baseline(h: HostInputs, budget_s: float = 24.0):
    """The oracle as it stands (plain C) on a bounded sample, on every host
    core the process may use and on one core."""
    import oracle
    oracle.build()
    n = host_threads()
    v_n, r_n, s_n = _oracle_rate(h, n, budget_s * 0.5)
    v_1, r_1, s_1 = _oracle_rate(h, 1, budget_s * 0.5)
    return {"value": v_n, "unit": "GB/s", "cores": n, "kind": "oracle", "rows_per_s": r_n,
            "sample": s_n, "cpu": host_cpu(),
            "single_thread": {"value": v_1, "unit": "GB/s", "cores": 1, "rows_per_s": r_1,
                              "sample": s_1}}


# ------------------------------------------------------------------- arms

def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, rank 0 only, bounded sample per step."""
    if rank != 0:
        return
    h = HostInputs()
    import oracle
    oracle.build()
    budget = float(os.environ.get("DAN_REFERENCE_BUDGET_S", "120"))
    nthr = host_threads()
    dt1, _, _ = oracle_sample(h, 8 * nthr, nthr)
    per_step = budget / max(1, args.steps + args.warmup)
    rows = int(max(1, min(T_ROWS, 8 * nthr * per_step / max(dt1, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(h, rows, nthr)
    t_all, b_all, r_all = 0.0, 0.0, 0
    for _ in range(args.steps):
        dt, b, r = oracle_sample(h, rows, nthr)
        t_all += dt
        b_all += b
        r_all += r
    value = b_all / t_all / 1e9
    sample = (f"each step: the first {rows} rows of each [1,4216,4096] workload and {rows} "
              f"tokens of the QKV epilogue, plain C oracle, rows split over {nthr} thread(s)")
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_all * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthr, "kind": "oracle",
                             "sample": sample, "cpu": host_cpu()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "rows_per_s": r_all / t_all}
    print(json.dumps(line), flush=True)


METRIC = "GB/s and % of HBM peak for rms/ln_modulate at (1,4216,4096) bf16; rows/s"


def time_graphs(graphs, steps, stream):
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def time_steps(round_graph, step_graphs, steps, stream):
    """Device time of exactly `steps` steps: full rounds of NSETS steps from
    one graph, then the remaining steps one graph each."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps // NSETS):
        round_graph.replay()
    for i in range(steps % NSETS):
        step_graphs[i].replay()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def run_ours(args, rank, world, dist):
    import torch
    from dit_adaln_norm_gb300 import build as dan_build
    from dit_adaln_norm_gb300 import ops

    dan_build.build()
    ops.load()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    h = HostInputs()
    sets = [DeviceSet(h, dev) for _ in range(NSETS)]
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for s in sets:  # eager warm-up (loads, occupancy queries) before capture
            s.step()
        torch.cuda.synchronize()
        # one graph runs NSETS consecutive steps, one per buffer set; steps
        # beyond a multiple of NSETS replay single-step graphs
        round_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(round_graph, stream=stream):
            for s in sets:
                s.step()
        step_graphs = []
        for s in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                s.step()
            step_graphs.append(g)
        # per-kernel graphs: `reps` launches of one kernel cycling through the
        # buffer sets, so no launch finds its input in L2
        per_kernel_graphs = {}
        reps = 4 * NSETS
        for name in KERNELS:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    sets[i % NSETS].launch(name)
            per_kernel_graphs[name] = [g]
    torch.cuda.synchronize()

    try:
        sel = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        sel = str(local)
    clocks = ClockSampler(sel)
    clocks.start()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, NSETS)):  # every graph replays once before timing
            step_graphs[i % NSETS].replay()
        round_graph.replay()
        barrier()
        t0 = time.time()
        elapsed = time_steps(round_graph, step_graphs, args.steps, stream)
        t1 = time.time()
        barrier()
    clocks.mark(t0, t1)

    # per-kernel launch durations: each kernel alone, graph of `reps` launches
    kb = kernel_bytes()
    per_kernel = {}
    n_iter = max(10, min(400, args.steps // 4))
    with torch.cuda.stream(stream):
        for name in KERNELS:
            gs = per_kernel_graphs[name]
            for i in range(3):
                gs[0].replay()
            torch.cuda.synchronize()
            t0 = time.time()
            el = time_graphs(gs, n_iter, stream)
            clocks.mark(t0, time.time())
            us = el / (n_iter * reps) * 1e6
            b, r = kb[name]
            per_kernel[name] = {"us_per_launch": us, "gbs": b / us / 1e3, "rows_per_s": r / us * 1e6,
                                "bytes_per_launch": b, "rows_per_launch": r}
    configs = None
    if not args.no_configs:
        t0 = time.time()
        configs = time_configs(dev, stream)
        clocks.mark(t0, time.time())
    clock_info = clocks.stop()

    # e2e through the public API with pinned host buffers: every step copies
    # its inputs in, runs the 4 launches and copies its outputs back.  Steps
    # are pipelined over E2E_SETS buffer sets and three streams (copy in,
    # compute, copy out), so one step's copies overlap its neighbours' work.
    e2e = None
    if not args.no_e2e:
        pipe = sets[:E2E_SETS]
        # one pinned host image of a set's inputs, one of its outputs per set
        h_in = pipe[0].in_buf.cpu().pin_memory()
        h_out = [torch.empty(s.out_buf.shape, dtype=torch.uint8, pin_memory=True) for s in pipe]
        h2d = h_in.numel()
        d2h = h_out[0].numel()
        e2e_steps = max(4, min(E2E_MAX_STEPS, args.steps // 20))
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()

        def e2e_run(n):
            """Issue n pipelined steps; returns the last event of the copy-out stream."""
            consumed = [None] * len(pipe)  # compute of the previous step on this set done
            drained = [None] * len(pipe)   # copy-out of the previous step on this set done
            for i in range(n):
                k = i % len(pipe)
                s = pipe[k]
                with torch.cuda.stream(s_in):
                    if consumed[k] is not None:
                        s_in.wait_event(consumed[k])
                    s.in_buf.copy_(h_in, non_blocking=True)
                    loaded = ev()
                    loaded.record(s_in)
                with torch.cuda.stream(stream):
                    stream.wait_event(loaded)
                    if drained[k] is not None:
                        stream.wait_event(drained[k])
                    s.step()
                    consumed[k] = ev()
                    consumed[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(consumed[k])
                    h_out[k].copy_(s.out_buf, non_blocking=True)
                    drained[k] = ev()
                    drained[k].record(s_out)
            return drained

        e2e_run(len(pipe))
        barrier()
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record(s_in)
        drained = e2e_run(e2e_steps)
        for d in drained:
            s_out.wait_event(d)
        en.record(s_out)
        en.synchronize()
        e2e_el = st.elapsed_time(en) / 1e3
        barrier()
        e2e = (e2e_el, e2e_steps, h2d, d2h)

    elapsed = max_over_ranks(elapsed, dist, dev)
    if e2e is not None:
        e2e = (max_over_ranks(e2e[0], dist, dev),) + e2e[1:]
    if rank != 0:
        return

    agg = aggregate(elapsed, args.steps, world)
    peak, peak_kind = hbm_peak()
    dom = max(KERNELS, key=lambda n: per_kernel[n]["us_per_launch"])
    pk = per_kernel[dom]
    traffic = load_traffic(dom)
    # every kernel of the step beside the dominant one (the metric names the
    # ln and rms kernels at the step's shape), and every configuration's
    # fraction of peak; the full configuration table goes to a side file
    step_kernels = {n: {"workload": KERNEL_WORKLOADS[n], "us": round(v["us_per_launch"], 3),
                        "achieved": round(v["gbs"], 1), "frac": round(v["gbs"] / peak, 4),
                        "traffic": load_traffic(n)}
                    for n, v in per_kernel.items()}
    configs_frac = None
    if configs is not None:
        configs_frac = {CONFIG_IDS.get(n, n): round(v["gbs"] / peak, 3) for n, v in configs.items()}
        table = {n: dict(v, hbm_frac=v["gbs"] / peak) for n, v in configs.items()}
        if args.configs_out:
            with open(args.configs_out, "w") as fh:
                json.dump({"peak_gbs": peak, "configs": table}, fh, indent=1)
        for n, v in table.items():
            print(f"config {n}: {v['us_per_launch']:.2f} us, {v['gbs']:.0f} GB/s, "
                  f"{v['hbm_frac']:.3f} of peak", file=sys.stderr)
    line = {
        "metric": METRIC, "value": agg["gbs"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": agg["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes()[0],
                   "rows_per_step": step_bytes()[1],
                   "l2": "4 rotating buffer sets (~1.8 GB), >= 200 MB between two uses "
                         "of a buffer (L2 129 MB)",
                   "graph": "4-step CUDA graphs, programmatic dependent launch"},
        "hbm_frac": agg["gbs"] / world / peak, "rows_per_s": agg["rows_per_s"],
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": pk["gbs"], "peak": peak,
                     "peak_kind": f"{peak_kind} (copy, MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback",
                     "unit": "GB/s", "frac": pk["gbs"] / peak,
                     "traffic": traffic, "per_kernel": step_kernels,
                     "configs_frac": configs_frac},
        "gpu_launches": len(KERNELS) * args.steps,
        "clocks": clock_info,
    }
    if e2e is not None:
        e2e_el, e2e_steps, h2d, d2h = e2e
        b, _ = step_bytes()
        line["e2e"] = {"value": world * b * e2e_steps / e2e_el / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_el * 1e3 / e2e_steps}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(h)
    print(json.dumps(line), flush=True)


# ------------------------------------------------- every configuration

# The kernel configurations of the path: the metric's shapes and the
# pages' other sites (FLUX.1 LayerNorm sites at D = 3072, the CFG batch of
# two, the ERNIE RMS with weight at the larger hidden sizes), and the
# variants built beyond them (LayerNorm + FP8, gated LayerNorm, QK with the
# neox rotation and head_dim 64).  Each is timed alone; these are
# per-kernel figures, not part of the step.  (name, kind, B, T, D, flag):
# flag is the RMS weight, or for "qk" the neox rotation with D = head_dim.
# Short names of the configurations for the JSON line (the full names label
# the side file and the per-configuration lines on stderr).
CONFIG_IDS = {
    "C1 rms [1,128,2048]": "C1", "C1' rms [1,4216,4096]": "C1'", "C2a ln [1,4096,3072]": "C2a",
    "C2b ln [1,512,3072]": "C2b", "C2c ln [1,4608,3072]": "C2c", "C2d ln [1,4093,3072]": "C2d",
    "C2' ln [1,4216,4096]": "C2'", "C3 gated [1,4216,4096]": "C3", "C4 ln CFG [2,1140,4096]": "C4",
    "C5 qk 256+4096 tokens x 24 heads x 128": "C5",
    "N4 rms+weight [1,4216,6144]": "N4 rms 6144", "N4 rms+weight [1,4216,8192]": "N4 rms 8192",
    "N4 gated [1,4216,8192]": "N4 gated 8192", "N1 ln+fp8 [1,4216,4096]": "N1 4096",
    "N1 ln+fp8 [1,4096,3072]": "N1 3072", "N2 gated ln [1,4216,4096]": "N2 gated ln 4096",
    "N2 gated ln [1,4096,3072]": "N2 gated ln 3072",
    "N3 qk neox 256+4096 tokens x 24 heads x 128": "N3 neox hd128",
    "N3 qk 256+4096 tokens x 48 heads x 64": "N3 hd64",
    "N3 qk neox 256+4096 tokens x 48 heads x 64": "N3 neox hd64",
    "N2 gated residual, [1,3072,4096] residual layout": "N2 resid T4096",
    "N2 gated residual, [1,3072,4093] residual layout (odd T)": "N2 resid T4093",
}

CONFIGS = [
    ("C1 rms [1,128,2048]", "rms", 1, 128, 2048, False),
    ("C1' rms [1,4216,4096]", "rms", 1, 4216, 4096, False),
    ("C2a ln [1,4096,3072]", "ln", 1, 4096, 3072, False),
    ("C2b ln [1,512,3072]", "ln", 1, 512, 3072, False),
    ("C2c ln [1,4608,3072]", "ln", 1, 4608, 3072, False),
    ("C2d ln [1,4093,3072]", "ln", 1, 4093, 3072, False),
    ("C2' ln [1,4216,4096]", "ln", 1, 4216, 4096, False),
    ("C3 gated [1,4216,4096]", "gated", 1, 4216, 4096, False),
    ("C4 ln CFG [2,1140,4096]", "ln", 2, 1140, 4096, False),
    ("C5 qk 256+4096 tokens x 24 heads x 128", "qk", 1, 0, 128, False),
    ("N4 rms+weight [1,4216,6144]", "rms", 1, 4216, 6144, True),
    ("N4 rms+weight [1,4216,8192]", "rms", 1, 4216, 8192, True),
    ("N4 gated [1,4216,8192]", "gated", 1, 4216, 8192, False),
    ("N1 ln+fp8 [1,4216,4096]", "lnfp8", 1, 4216, 4096, False),
    ("N1 ln+fp8 [1,4096,3072]", "lnfp8", 1, 4096, 3072, False),
    ("N2 gated ln [1,4216,4096]", "gatedln", 1, 4216, 4096, False),
    ("N2 gated ln [1,4096,3072]", "gatedln", 1, 4096, 3072, False),
    ("N3 qk neox 256+4096 tokens x 24 heads x 128", "qk", 1, 0, 128, True),
    ("N3 qk 256+4096 tokens x 48 heads x 64", "qk", 1, 0, 64, False),
    ("N3 qk neox 256+4096 tokens x 48 heads x 64", "qk", 1, 0, 64, True),
    ("N2 gated residual, [1,3072,4096] residual layout", "resid_t", 1, 4096, 3072, False),
    ("N2 gated residual, [1,3072,4093] residual layout (odd T)", "resid_t", 1, 4093, 3072, False),
]


def config_bytes(kind, B, T, D, weight):
    """Algorithmic bytes and rows of one launch of a configuration."""
    if kind == "qk":  # D is head_dim; 24 heads of 128 or 48 of 64
        heads, tok = 24 * 128 // D, T_TXT + T_IMG
        return 2 * tok * 3 * heads * D * 2 + 4 * D * 2 + tok * D * 4, tok
    rows, nvec = B * T, {"rms": 2, "ln": 2, "gated": 3, "lnfp8": 2, "gatedln": 3, "resid_t": 1}[kind]
    io = {"rms": 4, "ln": 4, "gated": 8, "lnfp8": 3, "gatedln": 8, "resid_t": 6}[kind]
    return io * rows * D + nvec * B * D * 2 + (D * 2 if weight else 0), rows


def time_configs(dev, stream, min_bytes=260 << 20, max_sets=16, n_repeats=10, eager_only=0):
    """Launch time of every configuration: a graph of launches cycling over
    enough buffer sets that ~2x L2 of other traffic separates two uses of a
    buffer (up to max_sets; smaller configurations stay L2-resident and say
    so).  Inputs are drawn on the device (normal, seeded): the kernels'
    time does not depend on the values.  Each configuration is timed as
    n_repeats repeats of at least 100 launches; the median repeat is
    reported, with the fastest and slowest.  eager_only = k > 0 instead runs
    each configuration k times without graphs or timing (for an ncu
    capture of every configuration's DRAM traffic) and returns None."""
    import torch
    from dit_adaln_norm_gb300 import ops
    from dit_adaln_norm_gb300.synth import split_qkv
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    rnd = lambda *shape, std=1.0: (torch.randn(*shape, generator=g, device=dev) * std).to(torch.bfloat16)
    out = {}
    for name, kind, B, T, D, weight in CONFIGS:
        nbytes, rows = config_bytes(kind, B, T, D, weight)
        nsets = max(2, min(max_sets, -(-min_bytes // nbytes)))
        sets = []
        for _ in range(nsets):
            if kind == "qk":
                hd, heads = D, 24 * 128 // D
                txt, img = rnd(T_TXT, 3 * heads * hd), rnd(T_IMG, 3 * heads * hd)
                w = (1.0 + rnd(4, hd, std=0.05).float()).to(torch.bfloat16)
                sets.append(dict(txt=txt, img=img, w=w,
                                 out=tuple(torch.empty((T_TXT + T_IMG, heads, hd),
                                                       dtype=torch.bfloat16, device=dev)
                                           for _ in range(3))))
            else:
                emb = rnd(B, 6 * D, std=0.1)
                ydt = torch.uint8 if kind == "lnfp8" else torch.bfloat16
                st = dict(x=rnd(B, T, D), emb=emb, y=torch.empty(B, T, D, dtype=ydt, device=dev),
                          w=(1.0 + rnd(D, std=0.05).float()).to(torch.bfloat16) if weight else None)
                if kind == "resid_t":  # residual [B, D, T], update [B, T, D]
                    st = dict(x=rnd(B, D, T), h=rnd(B, T, D), emb=emb,
                              y=torch.empty(B, D, T, dtype=torch.bfloat16, device=dev))
                if kind in ("gated", "gatedln"):
                    st.update(h=rnd(B, T, D), r_out=torch.empty(B, T, D, dtype=torch.bfloat16, device=dev))
                sets.append(st)
        if kind == "qk":
            from dit_adaln_norm_gb300 import synth
            rope_t = torch.from_numpy(synth.rope_table(T_TXT, D)).to(dev)
            rope_i = torch.from_numpy(synth.rope_table(T_IMG, D, pos0=T_TXT)).to(dev)

        def launch(st):
            if kind == "qk":
                w, hd = st["w"], D
                heads = 24 * 128 // hd
                ops.qk_norm_rope_epilogue(split_qkv(st["txt"], heads, hd),
                                          split_qkv(st["img"], heads, hd), w[0], w[1], w[2], w[3],
                                          rope_t, rope_i, EPS, EPS, heads, out=st["out"],
                                          head_dim=hd, neox=weight)
                return
            vec = lambda i: st["emb"][:, i * D:(i + 1) * D]
            if kind == "rms":
                ops.rms_modulate(st["x"], vec(0), vec(1), EPS, weight=st["w"], out=st["y"])
            elif kind == "ln":
                ops.ln_modulate(st["x"], vec(0), vec(1), EPS, out=st["y"])
            elif kind == "lnfp8":
                ops.ln_modulate_fp8(st["x"], vec(0), vec(1), 0.05, EPS, out=st["y"])
            elif kind == "resid_t":
                ops.gated_residual_transposed(st["x"], st["h"], vec(2), out=st["y"])
            elif kind == "gatedln":
                ops.gated_ln_modulate(st["x"], st["h"], vec(0), vec(1), vec(2), EPS,
                                      r_out=st["r_out"], out=st["y"])
            else:
                ops.gated_rms_modulate(st["x"], st["h"], vec(0), vec(1), vec(2), EPS,
                                       r_out=st["r_out"], out=st["y"])

        reps = max(32, nsets)
        torch.cuda.synchronize()  # inputs were drawn on the default stream
        if eager_only:
            with torch.cuda.stream(stream):
                for i in range(eager_only):
                    launch(sets[i % nsets])
            torch.cuda.synchronize()
            del sets
            torch.cuda.empty_cache()
            continue
        with torch.cuda.stream(stream):
            for st in sets:
                launch(st)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(reps):
                    launch(sets[i % nsets])
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            # repeats of >= 100 launches each; the median repeat is reported
            per = -(-100 // reps)
            samples = [time_graphs([graph], per, stream) / (per * reps) * 1e6
                       for _ in range(n_repeats)]
        us = statistics.median(samples)
        out[name] = {"us_per_launch": us, "gbs": nbytes / us / 1e3, "rows_per_s": rows / us * 1e6,
                     "bytes_per_launch": nbytes, "rows_per_launch": rows, "buffer_sets": nsets,
                     "l2_resident": nsets * nbytes < min_bytes, "repeats": n_repeats,
                     "launches_per_repeat": per * reps,
                     "us_min_max": [round(min(samples), 3), round(max(samples), 3)]}
        del sets, graph
        torch.cuda.empty_cache()
    return None if eager_only else out


def _strip_comments(src: str) -> str:
    """C/C++ source without comments and blank lines (string literals kept)."""
    import re
    pattern = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)
    out = pattern.sub(lambda m: m.group(0) if m.group(0).startswith('"') else "", src)
    return "\n".join(line.rstrip() for line in out.splitlines() if line.strip())


def kernel_sources_digest():
    """sha256 over the CUDA sources with their comments removed, to tie
    stored counters to the code they were taken on (a comment edit keeps
    the digest; any code change voids it)."""
    import hashlib
    d = hashlib.sha256()
    csrc = os.path.join(ROOT, "dit_adaln_norm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            d.update(f.encode())
            d.update(_strip_comments(open(os.path.join(csrc, f)).read()).encode())
    return d.hexdigest()


def load_traffic(kernel):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    summary, or None when the counters were taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        data = json.load(open(path))
    except (OSError, ValueError):
        return None
    if data.get("sources_sha256") != kernel_sources_digest():
        return None
    return data.get("dram_bytes_per_launch", {}).get(kernel)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs-out", default="bench_configs.json",
                    help="file for the full per-configuration table ('' for none)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration kernel timings")
    ap.add_argument("--config-launches", type=int, default=0,
                    help="only launch every configuration this many times, untimed (for ncu)")
    ap.add_argument("--config-filter", default="",
                    help="keep only the configurations whose name contains one of these |-separated texts")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.config_filter:
        keep = args.config_filter.split("|")
        CONFIGS[:] = [c for c in CONFIGS if any(k in c[0] for k in keep)]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    if args.config_launches > 0:
        import torch
        from dit_adaln_norm_gb300 import build as dan_build
        dan_build.build()
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        time_configs(dev, torch.cuda.Stream(device=dev), eager_only=args.config_launches)
        print(json.dumps({"config_launches": args.config_launches,
                          "configs": [c[0] for c in CONFIGS]}))
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
