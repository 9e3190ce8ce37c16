"""Benchmark of the decode-row trellis projection on one GB300 per process.

Workload: the LM head, 5120 -> 129,280 at 4 bits per weight, one call each at
1, 8 and 16 rows per step (fp32 logits), on seeded synthetic inputs shaped
like the page's ("hip exl3: the input rotation and trellis linear for decode
rows", section "What this changes": x ~ N(0,1) fp16, suh/svh random sign *
U[0.5,1.5], uniformly random packed trellis bits).

A step is the whole hot path for each row count: the rotation of the rows
and the trellis linear, by default as one call (tf_rot_in_linear: one launch
that rotates, then sums; `--calls separate` times tf_rot_in then
tf_trellis_linear, two launches). The weights are in the k-tile-major order of the packed tiles
(`--layout strips` times the library's strips order instead, repacked once
at load time, outside the timed region, through the two calls). The packed weights
(331 MB each) exceed the 129 MB L2; two copies alternate between calls, so no
call finds its weights in L2.

Metric: weight GB/s = packed weight bytes streamed / time, over K steps with
nothing recorded between the launches. The roofline is HBM: the fraction is
the linear's algorithmic bytes per launch (packed weights + xr + svh + y)
over its CUDA-event time, against the measured HBM copy bandwidth; those
per-launch times come from a second timed pass of the K steps with an event
pair around each call (the fused call, or the rot_in and linear pair). The
decode's issue-slot view (lane operations per second against the SMs' issue
peak) is reported beside it under "alu".

Also measured in the same run, outside the headline: every other
configuration the page's projections give (wk, wkv at 1/4/16 rows, the bit
width sweep at 8 rows, the head at 6 bits and 64 rows) under "by_config",
each with time, weight GB/s, rows/s and the HBM fraction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: the path has no exchange step; N processes run N independent
replicas (weak scaling) and rank 0 reports the aggregate.
"""

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

IN_F, OUT_F, BITS = 5120, 129280, 4
ROWS = (1, 8, 16)
WORKLOAD = "LM head 5120->129280, 4 bits/weight, rows {1,8,16} per step, fp32 logits"
METRIC = "weight GB/s and % of HBM peak, trellis linear 5120->129280 @4b, 1-16 rows"
KERNEL_SOURCES = ("linear_mma.cu", "linear_mma.cuh", "linear_tc.cuh", "decode.cuh", "epilogue.cuh", "ptx.cuh",
                  "kernels.h", "rot_block.cuh")
DOMINANT_KERNEL = "trellis_linear_tc_kernel"
L2_BYTES = 129 * 1024 * 1024

# The other configurations of the page's projections, timed in the same run
# (not part of the headline): (name, in, out, bits, rows, out dtype).
CONFIGS = [
    ("wk 512->128", 512, 128, 4, (1,), "fp16"),
    ("wkv 6144->25600", 6144, 25600, 4, (1, 4, 16), "fp16"),
    ("wkv sweep 2b", 6144, 25600, 2, (8,), "fp16"),
    ("wkv sweep 3b", 6144, 25600, 3, (8,), "fp16"),
    ("wkv sweep 4b", 6144, 25600, 4, (8,), "fp16"),
    ("wkv sweep 5b", 6144, 25600, 5, (8,), "fp16"),
    ("wkv sweep 6b", 6144, 25600, 6, (8,), "fp16"),
    ("wkv sweep 8b", 6144, 25600, 8, (8,), "fp16"),
    ("head 6b", 5120, 129280, 6, (64,), "fp32"),
]


def weight_bytes(i=IN_F, o=OUT_F, b=BITS):
    return i * o * b // 8


def launch_bytes(rows, i=IN_F, o=OUT_F, b=BITS, out_elem=4, fused=False):
    """Algorithmic bytes of one linear call: packed weights (streamed once per
    pass of up to 128 rows), fp16 xr, fp16 svh, the output. The fused call
    reads fp16 x in place of xr and also reads suh and writes xr."""
    passes = max(1, math.ceil(rows / 128))
    extra = (i * 2 + rows * i * 2) if fused else 0
    return passes * weight_bytes(i, o, b) + rows * i * 2 + o * 2 + rows * o * out_elem + extra


# Lane operations the method's decode needs per weight: window cut, 32-bit
# multiply, byte sum, fp16 fma.
DECODE_OPS_PER_WEIGHT = 4


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh)
    return None


def measured_peaks():
    d = _peaks()
    if d is not None:
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def max_sm_mhz():
    d = _peaks()
    if d is not None and d.get("sm_max_mhz"):
        return float(d["sm_max_mhz"])
    return 2070.0


def alu_peak_tops(num_sms):
    """Issue-slot peak in tera lane-ops/s: one warp instruction per cycle in
    each of an SM's four sub-partitions."""
    return num_sms * 4 * 32 * max_sm_mhz() * 1e6 / 1e12


def code_only(text):
    """C++/CUDA source without its comments, trailing blanks and empty lines,
    so that the kernel hash changes with the code and not with its comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def kernel_hash(read=None):
    """Hash of the kernel sources' code (comments excluded). `read(name)`
    returns a source's text (default: the files in csrc/)."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "trellis_quantized_linear_rot_gb300", "csrc", name), encoding="utf-8") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(read(f)).encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources (else None).
    Returns {rows: bytes}."""
    path = os.path.join(ROOT, "profiles", "trellis_linear_head_4b.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    if d.get("kernel_hash") != kernel_hash():
        return None
    per = d.get("dram_bytes_per_launch_by_rows")
    if isinstance(per, dict):
        return {int(k): v for k, v in per.items()}
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(bytes_per_step, steps, world, ms_total):
    """Whole-job weight GB/s of N independent replicas: every rank streams the
    same bytes per step; the job takes the slowest rank's time."""
    return bytes_per_step * steps * world / (ms_total * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ CPU baseline
def oracle_sample(n_blocks, rows_list, stream=0):
    """The oracle on a bounded sample of the workload: n_blocks output blocks
    of 128 over all 5120 inputs (a packed stream of the same distribution,
    `stream` picking another seeded one), for each row count: rot_in,
    decode, float64 linear and output rotation. Returns (seconds, packed
    weight bytes covered)."""
    import numpy as np
    from oracle import exl3 as o
    from trellis_quantized_linear_rot_gb300 import synth
    g = np.random.Generator(np.random.PCG64(synth.SEED_TRELLIS + 2 + BITS + 1000 * stream))
    tr = g.integers(0, 2**32, size=IN_F * 128 * n_blocks * BITS // 32, dtype=np.uint32)
    x = synth.make_x(max(rows_list), IN_F, synth.SEED_X + 2)
    suh = synth.make_scale(IN_F, synth.SEED_SUH + 2)
    svh = synth.make_scale(128 * n_blocks, synth.SEED_SVH + 2)
    t0 = time.perf_counter()
    covered = 0
    for rows in rows_list:
        xr = o.rot_in_f32(x[:rows], suh)
        w = o.decode_matrix(tr, IN_F, 128 * n_blocks, BITS)
        o.linear_f64(xr, w, svh)
        covered += weight_bytes(IN_F, 128 * n_blocks)
    return time.perf_counter() - t0, covered


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _oracle_job(job):
    return oracle_sample(*job)


class OraclePool:
    """The oracle on `workers` host cores: one worker process per core,
    started with spawn (never forked from a process that has used the GPU),
    each with its BLAS limited to one thread, each timing its own seeded
    sample."""

    ONE_THREAD = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, workers):
        import multiprocessing as mp
        self.workers = workers
        saved = {k: os.environ.get(k) for k in self.ONE_THREAD}
        for k in self.ONE_THREAD:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(workers)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.run(1)  # imports in every worker

    def run(self, n_blocks_each, rows_list=None):
        """Wall seconds for all workers' samples, and the bytes they covered."""
        rows_list = tuple(rows_list or ROWS)
        jobs = [(n_blocks_each, rows_list, w) for w in range(self.workers)]
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_job, jobs)
        return time.perf_counter() - t0, sum(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def sample_text(n_blocks, workers):
    return ("per worker: %d of 1010 output blocks (5120x128 weights each) for each of rows {%s}; "
            "%d single-threaded worker%s" % (n_blocks, ",".join(str(r) for r in ROWS), workers,
                                              "" if workers == 1 else "s"))


def cpu_baseline(all_blocks=60, one_blocks=6):
    """The oracle's weight GB/s on every host core (one single-threaded worker
    per core) and on one core, on the same sample definition as the
    reference arm."""
    pool = OraclePool(cpu_threads())
    secs, covered = pool.run(all_blocks)
    pool.close()
    one = OraclePool(1)
    secs1, covered1 = one.run(one_blocks)
    one.close()
    return {"value": covered / secs / 1e9, "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
            "sample": sample_text(all_blocks, pool.workers) + ", %.1f s wall" % secs,
            "host_threads_available": cpu_threads(),
            "one_core": {"value": covered1 / secs1 / 1e9, "unit": "GB/s", "cores": 1,
                         "sample": sample_text(one_blocks, 1) + ", %.1f s wall" % secs1}}


def fused_calls(args):
    """Whether the step runs the fused call (the k-tile order only)."""
    return getattr(args, "calls", "separate") == "fused" and args.layout == "tiles"


def bench_config(args, world):
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "rows": list(ROWS), "in_features": IN_F, "out_features": OUT_F,
            "bits": BITS, "out_dtype": "fp32", "weight_bytes_per_call": weight_bytes(),
            "layout": args.layout,
            "calls": ("fused: tf_rot_in_linear, one launch per call" if fused_calls(args)
                      else "separate: tf_rot_in then tf_trellis_linear"),
            "l2": "inputs larger than L2: 331 MB packed weights per call, two copies alternated",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    """The oracle timed on the host cores, on the same workload and metric:
    each step is the same bounded sample as the cpu_baseline leg of our arm
    (whole output blocks over all inputs, for each row count), with the block
    count sized so that the whole run of warm-up and timed steps takes about
    two minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    pool = OraclePool(cpu_threads())
    t_cal, _ = pool.run(1)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n_blocks = int(max(1, min(60, per_step / max(t_cal, 1e-6))))
    for _ in range(args.warmup):
        pool.run(n_blocks)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        t, b = pool.run(n_blocks)
        total_t += t
        total_b += b
    pool.close()
    value = total_b / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(args, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
                         "sample": sample_text(n_blocks, pool.workers) + " per step",
                         "host_threads_available": cpu_threads()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------------ GPU arm
def time_config(tf, dev, name, i_f, o_f, bits, rows_list, out_dtype, layout, iters, peak):
    """One configuration: the linear alone (xr already rotated), weight
    copies alternated so that their total exceeds twice the L2. Returns
    {rows: figures}."""
    import numpy as np
    import torch
    from trellis_quantized_linear_rot_gb300 import synth
    c = [c[0] for c in CONFIGS].index(name)
    w0 = torch.from_numpy(synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + 10 + c).view(np.int32)).to(dev)
    if layout == "strips":
        w0 = tf.tf_trellis_to_strips(w0, i_f, o_f, bits)
    n_copies = max(2, math.ceil(2 * L2_BYTES / max(1, weight_bytes(i_f, o_f, bits))))
    n_copies = min(n_copies, 64)
    ws = [w0] + [w0.clone() for _ in range(n_copies - 1)]
    lin = tf.tf_trellis_linear_strips if layout == "strips" else tf.tf_trellis_linear
    R = max(rows_list)
    x = torch.from_numpy(synth.make_x(R, i_f, synth.SEED_X + 10 + c)).to(dev)
    suh = torch.from_numpy(synth.make_scale(i_f, synth.SEED_SUH + 10 + c)).to(dev)
    svh = torch.from_numpy(synth.make_scale(o_f, synth.SEED_SVH + 10 + c)).to(dev)
    xr = tf.tf_rot_in(x, suh)
    dt = {"fp16": torch.float16, "fp32": torch.float32}[out_dtype]
    st = torch.cuda.current_stream()
    out = {}
    for r in rows_list:
        y = torch.empty((r, o_f), dtype=dt, device=dev)
        for k in range(3):
            lin(xr[:r], ws[k % n_copies], svh, bits, o_f, y=y)
        evs = []
        for k in range(iters):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            lin(xr[:r], ws[k % n_copies], svh, bits, o_f, y=y)
            e1.record(st)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        us = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3
        # The same calls replayed from a CUDA graph (16 calls a replay): the
        # device time of a call without the host's per-call launch cost,
        # which bounds the eager figure of the small layers.
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(st)
        with torch.cuda.graph(g, stream=side):
            for k in range(16):
                lin(xr[:r], ws[k % n_copies], svh, bits, o_f, y=y)
        torch.cuda.synchronize()
        g.replay()
        gevs = []
        for k in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            g.replay()
            e1.record(st)
            gevs.append((e0, e1))
        torch.cuda.synchronize()
        gus = statistics.median(e0.elapsed_time(e1) for e0, e1 in gevs) * 1e3 / 16
        del g
        lb = launch_bytes(r, i_f, o_f, bits, 2 if out_dtype == "fp16" else 4)
        out[str(r)] = {"us_median": us, "weight_gbs": weight_bytes(i_f, o_f, bits) * math.ceil(r / 128) / us / 1e3,
                       "rows_per_s": r / (us * 1e-6), "hbm_frac": lb / us / 1e3 / peak,
                       "graph_us_per_call": gus}
    tf.tf_device_error()
    del ws
    return {"in_features": i_f, "out_features": o_f, "bits": bits, "out_dtype": out_dtype,
            "weight_copies": n_copies, "by_rows": out}


def run_ours(args):
    import numpy as np
    import torch
    import trellis_quantized_linear_rot_gb300 as tf
    from trellis_quantized_linear_rot_gb300 import synth

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    if args.only_configs:
        # Only the named configurations, nothing else on the device: the
        # command the per-configuration ncu captures use.
        names = [n.strip() for n in args.only_configs.split(",")]
        known = [c[0] for c in CONFIGS]
        for n in names:
            if n not in known:
                raise SystemExit("unknown configuration %r (known: %s)" % (n, ", ".join(known)))
        peak, _ = measured_peaks()
        by_config = {}
        for name, i_f, o_f, bits, rows_list, odt in CONFIGS:
            if name in names:
                by_config[name] = time_config(tf, dev, name, i_f, o_f, bits, rows_list, odt, args.layout,
                                              args.config_iters, peak)
        if rank == 0:
            print(json.dumps({"by_config": by_config}))
        if dist is not None:
            dist.destroy_process_group()
        return

    # Inputs (untimed): two copies of the packed weights, x for 16 rows.
    tr_np = synth.make_trellis(IN_F, OUT_F, BITS, synth.SEED_TRELLIS + 2 + BITS)
    tr0 = torch.from_numpy(tr_np.view(np.int32)).to(dev)
    del tr_np
    if args.layout == "strips":
        tr0 = tf.tf_trellis_to_strips(tr0, IN_F, OUT_F, BITS)
    tr1 = tr0.clone()
    linear = tf.tf_trellis_linear_strips if args.layout == "strips" else tf.tf_trellis_linear
    trs = (tr0, tr1)
    fused = fused_calls(args)
    x = torch.from_numpy(synth.make_x(max(ROWS), IN_F, synth.SEED_X + 2)).to(dev)
    suh = torch.from_numpy(synth.make_scale(IN_F, synth.SEED_SUH + 2)).to(dev)
    svh = torch.from_numpy(synth.make_scale(OUT_F, synth.SEED_SVH + 2)).to(dev)
    xrs = {r: torch.empty((r, IN_F), dtype=torch.float16, device=dev) for r in ROWS}
    ys = {r: torch.empty((r, OUT_F), dtype=torch.float32, device=dev) for r in ROWS}
    ev = {r: [] for r in ROWS}
    call = [0]

    def step(record, fused=fused):
        # With `record`, an event pair brackets rot_in and the linear (an
        # event recorded between them would cut the programmatic dependent
        # launch that lets the linear's prologue overlap rot_in; rot_in is
        # ~2 % of the pair, so the linear's figures are slightly
        # conservative).
        for r in ROWS:
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            t = trs[call[0] % 2]
            call[0] += 1
            if fused:
                tf.tf_rot_in_linear(x[:r], suh, t, svh, BITS, OUT_F, xr=xrs[r], y=ys[r])
            else:
                tf.tf_rot_in(x[:r], suh, xr=xrs[r])
                linear(xrs[r], t, svh, BITS, OUT_F, y=ys[r])
            if record:
                e1.record(stream)
                ev[r].append((e0, e1))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    tf.tf_device_error()
    barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # Untimed steps for --load-s seconds first, so that the clock samples
        # (every 20 ms) see the GPU under this load even when the timed
        # region itself is a few milliseconds.
        t_load = time.perf_counter()
        while time.perf_counter() - t_load < args.load_s:
            for _ in range(16):
                step(False)
            torch.cuda.synchronize()
        barrier()
        # The headline: K steps with nothing between the launches, so that
        # each launch overlaps the end of the kernel before it (programmatic
        # dependent launch).
        start.record(stream)
        for _ in range(args.steps):
            step(False)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
        # The per-launch figures: a second timed pass of the same K steps
        # with an event pair around each (rot_in, linear) pair. The events cut
        # the overlap between launches.
        for _ in range(args.steps):
            step(True)
        torch.cuda.synchronize()
        # The same K steps through the other form of the call (the fused
        # rotation + linear when the headline runs the two calls, and the
        # other way round), reported beside the headline.
        alt_ms = None
        if args.layout == "tiles":
            for _ in range(args.warmup):
                step(False, fused=not fused)
            torch.cuda.synchronize()
            barrier()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(args.steps):
                step(False, fused=not fused)
            a1.record(stream)
            torch.cuda.synchronize()
            alt_ms = max_over_ranks(a0.elapsed_time(a1), dist, dev)
    barrier()
    tf.tf_device_error()
    ms_total = max_over_ranks(start.elapsed_time(stop), dist, dev)
    ms_step = ms_total / args.steps
    bytes_step = weight_bytes() * len(ROWS)
    value = replica_value(bytes_step, args.steps, world, ms_total)

    # The dominant kernel: the linear launches, timed by events on their
    # stream over the second timed pass.
    peak, peak_kind = measured_peaks()
    per_rows = {}
    dur_sum, byte_sum, launches = 0.0, 0, 0
    for r in ROWS:
        ds = [a.elapsed_time(b) for a, b in ev[r]]
        us = statistics.median(ds) * 1e3
        per_rows[str(r)] = {"us_median": us, "weight_gbs": weight_bytes() / us / 1e3, "rows_per_s": r / (us * 1e-6),
                            "hbm_gbs": launch_bytes(r, fused=fused) / us / 1e3, "hbm_frac": launch_bytes(r, fused=fused) / us / 1e3 / peak}
        dur_sum += sum(ds)
        byte_sum += launch_bytes(r, fused=fused) * len(ds)
        launches += len(ds)
    achieved = byte_sum / (dur_sum * 1e-3) / 1e9
    traffic = profiled_traffic()
    traffic_avg = (sum(traffic[r] for r in ROWS) / len(ROWS)) if traffic and all(r in traffic for r in ROWS) else None
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = alu_peak_tops(num_sms)
    alu_achieved = IN_F * OUT_F * DECODE_OPS_PER_WEIGHT * launches / (dur_sum * 1e-3) / 1e12

    # End to end through the public API from pinned host memory: every step
    # copies the rows of x its calls take in (one copy, the largest call's
    # rows; each call reads its first rows), and the step's logits out on a
    # copy stream that waits for the step's last call, so that the read
    # overlaps the next step; the timed region ends when every copy has
    # landed.
    x_host = torch.from_numpy(synth.make_x(max(ROWS), IN_F, synth.SEED_X + 2)).pin_memory()
    y_host = {r: torch.empty((r, OUT_F), dtype=torch.float32).pin_memory() for r in ROWS}
    e2e_steps = max(2, min(args.steps, 200))
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        x_dev = x_host.to(dev, non_blocking=True)
        ys_step = []
        for r in ROWS:
            if fused:
                _, y = tf.tf_rot_in_linear(x_dev[:r], suh, trs[call[0] % 2], svh, BITS, OUT_F,
                                           out_dtype=torch.float32)
            else:
                xr = tf.tf_rot_in(x_dev[:r], suh)
                y = linear(xr, trs[call[0] % 2], svh, BITS, OUT_F, out_dtype=torch.float32)
            call[0] += 1
            ys_step.append((r, y))
        # One event after the step's last call: an event recorded between two
        # launches would cut their overlap. The step's logits then go back on
        # the copy stream while the next step computes.
        done = torch.cuda.Event()
        done.record(stream)
        copy_stream.wait_event(done)
        with torch.cuda.stream(copy_stream):
            for r, y in ys_step:
                y_host[r].copy_(y, non_blocking=True)
        for r, y in ys_step:
            y.record_stream(copy_stream)

    e2e_s = float("nan")
    if not args.no_e2e:
        e2e_step()
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    e2e_value = replica_value(bytes_step, e2e_steps, world, e2e_s * 1e3) if not args.no_e2e else None

    # The other configurations (untimed for the headline).
    by_config = None
    if not args.no_configs and rank == 0:
        del trs, tr0, tr1
        torch.cuda.empty_cache()
        by_config = {}
        for name, i_f, o_f, bits, rows_list, odt in CONFIGS:
            by_config[name] = time_config(tf, dev, name, i_f, o_f, bits, rows_list, odt, args.layout,
                                          args.config_iters, peak)
            torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (fp32 sums)", "data": "synthetic",
        "config": bench_config(args, world),
        "by_rows": per_rows,
        "other_calls": None if alt_ms is None else {
            "calls": ("separate: tf_rot_in then tf_trellis_linear" if fused
                      else "fused: tf_rot_in_linear, one launch per call"),
            "ms_per_step": alt_ms / args.steps,
            "value": replica_value(bytes_step, args.steps, world, alt_ms), "unit": "GB/s"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_avg, "peak_source": peak_kind,
                     "kernel": DOMINANT_KERNEL, "kernel_hash": kernel_hash(),
                     "timing": ("CUDA events around each fused (rotation + linear) call" if fused else
                                "CUDA events around each (rot_in, linear) pair") + " over a second pass of the K steps",
                     "bytes_per_launch": {str(r): launch_bytes(r, fused=fused) for r in ROWS},
                     "alu": {"achieved": alu_achieved, "peak": alu_peak, "unit": "Tops/s",
                             "frac": alu_achieved / alu_peak, "ops_per_weight": DECODE_OPS_PER_WEIGHT,
                             "peak_source": "%d SMs x 4 issue slots x 32 lanes x %.0f MHz" % (num_sms, max_sm_mhz())}},
        "clocks": clocks.summary(),
        "e2e": None if args.no_e2e else {
            "value": e2e_value, "unit": "GB/s",
            "h2d_bytes_per_step": max(ROWS) * IN_F * 2,
            "d2h_bytes_per_step": sum(r * OUT_F * 4 for r in ROWS)},
        "gpu_launches": (1 if fused else 2) * len(ROWS) * args.steps,
        "cpu_baseline": cpu,
        "by_config": by_config,
    }
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations")
    ap.add_argument("--config-iters", type=int, default=20)
    ap.add_argument("--only-configs", default="",
                    help="time only these configurations (comma-separated names), print their by_config "
                         "entries and nothing else (for per-configuration profiling)")
    ap.add_argument("--load-s", type=float, default=0.5,
                    help="untimed steps run under the clock sampler before the timed region (seconds)")
    ap.add_argument("--rows", default="1,8,16", help="row counts per step (default 1,8,16)")
    ap.add_argument("--calls", choices=["fused", "separate"], default="separate",
                    help="the headline step's calls: rot_in then the linear (default), or the fused rotation + "
                         "linear (the k-tile order only); the other form is timed beside it")
    ap.add_argument("--layout", choices=["tiles", "strips"], default="tiles",
                    help="weight storage order: the k-tile-major tiles (the default) or strips "
                         "(repacked once at load, untimed)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    global ROWS
    ROWS = tuple(int(r) for r in args.rows.split(","))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
