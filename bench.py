"""Benchmark of the decode-row trellis projection on one GB300 per process.

Workload: the LM head, 5120 -> 129,280 at 4 bits per weight, one call each at
1, 8 and 16 rows per step (fp32 logits), on seeded synthetic inputs shaped
like the page's ("hip exl3: the input rotation and trellis linear for decode
rows", section "What this changes": x ~ N(0,1) fp16, suh/svh random sign *
U[0.5,1.5], uniformly random packed trellis bits).

A step is the whole hot path for each row count: tf_rot_in then the trellis
linear. The weights are stored in the library's strips order (repacked once
from the k-tile-major tiles at load time, outside the timed region;
`--layout tiles` times the k-tile-major order instead). The packed weights
(331 MB each) exceed the 129 MB L2; two copies alternate between calls, so no
call finds its weights in L2.

Metric: weight GB/s = packed weight bytes streamed / time, with the fraction
of the measured HBM copy bandwidth it reaches. Prints one JSON line.

Roofline: the linear is bound by the decode's integer arithmetic, not by HBM.
Decoding one weight takes four 32-bit lane operations (cut its 16-bit window
out of the stream, multiply by the mul1 constant, sum the product's bytes, one
fp16 fma); an SM issues one warp instruction (32 lane operations) per cycle in
each of its four sub-partitions, so the peak is SMs x 4 x 32 x the maximum SM
clock. The line's "roofline" reports that bound (unit: tera lane-ops/s) and,
under "hbm", the fraction of the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: the path has no exchange step; N processes run N independent
replicas (weak scaling) and rank 0 reports the aggregate.
"""

import argparse
import hashlib
import json
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
                  "kernels.h")


def weight_bytes():
    return IN_F * OUT_F * BITS // 8


def launch_bytes(rows):
    """Algorithmic bytes of one linear launch: packed weights, fp16 xr, fp16
    svh, fp32 y."""
    return weight_bytes() + rows * IN_F * 2 + OUT_F * 2 + rows * OUT_F * 4


# Lane operations the method's decode needs per weight: window cut, 32-bit
# multiply, byte sum, fp16 fma.
DECODE_OPS_PER_WEIGHT = 4


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def max_sm_mhz():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        if d.get("sm_max_mhz"):
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
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "trellis_linear_head_4b.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


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
                 "--format=csv,noheader,nounits", "-lms", "50"],
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


def oracle_sample(n_blocks, rows_list, k_tiles=IN_F // 16, stream=0):
    """The oracle on a bounded sample of the workload: the weights of n_blocks
    output blocks of 128 over the first k_tiles * 16 inputs (decoded from a
    packed stream of the same distribution; `stream` picks another seeded
    stream), for each row count: rot_in, decode, float64 linear and output
    rotation. Returns (seconds, packed weight bytes covered)."""
    import numpy as np
    from oracle import exl3 as o
    from trellis_quantized_linear_rot_gb300 import synth
    i_s = 128 * max(1, k_tiles // 8)
    g = np.random.Generator(np.random.PCG64(synth.SEED_TRELLIS + 2 + BITS + 1000 * stream))
    tr = g.integers(0, 2**32, size=i_s * 128 * n_blocks * BITS // 32, dtype=np.uint32)
    x = synth.make_x(max(rows_list), i_s, synth.SEED_X + 2)
    suh = synth.make_scale(i_s, synth.SEED_SUH + 2)
    svh = synth.make_scale(128 * n_blocks, synth.SEED_SVH + 2)
    t0 = time.perf_counter()
    covered = 0
    for rows in rows_list:
        xr = o.rot_in_f32(x[:rows], suh)
        w = o.decode_matrix(tr, i_s, 128 * n_blocks, BITS)
        o.linear_f64(xr, w, svh)
        covered += i_s * 128 * n_blocks * BITS // 8
    return time.perf_counter() - t0, covered


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _oracle_job(job):
    return oracle_sample(*job)


class OraclePool:
    """The oracle on every host core: one worker process per core, started
    with spawn (never forked from a process that has used the GPU), each with
    its BLAS limited to one thread, each timing its own seeded sample."""

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
        self.run(1, ROWS[:1], 8)  # imports in every worker

    def run(self, n_blocks_each, rows_list, k_tiles):
        """Wall seconds for all workers' samples, and the bytes they covered."""
        jobs = [(n_blocks_each, tuple(rows_list), k_tiles, w) for w in range(self.workers)]
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_job, jobs)
        return time.perf_counter() - t0, sum(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def bench_config(args, world):
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "rows": list(ROWS), "in_features": IN_F, "out_features": OUT_F,
            "bits": BITS, "out_dtype": "fp32", "weight_bytes_per_call": weight_bytes(),
            "layout": args.layout,
            "l2": "inputs larger than L2: 331 MB packed weights per call, two copies alternated",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    """The oracle timed on the host cores, on the same workload and metric.
    Each step is a bounded sample of it (one output block over a slice of the
    inputs, for each row count), sized so that the whole run of warm-up and
    timed steps takes about two minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    pool = OraclePool(cpu_threads())
    t_cal, _ = pool.run(1, ROWS, 8)                    # 128 inputs x 128 outputs per worker
    per_step = 120.0 / max(1, args.steps + args.warmup)
    k_tiles = int(max(8, min(IN_F // 16, 8 * per_step / max(t_cal, 1e-6))))
    for _ in range(args.warmup):
        pool.run(1, ROWS, k_tiles)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        t, b = pool.run(1, ROWS, k_tiles)
        total_t += t
        total_b += b
    pool.close()
    value = total_b / total_t / 1e9
    sample = ("per worker and step: 1 of 1010 output blocks over %d of 5120 inputs per row count "
              "(rows {1,8,16}); %d single-threaded workers" % (128 * max(1, k_tiles // 8), pool.workers))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(args, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
                         "sample": sample, "host_threads_available": cpu_threads()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


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

    # Inputs (untimed): two copies of the packed weights, x for 16 rows.
    tr_np = synth.make_trellis(IN_F, OUT_F, BITS, synth.SEED_TRELLIS + 2 + BITS)
    tr0 = torch.from_numpy(tr_np.view(np.int32)).to(dev)
    del tr_np
    if args.layout == "strips":
        tr0 = tf.tf_trellis_to_strips(tr0, IN_F, OUT_F, BITS)
    tr1 = tr0.clone()
    linear = tf.tf_trellis_linear_strips if args.layout == "strips" else tf.tf_trellis_linear
    trs = (tr0, tr1)
    x = torch.from_numpy(synth.make_x(16, IN_F, synth.SEED_X + 2)).to(dev)
    suh = torch.from_numpy(synth.make_scale(IN_F, synth.SEED_SUH + 2)).to(dev)
    svh = torch.from_numpy(synth.make_scale(OUT_F, synth.SEED_SVH + 2)).to(dev)
    xrs = {r: torch.empty((r, IN_F), dtype=torch.float16, device=dev) for r in ROWS}
    ys = {r: torch.empty((r, OUT_F), dtype=torch.float32, device=dev) for r in ROWS}
    ev = {r: [] for r in ROWS}
    call = [0]

    def step(record):
        # The event pair brackets rot_in and the linear: an event recorded
        # between them would cut the programmatic dependent launch that lets
        # the linear's prologue overlap rot_in. rot_in is ~1 % of the pair.
        for r in ROWS:
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            tf.tf_rot_in(x[:r], suh, xr=xrs[r])
            t = trs[call[0] % 2]
            call[0] += 1
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
        start.record(stream)
        for _ in range(args.steps):
            step(True)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier()
    tf.tf_device_error()
    ms_total = max_over_ranks(start.elapsed_time(stop), dist, dev)
    ms_step = ms_total / args.steps
    bytes_step = weight_bytes() * len(ROWS)
    value = replica_value(bytes_step, args.steps, world, ms_total)

    # Dominant kernel: the linear launches, timed by events on their stream.
    per_rows = {}
    dur_sum, byte_sum, launches = 0.0, 0, 0
    for r in ROWS:
        ds = [a.elapsed_time(b) for a, b in ev[r]]
        per_rows[r] = {"us_median": statistics.median(ds) * 1e3,
                       "weight_gbs": weight_bytes() / (statistics.median(ds) * 1e-3) / 1e9}
        dur_sum += sum(ds)
        byte_sum += launch_bytes(r) * len(ds)
        launches += len(ds)
    achieved = byte_sum / (dur_sum * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    traffic = profiled_traffic()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = alu_peak_tops(num_sms)
    alu_achieved = IN_F * OUT_F * DECODE_OPS_PER_WEIGHT * launches / (dur_sum * 1e-3) / 1e12

    # End to end through the public API from pinned host memory: every call
    # copies its rows of x in, and its logits out on a copy stream that waits
    # for the call, so that the read of one call's logits overlaps the next
    # call; the timed region ends when every copy has landed.
    x_host = torch.from_numpy(synth.make_x(16, IN_F, synth.SEED_X + 2)).pin_memory()
    y_host = {r: torch.empty((r, OUT_F), dtype=torch.float32).pin_memory() for r in ROWS}
    e2e_steps = max(2, min(args.steps, 200))
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        for r in ROWS:
            xd = x_host[:r].to(dev, non_blocking=True)
            xr = tf.tf_rot_in(xd, suh)
            y = linear(xr, trs[call[0] % 2], svh, BITS, OUT_F, out_dtype=torch.float32)
            call[0] += 1
            done = torch.cuda.Event()
            done.record(stream)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                y_host[r].copy_(y, non_blocking=True)
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

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        n_blocks = 60
        pool = OraclePool(cpu_threads())
        secs, covered = pool.run(n_blocks, ROWS, IN_F // 16)
        pool.close()
        cpu = {"value": covered / secs / 1e9, "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
               "sample": "per worker: %d of 1010 output blocks (5120x128 weights each) for each of rows "
                         "{1,8,16}; %d single-threaded workers, %.1f s wall" % (n_blocks, pool.workers, secs),
               "host_threads_available": cpu_threads()}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (fp32 sums)", "data": "synthetic",
        "config": bench_config(args, world),
        "by_rows": per_rows,
        "roofline": {"bound": "alu", "achieved": alu_achieved, "peak": alu_peak, "unit": "Tops/s",
                     "frac": alu_achieved / alu_peak, "traffic": traffic,
                     "ops_per_weight": DECODE_OPS_PER_WEIGHT,
                     "peak_source": "%d SMs x 4 issue slots x 32 lanes x %.0f MHz" % (num_sms, max_sm_mhz()),
                     "kernel": "trellis_linear", "kernel_hash": kernel_hash(),
                     "hbm": {"achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                             "peak_source": peak_kind}},
        "clocks": clocks.summary(),
        "e2e": None if args.no_e2e else {
            "value": e2e_value, "unit": "GB/s",
            "h2d_bytes_per_step": sum(r * IN_F * 2 for r in ROWS),
            "d2h_bytes_per_step": sum(r * OUT_F * 4 for r in ROWS)},
        "gpu_launches": 2 * len(ROWS) * args.steps,
        "cpu_baseline": cpu,
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
    ap.add_argument("--rows", default="1,8,16", help="row counts per step (default 1,8,16)")
    ap.add_argument("--layout", choices=["tiles", "strips"], default="strips",
                    help="weight storage order: strips (repacked once at load, untimed; the default) "
                         "or the k-tile-major tiles")
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
