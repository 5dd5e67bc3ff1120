"""Throughput of the DP-SGD private-gradient step (norms -> clip -> clipped sum
-> noise -> /L) on GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 5] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole path over one
batch of synthetic records already resident in HBM: every
dp_norm_accumulate (one batched call), dp_clip_factors and
dp_clipped_noisy_grad.  The metric is clipped+noised examples per second over
all ranks.  Under torchrun each rank processes its own batch (weak scaling,
no collective on the data path of the timed step).

The default workload is the largest single-GPU configuration: one
Llama-3-8B-shaped decoder layer (LoRA rank 16 on q/k/v/o and gate/up, the
full-weight down_proj), B = 32 records of T = 2048 tokens.
"""

from __future__ import annotations

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

METRIC = "clipped+noised examples/sec per step; TFLOP/s & HBM GB/s as % of GB300 roofline"
UNIT = "examples/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=5, help="workload index 1..5 (default: 5, the largest)")
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's B (smaller cases for profiler captures)")
    p.add_argument("--int8-forward", action="store_true",
                   help="time the record-owned LLM.int8 forward on OPT-125M-shaped layers instead")
    p.add_argument("--floors", action="store_true",
                   help="also time a device copy of the step's input bytes (the read floor at this size)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=12.0)
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(kernel: str):
    """dram read+write bytes per launch from the committed ncu summary, or None
    when the kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != d["source_sha256"]:
        return None
    return d["bytes_per_launch"]


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_samples(self, n: int, timeout_s: float = 3.0):
        t0 = time.time()
        while self.proc is not None and len(self.lines) < n and time.time() - t0 < timeout_s:
            time.sleep(0.02)

    def mark(self) -> int:
        """Index of the last sample taken before the timed region starts."""
        self.wait_samples(1)
        return max(0, len(self.lines) - 1)

    def stop(self, since: int = 0):
        """Stop after one more sample arrives; summarise samples from `since` on."""
        if self.proc is None:
            return None
        self.wait_samples(len(self.lines) + 1, 1.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[since:]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


PIN_CHUNK = 1 << 30


def pinned_chunks(nbytes: int):
    """Pinned host memory for nbytes as (offset, uint8 tensor) pieces of 1 GiB.
    torch's pinned-memory allocator rounds one request up to a power of two
    (16 GB for the 11.6 GB of inputs of the Llama-shaped layer, held by every
    rank of a node at once); 1 GiB pieces waste less than one piece."""
    import torch
    return [(o, torch.empty(min(PIN_CHUNK, nbytes - o), dtype=torch.uint8, pin_memory=True))
            for o in range(0, nbytes, PIN_CHUNK)]


def max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the default process group (x itself
    without one): the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, B: int, steps: int, total_ms: float) -> float:
    """Examples per second of the whole job: every rank clips and noises its
    own B records each step (weak scaling), in the slowest rank's time."""
    return world * B * steps / (total_ms / 1e3)


# ----------------------------------------------------------- work accounting
def work_model(w):
    """Algorithmic work of one step, per phase (one batch of w.B records).

    Norm phase: ghost layers with T > 1 do the two symmetric Grams,
    B T^2 (d_in + d_out) flops (tensor); T = 1 and materialized layers read
    A and E once (HBM).  Gradient phase: ghost layers do the reweighted
    GEMM, 2 B T d_in d_out flops (tensor); materialized layers read their
    stored per-example gradients once and write G (HBM)."""
    import differentially_private_gb300 as dp
    esz = 4 if w.dtype == "f32" else 2
    norm_flops = norm_bytes = grad_flops = grad_bytes = 0
    for ly in w.layers:
        ab = w.B * ly.T * (ly.d_in + ly.d_out) * esz
        ncl = ly.d_out * ly.d_in + (ly.d_out if ly.has_bias else 0)
        if dp.dp_choose_path(ly.T, ly.d_in, ly.d_out) == dp.DP_PATH_GHOST:
            if ly.T == 1:
                norm_bytes += ab
            else:
                norm_flops += w.B * ly.T * ly.T * (ly.d_in + ly.d_out)
            grad_flops += 2 * w.B * ly.T * ly.d_in * ly.d_out
            grad_bytes += ab + 4 * ncl
        else:
            norm_bytes += ab
            grad_bytes += 4 * ncl * (w.B + 1)
    return {"norm_flops": norm_flops, "norm_bytes": norm_bytes, "grad_flops": grad_flops, "grad_bytes": grad_bytes}


def dominant_kernel(w, phase: str, bound: str) -> str:
    """The library kernel that dominates a phase of one step of workload w,
    given the bound the work model assigns to that phase (the runtime's own
    kernel choice restated from the layers' dtype and shapes)."""
    import torch
    import differentially_private_gb300 as dp
    ghost_T = [ly.T for ly in w.layers if dp.dp_choose_path(ly.T, ly.d_in, ly.d_out) == dp.DP_PATH_GHOST]
    if w.torch_dtype == torch.float32:
        # fp32 layers take the CUDA-core kernels: ghost or materialized norms, and
        # the reweighted sum (16 x 16 tiles below sixteen 64 x 64 tiles) or the
        # weighted sum of the stored per-example gradients
        ly = max(w.layers, key=lambda l: l.d_in * l.d_out)
        ghost = dp.dp_choose_path(ly.T, ly.d_in, ly.d_out) == dp.DP_PATH_GHOST
        tiles64 = -(-ly.d_in // 64) * -(-ly.d_out // 64)
        if phase == "norm":
            return "k_norm_ghost_cc" if ghost else "k_norm_mat_cc"
        return "k_grad_wsum" if not ghost else "k_grad_gemm_small" if tiles64 < 16 else "k_grad_gemm_cc"
    if phase == "norm":
        return ("k_ghost_gram_tc" if bound == "tensor"
                else "k_norm_t1_group" if ghost_T and all(t == 1 for t in ghost_T) else "k_mat_skinny_tc")
    # layers whose T is not a multiple of 64 are summed as one pre-scaled record,
    # the layers sharing K in one launch of k_sum_layers_pair_tc
    return ("k_grad_wsum" if bound == "hbm"
            else "k_sum_layers_pair_tc" if ghost_T and all(t % 64 for t in ghost_T)
            else "k_clipped_sum_fold_pair_tc")


# ------------------------------------------------------------ CPU oracle leg
def oracle_sample_rate(w, record, n_avail: int, budget_s: float):
    """Oracle throughput (examples/s) on a bounded sample of the workload.

    The oracle materializes every per-example gradient in float64.  Its
    per-record work (the record's norm over all layers, its clip factor and
    its clipped gradient added to the running sum S of every layer) is timed
    on the first b records, b growing until the budget is used or the n_avail
    records given are exhausted; the noise and the division,
    G = (S + sigma C z) / L, are timed on a sample of coordinates.  The
    full-batch step time is t_records * B / b + t_noise * P / p.
    record(l, i) returns record i of layer l as float64 arrays (A_i, E_i);
    fetching it is not timed."""
    import numpy as np
    from oracle import dpsgd, philox

    layers = [dpsgd.Layer(ly.d_in, ly.d_out, ly.has_bias) for ly in w.layers]
    t_rec = 0.0
    t0 = time.perf_counter()
    S = [np.zeros((ly.d_out, ly.d_in)) for ly in layers]
    Sb = [np.zeros(ly.d_out) if ly.has_bias else None for ly in layers]
    t_rec += time.perf_counter() - t0
    b = 0
    while b < min(w.B, n_avail) and (b == 0 or t_rec < budget_s * 0.8):
        rec = [record(l, b) for l in range(len(layers))]
        t0 = time.perf_counter()
        n2 = 0.0
        for ly, (A, E) in zip(layers, rec):
            n2 += dpsgd.record_sqnorm(A, E, ly.has_bias)
        c = dpsgd.clip_factors(np.array([n2]), w.C)[0]
        for l, (ly, (A, E)) in enumerate(zip(layers, rec)):
            g, bb = dpsgd.per_example_grad(A, E, ly.has_bias)
            S[l] += c * g
            if bb is not None:
                Sb[l] += c * bb
        t_rec += time.perf_counter() - t0
        b += 1
    P = w.ncoords
    p = min(P, 1 << 22)
    t0 = time.perf_counter()
    z = philox.normals(w.noise_seed, w.step, 0, p)
    done = 0
    for l, ly in enumerate(layers):
        if done >= p:
            break
        flat = S[l].reshape(-1) if Sb[l] is None else np.concatenate([S[l].reshape(-1), Sb[l]])
        m = min(flat.size, p - done)
        _ = (flat[:m] + w.sigma * w.C * z[done:done + m]) / float(w.B)
        done += m
    t_noise = (time.perf_counter() - t0) * P / p
    t_full = t_rec * w.B / b + t_noise
    cores = len(os.sched_getaffinity(0))
    sample = (f"oracle float64 on {b} of {w.B} records (per-record norm, clip factor, clipped gradient "
              f"added to the sum of every layer) timed, scaled to B; noise and division timed on {p} of "
              f"{P} coordinates, scaled to P")
    return w.B / t_full, cores, sample, t_full


def device_records(A_dev, E_dev):
    """record(l, i) over device tensors: record i of layer l copied to the host in float64."""
    import torch

    def record(l, i):
        return (A_dev[l][i].to("cpu", torch.float64).numpy(), E_dev[l][i].to("cpu", torch.float64).numpy())
    return record


def host_records(w, max_bytes: int = 2 << 30):
    """record(l, i) over inputs drawn on the CPU with the workload's recipe,
    keeping at most about max_bytes of them (the first records of a batch of
    that size: per-record work does not depend on B); returns (record, n)."""
    import torch
    from synthetic import generate_layer
    n = w.B if w.input_bytes <= max_bytes else max(2, int(w.B * max_bytes / w.input_bytes))
    ws = w.scaled(B=n)
    A_host, E_host = [], []
    for i in range(len(w.layers)):
        a, e = generate_layer(ws, i, "cpu")
        A_host.append(a)
        E_host.append(e)

    def record(l, i):
        return A_host[l][i].to(torch.float64).numpy(), E_host[l][i].to(torch.float64).numpy()
    return record, n


def config_dict(w, world: int) -> dict:
    """The workload's description, the same in both arms."""
    return {"workload": w.name, "B": w.B, "layers": len(w.layers), "T": sorted({ly.T for ly in w.layers}),
            "C": w.C, "sigma": w.sigma,
            "l2": (f"flushed before every timed step: {L2_FLUSH_BYTES >> 20} MB written, "
                   f"then {L2_FLUSH_BYTES >> 20} MB read"),
            "parallelism": f"replicas x{world}"}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


MANIFEST_KEYS = ("gpu", "compute_capability", "sms", "driver", "cuda", "torch", "library_version",
                 "library_sha256_16", "B", "T", "C", "sigma", "seed", "step", "L", "dtype", "chooser",
                 "kernels_per_step", "host")


def release_record(w, gpu: dict, lib: dict, kernels_per_step: dict, host: dict) -> dict:
    """Release record of a run: hardware and software (gpu: name,
    compute_capability, sms, driver, cuda, torch; lib: version, sha256_16),
    the step's public parameters (B, T, C, sigma, seed, step, L, dtype), the
    chooser's decision per layer (exact integer rule T^2 < d_in d_out), the
    kernels launched per step and the host the oracle ran on."""
    import differentially_private_gb300 as dp
    rec = dict(gpu)
    rec.update({
        "library_version": lib.get("version"), "library_sha256_16": lib.get("sha256_16"),
        "B": w.B, "T": [ly.T for ly in w.layers], "C": w.C, "sigma": w.sigma, "seed": w.noise_seed,
        "step": w.step, "L": float(w.B), "dtype": w.dtype,
        "chooser": [[ly.name, ly.d_in, ly.d_out, ly.T,
                     "ghost" if dp.dp_choose_path(ly.T, ly.d_in, ly.d_out) == dp.DP_PATH_GHOST else "materialize"]
                    for ly in w.layers],
        "kernels_per_step": kernels_per_step,
        "host": host,
    })
    return {k: rec.get(k) for k in MANIFEST_KEYS}


def manifest(w, dp, device, kernels_per_step: dict) -> dict:
    """The release record of this run, collected from the device, the driver and the library."""
    import torch
    props = torch.cuda.get_device_properties(device)
    try:
        drv = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(device.index or 0)], capture_output=True, text=True, timeout=20).stdout.strip()
    except (OSError, subprocess.SubprocessError):
        drv = None
    gpu = {"gpu": props.name, "compute_capability": f"{props.major}.{props.minor}",
           "sms": props.multi_processor_count, "driver": drv, "cuda": torch.version.cuda, "torch": torch.__version__}
    lib = {"version": dp.dp_version(), "sha256_16": hashlib.sha256(open(dp.LIB_PATH, "rb").read()).hexdigest()[:16]}
    host = {"cores": len(os.sched_getaffinity(0)), "cpu_model": cpu_model()}
    return release_record(w, gpu, lib, kernels_per_step, host)


# ------------------------------------------------------------------- arms
def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    record, n_avail = host_records(w)
    per = max(2.0, args.cpu_budget_s / max(1, args.steps + args.warmup) * 4)
    for _ in range(args.warmup):
        oracle_sample_rate(w, record, n_avail, min(per, 2.0))
    times = []
    rate, cores, sample = None, None, None
    for _ in range(args.steps):
        rate, cores, sample, t_full = oracle_sample_rate(w, record, n_avail, per)
        times.append(t_full)
    t_step = statistics.mean(times)
    value = w.B / t_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample + f"; inputs drawn on the host ({n_avail} records)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import differentially_private_gb300 as dp
    from synthetic import generate_layer

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dp.load_library()

    layers = [(ly.d_in, ly.d_out, ly.has_bias) for ly in w.layers]
    # all inputs in one device arena (256-byte aligned segments), so that the
    # end-to-end leg moves them with one host->device copy per step
    esz = 4 if w.dtype == "f32" else 2
    seg = lambda n: (n * esz + 255) // 256 * 256  # noqa: E731
    sizes = []
    for ly in w.layers:
        sizes += [w.B * ly.T * ly.d_in, w.B * ly.T * ly.d_out]
    arena = torch.empty(sum(seg(n) for n in sizes), dtype=torch.uint8, device=device)

    def carve(buf):
        # the layers' A and E as views of one arena, in layer order
        views, off = [], 0
        for n in sizes:
            views.append(buf[off:off + n * esz].view(w.torch_dtype))
            off += seg(n)
        return ([views[2 * i].view(w.B, ly.T, ly.d_in) for i, ly in enumerate(w.layers)],
                [views[2 * i + 1].view(w.B, ly.T, ly.d_out) for i, ly in enumerate(w.layers)])

    A_dev, E_dev = carve(arena)
    for i, ly in enumerate(w.layers):
        a, e = generate_layer(w, i, device)
        A_dev[i].copy_(a)
        E_dev[i].copy_(e)
        del a, e
    T_list = [ly.T for ly in w.layers]
    stream = torch.cuda.current_stream(device)
    pg = dp.PrivateGradient(layers, dtype=w.torch_dtype, device=local, stream=stream)
    _, clip, sq = pg.alloc_outputs(w.B)
    gsizes = [(n + 63) // 64 * 64 for (_, _, _, _, n) in pg.layers]
    garena = torch.empty(sum(gsizes), dtype=torch.float32, device=device)
    grads, off = [], 0
    for (_, _, _, _, n), gs in zip(pg.layers, gsizes):
        grads.append(garena[off:off + n])
        off += gs
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the dirty lines of
        # the write are written back here, before the timed step, not during it
        flush.zero_()
        flush_rd.sum()

    ctx = pg.ctx
    # the step's pointer arguments are marshalled once; every step makes the
    # same four C calls (begin, batched norms, clip factors, clipped noisy sum)
    prep = pg.prepare(A_dev, E_dev, T_list, outputs=(grads, clip, sq))

    def step(evs=None, after_phase=None):
        prep.run(w.C, w.sigma, w.noise_seed, w.step, events=evs, after_phase=after_phase)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    st = dp.dp_step_status(ctx)
    if st != dp.DP_OK:
        raise dp.DPError(st, "dp_step_status", dp.dp_last_error(ctx))

    K = args.steps
    # timed region: K steps, one event pair per step.  An event recorded
    # between two kernels of the step would serialize the dependent launches
    # of the step's later kernels, so the phase split is taken in a second
    # pass of K steps with events between the phases.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    since = clocks.mark()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n_launch0 = dp.dp_kernel_launches()
    per_kernel0 = dp.dp_kernel_launch_counts()
    for k in range(K):
        flush_l2()
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    n_launch = dp.dp_kernel_launches() - n_launch0
    per_kernel = {name: (cnt - per_kernel0[name]) / K for name, cnt in dp.dp_kernel_launch_counts().items()
                  if cnt != per_kernel0[name]}
    if world > 1:
        torch.distributed.barrier()
    for k in range(K):
        flush_l2()
        step(pevs[k])
    torch.cuda.synchronize()
    clk = clocks.stop(since)
    # SM clock at the end of each phase, from the device: two spins of a fixed
    # number of SM cycles right after the phase, timed with events on the
    # stream; the difference of their times cancels the launch and event
    # overheads (a third pass of K steps; not part of the timed region)
    short_cycles, long_cycles = 50_000, 250_000
    probes = {"norm": [], "clip": [], "grad": []}

    def probe(phase):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        torch.cuda._sleep(short_cycles)
        ev[1].record(stream)
        torch.cuda._sleep(long_cycles)
        ev[2].record(stream)
        probes[phase].append(ev)

    for k in range(K):
        flush_l2()
        step(after_phase=probe)
    torch.cuda.synchronize()

    def mhz(ev):
        dt_ms = ev[1].elapsed_time(ev[2]) - ev[0].elapsed_time(ev[1])
        return (long_cycles - short_cycles) / (dt_ms * 1e3) if dt_ms > 0 else float("nan")
    phase_mhz = {ph: statistics.median([mhz(ev) for ev in v]) for ph, v in probes.items() if v}
    if clk is not None:
        clk["sm_mhz_after_phase"] = phase_mhz
    st = dp.dp_step_status(ctx)
    if st != dp.DP_OK:
        raise dp.DPError(st, "dp_step_status", dp.dp_last_error(ctx))

    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    norm_ms = [e[0].elapsed_time(e[1]) for e in pevs]
    clip_ms = [e[1].elapsed_time(e[2]) for e in pevs]
    grad_ms = [e[2].elapsed_time(e[3]) for e in pevs]
    total_ms = max_over_ranks(sum(step_ms), device)
    value = job_throughput(world, w.B, K, total_ms)

    # roofline of the dominant phase
    peaks = load_peaks()
    wm = work_model(w)
    mn, mg = statistics.mean(norm_ms), statistics.mean(grad_ms)
    if mn >= mg:
        phase, t_ms, flops, bytes_ = "norm", mn, wm["norm_flops"], wm["norm_bytes"]
    else:
        phase, t_ms, flops, bytes_ = "grad", mg, wm["grad_flops"], wm["grad_bytes"]
    # fp32 layers run their arithmetic on the CUDA cores: 152 SMs x 128 fp32
    # lanes x 2 flops (FMA) x the SM clock's maximum
    alu = w.dtype == "f32"
    alu_tflops = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    cpeak = alu_tflops if alu else peaks["bf16_tflops"]
    tc_time = flops / (cpeak * 1e12)
    hb_time = bytes_ / (peaks["hbm_gbs"] * 1e9)
    if tc_time >= hb_time and flops > 0:
        ach = flops / (t_ms / 1e3) / 1e12
        roof = {"bound": "alu" if alu else "tensor", "achieved": ach, "peak": cpeak, "unit": "TFLOP/s",
                "frac": ach / cpeak}
    else:
        ach = bytes_ / (t_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    kernel_name = dominant_kernel(w, phase, roof["bound"])
    roof["traffic"] = kernel_traffic(f"{kernel_name}@{w.name}")
    roof["kernel"] = kernel_name
    roof["phase"] = phase
    roof["timing"] = f"mean {phase} phase of a second pass of {K} steps with events between the phases"
    roof["peak_source"] = ("derived: 152 SMs x 128 fp32 lanes x 2 flops x max SM clock"
                           if roof["bound"] == "alu" else peaks["source"])

    # what a plain copy of the step's input bytes reaches at this size (a
    # device-to-device copy of the input arena, L2 flushed first): the
    # fraction of the peak a launch of this size can reach, outside the library
    floors = None
    if args.floors:
        dst = torch.empty_like(arena)
        cp = []
        for _ in range(max(3, args.warmup)):
            dst.copy_(arena)
        for _ in range(K):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(arena)
            e1.record(stream)
            torch.cuda.synchronize()
            cp.append(e0.elapsed_time(e1))
        del dst
        t_cp = statistics.median(cp)
        eff = 2 * arena.numel() / (t_cp / 1e3) / 1e9 / peaks["hbm_gbs"]
        floors = {"input_bytes": arena.numel(), "copy_us": t_cp * 1e3, "copy_frac_of_peak": eff,
                  "read_floor_us": arena.numel() / (peaks["hbm_gbs"] * 1e9 * eff) * 1e6,
                  "ideal_read_us": arena.numel() / (peaks["hbm_gbs"] * 1e9) * 1e6}

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads G back.  Two schedules are
    # timed: the inputs of step k + 1 copied into a second device arena on a
    # second stream while step k computes (as a data loader would prefetch
    # the next batch), and copy, step and read-back one after the other on one
    # stream; the line reports the faster, both, and the host link's own rate
    e2e = None
    if not args.no_e2e:
        arena_pin = pinned_chunks(arena.numel())
        for o, c in arena_pin:
            c.copy_(arena[o:o + c.numel()])

        def h2d_copy(dst):
            for o, c in arena_pin:
                dst[o:o + c.numel()].copy_(c, non_blocking=True)

        garena_pin = torch.empty(garena.numel(), dtype=torch.float32, pin_memory=True)
        h2d = arena.numel()
        d2h = garena.numel() * 4
        ke = max(3, min(K, 10))

        def timed(fn):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        link_ms = min(timed(lambda: h2d_copy(arena)) for _ in range(3))
        d2h_link_ms = min(timed(lambda: garena_pin.copy_(garena, non_blocking=True)) for _ in range(3))

        copy_ev, read_ev = [], []

        def serial(n):
            for _ in range(n):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                ev[0].record(stream)
                h2d_copy(arena)
                ev[1].record(stream)
                step()
                ev[2].record(stream)
                garena_pin.copy_(garena, non_blocking=True)
                ev[3].record(stream)
                copy_ev.append((ev[0], ev[1]))
                read_ev.append((ev[2], ev[3]))

        arena2 = torch.empty_like(arena)
        A2, E2 = carve(arena2)
        preps = [prep, pg.prepare(A2, E2, T_list, outputs=(grads, clip, sq))]
        arenas = [arena, arena2]
        cstream = torch.cuda.Stream(device)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        freed = [torch.cuda.Event(), torch.cuda.Event()]

        def pipelined(n):
            cstream.wait_stream(stream)
            with torch.cuda.stream(cstream):
                h2d_copy(arenas[0])
                copied[0].record(cstream)
            for k in range(n):
                cur, nxt = k % 2, (k + 1) % 2
                if k + 1 < n:
                    with torch.cuda.stream(cstream):
                        if k >= 1:
                            cstream.wait_event(freed[nxt])     # step k - 1 is done with that arena
                        h2d_copy(arenas[nxt])
                        copied[nxt].record(cstream)
                stream.wait_event(copied[cur])
                preps[cur].run(w.C, w.sigma, w.noise_seed, w.step)
                freed[cur].record(stream)
                garena_pin.copy_(garena, non_blocking=True)

        serial(2)
        pipelined(2)
        copy_ev.clear()
        read_ev.clear()
        ser_ms = max_over_ranks(timed(lambda: serial(ke)), device)
        loop_copy_ms = statistics.median(a.elapsed_time(b) for a, b in copy_ev)
        loop_read_ms = statistics.median(a.elapsed_time(b) for a, b in read_ev)
        ems = max_over_ranks(timed(lambda: pipelined(ke)), device)
        st = dp.dp_step_status(ctx)
        if st != dp.DP_OK:
            raise dp.DPError(st, "dp_step_status", dp.dp_last_error(ctx))
        del arena2, A2, E2, preps, arena_pin
        pipe_value = job_throughput(world, w.B, ke, ems)
        ser_value = job_throughput(world, w.B, ke, ser_ms)
        # the faster of the two schedules (for a few KB of inputs the second
        # stream's synchronization costs more than the copy it hides)
        e2e = {"value": max(pipe_value, ser_value), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ke,
               "copies": ("next step's inputs copied on a second stream while the current step computes"
                          if pipe_value >= ser_value else "copy, step and read-back one after the other on one stream"),
               "pipelined_value": pipe_value, "serial_value": ser_value,
               "h2d_link_gbs": h2d / (link_ms / 1e3) / 1e9,
               "h2d_gbs_in_serial_loop": h2d / (loop_copy_ms / 1e3) / 1e9,
               "d2h_link_gbs": d2h / (d2h_link_ms / 1e3) / 1e9,
               "d2h_gbs_in_serial_loop": d2h / (loop_read_ms / 1e3) / 1e9}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, sample, _ = oracle_sample_rate(w, device_records(A_dev, E_dev), w.B, args.cpu_budget_s)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_dict(w, world),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": n_launch,
            "clocks": clk,
            "phases_ms": {"norm": mn, "clip": statistics.mean(clip_ms), "grad": mg,
                          "step_with_phase_events": statistics.mean([e[0].elapsed_time(e[3]) for e in pevs])},
            "manifest": manifest(w, dp, device, per_kernel),
            **({"floors": floors} if floors is not None else {}),
        }
        print(json.dumps(line), flush=True)
    pg.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_int8_forward(args):
    """The record-owned LLM.int8 forward of a frozen layer on OPT-125M-shaped
    inputs: 16 records x 256 rows of fp16 activations, d_model 768, with a
    few outlier entries (|a| >= 6) in a few columns of some records.  Times
    dp_int8_forward (all its launches) with CUDA events, 10 warm-up and K
    timed calls (both products warmed up), L2 flushed before each and the GPU kept busy while the host
    enqueues them (the host's enqueue time is reported apart); beside it, the same product through
    torch.matmul in fp16 (cuBLAS on the tensor cores, batched-LLM.int8-free
    and not record-isolated: context only).  Prints one JSON line per layer."""
    import torch
    from differentially_private_gb300.int8 import Int8Linear
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(9)
    records, rows, K = 16, 256, 768
    n = records * rows
    A = torch.randn(n, K, device=dev, generator=g)
    for r in range(0, records, 3):                      # outliers in a few columns of every third record
        A[r * rows + 5, 17] = 8.0
        A[r * rows + 90, 300 + r] = -7.5
    A = A.half()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one (the write-back
        # of the dirty lines happens here, not inside the timed calls)
        flush.zero_()
        flush_rd.sum()

    stream = torch.cuda.current_stream(dev)
    for N in (768, 3072):
        W = (torch.randn(N, K, device=dev, generator=g) * 0.03).half()
        lin = Int8Linear(W, stream=stream)
        for _ in range(10):
            lin(A, rows)
            torch.matmul(A, W.t())
        torch.cuda.synchronize()
        times, ref_times, host = [], [], []
        for _ in range(args.steps):
            # a spin first, so that the GPU time between the events is the
            # calls' own and not the host's time to enqueue them
            flush_l2()
            torch.cuda._sleep(2_000_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            h0 = time.perf_counter()
            lin(A, rows)
            host.append(time.perf_counter() - h0)
            e1.record(stream)
            flush_l2()
            torch.cuda._sleep(2_000_000)
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            torch.matmul(A, W.t())
            f1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
            ref_times.append(f0.elapsed_time(f1))
        t = statistics.median(times)
        ops = 2 * n * K * N
        line = {"metric": "record-owned LLM.int8 forward", "layer": f"{K}->{N}", "records": records,
                "rows_per_record": rows, "us_per_call": t * 1e3, "int8_tops": ops / (t / 1e3) / 1e12,
                "bytes_moved_min": n * K * 2 + N * K * (1 + 2) + n * N * 2,
                "host_enqueue_us": statistics.median(host) * 1e6,
                "torch_fp16_matmul_us": statistics.median(ref_times) * 1e3, "steps": args.steps,
                "l2": "flushed before every timed call"}
        print(json.dumps(line), flush=True)
    # the GPU's own int8 and bf16 tensor-core rates on a large product (cuBLAS
    # through torch): context for the int8 forward, whose exact integer
    # product runs on the bf16 tensor cores for K up to 4096
    rates = {}
    m = 8192
    for name, mk in (("int8", lambda: (torch.randint(-127, 128, (m, m), dtype=torch.int8, device=dev),
                                       torch.randint(-127, 128, (m, m), dtype=torch.int8, device=dev).t())),
                     ("bf16", lambda: (torch.randn(m, m, device=dev, dtype=torch.bfloat16),
                                       torch.randn(m, m, device=dev, dtype=torch.bfloat16).t()))):
        try:
            a, bm = mk()
            f = torch._int_mm if name == "int8" else torch.matmul
            for _ in range(3):
                f(a, bm)
            torch.cuda.synchronize()
            ts = []
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                f(a, bm)
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            rates[name + "_tops"] = 2 * m ** 3 / (min(ts) / 1e3) / 1e12
            del a, bm
        except (RuntimeError, AttributeError) as exc:
            rates[name + "_tops"] = f"unavailable: {type(exc).__name__}"
    print(json.dumps({"metric": "tensor-core rate, 8192^3 product (torch/cuBLAS), best of 10", **rates}), flush=True)
    return 0


def main():
    args = parse()
    if args.int8_forward:
        return run_int8_forward(args)
    from synthetic import by_index
    w = by_index(args.workload)
    if args.batch is not None:
        w = w.scaled(B=int(args.batch))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
