"""Benchmark of the packed varlen attention hot path on GB300.

One step = one pass of the whole varlen path over one batch:
  cu_seqlens from lengths -> pack q, k, v (padded -> flat) -> varlen
  attention -> unpack the output (flat -> padded).
The headline workload is the largest single-GPU config, the dynamic step
batch with classifier-free guidance (8 requests with image tokens from
{2304, 4096, 6889, 16384}, each doubled into a positive and a negative text
span: 16 sequences, 129,490 tokens, H=24, D=128, bf16 N(0,1)).  The single
edit request (256 + 32,768 tokens) and the mixed-resolution batch (4
requests) are timed the same way and reported under "configs".
The Token2Wav block-window variant (22 layers, n=2400, H=16, D=64, block 24)
is timed in the same run and reported under "block_window", and its fp32
form (the DiT's own dtype, classifier-free guidance as batch 2) under
"block_window_f32".

Rank 0 prints one JSON line.  Under torchrun each rank runs its own batch
(its own value seed) on its own GPU; no data moves between ranks (weak
scaling); the timed region is bracketed by a barrier and the slowest rank's
time is reported.

--impl reference times the CPU oracle (fp64 NumPy) on a bounded sample of the
same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "packed varlen attention useful TFLOP/s and % of GB300 bf16 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = "cfg_dynamic_batch"
SUB_WORKLOADS = ("single_edit", "mixed_res_mmdit")
# query rows per sequence of the CPU-oracle baseline sample, per workload
# (about 5-15 s of fp64 work each on 16 host cores)
CPU_ROWS = {"cfg_dynamic_batch": 512, "single_edit": 1024, "mixed_res_mmdit": 1024}
# FP32 FMA rate of one GB300: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            raw = json.load(f)
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"
    out = dict(FALLBACK_PEAKS)
    flat = {}

    def walk(d):   # numbers at any depth, by their own key
        if isinstance(d, dict):
            for k, v in d.items():
                if isinstance(v, (int, float)) and not isinstance(v, bool):
                    flat.setdefault(k, float(v))
                else:
                    walk(v)
    walk(raw)

    def find(keys):
        for k in keys:
            if k in flat:
                return flat[k]
        return None
    hbm = find(["hbm_gbs", "hbm_GBps", "hbm_gb_s"])
    bf = find(["bf16_tflops", "bf16_TFLOPs"])
    bfs = find(["bf16_tflops_sustained"])
    if hbm:
        out["hbm_gbs"] = hbm
    if bf:
        out["bf16_tflops"] = bf
    if bfs:
        out["bf16_tflops_sustained"] = bfs
    return out, ("measured" if (hbm or bf) else "fallback")


def _kernel_digest() -> str:
    """Hash of the sources of the dominant kernel (ties an ncu traffic figure
    to the code it was taken on)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "packed_varlen_gb300", "csrc")
    for name in ("attn_pair.cu", "varlen_items.cuh", "tc_ptx.cuh", "sched.cuh", "internal.h",
                 "tma_map.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled(digest: str, workload: str = WORKLOAD):
    """Figures of the attention kernel on `workload` from its committed ncu
    summary (DRAM bytes per launch, tensor-pipe utilisation, DRAM GB/s), if
    it was taken on the current kernel sources; else an empty dict."""
    path = os.path.join(ROOT, "profiles", f"varlen_attn_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return {}
    m_d = re.search(r"kernel_digest:\s*([0-9a-f]+)", text)
    if not m_d or m_d.group(1) != digest:
        return {}
    out = {}
    for key in ("dram_bytes_per_launch", "tensor_pipe_active_pct", "dram_gbs"):
        m = re.search(key + r":\s*([0-9.eE+]+)", text)
        if m:
            out[key] = float(m.group(1))
    return out


def rank_seed(rank: int, base: int = 1002) -> int:
    """Value seed of the batch a rank processes: every rank holds its own batch
    of the same shape (same lengths, weak scaling); no data moves between ranks."""
    return base + 7919 * rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's time: the job finishes when its last rank does."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class L2Flusher:
    """Empties L2 between timed iterations, outside the timed events: writes a
    buffer larger than L2 (evicting everything), then reads a second one so
    that the dirty lines of the write are written back before timing starts
    and L2 holds only clean lines."""

    def __init__(self, device, nbytes: int = L2_FLUSH_BYTES):
        self.w = torch.empty(nbytes // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def flush(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def block_window_flops(n, H, D, block, look_back, look_ahead):
    """Useful FLOPs of one block-window layer: 4*H*D per allowed (query, key)
    pair; a query of block i sees keys [(i-lb)*block, (i+la+1)*block) in [0, n)."""
    pairs = 0
    for i in range(-(-n // block)):
        rows = min(n, (i + 1) * block) - i * block
        keys = min(n, (i + look_ahead + 1) * block) - max(0, (i - look_back) * block)
        pairs += rows * keys
    return 4 * H * D * pairs


def oracle_sample(pw, rows_per_seq: int, seed: int = 0):
    """Bounded oracle sample on a padded workload: ``rows_per_seq`` random
    query rows of every sequence, all heads, against all of its keys; one
    sequence at a time so only that sequence is held in fp64.  Returns
    (seconds, useful FLOPs of the sample, description)."""
    import oracle
    rng = np.random.default_rng(seed)
    H, D = pw.H, pw.D
    scale = 1.0 / math.sqrt(D)
    flops, n_rows, dt = 0, 0, 0.0
    for b, L in enumerate(pw.lengths):
        r = np.sort(rng.choice(L, size=min(rows_per_seq, L), replace=False))
        q, k, v = (oracle.to_f64(t[b, :L]) for t in (pw.q, pw.k, pw.v))
        t0 = time.perf_counter()
        oracle.varlen_attention(q, k, v, [0, L], [0, L], scale, rows=r)
        dt += time.perf_counter() - t0
        flops += 4 * H * D * len(r) * L
        n_rows += len(r)
    desc = (f"{rows_per_seq} query rows per sequence x all {H} heads ({n_rows} rows) of the "
            f"{pw.name[:-len('_padded')]} batch against all keys, fp64 NumPy")
    return dt, flops, desc


def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    pw = workloads.varlen_padded(WORKLOAD, rank_seed(0))
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(pw, rows)
    times, flops, desc = [], 0, ""
    for i in range(args.steps):
        dt, flops, desc = oracle_sample(pw, rows, seed=i)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    cores = _cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": len(pw.lengths), "H": pw.H, "D": pw.D,
                   "tokens": sum(pw.lengths), "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def measure_varlen_config(pv, name, dev, args, flusher, rank, dist, ws, cpu_rows=None):
    """Time K steps of the varlen path on one config, inputs resident in HBM
    and L2 emptied between steps (outside the events); then the same K steps
    end to end with host buffers; then, if asked, the CPU oracle on a bounded
    sample.  Returns the fields of a bench line for this config."""
    pw = workloads.varlen_padded(name, rank_seed(rank))
    L = pw.lengths
    T, H, D, B, S = sum(L), pw.H, pw.D, len(L), pw.s_max
    flops = 4 * H * D * sum(x * x for x in L)
    stream = torch.cuda.current_stream()
    q_pad, k_pad, v_pad = pw.q.to(dev), pw.k.to(dev), pw.v.to(dev)
    lengths = torch.tensor(L, dtype=torch.int32, device=dev)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    qf = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    kf, vf, of = torch.empty_like(qf), torch.empty_like(qf), torch.empty_like(qf)
    out_pad = torch.zeros_like(q_pad)
    scale = 1.0 / math.sqrt(D)
    attn_ev = []

    def step(record=False):
        pv.cu_seqlens_from_lengths(lengths, out=cu)
        pv.pack(q_pad, cu, T, out=qf)
        pv.pack(k_pad, cu, T, out=kf)
        pv.pack(v_pad, cu, T, out=vf)
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        pv.varlen_attn_fwd(qf, kf, vf, cu, cu, max(L), max(L), scale=scale, out=of)
        if record:
            e1.record(stream)
            attn_ev.append((e0, e1))
        pv.unpack(of, cu, out_pad)

    launches_per_step = 6
    warm = max(3, args.warmup)
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    if pv.get_device_status() != 0:
        raise RuntimeError(f"device status error during the {name} warm-up")

    # ---- timed: K steps, L2 flushed between steps (outside the events) ------
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ev = []
    for _ in range(args.steps):
        flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(record=True)
        e1.record(stream)
        step_ev.append((e0, e1))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    if pv.get_device_status() != 0:
        raise RuntimeError(f"device status error during the {name} timed steps")
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    value = flops * ws * args.steps / (total_ms * 1e-3) / 1e12
    want_out = out_pad.cpu()
    del q_pad, k_pad, v_pad, qf, kf, vf, of, out_pad

    # ---- end to end: host buffers in, host result out ----------------------
    # the same job size as the device-timed value: K steps, copies included
    e2e_mean, h2d, d2h = run_e2e(pv, pw, dev, scale, max(3, args.steps), want_out)
    e2e_mean = max_over_ranks(e2e_mean, dist, dev)
    e2e_value = flops * ws / (e2e_mean * 1e-3) / 1e12
    del want_out

    peaks, peak_src = _peaks()
    attn_mean_ms = statistics.mean(attn_ms)
    achieved = flops / (attn_mean_ms * 1e-3) / 1e12
    digest = _kernel_digest()
    prof = _profiled(digest, name)
    cpu = None
    if cpu_rows and rank == 0 and ws == 1:
        dt, sflops, desc = oracle_sample(pw, cpu_rows)
        cpu = {"value": sflops / dt / 1e12, "unit": UNIT, "cores": _cpu_cores(),
               "kind": "oracle", "sample": desc, "seconds": dt}
    res = {
        "value": value, "unit": UNIT, "ms_per_step": total_ms / args.steps,
        "config": {"workload": name, "batch": B, "lengths": L, "tokens": T, "H": H, "D": D,
                   "s_max": S, "useful_flops_per_step": flops,
                   "step": "cu_seqlens + pack q,k,v + varlen attention + unpack",
                   "l2": "flushed between timed steps outside the events (512 MB write, then "
                         "512 MB read so L2 holds clean lines); padded inputs 3 x %.0f MB also "
                         "exceed L2" % (pw.q.numel() * 2 / 2**20),
                   "parallelism": f"{ws} independent batches (one per GPU)"},
        "pct_of_peak": 100.0 * value / peaks["bf16_tflops"],
        "roofline": {"kernel": "varlen_attn_fwd", "bound": "tensor",
                     "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     # context: the same launch against the power-capped
                     # sustained GEMM rate (back-to-back steps run the GPU
                     # at its power limit; the headline fraction is the
                     # burst one above)
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "launch_ms": attn_mean_ms, "traffic": prof.get("dram_bytes_per_launch"),
                     "ncu": {"tensor_pipe_active_pct": prof.get("tensor_pipe_active_pct"),
                             "dram_gbs": prof.get("dram_gbs"),
                             "source": f"profiles/varlen_attn_{name}.md"} if prof else None,
                     "kernel_digest": digest},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean,
                "how": "each sequence's real q/k/v rows from pinned host memory into the padded "
                       "device layout, step, real output rows back to pinned host memory; "
                       "copy-in/compute/copy-out on three streams, double-buffered, all K "
                       "steps inside the timed region (the first copy-in and the last "
                       "copy-out included)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    return res, pw


def run_ours(args):
    import packed_varlen_gb300 as pv

    ws, rank, local = _dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pv.load_library()
    pv.get_device_status()
    flusher = L2Flusher(dev)
    stream = torch.cuda.current_stream()
    no_cpu = args.no_cpu_baseline

    head, _ = measure_varlen_config(pv, WORKLOAD, dev, args, flusher, rank, dist, ws,
                                    None if no_cpu else CPU_ROWS[WORKLOAD])
    torch.cuda.empty_cache()
    # the other two large varlen configs, one GPU only (each a bench-line
    # object of its own; the scaling runs time the headline alone)
    subs = {}
    if ws == 1:
        for name in SUB_WORKLOADS:
            subs[name], _ = measure_varlen_config(pv, name, dev, args, flusher, rank, None, 1,
                                                  None if no_cpu else CPU_ROWS[name])
            torch.cuda.empty_cache()

    # ---- block-window variants (Token2Wav), timed per layer ------------------
    bw_meas = measure_block_window(pv, workloads.token2wav(), False, dev, flusher, stream)
    bw32_meas = measure_block_window(pv, workloads.token2wav_f32(), True, dev, flusher, stream)
    bw_meas["graph"] = measure_block_window_graph(pv, workloads.token2wav(), False, dev, flusher)
    bw32_meas["graph"] = measure_block_window_graph(pv, workloads.token2wav_f32(), True, dev,
                                                    flusher)
    if pv.get_device_status() != 0:
        raise RuntimeError("device status error during the block-window runs")
    cfg_meas = measure_cfg_combine(dev, 3072, 10, 3)
    rope_meas = measure_rope(dev, 10, 3)
    linear_meas = measure_linear(dev, 10, 3)

    peaks, _ = _peaks()
    if rank == 0:
        result = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": head["config"],
            "pct_of_peak": head["pct_of_peak"],
            "roofline": head["roofline"],
            "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "configs": subs,
            "block_window": dict(bw_meas, hbm_frac_own_block_layer=bw_meas["gbs_own_block_layer"]
                                 / peaks["hbm_gbs"],
                                 hbm_frac_graph=bw_meas["graph"]["gbs"] / peaks["hbm_gbs"]),
            "block_window_f32": dict(bw32_meas,
                                     hbm_frac_own_block_layer=bw32_meas["gbs_own_block_layer"]
                                     / peaks["hbm_gbs"],
                                     alu={"bound": "alu", "peak": FP32_PEAK_TFLOPS,
                                          "unit": "TFLOP/s",
                                          "achieved_neighbour_layer": bw32_meas["tflops_1_1"],
                                          "frac": bw32_meas["tflops_1_1"] / FP32_PEAK_TFLOPS,
                                          "peak_source": "152 SMs x 128 FP32 lanes x 2 FLOP "
                                                         "x 2.07 GHz"}),
            "cfg_combine": cfg_meas,
            "rope": rope_meas,
            "linear": linear_meas,
        }
        print(json.dumps(result), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_attn_only(args):
    """Attention kernel alone on one workload (for profiling runs): W + K
    launches on resident inputs, L2 flushed between launches."""
    import packed_varlen_gb300 as pv
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pv.load_library()
    pv.get_device_status()
    if args.workload in ("token2wav", "token2wav_f32"):
        return run_block_window_only(args, dev)
    if args.workload.startswith("cfg_combine"):
        return run_cfg_combine_only(args, dev)
    if args.workload in ("linear_qkv", "linear_out"):
        return run_linear_only(args, dev)
    if args.workload == "rope":
        print(json.dumps(measure_rope(dev, args.steps, args.warmup)), flush=True)
        return 0
    if args.workload in workloads.VARLEN_CONFIGS:
        w = workloads.VARLEN_CONFIGS[args.workload]()
    else:
        n = int(args.workload.split("_")[-1].rstrip("k")) * 1024
        w = workloads.random_varlen([n], None, 24, 128, seed=n, name=args.workload)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    cu = pv.cu_seqlens_from_lengths(torch.tensor(w.lengths_q, dtype=torch.int32, device=dev))
    out = torch.empty_like(q)
    flusher = L2Flusher(dev)
    flops = 4 * w.H * w.D * sum(a * b for a, b in zip(w.lengths_q, w.lengths_k))
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        pv.varlen_attn_fwd(q, k, v, cu, cu, max(w.lengths_q), max(w.lengths_k), out=out)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pv.varlen_attn_fwd(q, k, v, cu, cu, max(w.lengths_q), max(w.lengths_k), out=out)
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    if pv.get_device_status() != 0:
        raise RuntimeError("device status error")
    ms = statistics.median(a.elapsed_time(b) for a, b in ts)
    print(json.dumps({"workload": w.name, "lengths": w.lengths_q, "H": w.H, "D": w.D,
                      "attn_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}), flush=True)
    return 0


def run_e2e(pv, pw, dev, scale, steps, want_out):
    """The same step through the public API with host buffers, pipelined the
    way a serving loop would run it: each step copies every sequence's real
    q/k/v rows (what a request holds; the pack step never reads padding rows)
    from pinned host memory into the padded device layout, computes, and
    copies the real output rows back to pinned host memory.  Copy-in,
    compute and copy-out run on three streams with double-buffered device
    and output buffers, so step i+1's copy-in overlaps step i's compute.
    Returns (ms per step, H2D bytes per step, D2H bytes per step); the timed
    region spans all steps' copies."""
    L = pw.lengths
    B, S, H, D = len(L), pw.s_max, pw.H, pw.D
    row = H * D * 2
    T = sum(L)
    # per request: its own pinned [L_b, H, D] q, k, v (read-only, shared by
    # both pipeline buffers) and two pinned output buffers
    host_in = [[t[j, :L[j]].pin_memory() for j in range(B)] for t in (pw.q, pw.k, pw.v)]
    host_len = torch.tensor(L, dtype=torch.int32).pin_memory()
    host_out = [[torch.empty((L[j], H, D), dtype=torch.bfloat16).pin_memory() for j in range(B)]
                for _ in range(2)]
    dev_in = [[torch.zeros((B, S, H, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
              for _ in range(2)]
    dev_len = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
    dev_out = [torch.zeros((B, S, H, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    cu = [torch.empty(B + 1, dtype=torch.int32, device=dev) for _ in range(2)]
    flat = [[torch.empty((T, H, D), dtype=torch.bfloat16, device=dev) for _ in range(4)]
            for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    h2d = 3 * T * row + B * 4
    d2h = T * row

    def one(i, first):
        b = i % 2
        with torch.cuda.stream(s_in):
            if not first[b]:
                s_in.wait_event(ev_cmp[b])     # device inputs b free again
            dev_len[b].copy_(host_len, non_blocking=True)
            for t in range(3):
                for j in range(B):
                    dev_in[b][t][j, :L[j]].copy_(host_in[t][j], non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[b])
            if not first[b]:
                s_cmp.wait_event(ev_out[b])    # device output b read back already
            pv.cu_seqlens_from_lengths(dev_len[b], out=cu[b], stream=s_cmp)
            for t in range(3):
                pv.pack(dev_in[b][t], cu[b], T, out=flat[b][t], stream=s_cmp)
            pv.varlen_attn_fwd(flat[b][0], flat[b][1], flat[b][2], cu[b], cu[b], max(L), max(L),
                               scale=scale, out=flat[b][3], stream=s_cmp)
            pv.unpack(flat[b][3], cu[b], dev_out[b], stream=s_cmp)
            ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            for j in range(B):
                host_out[b][j].copy_(dev_out[b][j, :L[j]], non_blocking=True)
            ev_out[b].record(s_out)
        first[b] = False

    first = [True, True]
    for i in range(2):
        one(i, first)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        one(i, first)
    torch.cuda.current_stream(dev).wait_stream(s_out)
    e1.record(s_out)
    torch.cuda.synchronize()
    # the pipelined path must reproduce the plain step's output bit for bit
    got = host_out[(steps - 1) % 2]
    for j in range(B):
        if not torch.equal(got[j].view(torch.int16), want_out[j, :L[j]].view(torch.int16)):
            raise RuntimeError("pipelined end-to-end output differs from the device step")
    return e0.elapsed_time(e1) / steps, h2d, d2h


def measure_cfg_combine(dev, C, steps, warmup):
    """Segment-aware unpack + CFG combine alone on the CFG batch's layout with
    rows of C channels (64: latent channels, 3072: 24 x 128 attention output).
    Returns us per launch and HBM GB/s of the algorithmic bytes (positive and
    negative image rows read once, output rows written once)."""
    import packed_varlen_gb300 as pv
    seg = workloads.cfg_segments(C=C)
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=dev)
    cu = pv.cu_seqlens_from_lengths(i32(seg.lengths))
    flat = seg.flat.to(dev)
    args_t = (i32(seg.text), i32(seg.pos_seq), i32(seg.neg_seq),
              torch.tensor(seg.cfg_scale, device=dev), i32(seg.cfg_normalize))
    out = torch.zeros((len(seg.pos_seq), seg.img_max, C), dtype=torch.bfloat16, device=dev)
    n_img = [seg.lengths[p] - seg.text[p] for p in seg.pos_seq]
    nbytes = sum(n * C * 2 * (3 if q >= 0 else 2) for n, q in zip(n_img, seg.neg_seq))
    flusher = L2Flusher(dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        pv.cfg_combine(flat, cu, *args_t, seg.img_max, out=out)
    ts = []
    for _ in range(steps):
        flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pv.cfg_combine(flat, cu, *args_t, seg.img_max, out=out)
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    if pv.get_device_status() != 0:
        raise RuntimeError("device status error")
    us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ts)
    peaks, src = _peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"cfg dynamic batch, {len(n_img)} requests x (positive, negative), "
                        f"rows of {C} bf16", "image_rows": sum(n_img), "bytes": nbytes,
            "us": us, "gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"], "peak_source": src}


def measure_rope(dev, steps, warmup):
    """Request-local RoPE alone on the mixed-resolution batch's q and k (in
    place).  Algorithmic bytes: q and k read once and written once."""
    import packed_varlen_gb300 as pv
    w = workloads.mixed_res()
    q, k = w.q.to(dev), w.k.to(dev)
    cu = pv.cu_seqlens_from_lengths(torch.tensor(w.lengths_q, dtype=torch.int32, device=dev))
    nbytes = 2 * 2 * q.numel() * 2
    flusher = L2Flusher(dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        pv.rope_packed(q, k, cu, cu)
    ts = []
    for _ in range(steps):
        flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pv.rope_packed(q, k, cu, cu)
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    if pv.get_device_status() != 0:
        raise RuntimeError("device status error")
    us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ts)
    peaks, src = _peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": "mixed-resolution batch q and k, T=%d, H=24, D=128, in place" % q.shape[0],
            "bytes": nbytes, "us": us, "gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
            "peak_source": src}


def measure_linear(dev, steps, warmup, kinds=("qkv", "out")):
    """The batch-invariant packed-M projections of the mixed-resolution batch
    (x [T, 3072] times the fused QKV or the output weight, with bias), each
    launch after an L2 flush.  cuBLAS (torch's linear, not batch invariant)
    is timed on the same operands for context."""
    import packed_varlen_gb300 as pv
    peaks, src = _peaks()
    flusher = L2Flusher(dev)
    stream = torch.cuda.current_stream()
    res = {}
    for kind in kinds:
        w = workloads.mmdit_projection(kind)
        x, wt, b = w.x.to(dev), w.w.to(dev), w.bias.to(dev)
        y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
        flops = 2 * w.M * w.N * w.K

        def timed(fn):
            for _ in range(warmup):
                fn()
            ts = []
            for _ in range(steps):
                flusher.flush()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ts.append((e0, e1))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(c) for a, c in ts)

        ms = timed(lambda: pv.linear_bf16(x, wt, b, out=y))
        ms_cublas = timed(lambda: torch.nn.functional.linear(x, wt, b))
        if pv.get_device_status() != 0:
            raise RuntimeError("device status error")
        tf = flops / (ms * 1e-3) / 1e12
        res[kind] = {"workload": f"{w.name}: M={w.M} (requests {w.lengths}), N={w.N}, K={w.K}",
                     "flops": flops, "us": 1e3 * ms, "tflops": tf,
                     "frac": tf / peaks["bf16_tflops"], "peak_source": f"{src} bf16 dense (burst)",
                     "cublas_us": 1e3 * ms_cublas,
                     "cublas_tflops": flops / (ms_cublas * 1e-3) / 1e12}
    return res


def run_linear_only(args, dev):
    kind = args.workload.split("_", 1)[1]
    print(json.dumps(dict(measure_linear(dev, args.steps, args.warmup, kinds=(kind,)),
                          workload_name=args.workload)), flush=True)
    return 0


def measure_block_window(pv, bw, f32, dev, flusher, stream, reps=20):
    """Median time of each Token2Wav layer type with a clean L2 before every
    launch; bytes = q, k, v read once and out written once."""
    fn = pv.block_window_attn_fwd_f32 if f32 else pv.block_window_attn_fwd
    bq, bk, bv = bw.q.to(dev), bw.k.to(dev), bw.v.to(dev)
    bo = torch.empty_like(bq)
    for _ in range(3):
        for lb, la in bw.layers:
            fn(bq, bk, bv, bw.block, lb, la, out=bo)
    torch.cuda.synchronize()
    per_layer = {}
    for lb, la in sorted(set(bw.layers)):
        ts = []
        for _ in range(reps):
            flusher.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(bq, bk, bv, bw.block, lb, la, out=bo)
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        per_layer[(lb, la)] = statistics.median(a.elapsed_time(b) for a, b in ts)
    nbytes = 4 * bq.numel() * bq.element_size()
    total_us = sum(per_layer[l] for l in bw.layers) * 1e3
    flops = sum(block_window_flops(bw.n, bw.H, bw.D, bw.block, lb, la) * bw.batch
                for lb, la in bw.layers)
    n_own = sum(1 for l in bw.layers if l == (0, 0))
    t11 = block_window_flops(bw.n, bw.H, bw.D, bw.block, 1, 1) * bw.batch / (
        per_layer[(1, 1)] * 1e-3) / 1e12 if (1, 1) in per_layer else None
    return {
        "tflops_1_1": t11,
        "workload": f"token2wav {'fp32' if f32 else 'bf16'} batch={bw.batch} n={bw.n} "
                    f"H={bw.H} D={bw.D} block={bw.block}, {n_own} x (0,0) + "
                    f"{len(bw.layers) - n_own} x (1,1) layers",
        "us_per_layer": {f"{lb},{la}": 1e3 * ms for (lb, la), ms in per_layer.items()},
        "us_all_layers": total_us,
        "bytes_per_layer": nbytes,
        "gbs_own_block_layer": nbytes / (per_layer[(0, 0)] * 1e-3) / 1e9,
        "useful_tflops": flops / (total_us * 1e-6) / 1e12,
        "launches": len(bw.layers)}


def measure_block_window_graph(pv, bw, f32, dev, flusher, reps=10):
    """The 22 Token2Wav layers as one CUDA graph, each layer on its own q, k,
    v and out (22 x the layer's bytes, more than L2), the way the layers run
    inside the model: no per-launch host gaps or events between layers.  L2
    is emptied before each replay, outside the events."""
    fn = pv.block_window_attn_fwd_f32 if f32 else pv.block_window_attn_fwd
    n_layers = len(bw.layers)
    qs = [bw.q.to(dev) for _ in range(n_layers)]
    ks = [bw.k.to(dev) for _ in range(n_layers)]
    vs = [bw.v.to(dev) for _ in range(n_layers)]
    outs = [torch.empty_like(qs[0]) for _ in range(n_layers)]
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for i, (lb, la) in enumerate(bw.layers):   # warm-up outside the capture
            fn(qs[i], ks[i], vs[i], bw.block, lb, la, out=outs[i])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i, (lb, la) in enumerate(bw.layers):
            fn(qs[i], ks[i], vs[i], bw.block, lb, la, out=outs[i])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(reps):
        flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ts)
    nbytes = 4 * qs[0].numel() * qs[0].element_size()
    return {"us_all_layers": us, "us_per_layer": us / n_layers,
            "gbs": n_layers * nbytes / (us * 1e-6) / 1e9,
            "how": f"{n_layers} layers captured in one CUDA graph, each on its own "
                   f"q/k/v/out ({n_layers * nbytes / 2**20:.0f} MB in all), L2 emptied "
                   "before each replay"}


def run_cfg_combine_only(args, dev):
    C = 3072 if args.workload.endswith("3072") else 64
    print(json.dumps(dict(measure_cfg_combine(dev, C, args.steps, args.warmup),
                          workload_name=args.workload)), flush=True)
    return 0


def run_block_window_only(args, dev):
    """Block-window layers alone (profiling): median us per layer type with a
    clean L2 before each launch, and a one-CTA kernel for the launch floor."""
    import packed_varlen_gb300 as pv
    f32 = args.workload == "token2wav_f32"
    bw = workloads.token2wav_f32() if f32 else workloads.token2wav()
    fwd = pv.block_window_attn_fwd_f32 if f32 else pv.block_window_attn_fwd
    bq, bk, bv = bw.q.to(dev), bw.k.to(dev), bw.v.to(dev)
    bo = torch.empty_like(bq)
    flusher = L2Flusher(dev)
    stream = torch.cuda.current_stream()
    lens = torch.tensor([5, 7], dtype=torch.int32, device=dev)
    cu = torch.empty(3, dtype=torch.int32, device=dev)
    res = {}
    cases = [("0,0", lambda: fwd(bq, bk, bv, 24, 0, 0, out=bo)),
             ("1,1", lambda: fwd(bq, bk, bv, 24, 1, 1, out=bo)),
             ("floor", lambda: pv.cu_seqlens_from_lengths(lens, out=cu))]
    for name, fn in cases:
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flusher.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        res[name] = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ts)
    print(json.dumps({"workload": args.workload, "us": res}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="query rows per sequence per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attn-only", action="store_true",
                    help="time the attention kernel alone (profiling); not the bench line")
    ap.add_argument("--workload", default="single_8k",
                    help="with --attn-only: a varlen config name, single_<N>k, token2wav, token2wav_f32, "
                         "linear_qkv, linear_out, "
                         "cfg_combine, cfg_combine_3072 or rope")
    args = ap.parse_args()
    if args.attn_only:
        return run_attn_only(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
