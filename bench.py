"""Benchmark of the fused chunked linear + cross-entropy forward+backward.

One step = one lce_fwd_bwd call (label scan, per-chunk logits GEMM with the
log-sum-exp epilogue, slab merge + G rescale, dH/dW GEMM tiles, loss) over the
Llama-3-8B-shaped LM head: N=16384 tokens, D=4096, V=128256, chunk 1024, 5% of
rows ignore_index, synthetic seeded inputs (no dataset).

Prints one JSON line (rank 0). With --impl reference the fp64 CPU oracle is
timed instead on the host cores, one bounded row sample per step. Other
measurements: --frozen-w (the LM head frozen: no dW, 4NDV per step),
--dtype fp16, --workload / --chunk (the other head shapes and chunk sizes),
--path ce-logits (cross-entropy over given logits), --path norm (final RMSNorm
+ head + cross-entropy).

Multi-GPU (torchrun, --gpus N): every rank runs its own replica of the
workload (independent problems, weak scaling, no collective on the data path);
`value` is the tokens of all ranks over the slowest rank's time.
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

METRIC = "LCE fwd+bwd tokens/s at N=16384,D=4096,V=128256; % of bf16 tensor peak"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3-8b")
    ap.add_argument("--chunk", type=int, default=0, help="0: the workload's own chunk")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cublas", action="store_true",
                    help="skip the cuBLAS timing of the same GEMM shapes (after the timed region)")
    ap.add_argument("--ce-rows", type=int, default=0,
                    help="ce-logits path: rows of the logits (0: the workload's N)")
    ap.add_argument("--frozen-w", action="store_true",
                    help="fused path with W frozen (LCE_FROZEN_W: no dW, 4NDV per step), the "
                         "LoRA / QLoRA setting; the headline trains W")
    ap.add_argument("--low-memory", action="store_true",
                    help="one chunk buffer (LCE_LOW_MEMORY): no overlap of a chunk's logits GEMM "
                         "with the previous chunk's gradient GEMMs, about half the workspace")
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16",
                    help="H and W dtype of the fused path (the headline is bf16)")
    ap.add_argument("--path", choices=["fused", "separate", "ce-logits", "norm"], default="fused",
                    help="fused: the LM-head linear + CE forward+backward (the headline); "
                         "separate: lce_forward, then lce_backward recomputing the logits from the "
                         "saved lse (8NDV executed); "
                         "ce-logits: the CE over precomputed bf16 logits of the same workload "
                         "(gradient in place); norm: final RMSNorm + LM head + CE forward and "
                         "backward into the pre-norm hidden state (lce_norm_fwd_bwd)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """Slowest rank's time: all-reduce(MAX) when more than one rank runs."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of the SM clock, power and throttle reasons (every 100 ms)
    around the timed region. start() returns once the first sample has arrived, so
    the timed region is covered; the reported SM clock is the median over the
    samples taken under load (power at least 60 % of the highest sample)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int = 0):
        self.proc = None
        self.lines = []
        self.reader = None
        self.dev = device_index

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def start(self):
        import threading
        import torch
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
        except Exception:
            uuid = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            self.proc.wait()
        if self.reader:
            self.reader.join(timeout=5)
        rows = []
        smax = None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            rows.append((sm, pw, [nm for nm, v in zip(names, parts[4:8])
                                  if v.lower().startswith("active")]))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": smax, "samples": 0, "reasons": []}
        pmax = max(r[1] for r in rows)
        load = [r for r in rows if r[1] >= 0.6 * pmax]
        reasons = sorted({nm for r in load for nm in r[2]})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": smax,
                "power_w_max": pmax, "samples": len(rows), "samples_under_load": len(load),
                "reasons": reasons}


# ----------------------------------------------------------------- reference arm

def oracle_sample_rate(wl, rows: int, H64, W64, y):
    """Time the fp64 oracle's forward+backward over the first `rows` tokens."""
    from oracle import lce_oracle
    t0 = time.perf_counter()
    lce_oracle.forward_backward(H64[:rows], W64, y[:rows])
    return time.perf_counter() - t0


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def prepare_oracle_inputs(wl):
    import numpy as np
    from lce_synth import workload_inputs
    H, W, y = workload_inputs(wl)
    import torch
    return (H.to(torch.float64).numpy(), W.to(torch.float64).numpy(),
            y.numpy().astype(np.int64))


def calibrate_rows(wl, H64, W64, y, target_s: float) -> int:
    """Rows of the workload the oracle processes in about target_s seconds (the
    cost is linear in rows; the pilot is large enough for BLAS to be efficient)."""
    rows = min(wl.N, 128)
    t = oracle_sample_rate(wl, rows, H64, W64, y)
    want = int(rows * target_s / max(t, 1e-3))
    return max(16, min(wl.N, want))


def run_reference(args, wl, chunk):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    H64, W64, y = prepare_oracle_inputs(wl)
    rows = calibrate_rows(wl, H64, W64, y, target_s=2.0)
    for _ in range(args.warmup):
        oracle_sample_rate(wl, rows, H64, W64, y)
    times = [oracle_sample_rate(wl, rows, H64, W64, y) for _ in range(args.steps)]
    total = sum(times)
    value = rows * args.steps / total
    flops = 6.0 * wl.D * wl.V * rows
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, chunk, l2="host CPU run"),
        "tflops": flops * args.steps / total / 1e12,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(),
                         "kind": "oracle",
                         "sample": f"first {rows} of {wl.N} tokens of the workload per step "
                                   f"(fp64 numpy forward+backward incl. the full dW)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm

def workload_config(wl, chunk, l2, **extra):
    return {"workload": f"{wl.name} LM head N={wl.N} D={wl.D} V={wl.V} chunk={chunk}",
            "N": wl.N, "D": wl.D, "V": wl.V, "chunk": chunk,
            "ignored_rows": wl.n_ignored, "labels": wl.labels, "seed": wl.seed,
            "global_batch_tokens": wl.N, "l2": l2, "parallelism": "replicas", **extra}


def run_ours(args, wl, chunk):
    import torch
    import torch.distributed as dist

    import linear_cross_entropy_chunked_gb300 as lce
    from lce_synth import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    lce.build()
    peaks, peak_src = load_peaks()

    # inputs (each rank its own replica, seed offset by rank)
    H, W, y = make_inputs(wl.N, wl.D, wl.V, wl.seed + 1000 * rank, wl.labels, wl.n_ignored,
                          dtype=args.dtype)
    Hd, Wd, yd = H.to(dev), W.to(dev), y.to(dev)
    N, D, V = wl.N, wl.D, wl.V
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    mem0 = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    frozen = bool(args.frozen_w)
    low = bool(args.low_memory)
    ws_flags = (lce.FROZEN_W if frozen else 0) | (lce.LOW_MEMORY if low else 0)
    ws = lce.alloc_workspace(N, D, V, chunk, dev, ws_flags)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dH = torch.empty(N, D, dtype=Hd.dtype, device=dev)
    dW = None if frozen else torch.empty(V, D, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    separate = args.path == "separate"

    def step():
        if separate:
            lce.lce_forward(Hd, Wd, yd, chunk=chunk, loss=loss, lse=lse, ws=ws, stream=stream)
            lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, dH=dH, dW=dW, ws=ws, stream=stream,
                             compute_dW=not frozen, low_memory=low)
        else:
            lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, loss=loss, lse=lse, dH=dH, dW=dW, ws=ws,
                            stream=stream, compute_dW=not frozen, low_memory=low)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    st = lce.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    launches_per_step = lce.last_launch_count()
    extra_bytes = torch.cuda.max_memory_allocated(dev) - mem0 - (
        lse.numel() * 4 + dH.numel() * 2 + (0 if frozen else dW.numel() * 4) + 4)

    # ---- timed region: per-step CUDA events, L2 flushed between steps
    lce.profile_reset()
    lce.profile_enable(True)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_wall0 = time.perf_counter()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    lce.profile_enable(False)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)
    grad_ms, grad_n = lce.profile_read("grad")
    phase_ms, phase_n = lce.profile_read("phase")
    dh_ms, dh_n = lce.profile_read("dh")
    logit_ms, logit_n = lce.profile_read("logits")
    merge_ms, merge_n = lce.profile_read("merge")
    st = lce.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after timed steps")
    total_ms = max_over_ranks(total_ms, world, dev)

    ms_per_step = total_ms / args.steps
    tokens_per_s = job_tokens_per_s(world, N, args.steps, total_ms)
    flops_step = (4.0 if frozen else 6.0) * N * D * V
    tflops = flops_step / (ms_per_step / 1e3) / 1e12
    peak_burst = peaks.get("bf16_tflops", 1900.0)
    peak_sust = peaks.get("bf16_tflops_sustained", 1700.0)

    # dominant kernel. With two chunk buffers (the default) the chunks go in pairs
    # and it is the second chunk's gradient phase: its dH GEMM beside one dW
    # contraction over both chunks of the pair (one dW grid beside the dH kernel,
    # one behind it), timed together from fork to join: 6*C*D*V flops (2 for the
    # dH, 4 for the dW over 2C rows). The first chunk's dH GEMM runs beside the
    # second chunk's logits GEMM (kind "dh", 4*C*D*V), the first chunk's logits GEMM
    # alone (kind "logits"). With one buffer (or W frozen) it is a chunk's gradient phase:
    # the dH GEMM and the dW grids, 4*C*D*V flops (W frozen: the dH GEMM alone,
    # 2*C*D*V).
    nchunks = (N + chunk - 1) // chunk
    cdv = float(D) * V * N / nchunks
    overlapped = phase_n > 0
    if frozen and dh_n > 0:
        # W frozen, two chunk buffers: chunk k's dH GEMM with chunk k+1's logits GEMM
        # on the pairs it leaves free (4*C*D*V: 2 each)
        dom_ms, dom_n, dom_flops = dh_ms, dh_n, 4.0 * cdv
        dom_name = ("W frozen: lce_gemm_kernel<MODE_DH> (dH tiles of chunk k, 512 wide, split along "
                    "the vocabulary) beside lce_gemm_kernel<MODE_LSE_P> (logits tiles of chunk k+1: "
                    "one grid on the pairs the dH kernel leaves free, one behind it)")
    elif overlapped:
        dom_ms, dom_n, dom_flops = phase_ms, phase_n, 6.0 * cdv
        dom_name = ("gradient phase of the second chunk of a pair: lce_gemm_kernel<MODE_DH> (its "
                    "dH tiles, 512 wide) beside lce_gemm_kernel<MODE_BWD> (the dW tiles of both "
                    "chunks, K = 2 chunks: one grid beside the dH kernel, one behind it)")
    else:
        dom_ms, dom_n, dom_flops = grad_ms, grad_n, (2.0 if frozen else 4.0) * cdv
        dom_name = ("gradient phase, W frozen: lce_gemm_kernel<MODE_DH> (dH tiles, 512 wide, split "
                    "along the vocabulary) alone" if frozen else
                    "gradient phase: lce_gemm_kernel<MODE_DH> (dH tiles, 512 wide) + "
                    "lce_gemm_kernel<MODE_BWD> (dW tiles: one grid beside the dH kernel, one "
                    "behind it), concurrent")
    dom_avg_ms = dom_ms / max(dom_n, 1)
    dom_tflops = dom_flops / (dom_avg_ms / 1e3) / 1e12
    grad_avg_ms = grad_ms / max(grad_n, 1)
    grad_tflops = (2.0 if frozen else 4.0) * cdv / (grad_avg_ms / 1e3) / 1e12 if grad_n else None
    logit_avg_ms = logit_ms / max(logit_n, 1)
    logit_tflops = 2.0 * cdv / (logit_avg_ms / 1e3) / 1e12 if logit_n else None
    variant = "+".join(x for x in (("fp16" if args.dtype == "fp16" else ""),
                                   ("frozen_w" if frozen else ""), ("low_memory" if low else ""),
                                   ("separate" if separate else "")) if x)
    traffic = load_traffic(wl.name, chunk, variant)
    dom_traffic = traffic.get("phase" if overlapped else ("grad_frozen" if frozen else "grad"))
    # algorithmic bytes of the method (the minimum it must move) per step: read H, W
    # and y, write lse, dH and dW (fp32); a launch of the dominant kernel carries the
    # share of them that its flops are of the step's (a pair's phase: 6 of a chunk
    # pair's 12 C*D*V; a chunk's gradient phase: 4 of its 6)
    alg_bytes_step = (N * D * 2 + V * D * 2 + N * 8 + N * 4 + N * D * 2 +
                      (0 if frozen else V * D * 4))
    alg_bytes_launch = alg_bytes_step * dom_flops / flops_step
    # softmax / gather epilogue bytes of the fused path (beyond the GEMM operands):
    # P' written by the logits epilogue, then read and rewritten in place as G by the
    # prep kernel (3 x N x V x 2 B); the (max, sum) slab partials written and read
    # (2 x N x ceil(V/128) x 8 B, read once per 16384-column segment of a row:
    # L2-resident); target logits and lse (N x 12 B)
    elem = 2
    epi_bytes = 3.0 * N * V * elem + 2.0 * N * ((V + 127) // 128) * 8 + 12.0 * N
    merge_ms_step = merge_ms / args.steps
    sm_peak_clk = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e and not separate:
        e2e = run_e2e(args, lce, H, W, y, chunk, dev, stream, world, frozen, low=low)
        w_up = run_e2e(args, lce, H, W, y, chunk, dev, stream, world, frozen, upload_w=True,
                       low=low)
        e2e["with_weight_upload"] = {k: w_up[k] for k in (
            "value", "ms_per_step", "h2d_bytes_per_step", "h2d_ms_per_step_alone",
            "h2d_ms_per_step_under_load", "compute_ms_per_step_under_load")}
        dh_back = run_e2e(args, lce, H, W, y, chunk, dev, stream, world, frozen, low=low,
                          read_dh=True)
        e2e["with_dh_readback"] = {k: dh_back[k] for k in (
            "value", "ms_per_step", "h2d_bytes_per_step", "d2h_bytes_per_step",
            "compute_ms_per_step_under_load", "note")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
    cublas = None
    if world == 1 and not args.no_cublas and not separate and not frozen:
        cublas = cublas_same_shapes(Hd, Wd, chunk, stream)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "ms_per_step_median": statistics.median(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": args.dtype, "data": "synthetic",
            "config": workload_config(wl, chunk,
                                      l2="L2 flushed between steps (256 MB write); "
                                         "W 1.05 GB also exceeds L2",
                                      **({"frozen_w": True} if frozen else {}),
                                      **({"path": "lce_forward + lce_backward"} if separate
                                         else {}),
                                      chunk_buffers=1 if (low or frozen or nchunks == 1) else 2),
            "tflops": tflops,
            "flops_per_step": {"algorithmic": flops_step,
                               "executed": flops_step * (8.0 / 6.0 if separate and not frozen else
                                                         (6.0 / 4.0 if separate else 1.0)),
                               "note": ("lce_forward + lce_backward: the backward recomputes the "
                                        "logits (2NDV more)") if separate else
                                       "the fused call recomputes nothing: executed = algorithmic "
                                       "(lce_forward + lce_backward would execute 8NDV)"},
            "pct_of_bf16_peak": {"vs_burst": tflops / peak_burst, "vs_sustained": tflops / peak_sust,
                                 "flops": "4NDV algorithmic (W frozen: no dW)" if frozen
                                 else "6NDV algorithmic", "peak_source": peak_src},
            "peak_extra_hbm_bytes": int(extra_bytes),
            "workspace_bytes": int(ws.numel()),
            "roofline": {"kernel": dom_name, "bound": "tensor", "achieved": dom_tflops,
                         "peak": peak_burst,
                         "peak_kind": f"bf16_tflops, burst ({peak_src}; the launch is timed "
                                      f"inside the step, not alone: see frac_vs_sustained)",
                         "unit": "TFLOP/s", "frac": dom_tflops / peak_burst,
                         "peak_sustained": peak_sust, "frac_vs_sustained": dom_tflops / peak_sust,
                         "sm_mhz_median": {"this_run": clk.get("sm_mhz"),
                                           "peak_measurement": sm_peak_clk},
                         "traffic": dom_traffic,
                         "alg_bytes_per_launch": alg_bytes_launch,
                         "traffic_over_alg_bytes": (dom_traffic / alg_bytes_launch
                                                    if dom_traffic else None),
                         "alg_bytes_note": "the method's algorithmic bytes per step (read H, W, "
                                           "y; write lse, dH, dW fp32) x the launch's share of "
                                           "the step's flops",
                         "launch_ms": dom_avg_ms, "launches": dom_n,
                         "flops_per_launch": dom_flops},
            "kernels": {
                "phase": {"ms_per_launch": phase_ms / max(phase_n, 1), "launches": phase_n,
                          "tflops": dom_tflops if overlapped else None,
                          "share": phase_ms / total_ms},
                "grad": {"ms_per_launch": grad_avg_ms, "launches": grad_n,
                         "tflops": grad_tflops, "share": grad_ms / total_ms},
                "dh_with_next_logits": {"ms_per_launch": dh_ms / max(dh_n, 1), "launches": dh_n,
                                        "tflops": (4.0 * cdv / (dh_ms / max(dh_n, 1) / 1e3) / 1e12
                                                   if dh_n else None),
                                        "share": dh_ms / total_ms},
                "logits": {"ms_per_launch": logit_avg_ms, "launches": logit_n,
                           "tflops": logit_tflops, "share": logit_ms / total_ms},
                "prep": {"ms_per_launch": merge_ms / max(merge_n, 1), "launches": merge_n,
                         "share": merge_ms / total_ms},
            },
            "alg_bytes_per_step": alg_bytes_step,
            "epilogue": {"bytes_per_step": epi_bytes,
                         "what": "P' stored by the logits epilogue, read and rewritten in place "
                                 "as G by the prep kernel; slab (max, sum) partials written and "
                                 "read; target logits, lse, row losses",
                         "aux_kernels_ms_per_step": merge_ms_step,
                         "aux_kernels": "one prep launch per chunk: lse and row losses from the "
                                        "slab partials, P' -> G in place, H chunk transpose (the "
                                        "P' store itself runs inside the logits GEMM's epilogue)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "wall_s_timed_region": wall,
        }
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        if cublas:
            line["cublas_same_shapes"] = cublas
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def kernel_source_hash(files) -> str:
    """First 16 hex digits of the SHA-256 of the named csrc files, in order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_cross_entropy_chunked_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def cublas_same_shapes(Hd, Wd, chunk, stream, reps: int = 10):
    """cuBLAS (torch.matmul: bf16 or fp16 in and out) on the three GEMM shapes of a
    chunk pair, each timed alone with CUDA events after the timed region: the
    logits Z_c = H_c W^T (C x V, K = D), dH_c = G_c W (C x D, K = V) and dW = G^T H
    over a pair of chunks (V x D, K = 2C). A yardstick for the library's kernels,
    which do more on the same shapes (the logits kernel's slab LSE, target gather
    and P' store; the dW tiles' fp32 read-modify-write of dW) and run beside one
    another inside the step rather than alone."""
    import torch
    N, D = Hd.shape
    V = Wd.shape[0]
    C = min(chunk, N)
    C2 = min(2 * C, N)
    dev = Hd.device
    g = torch.Generator(device=dev).manual_seed(0)
    G = (torch.randn(C2, V, device=dev, generator=g) * 1e-4).to(Hd.dtype)
    Hc, H2 = Hd[:C], Hd[:C2]
    Z = torch.empty(C, V, dtype=Hd.dtype, device=dev)
    dHc = torch.empty(C, D, dtype=Hd.dtype, device=dev)
    dWb = torch.empty(V, D, dtype=Hd.dtype, device=dev)
    cases = {
        "logits": (lambda: torch.matmul(Hc, Wd.t(), out=Z), 2.0 * C * D * V,
                   f"[{C} x {D}] @ [{D} x {V}]"),
        "dH": (lambda: torch.matmul(G[:C], Wd, out=dHc), 2.0 * C * D * V,
               f"[{C} x {V}] @ [{V} x {D}]"),
        "dW": (lambda: torch.matmul(G.t(), H2, out=dWb), 2.0 * C2 * D * V,
               f"[{V} x {C2}] @ [{C2} x {D}]"),
    }
    # the library's dW output: fp32, added to the dW already there (beta = 1)
    dW32 = torch.zeros(V, D, dtype=torch.float32, device=dev)
    try:
        torch.addmm(dW32[:256], G.t()[:256], H2, out_dtype=torch.float32)
        cases["dW_fp32_accumulate"] = (
            lambda: torch.addmm(dW32, G.t(), H2, out_dtype=torch.float32), 2.0 * C2 * D * V,
            f"fp32 [{V} x {D}] + [{V} x {C2}] @ [{C2} x {D}]")
    except (TypeError, RuntimeError):
        pass
    out = {}
    with torch.cuda.stream(stream):
        for name, (fn, flops, shape) in cases.items():
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for a, b in evs:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize(dev)
            ms = statistics.median(a.elapsed_time(b) for a, b in evs)
            out[name] = {"shape": shape, "ms": ms, "tflops": flops / (ms / 1e3) / 1e12}
    del G, Z, dHc, dWb, dW32
    out["note"] = ("torch.matmul / addmm (cuBLAS) alone on each shape, bf16/fp16 output (the "
                   "dW_fp32_accumulate case: fp32 output added to an fp32 dW, as the library "
                   f"does), median of {reps}; the library's kernels on these shapes also run "
                   "their epilogues and share the GPU with each other inside the step (see "
                   "kernels)")
    return out


def load_traffic(workload: str = "", chunk: int = 0, variant: str = ""):
    """DRAM bytes per launch from the committed ncu summary, per kernel; a kernel is
    left out when its sources changed since the capture, when the capture was of
    another workload, chunk or variant of the path, or when the file is absent."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    out = {}
    for k, v in d.get("kernels", {}).items():
        if v.get("sha256_16") != kernel_source_hash(v.get("sources", [])):
            continue
        if workload and v.get("workload", workload) != workload:
            continue
        if chunk and v.get("chunk", chunk) != chunk:
            continue
        if v.get("variant", "") != variant:
            continue
        out[k] = v.get("dram_bytes_per_launch_bench")
    return out


def run_e2e(args, lce, H, W, y, chunk, dev, stream, world, frozen=False, upload_w=False,
            low=False, read_dh=False):
    """The same metric through the public API from pinned host buffers: every
    step copies its inputs host -> device and reads its loss back. The inputs
    of a loss step are the hidden states H and the labels y; the LM-head weight
    W is a parameter that stays on the device between steps (uploaded once,
    before the timed region), unless upload_w, which copies W every step too
    (the conservative variant). The copies of step k+1 run on a copy stream
    while step k computes (two device input buffers), as a training loop that
    prefetches its next batch would; the loss read-back runs on a third stream
    from one of two device loss slots, so a read-back queued behind a copy never
    holds up the next step. The timed region contains every step's copies and
    read-backs. read_dh: every step also reads its dH (N x D bf16) back to pinned
    host memory (from one of two device dH slots, on the read-back stream), as a
    caller whose next layer's backward runs elsewhere would."""
    import torch
    Hh, yh = H.pin_memory(), y.pin_memory()
    Wh = W.pin_memory() if upload_w else None
    W_dev = None if upload_w else W.to(dev)
    bufs = [(torch.empty_like(Hh, device=dev),
             torch.empty_like(Wh, device=dev) if upload_w else W_dev,
             torch.empty_like(yh, device=dev)) for _ in range(2)]
    N, D = H.shape
    V = W.shape[0]
    ws = lce.alloc_workspace(N, D, V, chunk, dev, (lce.FROZEN_W if frozen else 0) |
                             (lce.LOW_MEMORY if low else 0))
    loss_h = torch.empty(2, dtype=torch.float32).pin_memory()
    loss_slots = torch.empty(2, 4, dtype=torch.float32, device=dev)   # 16-byte aligned slots
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dH_slots = [torch.empty(N, D, dtype=H.dtype, device=dev) for _ in range(2 if read_dh else 1)]
    dH_h = [torch.empty(N, D, dtype=H.dtype).pin_memory() for _ in range(2)] if read_dh else None
    dW = None if frozen else torch.empty(V, D, dtype=torch.float32, device=dev)
    copy_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]

    # (start, end) events of every step's copies and compute: how long each took
    # under load, and whether the copies stayed hidden behind the compute
    spans = {"copy": [], "compute": []}

    def timed():
        return torch.cuda.Event(enable_timing=True)

    def h2d(k):
        b = bufs[k % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[k % 2])   # the step that last read this buffer
            e0, e1 = timed(), timed()
            e0.record(copy_stream)
            b[0].copy_(Hh, non_blocking=True)
            if upload_w:
                b[1].copy_(Wh, non_blocking=True)
            b[2].copy_(yh, non_blocking=True)
            e1.record(copy_stream)
            copied[k % 2].record(copy_stream)
        spans["copy"].append((e0, e1))

    def compute(k):
        b = bufs[k % 2]
        stream.wait_event(copied[k % 2])
        stream.wait_event(read_back[k % 2])   # this loss slot's last value has been read
        e0, e1 = timed(), timed()
        e0.record(stream)
        dH = dH_slots[k % len(dH_slots)]
        lce.lce_fwd_bwd(b[0], b[1], b[2], chunk=chunk, loss=loss_slots[k % 2, :1], lse=lse,
                        dH=dH, dW=dW, ws=ws, stream=stream, compute_dW=not frozen, low_memory=low)
        e1.record(stream)
        consumed[k % 2].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(consumed[k % 2])
            loss_h[k % 2].copy_(loss_slots[k % 2, 0], non_blocking=True)
            if read_dh:
                dH_h[k % 2].copy_(dH, non_blocking=True)
            read_back[k % 2].record(d2h_stream)
        spans["compute"].append((e0, e1))

    def run(steps):
        h2d(0)
        for k in range(steps):
            if k + 1 < steps:
                h2d(k + 1)
            compute(k)

    for ev in consumed + read_back:
        ev.record(stream)
    run(3)
    torch.cuda.synchronize(dev)
    # one step's copies alone (outside the timed region): the host link's rate on
    # this machine, which bounds E when the copies take longer than a step
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(copy_stream)
    h2d(0)
    c1.record(copy_stream)
    torch.cuda.synchronize(dev)
    copy_ms = c0.elapsed_time(c1)
    spans["copy"].clear()
    spans["compute"].clear()
    steps = max(3, args.steps // 2)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    a.record(stream)
    copy_stream.wait_event(a)        # the first step's copies start inside the timed region
    run(steps)
    stream.wait_event(read_back[(steps - 1) % 2])   # ... and the last loss is on the host
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b) / steps, world, dev)   # the slowest rank, as for value
    under_load = {k: statistics.mean(e0.elapsed_time(e1) for e0, e1 in v) for k, v in spans.items()}
    h2d_bytes = Hh.numel() * 2 + (Wh.numel() * 2 if upload_w else 0) + yh.numel() * 8
    d2h_bytes = 4 + (N * D * H.element_size() if read_dh else 0)
    return {"value": world * N / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": steps, "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "h2d_ms_per_step_alone": copy_ms, "h2d_gbs": h2d_bytes / copy_ms / 1e6,
            "h2d_ms_per_step_under_load": under_load["copy"],
            "compute_ms_per_step_under_load": under_load["compute"],
            "note": ("every step copies H, W and y" if upload_w else
                     "every step copies H and y (W, a parameter, stays resident)") +
                    " from pinned host memory (on a copy stream, overlapping the previous step's "
                    "compute) and reads its loss " + ("and its dH (N x D) " if read_dh else "") +
                    "back (on a third stream, from one of two device slots)" +
                    ("" if read_dh else "; dH and dW stay on the device, as in a training step")}


def run_ce_logits(args, wl):
    """Streaming cross-entropy over precomputed bf16 logits Z [N, V] (the tensor
    the pages say must not be materialised; here it is the input), forward +
    in-place gradient. HBM bound: algorithmic bytes = read Z + write dZ."""
    import torch
    import linear_cross_entropy_chunked_gb300 as lce
    rank, world, local = dist_env()
    dev = torch.device("cuda", torch.cuda.current_device())
    lce.build()
    peaks, peak_src = load_peaks()
    N, V = (args.ce_rows or wl.N), wl.V
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    Z = torch.randn(N, V, device=dev, generator=g).mul_(1.3).to(torch.bfloat16)
    yv = torch.randint(0, V, (N,), device=dev, generator=g)
    yv[torch.randperm(N, device=dev, generator=g)[:wl.n_ignored * N // wl.N]] = -100
    ws = torch.empty(1024 + 4 * N + 1024, dtype=torch.uint8, device=dev)
    loss = torch.empty(1, device=dev)
    lse = torch.empty(N, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        lce.ce_logits(Z, yv, inplace=True, loss=loss, lse=lse, ws=ws, stream=stream)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    lce.profile_reset()
    lce.profile_enable(True)
    for a, b in evs:
        a.record(stream)
        lce.ce_logits(Z, yv, inplace=True, loss=loss, lse=lse, ws=ws, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    lce.profile_enable(False)
    k_ms, k_n = lce.profile_read("merge")
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    kernel_ms = k_ms / max(k_n, 1)
    alg_bytes = 2.0 * N * V * 2
    gbs = alg_bytes / (kernel_ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "CE over precomputed bf16 logits, forward + in-place gradient, tokens/s",
        "value": world * N / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{wl.name} logits N={N} V={V} bf16 ({N * V * 2 / 1e9:.2f} GB)",
                   "N": N, "V": V, "l2": "logits (4.2 GB) exceed L2"},
        "roofline": {"kernel": "lce_ce_logits_cluster_kernel<bf16>", "bound": "hbm", "achieved": gbs,
                     "peak": peaks.get("hbm_gbs", 6800.0), "unit": "GB/s",
                     "frac": gbs / peaks.get("hbm_gbs", 6800.0),
                     "traffic": load_traffic(wl.name).get("ce_logits")
                                if N == wl.N else None,
                     "alg_bytes_per_launch": alg_bytes, "launch_ms": kernel_ms,
                     "peak_source": peak_src},
        "gpu_launches": 3 * args.steps,
    }), flush=True)


def run_norm(args, wl, chunk):
    """Final RMSNorm + LM head + cross-entropy, forward and backward to X, gamma and
    W, on the workload's shape (lce_norm_fwd_bwd). Inputs resident, L2 flushed
    between steps. The roofline is the gradient GEMM's, as on the fused path; the
    RMSNorm kernels are reported against HBM."""
    import torch
    import linear_cross_entropy_chunked_gb300 as lce
    from lce_synth import make_norm_inputs
    rank, world, local = dist_env()
    if rank != 0:
        return
    dev = torch.device("cuda", torch.cuda.current_device())
    lce.build()
    peaks, peak_src = load_peaks()
    N, D, V = wl.N, wl.D, wl.V
    X, g, W, y = make_norm_inputs(N, D, V, wl.seed, wl.labels, wl.n_ignored)
    Xd, gd, Wd, yd = X.to(dev), g.to(dev), W.to(dev), y.to(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    low = bool(args.low_memory)
    ws = torch.empty(lce.norm_workspace_size(N, D, V, chunk, lce.LOW_MEMORY if low else 0),
                     dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return lce.norm_fwd_bwd(Xd, gd, Wd, yd, eps=1e-6, chunk=chunk, ws=ws, loss=loss, lse=lse,
                                stream=stream, low_memory=low)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if lce.read_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    launches = lce.last_launch_count()
    lce.profile_reset()
    lce.profile_enable(True)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    lce.profile_enable(False)
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    grad_ms, grad_n = lce.profile_read("grad")
    phase_ms, phase_n = lce.profile_read("phase")
    norm_ms, norm_n = lce.profile_read("norm")
    nchunks = (N + chunk - 1) // chunk
    # the dominant launch set: the pair phase (dH of a pair's second chunk beside the
    # pair's dW: 6*C*D*V) with two chunk buffers, a chunk's gradient phase (4*C*D*V)
    # with one
    if phase_n > 0:
        grad_ms, grad_n, grad_flops = phase_ms, phase_n, 6.0 * D * V * N / nchunks
        grad_name = "pair phase (lce_gemm_kernel<MODE_DH> beside <MODE_BWD>, dW over K = 2 chunks)"
    else:
        grad_flops = 4.0 * D * V * N / nchunks
        grad_name = "gradient phase (lce_gemm_kernel<MODE_DH> + <MODE_BWD>)"
    grad_avg = grad_ms / max(grad_n, 1)
    peak_sust = peaks.get("bf16_tflops_sustained", 1700.0)
    # RMSNorm kernels per step: forward reads X and writes H (bf16); backward reads
    # X (bf16) and dH (fp32) and writes dX (bf16)
    norm_bytes = N * D * (2 + 2) + N * D * (2 + 4 + 2)
    norm_step_ms = norm_ms / args.steps
    norm_gbs = norm_bytes / (norm_step_ms / 1e3) / 1e9
    hbm = peaks.get("hbm_gbs", 6800.0)

    # the standalone RMSNorm kernels over all N rows at once (forward, then the
    # backward from an fp32 dH): algorithmic bytes as above
    dH32 = torch.randn(N, D, device=dev, generator=torch.Generator(device=dev).manual_seed(5))
    Hs = torch.empty_like(Xd)
    bws = torch.empty(4 * 256 * D, dtype=torch.uint8, device=dev)
    for _ in range(3):
        lce.rmsnorm_forward(Xd, gd, eps=1e-6)
        lce.rmsnorm_backward(Xd, gd, dH32, eps=1e-6, ws=bws)
    torch.cuda.synchronize(dev)
    lce.profile_reset()
    lce.profile_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        lce.rmsnorm_forward(Xd, gd, eps=1e-6)
        flush.zero_()
        lce.rmsnorm_backward(Xd, gd, dH32, eps=1e-6, ws=bws)
    torch.cuda.synchronize(dev)
    lce.profile_enable(False)
    sa_ms, sa_n = lce.profile_read("norm")
    sa_step = sa_ms / args.steps
    sa_gbs = norm_bytes / (sa_step / 1e3) / 1e9
    del dH32, Hs

    print(json.dumps({
        "metric": "RMSNorm + LM head + CE fwd+bwd (to X, gamma, W) tokens/s",
        "value": N / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(wl, chunk, l2="L2 flushed between steps (256 MB write)"),
                       eps=1e-6, gamma="1 + 0.1 N(0,1)", x_rows="N(0,1) * exp(0.5 N(0,1)) per row"),
        "tflops": 6.0 * N * D * V / (ms / 1e3) / 1e12,
        "roofline": {"kernel": grad_name, "bound": "tensor",
                     "achieved": grad_flops / (grad_avg / 1e3) / 1e12,
                     "peak": peaks.get("bf16_tflops", 1900.0), "unit": "TFLOP/s",
                     "frac": grad_flops / (grad_avg / 1e3) / 1e12 / peaks.get("bf16_tflops", 1900.0),
                     "peak_kind": f"bf16_tflops, burst ({peak_src})",
                     "traffic": None, "launch_ms": grad_avg},
        "norm_kernels": {"ms_per_step": norm_step_ms, "launches_per_step": norm_n / args.steps,
                         "alg_bytes_per_step": norm_bytes, "achieved_gbs": norm_gbs,
                         "peak_gbs": hbm, "frac": norm_gbs / hbm, "share": norm_step_ms / ms,
                         "what": "per-chunk launches inside lce_norm_fwd_bwd (1024 rows each)"},
        "norm_kernels_standalone": {"ms_fwd_plus_bwd": sa_step, "launches": sa_n / args.steps,
                                    "alg_bytes": norm_bytes, "achieved_gbs": sa_gbs,
                                    "peak_gbs": hbm, "frac": sa_gbs / hbm,
                                    "what": "lce_rmsnorm_forward + lce_rmsnorm_backward (fp32 dH) "
                                            "over all N rows, L2 flushed before each"},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }), flush=True)


def cpu_baseline(wl):
    H64, W64, y = prepare_oracle_inputs(wl)
    rows = calibrate_rows(wl, H64, W64, y, target_s=40.0)
    t = oracle_sample_rate(wl, rows, H64, W64, y)
    return {"value": rows / t, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"first {rows} of {wl.N} tokens of the workload (fp64 numpy forward+"
                      f"backward incl. the full dW), {t:.1f} s"}


def main():
    args = parse()
    from lce_synth import WORKLOADS
    wl = WORKLOADS[args.workload]
    chunk = args.chunk or (1024 if 1024 in wl.chunks else wl.chunks[0])
    if args.impl == "reference":
        run_reference(args, wl, chunk)
    elif args.path == "ce-logits":
        run_ce_logits(args, wl)
    elif args.path == "norm":
        run_norm(args, wl, chunk)
    else:
        run_ours(args, wl, chunk)


if __name__ == "__main__":
    main()
