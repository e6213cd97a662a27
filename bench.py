"""Benchmark of the Krea 2 single-stream DiT block forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1024px] [--impl ours|reference]

One step = one block forward (all kernels of the path) over one batch of the
workload, inputs resident in HBM. The workload is the 1024px stage (B=2, 64x64 image +
512 text tokens, d=3072, 24/8 heads x 128, F=8192, bf16). With N GPUs (torchrun, one
rank per GPU) every rank runs its own batch (weak scaling, no collective on the data
path); the time is the max over ranks.

Prints one JSON line: tokens/s (whole job), bf16 TFLOP/s and the fraction of the
measured dense bf16 peak; ``roofline`` for the dominant kernel (its per-launch CUDA-event
time inside the timed region); ``e2e`` measured through the C ABI with host buffers
(pinned H2D of the step's inputs and D2H of its output inside the timed region);
``cpu_baseline`` = the fp64 oracle timed on this host's cores on a bounded sample.
``--impl reference`` times that oracle as the reference arm instead.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DiT block fwd tokens/s & bf16 TFLOP/s at 1024px; % of GB300 dense tensor peak"
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ------------------------------------------------------------------ host-side helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (independent samples: weak scaling)."""
    return base_seed + 1000 * rank


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {**FALLBACK_PEAKS, "bf16_tflops_sustained": FALLBACK_PEAKS["bf16_tflops"], "source": "fallback"}


def profile_traffic(workload: str):
    """Per-launch DRAM traffic (read + write bytes) per kernel from the ncu summary committed
    under profiles/ for this workload; {} when there is none."""
    p = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.md")
    out = {}
    if not os.path.exists(p):
        return out
    for line in open(p):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 4 and cells[3].isdigit():
            out[cells[0]] = int(cells[3])
    return out


def kernel_work(cfg):
    """Algorithmic work of one launch of each kernel: (bound, amount, unit).
    FLOPs count a multiply-add as 2; bytes count each tensor read or written once."""
    T, d, hd, F = cfg.T, cfg.d, cfg.hd, cfg.F
    nq, nkv = cfg.n_q, cfg.n_kv
    n_qkvg = ((2 if cfg.gate_on else 1) * nq + 2 * nkv) * hd
    act = 2  # bf16 bytes; the residual stream h1 is fp32
    return {
        "norm1_modulate": ("hbm", 2.0 * T * d * act, "bytes"),
        "qkvg_gemm_qknorm_rope": ("tensor", 2.0 * T * d * n_qkvg, "flops"),
        "attention_gate": ("tensor", 4.0 * cfg.B * cfg.L * cfg.L * nq * hd, "flops"),
        "oproj_gemm_residual": ("tensor", 2.0 * T * nq * hd * d, "flops"),
        "norm2_modulate": ("hbm", T * d * (4.0 + act), "bytes"),
        "upgate_gemm_swiglu": ("tensor", 2.0 * T * d * 2 * F, "flops"),
        "down_gemm_residual": ("tensor", 2.0 * T * F * d, "flops"),
    }


FP8_OVER_BF16 = 2.0  # nominal dense e4m3 / bf16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0  # nominal dense fp4 / bf16 tensor throughput ratio (13.5 / 2.25 PFLOP/s)


def time_gemm8(args, cfg, case, dev, flush, bf16_ms, modes=(("tensor", "fp8_tensor"), ("row", "fp8_row"))):
    """The block with quantised GEMMs (8-bit e4m3 operands under both scalings; NVFP4 with
    modes=(("nvfp4", "nvfp4"),)), same workload and timing protocol as the headline: per
    mode, ms per step, tokens/s, the speed-up over the bf16 block and per-kernel times
    (GEMM rates against the mode's peak: the measured bf16 peak times the nominal ratio)."""
    import torch

    import diffusion_transformer_block_gb300 as kd
    from diffusion_transformer_block_gb300.runner import DitBlock

    world, _, _ = dist_env()
    peaks = load_peaks()
    work = kernel_work(cfg)
    x_img = case.dev["x_img"].to(dev).contiguous()
    x_txt = case.dev["x_txt"].to(dev).contiguous()
    res = {}
    for scaling, mode in modes:
        ratio = FP4_OVER_BF16 if mode == "nvfp4" else FP8_OVER_BF16
        peak_key = "frac_of_fp4_peak" if mode == "nvfp4" else "frac_of_fp8_peak"
        blk = DitBlock(max_batch=cfg.B, max_seq=cfg.L, d=cfg.d, n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, F=cfg.F,
                       img_h_max=cfg.img_h, img_w_max=cfg.img_w, gate_on=cfg.gate_on, mode=mode, device=str(dev))
        blk.set_weights({k: case.dev[k] for k in ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w",
                                                  "norm2_w", "q_norm_w", "k_norm_w", "mod_bias")})
        blk.set_temb_weights({k: case.dev["temb." + k] for k in ("w1", "b1", "w2", "b2")})
        ms = blk.timestep_embed(case.dev["t"].to(dev))
        out = torch.empty(cfg.B, cfg.L, cfg.d, device=dev, dtype=torch.bfloat16)
        stream = torch.cuda.current_stream(dev)
        for _ in range(args.warmup):
            flush.zero_()
            blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out=out, stream=stream)
        torch.cuda.synchronize()
        kd.krea_dit_block_set_timing(blk.handle, True)
        kd.krea_dit_block_timing_reset(blk.handle)
        steps = max(3, min(args.steps, 20))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out=out, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        ktimes = kd.krea_dit_block_kernel_times(blk.handle)
        st, site = kd.krea_dit_block_device_status(blk.handle)
        if st != kd.KREA_DIT_OK:
            raise RuntimeError(f"{mode} device status: {kd.krea_dit_status_string(st)} (site {site})")
        step_ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), world) / steps
        kernels = {}
        for name, (tot, n) in ktimes.items():
            k = {"launches": n, "avg_ms": tot / n}
            b, amount, _ = work.get(name, ("", 0.0, ""))
            if b == "tensor" and "gemm" in name:
                k["tflops"] = amount / (k["avg_ms"] / 1000.0) / 1e12
                k[peak_key] = k["tflops"] / (ratio * peaks["bf16_tflops"])
            kernels[name] = k
        res[scaling] = {"ms_per_step": step_ms, "tokens_per_s": world * cfg.T / (step_ms / 1000.0),
                        "speedup_vs_bf16": bf16_ms / step_ms, "kernels": kernels,
                        "gpu_launches_per_step": sum(v["launches"] for v in kernels.values()) / steps}
        kd.krea_dit_block_set_timing(blk.handle, False)
        blk.close()
    if any(m == "nvfp4" for _, m in modes):
        res["how"] = ("krea_dit_block_forward4 on the headline workload, NVFP4 weights cast once before timing; "
                      "CUDA events per step, L2 flushed before each step outside the events; fp4 peak = measured "
                      f"bf16 peak x {FP4_OVER_BF16} (nominal ratio)")
    else:
        res["how"] = ("krea_dit_block_forward8 on the headline workload, e4m3 weights cast once before timing; "
                      "CUDA events per step, L2 flushed before each step outside the events; fp8 peak = measured "
                      f"bf16 peak x {FP8_OVER_BF16} (nominal ratio)")
    return res


def time_backward(args, cfg, blk, case, dev, flush, x_img, x_txt, ms):
    """The block backward (gradients of input, weights and modulation; the forward is
    recomputed inside the call), same workload and timing protocol as the headline."""
    import torch

    import dit_inputs as di
    import diffusion_transformer_block_gb300 as kd

    world, _, _ = dist_env()
    peaks = load_peaks()
    _, dout = di.make_dout(cfg)
    dout = dout.to(dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: blk.backward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, dout,  # noqa: E731
                                stream=stream)
    for _ in range(2):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    kd.krea_dit_block_set_timing(blk.handle, True)
    kd.krea_dit_block_timing_reset(blk.handle)
    steps = max(3, min(args.steps, 10))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    ktimes = kd.krea_dit_block_kernel_times(blk.handle)
    kd.krea_dit_block_set_timing(blk.handle, False)
    st, site = kd.krea_dit_block_device_status(blk.handle)
    if st != kd.KREA_DIT_OK:
        raise RuntimeError(f"backward device status: {kd.krea_dit_status_string(st)} (site {site})")
    ms_step = reduce_max(sum(a.elapsed_time(b) for a, b in evs), world) / steps
    flops = di.config_backward_flops(cfg)
    return {"ms_per_step": ms_step, "tokens_per_s": world * cfg.T / (ms_step / 1000.0),
            "tflops": flops / (ms_step / 1000.0) / 1e12,
            "frac_of_peak": flops / (ms_step / 1000.0) / 1e12 / peaks["bf16_tflops"],
            "flops_per_step": flops,
            "kernels_ms_per_step": {k: tot / steps for k, (tot, n) in ktimes.items()},
            "launches_per_step": sum(n for tot, n in ktimes.values()) / steps,
            "how": "krea_dit_block_backward (forward recomputed inside), CUDA events per step, L2 flushed before "
                   "each step outside the events; TFLOP/s counts the backward's algorithmic FLOPs only "
                   "(2x the projections, 2.5x the attention contractions), not the recomputation"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.perf_counter())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = getattr(self, "t_begin", None)
        t1 = getattr(self, "t_end", None)
        for ts, ln in self.lines:
            if t0 is not None and t1 is not None and not (t0 <= ts <= t1 + self.PERIOD_MS / 1000.0):
                continue  # keep samples taken during the timed region only
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing
def time_oracle(cfg, rows_per_step: int, seed: int):
    """Time the fp64 oracle on one batch element of ``cfg``: keys/values for all L
    tokens, every other step of the block for ``rows_per_step`` query rows.
    Returns (seconds, tokens credited = rows_per_step, threads)."""
    import numpy as np

    import dit_inputs as di
    import oracle

    one = cfg.replace(B=1, seed=seed)
    case = di.make_case(one)
    ms = oracle.mod_shared_for(case)
    rows = [np.sort(np.random.default_rng(seed).choice(one.L, size=min(rows_per_step, one.L), replace=False))]
    t0 = time.perf_counter()
    oracle.run_case(case, rows=rows if rows_per_step < one.L else None, mod_shared=ms)
    dt = time.perf_counter() - t0
    return dt, len(rows[0]), blas_threads()


def host_cpu() -> dict:
    """The host's logical CPU count and CPU model (lscpu's model name, else
    /proc/cpuinfo's model name or implementer/part codes, else the platform string)."""
    import platform

    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            info = open("/proc/cpuinfo").read()
            m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
            if m:
                model = m.group(1).strip()
            else:
                imp = re.search(r"^CPU implementer\s*:\s*(\S+)$", info, re.M)
                part = re.search(r"^CPU part\s*:\s*(\S+)$", info, re.M)
                if imp and part:
                    model = f"implementer {imp.group(1)} part {part.group(1)}"
        except Exception:
            pass
    return {"nproc": os.cpu_count() or 1, "model": model or platform.processor() or platform.machine()}


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm
def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    rows = args.ref_rows
    for _ in range(args.warmup):
        time_oracle(cfg, rows, cfg.seed)
    total, tokens, threads = 0.0, 0, 1
    for i in range(args.steps):
        dt, n, threads = time_oracle(cfg, rows, cfg.seed + i)
        total += dt
        tokens += n
    value = tokens / total
    flops_per_token = 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "L": cfg.L, "d_model": cfg.d, "n_q": cfg.n_q,
                   "n_kv": cfg.n_kv, "head_dim": cfg.hd, "ffn": cfg.F},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", **host_cpu(),
                         "sample": f"one batch element of {cfg.name}: K/V for all {cfg.L} tokens, the rest of the "
                                   f"block for {rows} query rows per step (tokens credited = rows)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del flops_per_token
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args, cfg):
    import torch

    import dit_inputs as di
    import diffusion_transformer_block_gb300 as kd
    from diffusion_transformer_block_gb300.runner import DitBlock

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    case = di.make_case(cfg.replace(seed=shard_seed(cfg.seed, rank)))
    blk = DitBlock(max_batch=cfg.B, max_seq=cfg.L, d=cfg.d, n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, F=cfg.F,
                   img_h_max=cfg.img_h, img_w_max=cfg.img_w, gate_on=cfg.gate_on, mode="bf16", device=str(dev))
    blk.set_weights({k: case.dev[k] for k in ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w",
                                              "q_norm_w", "k_norm_w", "mod_bias")})
    blk.set_temb_weights({k: case.dev["temb." + k] for k in ("w1", "b1", "w2", "b2")})
    x_img = case.dev["x_img"].to(dev).contiguous()
    x_txt = case.dev["x_txt"].to(dev).contiguous()
    t = case.dev["t"].to(dev)
    stream = torch.cuda.current_stream(dev)
    ms = blk.timestep_embed(t)
    out = torch.empty(cfg.B, cfg.L, cfg.d, device=dev, dtype=torch.bfloat16)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)

    def step():
        blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out=out, stream=stream)

    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st, site = kd.krea_dit_block_device_status(blk.handle)
    if st != kd.KREA_DIT_OK:
        raise RuntimeError(f"device status after warm-up: {kd.krea_dit_status_string(st)} (site {site})")

    # ---- timed region: K steps, L2 flushed before each (outside the step's events)
    kd.krea_dit_block_set_timing(blk.handle, True)
    kd.krea_dit_block_timing_reset(blk.handle)
    clocks = ClockSampler(local)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    time.sleep(0.3)  # let the sampler start
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    clocks.mark("t_begin")
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t_end")
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ktimes = kd.krea_dit_block_kernel_times(blk.handle)
    kd.krea_dit_block_set_timing(blk.handle, False)
    total_ms = sum(step_ms)
    total_ms_max = reduce_max(total_ms, world)
    st, site = kd.krea_dit_block_device_status(blk.handle)
    if st != kd.KREA_DIT_OK:
        raise RuntimeError(f"device status after timing: {kd.krea_dit_status_string(st)} (site {site})")

    # ---- end to end through the C ABI with host buffers: every step uploads its inputs
    # from pinned host memory and downloads its output (krea_dit_block_forward_host, which
    # overlaps step i's compute with step i+1's upload and step i-1's download)
    kd.krea_dit_block_enable_host_io(blk.handle)
    h_img = case.dev["x_img"].contiguous().pin_memory()
    h_txt = case.dev["x_txt"].contiguous().pin_memory()
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))

    def host_step(i):
        kd.krea_dit_block_forward_host(blk.handle, h_img, h_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms,
                                       blk._wstruct, h_out[i % 2], stream)

    for i in range(3):
        host_step(i)
    kd.krea_dit_block_host_sync(blk.handle)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        host_step(i)
    kd.krea_dit_block_host_sync(blk.handle)
    torch.cuda.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, world)
    e2e_ms = 1000.0 * e2e_s
    h2d = h_img.numel() * h_img.element_size() + h_txt.numel() * h_txt.element_size()
    d2h = h_out[0].numel() * h_out[0].element_size()

    # ---- a stack of blocks (distinct weight buffers per block) in place on the joint
    # sequence: eager launches vs one CUDA-graph launch per stack; x is reset and L2
    # flushed before each stack, outside its events
    stack = None
    if args.stack_blocks > 0:
        nb = args.stack_blocks
        sw = blk.stack_weights([{k: v.clone() for k, v in blk.w.items()} for _ in range(nb)])
        x0 = torch.cat([x_txt, x_img], dim=1).contiguous()
        xs = x0.clone()
        gstream = torch.cuda.Stream(dev)
        torch.cuda.synchronize()
        graph = blk.stack_graph(xs, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw, gstream)
        k_stack = max(3, min(args.steps, 20))

        def time_stack(run, st):
            for _ in range(2):
                xs.copy_(x0)
                flush.zero_()
                run()
            torch.cuda.synchronize()
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(k_stack)]
            for a, b in pairs:
                with torch.cuda.stream(st):
                    xs.copy_(x0)
                    flush.zero_()
                    a.record(st)
                    run()
                    b.record(st)
            torch.cuda.synchronize()
            return reduce_max(sum(a.elapsed_time(b) for a, b in pairs), world) / k_stack

        eager_ms = time_stack(lambda: blk.stack_forward(xs, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw,
                                                        stream=stream), stream)
        graph_ms = time_stack(lambda: graph.launch(gstream), gstream)
        graph.close()
        stack = {"blocks": nb, "stacks_timed": k_stack, "eager_ms_per_stack": eager_ms,
                 "graph_ms_per_stack": graph_ms, "graph_ms_per_block": graph_ms / nb,
                 "tokens_per_s_graph": world * cfg.T / (graph_ms / 1000.0),
                 "tflops_graph": world * di.config_flops(cfg) * nb / (graph_ms / 1000.0) / 1e12,
                 "how": "krea_dit_stack_forward (eager) and one krea_dit_graph_launch of the captured stack, "
                        "in place on the joint sequence; CUDA events around each stack"}
        del sw

    backward = None
    if not args.no_backward:
        backward = time_backward(args, cfg, blk, case, dev, flush, x_img, x_txt, ms)

    gemm8 = None
    if not args.no_gemm8:
        gemm8 = time_gemm8(args, cfg, case, dev, flush, total_ms_max / args.steps)
    nvfp4 = None
    if not args.no_nvfp4:
        nvfp4 = time_gemm8(args, cfg, case, dev, flush, total_ms_max / args.steps, modes=(("nvfp4", "nvfp4"),))

    # ---- numbers
    tokens_per_step = cfg.T
    ms_per_step = total_ms_max / args.steps
    value = world * tokens_per_step * args.steps / (total_ms_max / 1000.0)
    flops = di.config_flops(cfg)
    tflops = world * flops * args.steps / (total_ms_max / 1000.0) / 1e12
    peaks = load_peaks()
    work = kernel_work(cfg)
    per_kernel = {}
    for name, (tot, n) in ktimes.items():
        per_kernel[name] = {"launches": n, "avg_ms": tot / n, "share": tot / max(sum(v[0] for v in ktimes.values()),
                                                                                1e-12)}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["avg_ms"] * per_kernel[k]["launches"])
    bound, amount, unit = work[dom]
    avg_s = per_kernel[dom]["avg_ms"] / 1000.0
    if bound == "tensor":
        achieved, peak, runit = amount / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, runit = amount / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
    for name, pk in per_kernel.items():
        b, a, _ = work.get(name, ("", 0.0, ""))
        if b == "tensor":
            pk["tflops"] = a / (pk["avg_ms"] / 1000.0) / 1e12
            pk["frac_of_peak"] = pk["tflops"] / peaks["bf16_tflops"]
        elif b == "hbm":
            pk["gbs"] = a / (pk["avg_ms"] / 1000.0) / 1e9
            pk["frac_of_peak"] = pk["gbs"] / peaks["hbm_gbs"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, n, threads = time_oracle(cfg, args.cpu_rows, cfg.seed)
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle", **host_cpu(),
               "sample": f"one batch element of {cfg.name}: K/V for all {cfg.L} tokens, the rest of the block for "
                         f"{n} query rows ({dt:.1f} s; tokens credited = rows)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "img": f"{cfg.img_h}x{cfg.img_w}", "n_txt": cfg.n_txt,
                   "L": cfg.L, "d_model": cfg.d, "n_q": cfg.n_q, "n_kv": cfg.n_kv, "head_dim": cfg.hd,
                   "ffn": cfg.F, "gate_on": cfg.gate_on, "global_batch": cfg.B * world, "parallelism": f"dp{world}",
                   "l2": "flushed before every timed step (256 MB write outside the step's events)",
                   "flops_per_step": flops},
        "tflops": tflops,
        "frac_of_peak": tflops / peaks["bf16_tflops"],
        "peak_source": f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s (burst)",
        "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": runit,
                     "frac": achieved / peak, "traffic": profile_traffic(cfg.name).get(dom),
                     "algorithmic": {"amount_per_launch": amount, "unit": unit}},
        "kernels": per_kernel,
        "cpu_baseline": cpu,
        "e2e": {"value": world * tokens_per_step * e2e_steps / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "krea_dit_block_forward_host per step (pinned host in/out), wall clock over the steps "
                       "with device and copy streams synchronised on both sides"},
        "stack": stack,
        "gemm8": gemm8,
        "nvfp4": nvfp4,
        "backward": backward,
        "clocks": clk,
        "gpu_launches": sum(pk["launches"] for pk in per_kernel.values()),
        "wall_s_timed_region": wall,
    }
    if rank == 0:
        print(json.dumps(line))
    blk.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="1024px")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=4608, help="query rows of the CPU-baseline oracle sample")
    ap.add_argument("--ref-rows", type=int, default=1024, help="query rows per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gemm8", action="store_true", help="skip the 8-bit GEMM measurement")
    ap.add_argument("--no-nvfp4", action="store_true", help="skip the NVFP4 GEMM measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the block-backward measurement")
    ap.add_argument("--stack-blocks", type=int, default=8, help="blocks of the stack / CUDA-graph measurement (0: skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import dit_inputs as di

    cfg = di.CONFIGS[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
