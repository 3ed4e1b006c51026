#!/usr/bin/env python
"""Throughput of the DFlash draft-and-verify step on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input: KV injection
of the previous step's accepted positions, one block-diffusion draft pass (B = 16), the
synthetic target's agreement plant, greedy verification. Default workload: the
Qwen3-8B-shaped 5-layer drafter, batch 1, 2048 injected context positions, B = 16,
planted agreement p = 0.8 (configs of the draft-step benchmark: seeded synthetic
weights N(0, 0.02) and hidden states N(0, 1); no trained weights or datasets).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]

Prints one JSON line (rank 0). With --impl reference the CPU oracle is timed instead.
Timing: W untimed steps, then exactly K steps as CUDA-graph replays between CUDA events
on the launching stream, barrier + synchronize on both sides, max over ranks. The
weights streamed every step (3.4 GB) are far larger than L2 (129 MB), so no flush is
needed between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft+verify steps/s and drafted tok/s (B=16) with HBM/tensor roofline fraction"
UNIT = "steps/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default="qwen3-8b-b1-ctx2048-B16")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=30.0)
    ap.add_argument("--trace-steps", type=int, default=10)
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the block-size draft sweep and the fused target-verify measurement")
    ap.add_argument("--attn-mode", type=int, default=0, choices=[0, 1, 2, 3],
                    help="attention kernel (DFLASH_OPT_ATTN_MODE): 0 chosen by shape, 1 clusters, "
                         "2 flat split on the tensor cores where the shape allows, 3 flat on mma.sync")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ algorithmic traffic

def proj_bytes_flops(s, batch, B, tau):
    """Algorithmic (bytes, flops) of each projection: the weight read once, the activation
    rows read once, the outputs written once. bf16 activation operands are two planes
    (high and low, 4 bytes per value); q and the K and V cache entries are fp16 (2 bytes);
    the residual stream is fp32 (read and written by O and down). FLOPs count one product
    per weight and row (the low plane's second product is not counted)."""
    H, d, I, V = s.hidden, s.head_dim, s.intermediate, s.vocab
    rows = batch * B
    kin = s.n_taps * s.target_hidden
    kvd = s.n_kv_heads * d
    kv = 2 * s.n_layers * kvd
    nqkv = (s.n_heads + 2 * s.n_kv_heads) * d
    nqd = s.n_heads * d
    return {
        "fc": (2 * H * kin + 2 * tau * kin + 4 * tau * H, 2 * tau * H * kin),
        "kv": (2 * kv * H + 4 * tau * H + 2 * tau * kv, 2 * tau * kv * H),
        "qkv": (2 * nqkv * H + 4 * rows * H + rows * (2 * nqd + 4 * kvd), 2 * rows * nqkv * H),
        "o": (2 * H * nqd + 4 * rows * nqd + 12 * rows * H, 2 * rows * H * nqd),
        "gateup": (2 * 2 * I * H + 4 * rows * (H + I), 2 * rows * 2 * I * H),
        "down": (2 * H * I + 4 * rows * I + 12 * rows * H, 2 * rows * H * I),
        "lm_head": (2 * V * H + 4 * rows * H + 4 * batch * (B - 1), 2 * batch * (B - 1) * V * H),
    }


def attn_bytes_flops(s, batch, B, n_ctx):
    """K and V (fp16) read once per layer per sequence (context plus block keys), q (fp16)
    read, o (two bf16 planes) written."""
    kvb = 4 * (n_ctx + B) * s.n_kv_heads * s.head_dim * batch
    qo = 6 * batch * B * s.n_heads * s.head_dim
    fl = 4 * batch * B * s.n_heads * s.head_dim * (n_ctx + B)
    return kvb + qo, fl


def _passes(rows, width):
    return [(r0, min(width, rows - r0)) for r0 in range(0, rows, width)]


def launch_plan(s, batch, B, tau, n_ctx, n_sms=152, one_pass=False, chain_max=8):
    """Launch order of one step by call: (label, kind, bytes, flops). kind "gemv" marks the
    chained kernel (one launch runs up to `chain_max` phases, the handle's
    DFLASH_OPT_CHAIN_MAX, for one pass of at most 256 rows); attention is a launch of its own
    between chains. Injection runs in passes of a width fixed by max_batch * max_block.
    Mirrors the library's grouping. With one_pass every projection covers all rows at once:
    the method's own traffic, each weight once."""
    ab = attn_bytes_flops(s, batch, B, n_ctx)
    rows = batch * B
    nb = 1
    while nb * 16 < min(rows, 256):
        nb *= 2
    inject = []
    for _, pr in _passes(rows, rows if one_pass else 16 * nb):   # tau accepted rows per sequence, padded to B
        pj = proj_bytes_flops(s, 1, pr, tau * pr / B)
        inject.append(("fc+kv", "gemv", *tuple(map(sum, zip(pj["fc"], pj["kv"])))))
    draft = [("embed", "small", 2 * s.hidden * batch * (1 + 6 * B), 0)]
    segments = [["qkv"]]
    for l in range(s.n_layers):
        segments += ["attn", ["o", "gateup", "down", "qkv" if l + 1 < s.n_layers else "lm_head"]]
    for seg in segments:
        if seg == "attn":
            draft.append(("attn", "attn", *ab))
            continue
        for _, pr in _passes(rows, rows if one_pass else 256):
            pj = proj_bytes_flops(s, 1, pr, 1)
            if "lm_head" in seg:   # the LM head of a pass covers its rows' drafted slots
                pj["lm_head"] = proj_bytes_flops(s, pr // B if pr >= B else 1, B, 1)["lm_head"]
            for i in range(0, len(seg), chain_max):
                cur = seg[i:i + chain_max]
                draft.append(("+".join(cur), "gemv", sum(pj[n][0] for n in cur), sum(pj[n][1] for n in cur)))
    return {"inject": inject, "draft": draft,
            "verify": [("verify", "small", 4 * batch * B * s.vocab, 0)]}


def measured_traffic(launch, workload):
    """DRAM bytes per launch that ncu measured for this launch kind (profiles/traffic.json),
    or None when no capture covers it or the kernel sources changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        t = json.load(f)
    if t.get("launch") != launch or t.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for src in t["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return t["traffic_bytes"] if h.hexdigest() == t["sources_sha256"] else None


def step_bytes_flops(s, batch, B, n_ctx, tau):
    """Algorithmic bytes and FLOPs of one step: every weight read once, K/V read once per
    layer, activations and logits once (however the library splits rows into passes)."""
    byt = fl = 0
    for call in launch_plan(s, batch, B, tau, n_ctx, one_pass=True).values():
        for _, kind, b, f in call:
            byt += b
            fl += f
    return byt, fl


# ------------------------------------------------------------------ clocks

class NvmlClockSampler:
    """SM clock, power and clock-event reasons of this process's GPU, read through NVML
    (NVIDIA's management library, loaded with ctypes) every `period_ms` from a thread.
    Only reads; changes no setting. Raises in __init__ when NVML is not usable."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, pci_bus_id: str, period_ms=1.0):
        import ctypes
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + pci_bus_id)
        try:
            self._reasons = self.nv.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.period = period_ms / 1e3
        self.samples = []
        self._stop = False
        self._t = None

    def _read_one(self):
        import ctypes
        clk, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        self._reasons(self.h, ctypes.byref(rs))
        return float(clk.value), pw.value / 1e3, int(rs.value)

    def _loop(self):
        while not self._stop:
            self.samples.append((time.monotonic(), *self._read_one()))
            time.sleep(self.period)

    def start(self):
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()

    def stop(self):
        self._stop = True
        if self._t:
            self._t.join(timeout=2)

    def summary(self, t0, t1, gpu_index=None):
        inside = [r for r in self.samples if t0 <= r[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "no NVML sample inside the timed region"}
        reasons = sorted({n for r in inside for bit, n in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(r[2] for r in inside), "reasons": reasons, "samples": len(inside),
                "note": "NVML, sampled every ~1 ms during the timed region"}


def clock_sampler():
    """NVML sampler for the current CUDA device, else the nvidia-smi one."""
    try:
        import torch
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        return NvmlClockSampler(bus)
    except Exception:
        return ClockSampler()


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, period_ms=20):
        self.samples = []
        self.proc = None
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.period_ms)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, gpu_index=None):
        rows = [(t, r) for t, r in self.samples if len(r) >= 9 and (gpu_index is None or r[0] == str(gpu_index))]
        inside = [r for t, r in rows if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside and rows:   # a very short region: take the samples nearest to it
            rows.sort(key=lambda tr: min(abs(tr[0] - t0), abs(tr[0] - t1)))
            inside = [r for _, r in rows[:3]]
            note = "timed region shorter than the sampling period; nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------------ CPU oracle runs

def oracle_steps(shape, bits, w, seed, n_steps, budget_s, ctx_hidden_bits, step_hidden_bits, noise, masks):
    """Run the oracle on one sequence of the workload: an untimed prefill of the context,
    then up to n_steps timed steps (inject previous tau rows, draft, verify) within budget_s.
    Returns (steps_done, seconds)."""
    import numpy as np
    from oracle.dflash_ref import Oracle
    from synth import inputs as I
    o = Oracle(shape, bits)
    st = o.new_sequence(w.ctx + (n_steps + 2) * w.block + w.block, last_token=1)
    o.inject(st, ctx_hidden_bits)
    tau_prev = 0
    done, t_used = 0, 0.0
    while done < n_steps:
        t0 = time.perf_counter()
        if tau_prev:
            o.inject(st, step_hidden_bits[:, :tau_prev])
        r = o.draft(st, w.block)
        T = I.plant_logits(noise[None], r.drafted[None], masks[done % len(masks)][None])[0]
        v = o.verify(st, T, r.drafted)
        tau_prev = v.accept_len
        t_used += time.perf_counter() - t0
        done += 1
        if t_used > budget_s:
            break
    return done, t_used


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------ main arms

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device="cuda") -> float:
    """The largest of every rank's x (the job's time is its slowest replica's)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ws: int, batch: int, steps: int, seconds: float) -> float:
    """Whole-job steps/s: every rank ran `steps` steps of `batch` sequences in `seconds`."""
    return ws * batch * steps / seconds


def workload_config(w, ws, seed):
    """The `config` object of the JSON line, the same for both arms: what the workload is."""
    from synth import weight_bytes
    from synth import inputs as I
    s = w.shape
    wb = weight_bytes(s)
    return {"workload": w.name, "batch_per_gpu": w.batch, "block": w.block,
            "ctx": int(I.ragged_ctx(w, seed).mean()),
            "drafter": f"H{s.hidden} L{s.n_layers} nq{s.n_heads} nkv{s.n_kv_heads} d{s.head_dim} "
                       f"I{s.intermediate} V{s.vocab} k{s.n_taps}",
            "p_plant": w.p_plant, "parallelism": f"replicas x{ws}",
            "l2": f"inputs larger than L2: {sum(v for k, v in wb.items() if k != 'embed_row') / 1e9:.2f} "
                  "GB of weights streamed per step, no flush"}


def run_reference(a):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import numpy as np
    from synth import WORKLOADS
    from synth import inputs as I
    w = WORKLOADS[a.workload]
    s = w.shape
    weights = I.make_weights(s, a.seed)
    bits = weights.bits()
    ctx_bits = I.bf16_bits(I.make_hidden(s, w.ctx, a.seed, "ctx"))
    step_bits = I.bf16_bits(I.make_hidden(s, w.block, a.seed, "step"))
    noise = I.make_logit_noise(1, w.block, s.vocab, a.seed).numpy()[0][None]
    masks = [I.make_plant_mask(1, w.block, w.p_plant, a.seed, f"plant.{i}")[0] for i in range(8)]
    # W untimed steps, then exactly K timed steps; each step one sequence of the workload
    # (for the batch-1 workloads, the whole step)
    if a.warmup > 0:
        oracle_steps(s, bits, w, a.seed, a.warmup, float("inf"), ctx_bits, step_bits, noise[0], masks)
    n, secs = oracle_steps(s, bits, w, a.seed, a.steps, float("inf"), ctx_bits, step_bits, noise[0], masks)
    v = n / secs
    cores = cpu_cores()
    sample = (f"{n} oracle steps of the {w.name} workload (inject + B={w.block} draft + verify, fp64 NumPy, "
              f"one sequence of {w.batch}) after an untimed prefill of {w.ctx} positions and {a.warmup} "
              f"untimed warm-up steps")
    ws, _, _ = dist_info()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": a.gpus, "steps": n,
        "warmup": a.warmup, "ms_per_step": 1e3 * secs / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(w, ws, a.seed),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_cuda(a):
    import numpy as np
    import torch
    import torch.distributed as dist

    from block_diffusion_drafter_kv_gb300 import binding as BND
    from block_diffusion_drafter_kv_gb300.build import build
    from synth import WORKLOADS
    from synth import inputs as I

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        build()
    if ws > 1:
        dist.barrier()
    build()
    w = WORKLOADS[a.workload]
    s, B, batch = w.shape, w.block, w.batch
    log = (lambda *m: print(*m, file=sys.stderr, flush=True)) if rank == 0 else (lambda *m: None)
    t_setup = time.time()
    weights_cpu = I.make_weights(s, a.seed)
    weights = weights_cpu.to("cuda")
    ctx_lens = I.ragged_ctx(w, a.seed + rank)
    ctx_max = int(ctx_lens.max())
    cap = ctx_max + (a.warmup + a.steps + a.trace_steps + 4) * B + B
    dr = BND.Drafter(s, weights, max_block=B, max_batch=batch, kv_capacity=cap)
    dr.set_option(BND.OPT_ATTN_MODE, a.attn_mode)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    log(f"[bench] weights ready in {time.time() - t_setup:.1f}s; prefill {ctx_max} positions x {batch}")
    # prefill: inject the whole context of every sequence
    # context hidden states N(0,1), drawn on the device from a seeded generator (up to
    # 10 GB for the batched workload; the oracle's CPU baseline draws its own)
    hid_ctx = torch.empty(s.n_taps, batch * ctx_max, s.target_hidden, dtype=torch.bfloat16, device="cuda")
    hid_ctx.normal_(generator=torch.Generator(device="cuda").manual_seed(a.seed * 1000 + rank))
    n_ctx = torch.as_tensor(ctx_lens, dtype=torch.int32, device="cuda")
    pf0, pf1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        pf0.record(stream)
        dr.inject(hid_ctx, ctx_max, n_ctx, batch)
        pf1.record(stream)
        dr.last_token[:batch].copy_(torch.as_tensor(I.initial_tokens(batch, s.vocab, a.seed + rank)))
    stream.synchronize()
    prefill = {"positions": int(ctx_lens.sum()), "pass_rows": dr.get_option(BND.OPT_INJECT_PASS_ROWS),
               "us": 1e3 * pf0.elapsed_time(pf1)}
    if not a.no_sweep and dr.get_option(BND.OPT_INJECT_PASS_ROWS) < 128:
        # the same prefill through 128-row passes (a handle of its own: the width is fixed
        # per handle), each pass streaming the fusion and K/V weights once
        wide = BND.Drafter(s, weights, max_block=B, max_batch=batch, kv_capacity=cap)
        wide.set_option(BND.OPT_INJECT_PASS_ROWS, 128)
        with torch.cuda.stream(stream):
            wide.inject(hid_ctx, ctx_max, n_ctx, batch)   # warm-up
            wide.len.zero_()
            pf0.record(stream)
            wide.inject(hid_ctx, ctx_max, n_ctx, batch)
            pf1.record(stream)
        stream.synchronize()
        prefill["us_128_row_passes"] = 1e3 * pf0.elapsed_time(pf1)
        wide.close()
        del wide
    log(f"[bench] prefill: {json.dumps(prefill)}")
    del hid_ctx
    len0 = dr.len.clone()
    last0 = dr.last_token.clone()
    # per-step inputs, resident in HBM before timing
    n_masks = a.warmup + a.steps + a.trace_steps + 2
    p = I.per_seq_p(w, a.seed + rank)
    masks_np = np.stack([I.make_plant_mask(batch, B, p, a.seed + rank, f"plant.{i}") for i in range(n_masks)])
    hid_step_cpu = I.make_hidden(s, batch * B, a.seed + rank, "step")
    noise_cpu = I.make_logit_noise(batch, B, s.vocab, a.seed + rank)
    hid_step = hid_step_cpu.cuda()
    noise = noise_cpu.cuda()
    masks = torch.as_tensor(masks_np, device="cuda")
    accept = torch.zeros(batch, dtype=torch.int32, device="cuda")
    drafted = torch.zeros(batch, max(B - 1, 1), dtype=torch.int32, device="cuda")
    committed = torch.zeros(batch, B, dtype=torch.int32, device="cuda")
    step_ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
    saved = torch.zeros(2 * batch * B, dtype=torch.int32, device="cuda")
    launches = {}

    def inject_draft():
        dr.inject(hid_step, B, accept, batch)
        launches["inject"] = dr.last_launch_count()
        dr.draft(batch, B, drafted)
        launches["draft"] = dr.last_launch_count()

    def plant_verify():
        BND.synth_plant(noise, drafted, masks, n_masks, step_ctr, batch, B, 10.0, saved)
        dr.verify(noise, drafted, batch, B, accept, committed)
        launches["verify"] = dr.last_launch_count()
        BND.synth_unplant(noise, step_ctr, n_masks, batch, B, saved)
        launches["synthetic_target"] = 2

    def reset():
        dr.len.copy_(len0)
        dr.last_token.copy_(last0)
        accept.zero_()
        step_ctr.zero_()

    with torch.cuda.stream(stream):   # eager run once (also loads the modules) before capture
        inject_draft()
        plant_verify()
    stream.synchronize()
    assert dr.device_error(stream=stream) == 0, "device error flag after the eager step"
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        inject_draft()
        plant_verify()
    per_step_launches = sum(launches.values())
    with torch.cuda.stream(stream):
        reset()
    stream.synchronize()

    # ---------------------------------------------------------------- timed region
    clocks = clock_sampler()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            g_step.replay()
        reset()
    stream.synchronize()
    len_start = int(dr.len[:batch].sum())
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    th0 = time.monotonic()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(a.steps):
            g_step.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    th1 = time.monotonic()
    if ws > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    time.sleep(0.1)
    clocks.stop()
    err = dr.device_error(stream=stream)
    len_end = int(dr.len[:batch].sum())
    tau_sum = (len_end - len_start) + int(accept[:batch].sum())
    mean_tau = tau_sum / (a.steps * batch)
    ms_total = max_over_ranks(ms_total, ws)
    ms_step = ms_total / a.steps
    value = job_rate(ws, batch, a.steps, ms_total / 1e3)
    n_avg = len_start / batch + (len_end - len_start) / (2.0 * batch)
    tau_avg = mean_tau
    byt, fl = step_bytes_flops(s, batch, B, n_avg, tau_avg)
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    tens = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    t_hbm = byt / (hbm * 1e9)
    t_ten = fl / (tens * 1e12)
    step_roof = {"bound": "hbm" if t_hbm >= t_ten else "tensor", "bytes": byt, "flops": fl,
                 "achieved_gbs": byt / (ms_step * 1e-3) / 1e9,
                 "frac": max(t_hbm, t_ten) / (ms_step * 1e-3), "peak_gbs": hbm,
                 "peak_kind": f"{pk_kind} hbm_gbs"}
    log(f"[bench] {ms_step * 1e3:.1f} us/step, mean tau {mean_tau:.2f}, step roofline {step_roof['frac']:.3f}")

    # ---------------------------------------------------------------- draft latency alone
    # One dflash_draft_block call (embed, projection chains, attention, LM head and argmax)
    # captured in a graph and replayed back to back; it reads the cache and length, writes
    # only the block's scratch and the drafts, so replays are identical.
    g_draft = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_draft, stream=stream):
        dr.draft(batch, B, drafted)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_draft.replay()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_draft = 20
    with torch.cuda.stream(stream):
        d0.record(stream)
        for _ in range(n_draft):
            g_draft.replay()
        d1.record(stream)
    torch.cuda.synchronize()
    draft_ms = d0.elapsed_time(d1) / n_draft
    log(f"[bench] draft alone: {draft_ms * 1e3:.1f} us")
    # the same for every block size of the sweep (the block rides in the N operand of every
    # weight stream, so the draft's cost should barely depend on it)
    draft_by_block = {}
    for Bs in (() if a.no_sweep else (4, 8, 12, 16)):
        if Bs > B:
            continue
        if Bs == B:
            draft_by_block[str(Bs)] = draft_ms
            continue
        gB = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gB, stream=stream):
            dr.draft(batch, Bs, drafted)
        with torch.cuda.stream(stream):
            for _ in range(3):
                gB.replay()
            d0.record(stream)
            for _ in range(n_draft):
                gB.replay()
            d1.record(stream)
        torch.cuda.synchronize()
        draft_by_block[str(Bs)] = d0.elapsed_time(d1) / n_draft
        del gB
    log("[bench] draft by block: " + json.dumps({k: round(v * 1e3, 1) for k, v in draft_by_block.items()}))

    # ---------------------------------------------------------------- fused target-side verify
    # dflash_verify_greedy_hidden on a synthetic target head of this workload's size (final
    # norm gain 1 + N(0, 0.1), LM head N(0, 0.02) [V][Ht] bf16, hidden states N(0, 1)): the
    # target's norm, LM head and argmax of every block position, then the acceptance.
    fused = None
    if s.target_hidden <= 8192 and not a.no_sweep:
        gt = torch.Generator(device="cuda").manual_seed(a.seed + 99)
        t_gain = (1.0 + 0.1 * torch.randn(s.target_hidden, generator=gt, device="cuda")).to(torch.bfloat16)
        t_lm = (0.02 * torch.randn(s.vocab, s.target_hidden, generator=gt, device="cuda")).to(torch.bfloat16)
        t_hid = torch.randn(batch * B, s.target_hidden, generator=gt, device="cuda").to(torch.bfloat16)
        g_fv = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fv, stream=stream):
            dr.verify_hidden(t_hid, t_gain, t_lm, drafted, batch, B, accept, committed)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_fv.replay()
            d0.record(stream)
            for _ in range(n_draft):
                g_fv.replay()
            d1.record(stream)
        torch.cuda.synchronize()
        fv_ms = d0.elapsed_time(d1) / n_draft
        fv_bytes = 2 * s.vocab * s.target_hidden + 2 * batch * B * s.target_hidden
        fused = {"us": fv_ms * 1e3, "bytes": fv_bytes, "achieved_gbs": fv_bytes / (fv_ms * 1e-3) / 1e9,
                 "frac_of_hbm": fv_bytes / (fv_ms * 1e-3) / 1e9 / float(peaks()[0]["hbm_gbs"]),
                 "what": "dflash_verify_greedy_hidden: target final norm + LM head + argmax + acceptance"}
        del g_fv, t_lm
        log(f"[bench] fused target verify: {fv_ms * 1e3:.1f} us")
        with torch.cuda.stream(stream):
            reset()
        stream.synchronize()

    # ---------------------------------------------------------------- traced pass (per-kernel)
    kern = {}
    roof = None
    if a.trace_steps > 0:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(64)]
        for ev in evs:              # torch creates the CUDA event on its first record
            ev.record(stream)
        stream.synchronize()
        dr.trace_events(evs)
        plan = launch_plan(s, batch, B, tau_avg, n_avg, chain_max=dr.get_option(BND.OPT_CHAIN_MAX))
        with torch.cuda.stream(stream):
            reset()
        stream.synchronize()
        acc_t = {}

        def collect(call, n):
            torch.cuda.synchronize()
            assert n == len(plan[call]), f"{call}: {n} launches, plan has {len(plan[call])}"
            for i, (lab, kind, b, f) in enumerate(plan[call]):
                acc_t.setdefault((lab, kind, b), []).append(evs[i].elapsed_time(evs[i + 1]))

        for _ in range(a.trace_steps):
            with torch.cuda.stream(stream):
                dr.inject(hid_step, B, accept, batch)
            collect("inject", dr.last_launch_count())
            with torch.cuda.stream(stream):
                dr.draft(batch, B, drafted)
            collect("draft", dr.last_launch_count())
            with torch.cuda.stream(stream):
                BND.synth_plant(noise, drafted, masks, n_masks, step_ctr, batch, B, 10.0, saved)
                dr.verify(noise, drafted, batch, B, accept, committed)
            collect("verify", dr.last_launch_count())
            with torch.cuda.stream(stream):
                BND.synth_unplant(noise, step_ctr, n_masks, batch, B, saved)
        dr.trace_events([])
        stream.synchronize()
        sum_b = sum_t = 0.0
        for (lab, kind, b), ts in acc_t.items():
            us = 1e3 * sum(ts) / len(ts)
            k = kern.setdefault(lab, {"us": 0.0, "launches_per_step": 0, "bytes": 0})
            n_per = len(ts) // a.trace_steps
            k["us"] = round((k["us"] * k["launches_per_step"] + us * n_per) / (k["launches_per_step"] + n_per), 2)
            k["launches_per_step"] += n_per
            k["bytes"] = b
            k["gbs"] = round(b / (k["us"] * 1e-6) / 1e9, 1) if b else None
            if kind == "gemv":
                sum_b += b * len(ts)
                sum_t += sum(ts) * 1e-3
        # the dominant kernel: the gemv launch kind with the largest share of the step
        dom = max((lab for (lab, kind, _) in acc_t if kind == "gemv"),
                  key=lambda lab: kern[lab]["us"] * kern[lab]["launches_per_step"])
        achieved = kern[dom]["bytes"] / (kern[dom]["us"] * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": f"gemv_kernel, launch {dom} (weight-streaming tcgen05 GEMM chain)",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": measured_traffic(dom, w.name), "peak_kind": f"{pk_kind} hbm_gbs (copy bandwidth)",
                "algorithmic_bytes": kern[dom]["bytes"], "us_per_launch": kern[dom]["us"],
                "all_gemv_launches": {"achieved": round(sum_b / sum_t / 1e9, 1),
                                      "frac": round(sum_b / sum_t / 1e9 / hbm, 4)},
                "timing": "per-launch CUDA events on the launching stream, one traced step"}
        log("[bench] per-kernel: " + json.dumps(kern))
        with torch.cuda.stream(stream):
            reset()
        stream.synchronize()

    # ---------------------------------------------------------------- in-graph attention (timeline)
    # The traced pass serialises launches; here one graph-replayed step records per-CTA
    # %globaltimer stamps instead, and each attention launch is charged the time from the
    # last CTA exit of the launch before it to its own last CTA exit (the time it adds to
    # the step, programmatic overlap included).
    attn_graph = None
    if a.trace_steps > 0:
        rec = torch.zeros(32768, 37, dtype=torch.int64, device="cuda")
        dr.timeline(rec)
        g_tl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_tl, stream=stream):
            inject_draft()
            plant_verify()
        used = dr.timeline_used()
        dr.timeline(None)
        if used <= rec.shape[0]:
            with torch.cuda.stream(stream):
                reset()
                g_tl.replay()   # warm
                reset()
                rec.zero_()
                g_tl.replay()
                reset()
            stream.synchronize()
            r = rec[:used].cpu().numpy()
            lid = r[:, 0] & 0xFFFFFFFF
            kind = r[:, 0] >> 32
            ends = {int(l): int(r[lid == l, 36].max()) for l in np.unique(lid)}
            order = sorted(ends)
            adds = [ends[l] - ends[order[i - 1]] for i, l in enumerate(order)
                    if i > 0 and int(kind[lid == l][0]) == 2]
            if adds:
                ab_bytes = attn_bytes_flops(s, batch, B, n_avg)[0]
                us = 1e-3 * float(np.mean(adds))
                attn_graph = {"us_per_layer": round(us, 2), "bytes": ab_bytes,
                              "achieved_gbs": round(ab_bytes / (us * 1e-6) / 1e9, 1),
                              "frac_of_hbm": round(ab_bytes / (us * 1e-6) / 1e9 / hbm, 4),
                              "layers": len(adds),
                              "how": "one graph-replayed step with per-CTA timeline stamps: last CTA exit "
                                     "of each attention launch minus that of the launch before it"}
                log(f"[bench] attention in graph: {us:.1f} us per layer")
        del g_tl, rec

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not a.no_e2e:
        hid_host = hid_step_cpu.pin_memory()
        noise_host = noise_cpu.clone().pin_memory()
        logits_dev = torch.empty_like(noise)
        drafted_host = torch.empty(drafted.shape, dtype=torch.int32).pin_memory()
        acc_host = torch.empty(batch, dtype=torch.int32).pin_memory()
        com_host = torch.empty(batch, B, dtype=torch.int32).pin_memory()
        gA, gB = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gA, stream=stream):
            dr.inject(hid_step, B, accept, batch)
            dr.draft(batch, B, drafted)
        with torch.cuda.graph(gB, stream=stream):
            dr.verify(logits_dev, drafted, batch, B, accept, committed)
        with torch.cuda.stream(stream):
            reset()
        stream.synchronize()
        nh = noise_host.numpy()

        def e2e_step(k):
            with torch.cuda.stream(stream):
                hid_step.copy_(hid_host, non_blocking=True)
                gA.replay()
                drafted_host.copy_(drafted, non_blocking=True)
            stream.synchronize()
            d = drafted_host.numpy()
            m = masks_np[k % n_masks]
            planted = []
            for si in range(batch):
                for i in range(B - 1):
                    if m[si, i]:
                        planted.append((si, i, int(d[si, i])))
                        nh[si, i, int(d[si, i])] += np.float32(10.0)
            with torch.cuda.stream(stream):
                logits_dev.copy_(noise_host, non_blocking=True)
                gB.replay()
                acc_host.copy_(accept, non_blocking=True)
                com_host.copy_(committed, non_blocking=True)
            stream.synchronize()
            for si, i, tk in planted:
                nh[si, i, tk] -= np.float32(10.0)

        for k in range(min(a.warmup, 3)):
            e2e_step(k)
        with torch.cuda.stream(stream):
            reset()
        stream.synchronize()
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for k in range(a.steps):
            e2e_step(k)
        t1 = time.perf_counter()
        el = t1 - t0
        el = max_over_ranks(el, ws)
        e2e = {"value": job_rate(ws, batch, a.steps, el), "unit": UNIT,
               "h2d_bytes_per_step": hid_host.numel() * 2 + noise_host.numel() * 4,
               "d2h_bytes_per_step": drafted_host.numel() * 4 + acc_host.numel() * 4 + com_host.numel() * 4,
               "ms_per_step": 1e3 * el / a.steps,
               "path": "C ABI calls with pinned host buffers; host plants the synthetic target's agreement"}

    # ---------------------------------------------------------------- CPU baseline (oracle)
    cpu = None
    if rank == 0 and ws == 1 and not a.no_cpu_baseline:
        ctx_bits = I.bf16_bits(I.make_hidden(s, w.ctx, a.seed, "ctx"))
        step_bits = I.bf16_bits(hid_step_cpu[:, :B])
        masks_l = [masks_np[i][0] for i in range(len(masks_np))]
        t0 = time.perf_counter()
        n, secs = oracle_steps(s, weights_cpu.bits(), w, a.seed, 50, a.cpu_budget_s, ctx_bits, step_bits,
                               noise_cpu.numpy()[0], masks_l)
        log(f"[bench] oracle: {n} steps in {secs:.1f}s (+ prefill, total {time.perf_counter() - t0:.1f}s)")
        cpu = {"value": n / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n} oracle steps of this workload (one sequence: inject + B={B} draft + verify, fp64 "
                         f"NumPy) after an untimed prefill of {w.ctx} positions"}

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
    clk = clocks.summary(th0, th1, gpu_index if gpu_index.isdigit() else None)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) hidden states and logits)",
            "config": workload_config(w, ws, a.seed),
            "launch": "one CUDA graph per step, programmatic dependent launch between kernels",
            "attn_mode": a.attn_mode,
            "drafted_tok_per_s": value * (B - 1), "committed_tok_per_s": value * mean_tau, "mean_tau": mean_tau,
            "draft_ms": draft_ms, "draft_ms_by_block": draft_by_block, "fused_target_verify": fused,
            "prefill": prefill,
            "draft_flatness": (max(draft_by_block.values()) / min(draft_by_block.values())) if draft_by_block else None,
            "roofline": roof, "step_roofline": step_roof, "kernels": kern, "attention_in_graph": attn_graph,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": per_step_launches * a.steps, "launches_per_step": launches,
            "clocks": clk, "device_error": err,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_cuda(a)


if __name__ == "__main__":
    main()
