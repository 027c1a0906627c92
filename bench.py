"""Benchmark of the paged KV-cache attention hot path on GB300.

One step = one pass of the whole hot path over the big-pool workload: a 20,000-token request whose 23
blocks sit at the top (blocks 2,577-2,599) of a 2,600-block pool (block_size 880, 4 KV heads,
head_dim 256, 16 query heads), its last 2,048-token causal chunk prefilled
  (1) exact QK over the bf16 pool                                  [paged_prefill_attn]
  (2) int8 QK: quantize the chunk's 2,048 new K rows, then attend  [kv_int8_stats_quant + paged_prefill_attn]
  (3) fp8 e4m3 KV: dequantize [0, 20,000) into the dense bf16 scratch, then attend
                                                                   [kv_fp8_dequant_dense + paged_prefill_attn]
and an 8-token speculative verify of the same request over an int8 per-token-head copy of its
cache at the same blocks                                           [spec_verify_attn_partial + combine].
`value` = attention tokens per second over the whole step (3 x 2,048 prefill + 8 verify tokens).
The line also carries per-kernel rates (prefill TFLOP/s against the bf16 tensor peak, HBM GB/s of
the quant / dequant / verify passes) and, measured in the same run outside the step, the 32-request
verify batch (lognormal 4k-80k prefixes, median 16k) as verify HBM GB/s.

--impl reference times the CPU oracle (the reference arm of this build) on a bounded sample of the
same step. Inputs are seeded and synthetic; no dataset or weights are involved.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import workloads as W  # noqa: E402

METRIC = "paged prefill-attn tok/s & TFLOP/s (% tensor peak); verify-attn HBM GB/s"
CHUNK = W.BIGPOOL_CHUNK
L = W.BIGPOOL_L
T_VERIFY = 8
SPLIT = 4096  # verify split for the CPU oracle's sample (any split gives the same result)
HQ, HKV, D, BS = 16, 4, 256, W.BIGPOOL_BS
FLOP_PER_PAIR = 4 * D * HQ  # QK and PV, 2 flops per MAC, all 16 query heads


def prefill_pairs(seq_len, q_len):
    """causal (query, key) pairs of a chunk: queries at seq_len-q_len .. seq_len-1."""
    s = seq_len - q_len
    return q_len * s + q_len * (q_len + 1) // 2


def pick_split(seq_lens, n_sms, hkv=HKV):
    """split_tokens for a verify launch: the largest of 4096, 2048, 1024, 512 that still gives at
    least two CTAs per SM (larger splits mean fewer partials to write and combine; smaller ones fill
    the GPU when there are few or short requests)."""
    split = 4096
    while split > 512 and hkv * sum(math.ceil(int(s) / split) for s in seq_lens) < 2 * n_sms:
        split //= 2
    return split


def verify_bytes(seq_lens, T=T_VERIFY, hq=HQ):
    """algorithmic HBM bytes of a verify batch: int8 K and V (2*Hkv*D per token), their fp32
    per-token-head scales (2*Hkv*4), q and out bf16 (T*Hq*D*2 each) per request."""
    return sum(int(s) * (2 * HKV * D + 2 * HKV * 4) + 2 * T * hq * D * 2 for s in seq_lens)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()  # median SM clock under load, max clock, active slowdown reasons
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

class Workload:
    """Device-resident inputs of one step (built once; not timed)."""

    def __init__(self, torch, pkv, dev):
        from _devsetup import device_meta, device_pool, device_q, device_scale_pool, u16_to_bf16
        self.torch, self.pkv = torch, pkv
        # (1)/(2): bf16 pool, request at the top
        p = W.bigpool(top=True, q_len=CHUNK)
        self.p = p
        self.k, self.v = device_pool(p, "k"), device_pool(p, "v")
        self.bt, self.sl, self.qsl = device_meta(p)
        self.q = device_q(p)
        self.out = [torch.empty_like(self.q) for _ in range(3)]
        self.k8 = torch.zeros((1, L, HKV, D), dtype=torch.int8, device=dev)
        self.k8s = torch.zeros((1, L, HKV), dtype=torch.float32, device=dev)
        self.k16 = torch.zeros((1, L, HKV, D), dtype=torch.float16, device=dev)  # fp16 copy of the codes
        self.pos_begin = torch.tensor([L - CHUNK], dtype=torch.int32, device=dev)
        self.zero = torch.zeros(1, dtype=torch.int32, device=dev)
        # the earlier chunks' int8 K rows (quantized by previous steps of a real prefill)
        pkv.kv_int8_stats_quant(self.k, self.bt, self.zero, self.sl, L, self.k8, self.k8s, k16=self.k16)
        # (3): the same request as e4m3 codes (values N(0,1)*0.5: codes of N(0,1), per-tensor scale 0.5)
        pf = W.make_problem("bench_fp8", seed=2, seq_lens=[L], q_lens=[CHUNK], num_blocks=W.BIGPOOL_BLOCKS,
                            block_size=BS, kv_dtype="e4m3", placement="explicit",
                            block_lists=[p.requests[0].blocks])
        self.kf, self.vf = device_pool(pf, "k"), device_pool(pf, "v")
        self.fscale = torch.tensor([0.5], dtype=torch.float32, device=dev)
        self.kd = torch.empty((1, L, HKV, D), dtype=torch.bfloat16, device=dev)
        self.vd = torch.empty_like(self.kd)
        self.ident = torch.zeros((1, 1), dtype=torch.int32, device=dev)
        # (4): verify of the same request over an int8 per-token-head pool at the same blocks
        nbv = (L + T_VERIFY + BS - 1) // BS
        first = W.BIGPOOL_BLOCKS - nbv
        pv = W.make_problem("bench_verify", seed=62, seq_lens=[L + T_VERIFY], q_lens=[T_VERIFY],
                            num_blocks=W.BIGPOOL_BLOCKS, block_size=BS, kv_dtype="int8", placement="explicit",
                            block_lists=[np.arange(first, first + nbv)], softmax_scale=1.0 / 16.0)
        self.pv = pv
        self.vk, self.vv = device_pool(pv, "k"), device_pool(pv, "v")
        self.vks, self.vvs = device_scale_pool(pv, "k"), device_scale_pool(pv, "v")
        self.vbt, self.vsl, _ = device_meta(pv)
        self.vq = device_q(pv)
        self.split = pick_split([L + T_VERIFY], torch.cuda.get_device_properties(dev).multi_processor_count)
        S = pkv.splits_needed(L + T_VERIFY, self.split)
        self.po = torch.empty((S, T_VERIFY, HQ, D), dtype=torch.float32, device=dev)
        self.pl = torch.empty((S, T_VERIFY, HQ), dtype=torch.float32, device=dev)
        self.vout = torch.empty_like(self.vq)
        self.host_q = None
        # the persistent prefill launch (one CTA per SM: full waves of whole query tiles, the last
        # partial wave cut into key ranges and merged) needs a workspace; every prefill uses it
        self.ws = torch.empty(pkv.paged_prefill_workspace_bytes(), dtype=torch.uint8, device=dev)
        del u16_to_bf16

    def step(self, ev=None):
        """Enqueue one step; ev: optional list of (name, start, end) CUDA event pairs to record."""
        pkv, s = self.pkv, self.p.softmax_scale

        def rec(name, fn):
            if ev is None:
                fn()
            else:
                a, b = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                ev.append((name, a, b))

        rec("prefill_bf16", lambda: pkv.paged_prefill_attn(self.q, self.k, self.v, self.bt, self.sl, self.qsl, CHUNK,
                                                           s, self.out[0], workspace=self.ws))
        rec("int8_quant", lambda: pkv.kv_int8_stats_quant(self.k, self.bt, self.pos_begin, self.sl, CHUNK, self.k8,
                                                          self.k8s, k16=self.k16))
        rec("prefill_int8", lambda: pkv.paged_prefill_attn(self.q, None, self.v, self.bt, self.sl, self.qsl, CHUNK, s,
                                                           self.out[1], qk_mode=pkv.PKV_QK_INT8, k8_scale=self.k8s,
                                                           k16=self.k16, workspace=self.ws))
        rec("fp8_dequant", lambda: pkv.kv_fp8_dequant_dense(self.kf, self.vf, self.bt, self.sl, self.fscale,
                                                            self.fscale, self.kd, self.vd))
        rec("prefill_fp8_dense", lambda: pkv.paged_prefill_attn(self.q, self.kd, self.vd, self.ident, self.sl,
                                                                self.qsl, CHUNK, s, self.out[2], workspace=self.ws))
        rec("verify_partial", lambda: pkv.spec_verify_attn_partial(self.vq, self.vk, self.vv, self.vks, self.vvs,
                                                                   self.vbt, self.vsl, T_VERIFY, self.pv.softmax_scale,
                                                                   self.split, self.po, self.pl))
        rec("verify_combine", lambda: pkv.spec_verify_combine(self.po, self.pl, self.vsl, T_VERIFY, self.split,
                                                              self.vout))

    LAUNCHES_PER_STEP = 10  # 3 prefills x (persistent kernel + merge), quant, dequant, verify partial + combine
    TOKENS_PER_STEP = 3 * CHUNK + T_VERIFY


def algorithmic():
    pairs = prefill_pairs(L, CHUNK)
    return {
        "prefill_flops": pairs * FLOP_PER_PAIR,
        "int8_quant_bytes": CHUNK * HKV * (2 * D + D + 4 + 2 * D),  # bf16 in; int8 + scale + fp16 copy out
        "fp8_dequant_bytes": L * HKV * D * 2 * (1 + 2),
        "verify_bytes": verify_bytes([L + T_VERIFY]),
    }


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    from __graft_entry__ import build
    build()
    import paged_kv_cache_int64_gb300 as pkv

    wl = Workload(torch, pkv, dev)
    alg = algorithmic()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 512 MB > 129 MB L2

    # warm-up (also the first call of every kernel: attribute setup, module load)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # timed region: K steps, L2 flushed before each (outside the step's events)
    step_ms, per_kernel = [], {}
    barrier()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            evs = []
            a.record()
            wl.step(evs)
            b.record()
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
            for name, x, y in evs:
                per_kernel.setdefault(name, []).append(x.elapsed_time(y))
        barrier()
        wall = time.perf_counter() - t_wall
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    # end-to-end through the public API from pinned host memory
    e2e = run_e2e(torch, pkv, wl, args, dev)

    # verify batch (32 requests), measured in the same run, outside the step
    vb = run_verify_batch(torch, pkv, dev, flush, args) if not args.skip_batch else None
    # the two fp8 prefill paths on the step's fp8 chunk: dequantize once into the dense scratch, or
    # dequantize every tile inside the prefill
    fp8_paths = run_fp8_paths(torch, pkv, wl, flush, args)
    prefill_launches = run_prefill_launches(torch, pkv, wl, flush, args)
    quant_full = run_quant_full_context(torch, pkv, wl, flush, args)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks = load_peaks()
    mean = {k: statistics.mean(v) for k, v in per_kernel.items()}
    pf_tflops = {k: alg["prefill_flops"] / (mean[k] * 1e-3) / 1e12 for k in mean if k.startswith("prefill")}
    dominant = max(mean, key=mean.get)
    traffic = load_traffic(dominant)
    if dominant.startswith("prefill"):
        achieved = pf_tflops[dominant]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic, "kernel": dominant,
                "peak_source": peaks["source"] + " (bf16 dense, burst)"}
    else:
        byts = {"int8_quant": alg["int8_quant_bytes"], "fp8_dequant": alg["fp8_dequant_bytes"],
                "verify_partial": alg["verify_bytes"]}.get(dominant, 0)
        achieved = byts / (mean[dominant] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": dominant,
                "peak_source": peaks["source"]}
    value = whole_job_value(wl.TOKENS_PER_STEP, args.steps, world, total_ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "bigpool_20000_last_chunk_2048: 2,600-block pool, block_size 880, request on blocks "
                               "2577-2599, 16 q / 4 kv heads, head_dim 256; step = bf16 + int8-QK + fp8-dense (persistent launch) "
                               "prefill of the chunk and an 8-token int8-KV verify",
                   "tokens_per_step": wl.TOKENS_PER_STEP, "l2": "flushed before every step (512 MB write)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "per_kernel_ms": {k: round(v, 4) for k, v in mean.items()},
        "prefill_attn": {k: {"tok_s": round(CHUNK / (mean[k] * 1e-3), 1), "tflops": round(v, 2),
                             "frac_bf16_peak": round(v / peaks["bf16_tflops"], 4)} for k, v in pf_tflops.items()},
        "hbm_passes": {
            "int8_quant": _gbs(alg["int8_quant_bytes"], mean.get("int8_quant"), peaks),
            "fp8_dequant": _gbs(alg["fp8_dequant_bytes"], mean.get("fp8_dequant"), peaks),
            "verify_single_request": _gbs(alg["verify_bytes"], mean.get("verify_partial", 0) +
                                          mean.get("verify_combine", 0), peaks),
            "int8_quant_full_context": quant_full,
        },
        "verify_batch": vb,
        "fp8_prefill_paths": fp8_paths,
        "prefill_launches": prefill_launches,
        "e2e": e2e,
        "gpu_launches": wl.LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, sample_tokens=args.cpu_sample)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The slowest rank's timing (every rank holds its own replica of the workload)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_step: int, steps: int, world: int, max_total_ms: float) -> float:
    """Weak scaling: all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_step * steps / (max_total_ms * 1e-3)


def _gbs(nbytes, ms, peaks):
    if not ms:
        return None
    g = nbytes / (ms * 1e-3) / 1e9
    return {"gbs": round(g, 1), "frac_hbm": round(g / peaks["hbm_gbs"], 4), "ms": round(ms, 4)}


def load_traffic(kernel):
    """dram read + write bytes per launch of `kernel` from the committed ncu capture, or None when
    there is none or the kernel source has changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            ent = json.load(f).get(kernel)
        if not ent:
            return None
        with open(os.path.join(ROOT, ent["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != ent["source_sha256"]:
                return None
        return int(ent["dram_bytes_per_launch"])
    except Exception:
        return None


def run_e2e(torch, pkv, wl, args, dev):
    """Same step through the public API with host buffers: every step copies its q (and verify q)
    in from pinned memory and every output back, inside the timed region. The copies run on their
    own streams, pipelined as a serving loop would: two sets of device inputs and outputs alternate,
    so step i+1's inputs land and step i's outputs leave while the kernels of the other step run."""
    hq = wl.q.cpu().pin_memory()
    hvq = wl.vq.cpu().pin_memory()
    houts = [torch.empty_like(o, device="cpu").pin_memory() for o in wl.out]
    hvout = torch.empty_like(wl.vout, device="cpu").pin_memory()
    h2d = hq.numel() * 2 + hvq.numel() * 2
    d2h = sum(o.numel() * 2 for o in houts) + hvout.numel() * 2
    steps = max(1, args.steps)
    bufs = [(wl.q, wl.vq, wl.out, wl.vout),
            (torch.empty_like(wl.q), torch.empty_like(wl.vq), [torch.empty_like(o) for o in wl.out],
             torch.empty_like(wl.vout))]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for i in range(steps):
        k = i & 1
        q, vq, outs, vout = bufs[k]
        with torch.cuda.stream(s_in):  # inputs of step i, once step i-2 no longer reads this set
            s_in.wait_event(a)
            if i >= 2:
                s_in.wait_event(ev_done[k])
            q.copy_(hq, non_blocking=True)
            vq.copy_(hvq, non_blocking=True)
            ev_in[k].record(s_in)
        comp.wait_event(ev_in[k])
        if i >= 2:
            comp.wait_event(ev_out[k])  # step i-2's outputs have left this set
        wl.q, wl.vq, wl.out, wl.vout = q, vq, outs, vout
        wl.step()
        ev_done[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            for h, o in zip(houts, outs):
                h.copy_(o, non_blocking=True)
            hvout.copy_(vout, non_blocking=True)
            ev_out[k].record(s_out)
    comp.wait_event(ev_out[(steps - 1) & 1])
    b.record(comp)
    b.synchronize()
    wl.q, wl.vq, wl.out, wl.vout = bufs[0]
    ms = a.elapsed_time(b)
    return {"value": round(wl.TOKENS_PER_STEP * steps / (ms * 1e-3), 1), "unit": "tok/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": "copies on their own streams, two alternating sets of device inputs/outputs",
            "l2": "not flushed between steps (a serving loop), unlike the device-timed step"}


def run_quant_full_context(torch, pkv, wl, flush, args):
    """kv_int8_stats_quant over the request's whole 20,000-token context (a from-scratch prefill's
    quantization, 80,000 rows: 103 MB moved) rather than one 2,048-token chunk, whose 10 MB pass
    is launch- and latency-bound."""
    peaks = load_peaks()
    nbytes = L * HKV * (2 * D + D + 4 + 2 * D)

    def fn():
        pkv.kv_int8_stats_quant(wl.k, wl.bt, wl.zero, wl.sl, L, wl.k8, wl.k8s, k16=wl.k16)

    for _ in range(max(3, args.warmup)):
        fn()
    ts = []
    for _ in range(max(5, min(args.steps, 50))):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return _gbs(nbytes, statistics.mean(ts), peaks)


def run_prefill_launches(torch, pkv, wl, flush, args):
    """The step's bf16 and int8-QK prefills launched both ways: one CTA per query tile (no
    workspace) and the persistent grid the step uses. CUDA events, L2 flushed before each call."""
    s = wl.p.softmax_scale
    out = torch.empty_like(wl.q)
    calls = {
        "bf16": lambda ws: pkv.paged_prefill_attn(wl.q, wl.k, wl.v, wl.bt, wl.sl, wl.qsl, CHUNK, s, out, workspace=ws),
        "int8": lambda ws: pkv.paged_prefill_attn(wl.q, None, wl.v, wl.bt, wl.sl, wl.qsl, CHUNK, s, out,
                                                  qk_mode=pkv.PKV_QK_INT8, k8_scale=wl.k8s, k16=wl.k16, workspace=ws),
    }
    flops = algorithmic()["prefill_flops"]
    res = {}
    for name, fn in calls.items():
        for ws in (None, wl.ws):
            for _ in range(max(3, args.warmup)):
                fn(ws)
        t = {"per_query_tile": [], "persistent": []}
        for _ in range(max(5, min(args.steps, 30))):
            for kind, ws in (("per_query_tile", None), ("persistent", wl.ws)):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn(ws)
                b.record()
                b.synchronize()
                t[kind].append(a.elapsed_time(b))
        res[name] = {k: {"ms": round(statistics.mean(v), 4),
                         "tflops": round(flops / (statistics.mean(v) * 1e-3) / 1e12, 2)} for k, v in t.items()}
    return res


def run_fp8_paths(torch, pkv, wl, flush, args):
    """Chunk of 2,048 queries at the end of the 20,000-token e4m3 context, both fp8 prefill paths:
    kv_fp8_dequant_dense + bf16 prefill on the scratch, against paged_prefill_attn_fp8 (per-tile
    dequantization). CUDA events, L2 flushed before every repetition."""
    s = wl.p.softmax_scale
    out = torch.empty_like(wl.q)

    def dense():
        pkv.kv_fp8_dequant_dense(wl.kf, wl.vf, wl.bt, wl.sl, wl.fscale, wl.fscale, wl.kd, wl.vd)

    def dense_attn():
        pkv.paged_prefill_attn(wl.q, wl.kd, wl.vd, wl.ident, wl.sl, wl.qsl, CHUNK, s, out, workspace=wl.ws)

    def fused():
        pkv.paged_prefill_attn_fp8(wl.q, wl.kf, wl.vf, wl.fscale, wl.fscale, wl.bt, wl.sl, wl.qsl, CHUNK, s, out,
                                   workspace=wl.ws)

    for _ in range(max(3, args.warmup)):
        dense(); dense_attn(); fused()
    t = {"dequant": [], "attn": [], "fused": []}
    for _ in range(max(5, min(args.steps, 50))):
        for name, fn in (("dequant", dense), ("attn", dense_attn), ("fused", fused)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            t[name].append(a.elapsed_time(b))
    m = {k: statistics.mean(v) for k, v in t.items()}
    flops = algorithmic()["prefill_flops"]
    tf = lambda ms: round(flops / (ms * 1e-3) / 1e12, 2)
    return {"dense": {"dequant_ms": round(m["dequant"], 4), "attn_ms": round(m["attn"], 4),
                      "total_ms": round(m["dequant"] + m["attn"], 4), "attn_tflops": tf(m["attn"]),
                      "tflops_incl_dequant": tf(m["dequant"] + m["attn"])},
            "fused": {"ms": round(m["fused"], 4), "tflops": tf(m["fused"])},
            "note": "each dense-path step dequantizes the request's whole context [0, seq_len) once"}


def run_verify_batch(torch, pkv, dev, flush, args):
    """32-request verify batch (distinct blocks): HBM GB/s of partial + combine. The same cache also
    serves two other query geometries: a one-token decode step (T = 1, 16/4 heads) and the pages'
    24/4 heads with T = 8 (48 query columns per KV head, two CTAs per key range)."""
    from _devsetup import device_meta, device_pool, device_q, device_scale_pool, u16_to_bf16
    p = W.verify_batch()
    k, v = device_pool(p, "k"), device_pool(p, "v")
    ks, vs = device_scale_pool(p, "k"), device_scale_pool(p, "v")
    bt, _, _ = device_meta(p)
    peaks = load_peaks()

    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def measure(q, seq_lens, T, hq):
        sld = torch.from_numpy(np.asarray(seq_lens, dtype=np.int32)).to(dev)
        split = pick_split(seq_lens, n_sms)
        S = pkv.splits_needed(int(max(seq_lens)), split)
        po = torch.empty((S, q.shape[0], hq, D), dtype=torch.float32, device=dev)
        pl = torch.empty((S, q.shape[0], hq), dtype=torch.float32, device=dev)
        out = torch.empty_like(q)
        for _ in range(max(3, args.warmup)):
            pkv.spec_verify_attn_partial(q, k, v, ks, vs, bt, sld, T, p.softmax_scale, split, po, pl)
            pkv.spec_verify_combine(po, pl, sld, T, split, out)
        times, tp, tc = [], [], []
        for _ in range(max(5, args.steps)):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            pkv.spec_verify_attn_partial(q, k, v, ks, vs, bt, sld, T, p.softmax_scale, split, po, pl)
            e[1].record()
            pkv.spec_verify_combine(po, pl, sld, T, split, out)
            e[2].record()
            e[2].synchronize()
            times.append(e[0].elapsed_time(e[2]))
            tp.append(e[0].elapsed_time(e[1]))
            tc.append(e[1].elapsed_time(e[2]))
        nbytes = verify_bytes(seq_lens, T, hq)
        ms = statistics.mean(times)
        g = nbytes / (ms * 1e-3) / 1e9
        gp = nbytes / (statistics.mean(tp) * 1e-3) / 1e9
        return {"requests": p.num_reqs, "T": T, "q_heads": hq, "sum_seq_len": int(np.sum(seq_lens)),
                "algorithmic_bytes": int(nbytes), "ms": round(ms, 4), "gbs": round(g, 1),
                "frac_hbm": round(g / peaks["hbm_gbs"], 4), "partial_ms": round(statistics.mean(tp), 4),
                "partial_gbs": round(gp, 1), "combine_ms": round(statistics.mean(tc), 4), "split_tokens": split}

    res = measure(device_q(p), p.seq_lens, T_VERIFY, HQ)
    res["partial_dram_bytes"] = load_traffic("verify_partial")  # ncu capture of this batch's partial launch
    # decode: the first token of each request's verify window, alone
    dec_lens = p.seq_lens - (T_VERIFY - 1)
    res["decode_t1"] = measure(u16_to_bf16(W.bf16_normal(7, (p.num_reqs, HQ, D))).to(dev), dec_lens, 1, HQ)
    q24 = u16_to_bf16(W.bf16_normal(8, (p.num_reqs * T_VERIFY, 24, D))).to(dev)
    res["heads_24x4"] = measure(q24, p.seq_lens, T_VERIFY, 24)
    return res


# ----------------------------------------------------------------------------------------------
# CPU oracle (baseline arm)
# ----------------------------------------------------------------------------------------------

def cpu_baseline(args, sample_tokens=None):
    """Time the oracle on a bounded sample of one step and scale to the step's tokens.

    Sample: `sample_tokens` query tokens (all 16 heads) of each of the three prefill passes, the
    int8 quantization and fp8 dequantization of the matching share of rows, and the whole 8-token
    verify; each part's time is scaled by (full units / sampled units)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    if not sample_tokens:
        sample_tokens = os.cpu_count() or 1
    cores = min(os.cpu_count() or 1, sample_tokens)
    p = W.bigpool(top=True, q_len=CHUNK)
    kp, vp = p.pool_numpy("k"), p.pool_numpy("v")
    bt = p.block_table(fill=0)
    toks = np.linspace(0, CHUNK - 1, sample_tokens).astype(int)
    parts = {}

    def timed(name, fn, scale):
        t0 = time.perf_counter()
        fn()
        parts[name] = (time.perf_counter() - t0) * scale

    pool = ThreadPoolExecutor(max_workers=cores)

    def over_tokens(mode, k8=None, ks=None, kpool=kp, vpool=vp, table=bt):
        futs = [pool.submit(oracle.paged_prefill_attn, p.q, kpool, vpool, table, p.seq_lens, p.query_start_loc, HQ,
                            p.softmax_scale, mode, k8, ks, int(t), int(t) + 1) for t in toks]
        return [f.result() for f in futs]

    # A1 over the sampled share of the chunk's new rows, then int8 prefill of the sampled tokens
    k8, ks = oracle.kv_int8_stats_quant(kp, bt, [0], [L], BS, L)  # earlier positions (setup, untimed)
    n_q = max(1, CHUNK * sample_tokens // CHUNK)
    timed("int8_quant", lambda: oracle.kv_int8_stats_quant(kp, bt, [L - n_q], [L], BS, L), CHUNK / n_q)
    timed("prefill_bf16", lambda: over_tokens(0), CHUNK / sample_tokens)
    timed("prefill_int8", lambda: over_tokens(1, k8, ks), CHUNK / sample_tokens)
    # A4 on a share of positions; the dense scratch for the sampled fp8 prefill tokens
    pf = W.make_problem("bench_fp8", seed=2, seq_lens=[L], q_lens=[CHUNK], num_blocks=W.BIGPOOL_BLOCKS,
                        block_size=BS, kv_dtype="e4m3", placement="explicit", block_lists=[p.requests[0].blocks])
    fk, fv = pf.pool_numpy("k"), pf.pool_numpy("v")
    n_d = 2000
    timed("fp8_dequant", lambda: oracle.kv_fp8_dequant_dense(fk, fv, bt, [n_d], n_d, 0.5, 0.5), L / n_d)
    kd, vd = oracle.kv_fp8_dequant_dense(fk, fv, bt, [L], L, 0.5, 0.5)
    ident = np.zeros((1, 1), np.int32)
    timed("prefill_fp8_dense", lambda: over_tokens(0, kpool=kd.reshape(1, L, HKV, D), vpool=vd.reshape(1, L, HKV, D),
                                                   table=ident), CHUNK / sample_tokens)
    # verify: the whole 8-token verify of the request
    nbv = (L + T_VERIFY + BS - 1) // BS
    pv = W.make_problem("bench_verify", seed=62, seq_lens=[L + T_VERIFY], q_lens=[T_VERIFY],
                        num_blocks=W.BIGPOOL_BLOCKS, block_size=BS, kv_dtype="int8", placement="explicit",
                        block_lists=[np.arange(W.BIGPOOL_BLOCKS - nbv, W.BIGPOOL_BLOCKS)], softmax_scale=1.0 / 16.0)
    vargs = (pv.q, pv.pool_numpy("k"), pv.pool_numpy("v"), pv.scale_pool_numpy("k"), pv.scale_pool_numpy("v"),
             pv.block_table(fill=0), pv.seq_lens)

    def verify():
        S = math.ceil((L + T_VERIFY) / SPLIT)
        po, pl = oracle.spec_verify_partial(*vargs, T_VERIFY, HQ, pv.softmax_scale, SPLIT, S)
        oracle.spec_verify_combine(po, pl, pv.seq_lens, T_VERIFY, SPLIT)

    timed("verify", verify, 1.0)
    pool.shutdown()
    step_s = sum(parts.values())
    return {"value": round(Workload.TOKENS_PER_STEP / step_s, 3), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample_tokens} query tokens x 16 heads of each prefill pass, {n_q} quantized rows, "
                      f"{n_d} dequantized positions, the full 8-token verify; each scaled to one step",
            "part_seconds_per_step": {k: round(v, 3) for k, v in parts.items()}}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; W untimed steps are not needed
    vals = []
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(args, sample_tokens=args.cpu_sample)
        vals.append(last["value"])
    value = statistics.mean(vals)
    line = {"metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * Workload.TOKENS_PER_STEP / value, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": "bigpool_20000_last_chunk_2048 (bounded sample per step)",
                       "tokens_per_step": Workload.TOKENS_PER_STEP},
            "cpu_baseline": {k: last[k] for k in ("kind", "cores", "sample")} | {"value": round(value, 3)},
            "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ncu_case(args):
    """A small, self-contained case of one kernel for profiler capture (not a bench line): the big-pool
    request (20,000 tokens, last 2,048-token chunk) in a 64-block pool (the request's 23 blocks at its
    top), or the 32-request verify batch, launched `--steps` times after `--warmup` launches."""
    import torch
    from __graft_entry__ import build
    build()
    import paged_kv_cache_int64_gb300 as pkv
    from _devsetup import device_meta, device_pool, device_q, device_scale_pool
    dev = "cuda:0"
    torch.cuda.set_device(0)
    case = args.ncu_case
    if case == "verify":
        p = W.verify_batch()
        k, v = device_pool(p, "k"), device_pool(p, "v")
        ks, vs = device_scale_pool(p, "k"), device_scale_pool(p, "v")
        bt, sl, _ = device_meta(p)
        q = device_q(p)
        split = pick_split(p.seq_lens, torch.cuda.get_device_properties(dev).multi_processor_count)
        S = pkv.splits_needed(int(p.seq_lens.max()), split)
        po = torch.empty((S, q.shape[0], HQ, D), dtype=torch.float32, device=dev)
        pl = torch.empty((S, q.shape[0], HQ), dtype=torch.float32, device=dev)
        out = torch.empty_like(q)

        def fn():
            pkv.spec_verify_attn_partial(q, k, v, ks, vs, bt, sl, T_VERIFY, p.softmax_scale, split, po, pl)
            pkv.spec_verify_combine(po, pl, sl, T_VERIFY, split, out)
    else:
        nb = 64
        kv_dtype = "e4m3" if case == "fp8_dequant" else "bf16"
        p = W.make_problem("ncu", seed=2, seq_lens=[L], q_lens=[CHUNK], num_blocks=nb, block_size=BS,
                           kv_dtype=kv_dtype, placement="explicit", block_lists=[np.arange(nb - 23, nb)],
                           softmax_scale=1.0 / 16.0)
        k, v = device_pool(p, "k"), device_pool(p, "v")
        bt, sl, qsl = device_meta(p)
        q = device_q(p)
        out = torch.empty_like(q)
        k8 = torch.zeros((1, L, HKV, D), dtype=torch.int8, device=dev)
        k8s = torch.zeros((1, L, HKV), dtype=torch.float32, device=dev)
        zero = torch.zeros(1, dtype=torch.int32, device=dev)
        pb = torch.tensor([L - CHUNK], dtype=torch.int32, device=dev)
        k16 = torch.zeros((1, L, HKV, D), dtype=torch.float16, device=dev)
        if case == "prefill_int8":
            pkv.kv_int8_stats_quant(k, bt, zero, sl, L, k8, k8s, k16=k16)
        kd = torch.empty((1, L, HKV, D), dtype=torch.bfloat16, device=dev)
        vd = torch.empty_like(kd)
        sc = torch.tensor([0.5], dtype=torch.float32, device=dev)
        ws = torch.empty(pkv.paged_prefill_workspace_bytes(), dtype=torch.uint8, device=dev)
        fns = {
            "prefill_bf16": lambda: pkv.paged_prefill_attn(q, k, v, bt, sl, qsl, CHUNK, p.softmax_scale, out),
            "prefill_bf16_persistent": lambda: pkv.paged_prefill_attn(q, k, v, bt, sl, qsl, CHUNK, p.softmax_scale,
                                                                      out, workspace=ws),
            "prefill_int8": lambda: pkv.paged_prefill_attn(q, None, v, bt, sl, qsl, CHUNK, p.softmax_scale, out,
                                                           qk_mode=pkv.PKV_QK_INT8, k8_scale=k8s, k16=k16,
                                                           workspace=ws),
            "int8_quant": lambda: pkv.kv_int8_stats_quant(k, bt, pb, sl, CHUNK, k8, k8s, k16=k16),
            "fp8_dequant": lambda: pkv.kv_fp8_dequant_dense(k, v, bt, sl, sc, sc, kd, vd),
        }
        fn = fns[case]
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": case, "launches": args.warmup + args.steps, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=0, help="query tokens per prefill pass (0: one per core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-batch", action="store_true")
    ap.add_argument("--ncu-case", choices=["prefill_bf16", "prefill_bf16_persistent", "prefill_int8", "int8_quant",
                                           "fp8_dequant", "verify"],
                    help="run one kernel on a small case for profiler capture instead of the bench")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
