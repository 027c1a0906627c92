"""Benchmark of the paged KV-cache attention hot path on GB300.

One step = one pass of the whole hot path over the pages' workloads, inputs resident on the device:
  big pool     exact-QK prefill of the last 2,048-token chunk of a 20,000-token request whose 23
               blocks are the top of a 2,600-block bf16 pool (block 880)        [paged_prefill_attn]
  int8 prefill a 24,576- and a 47,104-token context, each in 2,048-token chunks over a 2,600-block
               bf16 pool with a random table; every chunk quantizes its new K rows, then attends
               with int8 QK                       [kv_int8_stats_quant + paged_prefill_attn, int8 QK]
  fp8 prefill  a 32,768-token context of e4m3 K/V (per-tensor scales 0.5) in 2,048-token chunks;
               every chunk dequantizes [0, seq_len) into the dense bf16 scratch, then attends on
               it (identity table, block_size = 32,768)  [kv_fp8_dequant_dense + paged_prefill_attn]
  verify       32 requests, cached prefixes lognormal 4k-80k (median 16k), 8 draft tokens each,
               int8 per-token-head KV, block 880, split-KV partials and their log-sum-exp merge
                                                     [spec_verify_attn_partial + spec_verify_combine]
16 query / 4 KV heads and head_dim 256 throughout; the prefills use the persistent launch.
`value` = attention tokens per second over the step (prefilled tokens + verified draft tokens);
the line also carries, per workload, tok/s, TFLOP/s against the bf16 tensor peak and the HBM GB/s
of the quant / dequant / verify passes, and measurements taken outside the step (launch variants,
the fused fp8 prefill, other verify geometries and pools, whole-context quantization, cache writes).

--impl reference times the CPU oracle (the reference arm of this build) on a bounded sample of the
same workloads. Inputs are seeded and synthetic; no dataset or weights are involved.
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
T_VERIFY = 8
HQ, HKV, D, BS = 16, 4, 256, W.BIGPOOL_BS
POOL_BLOCKS = W.BIGPOOL_BLOCKS
FLOP_PER_PAIR = 4 * D * HQ  # QK and PV, 2 flops per MAC, all 16 query heads
INT8_CONTEXTS = (24576, 47104)
FP8_CONTEXT = 32768
QUANT_BYTES_PER_ROW = 2 * D + D + 4       # bf16 row in; int8 row + fp32 scale out (772 B)
K16_BYTES_PER_ROW = 2 * D                 # the optional fp16 copy of the codes (overhead)
DEQUANT_BYTES_PER_TOKEN = HKV * D * 2 * 3  # K and V: 1 B e4m3 in, 2 B bf16 out (6,144 B)


def prefill_pairs(seq_len, q_len):
    """causal (query, key) pairs of a chunk: queries at seq_len-q_len .. seq_len-1."""
    s = seq_len - q_len
    return q_len * s + q_len * (q_len + 1) // 2


def pick_split(pkv, seq_lens, n_sms, T=None, hq=None, hkv=HKV):
    """split_tokens for a verify launch: the library's planner (spec_verify_pick_split), which
    models the launch as a longest-first list schedule of its CTAs over the SMs from the batch's
    sequence lengths and returns the split with the shortest modelled time."""
    split = pkv.spec_verify_pick_split(seq_lens, T_VERIFY if T is None else T, HQ if hq is None else hq, hkv, n_sms)
    if split <= 0:
        raise ValueError("spec_verify_pick_split rejected the batch")
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
# the workloads of one step (host side: shared by the GPU arm and the oracle sample)
# ----------------------------------------------------------------------------------------------

def bigpool_problem():
    return W.bigpool(top=True, q_len=CHUNK)


def int8_problem(ctx):
    return W.make_problem(f"int8_ctx{ctx}", seed=33, seq_lens=[ctx], q_lens=[ctx], num_blocks=POOL_BLOCKS,
                          block_size=BS, softmax_scale=1.0 / 16.0)


def fp8_problem():
    """e4m3 codes of N(0,1) draws with per-tensor scale 0.5: dequantized values N(0,1) * 0.5."""
    return W.make_problem(f"fp8_ctx{FP8_CONTEXT}", seed=44, seq_lens=[FP8_CONTEXT], q_lens=[FP8_CONTEXT],
                          num_blocks=POOL_BLOCKS, block_size=BS, kv_dtype="e4m3", softmax_scale=1.0 / 16.0)


FP8_SCALE = 0.5


def verify_problem(distinct=True):
    return W.verify_batch(distinct=distinct)


def step_tokens():
    return CHUNK + sum(INT8_CONTEXTS) + FP8_CONTEXT + 32 * T_VERIFY


def algorithmic(verify_seq_lens):
    """algorithmic work of one step, per kernel class: prefill FLOPs per workload, quant and
    dequant bytes, verify bytes."""
    a = {"bigpool": {"prefill_flops": prefill_pairs(W.BIGPOOL_L, CHUNK) * FLOP_PER_PAIR}}
    for ctx in INT8_CONTEXTS:
        sched = W.chunk_schedule(ctx)
        a[f"int8_ctx{ctx}"] = {"prefill_flops": sum(prefill_pairs(L, q) for L, q in sched) * FLOP_PER_PAIR,
                               "quant_bytes": ctx * HKV * QUANT_BYTES_PER_ROW,
                               "k16_bytes": ctx * HKV * K16_BYTES_PER_ROW}
    sched = W.chunk_schedule(FP8_CONTEXT)
    a[f"fp8_ctx{FP8_CONTEXT}"] = {"prefill_flops": sum(prefill_pairs(L, q) for L, q in sched) * FLOP_PER_PAIR,
                                  "dequant_bytes": sum(L for L, _ in sched) * DEQUANT_BYTES_PER_TOKEN}
    a["verify_batch32"] = {"bytes": verify_bytes(verify_seq_lens)}
    return a


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

class Step:
    """Device-resident inputs of one step (built once; not timed) and the step's launches."""

    def __init__(self, torch, pkv, dev):
        from _devsetup import device_meta, device_pool, device_q, device_scale_pool
        self.torch, self.pkv, self.dev = torch, pkv, dev
        i32 = lambda xs: torch.tensor(xs, dtype=torch.int32, device=dev)
        self.ws = torch.empty(pkv.paged_prefill_workspace_bytes(), dtype=torch.uint8, device=dev)
        self.items = []  # (workload, kernel, fn, h2d [(dev, rows)], d2h [(dev, rows)]) in launch order

        # big pool: bf16, request on the top blocks, last chunk
        p = bigpool_problem()
        k, v = device_pool(p, "k"), device_pool(p, "v")
        bt, sl, qsl = device_meta(p)
        q = device_q(p)
        out = torch.empty_like(q)
        self.bigpool = dict(p=p, k=k, v=v, bt=bt, sl=sl, qsl=qsl, q=q, out=out)
        self._add("bigpool", "prefill_bf16", self._dense_prefill_fn(q, k, v, bt, sl, qsl, CHUNK, p.softmax_scale, out),
                  q, out)

        # int8 prefill of whole contexts, chunk by chunk
        self.int8 = {}
        for ctx in INT8_CONTEXTS:
            p = int8_problem(ctx)
            k, v = device_pool(p, "k"), device_pool(p, "v")
            bt, _, _ = device_meta(p)
            q_all = device_q(p)
            out_all = torch.empty_like(q_all)
            k8 = torch.zeros((1, ctx, HKV, D), dtype=torch.int8, device=dev)
            ks = torch.zeros((1, ctx, HKV), dtype=torch.float32, device=dev)
            k16 = torch.zeros((1, ctx, HKV, D), dtype=torch.float16, device=dev)
            self.int8[ctx] = dict(p=p, k=k, v=v, bt=bt, q=q_all, out=out_all, k8=k8, ks=ks, k16=k16)
            name = f"int8_ctx{ctx}"
            for L, ql in W.chunk_schedule(ctx):
                sl, pb, qsl = i32([L]), i32([L - ql]), i32([0, ql])
                q, out = q_all[L - ql:L], out_all[L - ql:L]
                self._add(name, "int8_quant", self._quant_fn(k, bt, pb, sl, ql, k8, ks, k16))
                self._add(name, "prefill_int8", self._int8_prefill_fn(q, v, bt, sl, qsl, ql, p.softmax_scale, out, ks,
                                                                      k16), q, out)

        # fp8 prefill through the dense scratch, chunk by chunk
        p = fp8_problem()
        k, v = device_pool(p, "k"), device_pool(p, "v")
        bt, _, _ = device_meta(p)
        q_all = device_q(p)
        out_all = torch.empty_like(q_all)
        kd = torch.zeros((1, FP8_CONTEXT, HKV, D), dtype=torch.bfloat16, device=dev)
        vd = torch.zeros_like(kd)
        sc = torch.tensor([FP8_SCALE], dtype=torch.float32, device=dev)
        ident = torch.zeros((1, 1), dtype=torch.int32, device=dev)
        self.fp8 = dict(p=p, k=k, v=v, bt=bt, q=q_all, out=out_all, kd=kd, vd=vd, sc=sc, ident=ident)
        name = f"fp8_ctx{FP8_CONTEXT}"
        for L, ql in W.chunk_schedule(FP8_CONTEXT):
            sl, qsl = i32([L]), i32([0, ql])
            q, out = q_all[L - ql:L], out_all[L - ql:L]
            self._add(name, "fp8_dequant", self._dequant_fn(k, v, bt, sl, sc, kd, vd))
            self._add(name, "prefill_fp8_dense", self._dense_prefill_fn(q, kd, vd, ident, sl, qsl, ql, p.softmax_scale,
                                                                        out), q, out)

        # verify batch (distinct blocks)
        p = verify_problem()
        k, v = device_pool(p, "k"), device_pool(p, "v")
        ksp, vsp = device_scale_pool(p, "k"), device_scale_pool(p, "v")
        bt, sl, _ = device_meta(p)
        q = device_q(p)
        out = torch.empty_like(q)
        split = pick_split(pkv, p.seq_lens, torch.cuda.get_device_properties(dev).multi_processor_count)
        S = pkv.splits_needed(int(p.seq_lens.max()), split)
        po = torch.empty((S, q.shape[0], HQ, D), dtype=torch.float32, device=dev)
        pl = torch.empty((S, q.shape[0], HQ), dtype=torch.float32, device=dev)
        self.verify = dict(p=p, k=k, v=v, ksp=ksp, vsp=vsp, bt=bt, sl=sl, q=q, out=out, split=split)
        partial, combine = self._verify_fns(q, k, v, ksp, vsp, bt, sl, p.softmax_scale, split, po, pl, out)
        self._add("verify_batch32", "verify_partial", partial, q, None)
        self._add("verify_batch32", "verify_combine", combine, None, out)
        # prepare the earlier steps' state: every int8 context's codes (the chunks requantize their
        # own rows each step, so the state never changes)
        for fn in [it[2] for it in self.items]:
            fn()
        torch.cuda.synchronize()

    # Each launch's arguments are bound here, when the launch is created (a lambda written inline in
    # __init__ would read its variables when called, after later workloads have reused the names).
    def _quant_fn(self, k, bt, pb, sl, ql, k8, ks, k16):
        return lambda: self.pkv.kv_int8_stats_quant(k, bt, pb, sl, ql, k8, ks, k16=k16)

    def _int8_prefill_fn(self, q, v, bt, sl, qsl, ql, scale, out, ks, k16):
        return lambda: self.pkv.paged_prefill_attn(q, None, v, bt, sl, qsl, ql, scale, out, qk_mode=self.pkv.PKV_QK_INT8,
                                                   k8_scale=ks, k16=k16, workspace=self.ws)

    def _dequant_fn(self, k, v, bt, sl, sc, kd, vd):
        return lambda: self.pkv.kv_fp8_dequant_dense(k, v, bt, sl, sc, sc, kd, vd)

    def _dense_prefill_fn(self, q, kd, vd, ident, sl, qsl, ql, scale, out):
        return lambda: self.pkv.paged_prefill_attn(q, kd, vd, ident, sl, qsl, ql, scale, out, workspace=self.ws)

    def _verify_fns(self, q, k, v, ksp, vsp, bt, sl, scale, split, po, pl, out):
        pkv = self.pkv
        return (lambda: pkv.spec_verify_attn_partial(q, k, v, ksp, vsp, bt, sl, T_VERIFY, scale, split, po, pl),
                lambda: pkv.spec_verify_combine(po, pl, sl, T_VERIFY, split, out))

    def _add(self, workload, kernel, fn, q=None, out=None):
        self.items.append((workload, kernel, fn, q, out))

    def run(self, ev=None):
        """Enqueue one step; ev: optional list collecting (workload, kernel, start, end) events."""
        torch = self.torch
        for workload, kernel, fn, _, _ in self.items:
            if ev is None:
                fn()
                continue
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.append((workload, kernel, a, b))

    def launches_per_step(self):
        """kernels launched per step: a persistent prefill is the kernel and its merge."""
        return sum(2 if k.startswith("prefill") else 1 for _, k, _, _, _ in self.items)


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

    st = Step(torch, pkv, dev)
    alg = algorithmic(st.verify["p"].seq_lens)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 512 MB > 129 MB L2

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # timed region: K steps, L2 flushed before each (outside the step's events)
    step_ms, per = [], {}
    barrier()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            evs = []
            a.record()
            st.run(evs)
            b.record()
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
            acc = {}
            for wl, kern, x, y in evs:
                acc[(wl, kern)] = acc.get((wl, kern), 0.0) + x.elapsed_time(y)
            for key, ms in acc.items():
                per.setdefault(key, []).append(ms)
        barrier()
        wall = time.perf_counter() - t_wall
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    e2e = run_e2e(torch, pkv, st, args)
    extras = None if args.skip_extras else run_extras(torch, pkv, st, flush, args, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks = load_peaks()
    mean = {k: statistics.mean(v) for k, v in per.items()}  # ms per step of each (workload, kernel)
    workloads = summarize(mean, alg, peaks, st)
    # roofline: the kernel class with the most time per step, over all its launches in the step
    by_kernel = {}
    for (wl, kern), ms in mean.items():
        by_kernel[kern] = by_kernel.get(kern, 0.0) + ms
    dominant = max(by_kernel, key=by_kernel.get)
    roof = roofline(dominant, by_kernel, alg, peaks, st)
    value = whole_job_value(step_tokens(), args.steps, world, total_ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "pages' workloads, whole: big-pool chunk (2,048 of 20,000 tokens, blocks 2577-2599 "
                               "of 2,600, exact QK) + int8-QK prefill of 24,576- and 47,104-token contexts in 2,048 "
                               "chunks (quant per chunk) + fp8 prefill of a 32,768-token context in 2,048 chunks "
                               "(dense dequant per chunk) + 32-request 8-token int8 verify; 16 q / 4 kv heads, "
                               "head_dim 256, block 880",
                   "tokens_per_step": step_tokens(), "l2": "flushed before every step (512 MB write)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "workloads": workloads,
        "per_kernel_ms_per_step": {k: round(v, 4) for k, v in sorted(by_kernel.items())},
        "e2e": e2e,
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
        "extras": extras,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def summarize(mean, alg, peaks, st):
    """per-workload throughput and roofline fractions from the per-(workload, kernel) times."""
    out = {}
    tf = lambda flops, ms: flops / (ms * 1e-3) / 1e12
    gb = lambda nbytes, ms: nbytes / (ms * 1e-3) / 1e9

    ms = mean[("bigpool", "prefill_bf16")]
    f = alg["bigpool"]["prefill_flops"]
    out["bigpool_chunk2048"] = {"tokens": CHUNK, "ms": round(ms, 4), "tok_s": round(CHUNK / (ms * 1e-3), 1),
                                "tflops": round(tf(f, ms), 2), "frac_bf16_peak": round(tf(f, ms) / peaks["bf16_tflops"], 4)}
    for ctx in INT8_CONTEXTS:
        name = f"int8_ctx{ctx}"
        a = alg[name]
        pms, qms = mean[(name, "prefill_int8")], mean[(name, "int8_quant")]
        out[name] = {"tokens": ctx, "chunks": len(W.chunk_schedule(ctx)), "ms": round(pms + qms, 4),
                     "tok_s": round(ctx / ((pms + qms) * 1e-3), 1),
                     "tflops_incl_quant": round(tf(a["prefill_flops"], pms + qms), 2),
                     "prefill_ms": round(pms, 4), "prefill_tflops": round(tf(a["prefill_flops"], pms), 2),
                     "frac_bf16_peak": round(tf(a["prefill_flops"], pms) / peaks["bf16_tflops"], 4),
                     "quant_ms": round(qms, 4), "quant_gbs": round(gb(a["quant_bytes"], qms), 1),
                     "quant_frac_hbm": round(gb(a["quant_bytes"], qms) / peaks["hbm_gbs"], 4),
                     "quant_note": "772 B per (token, head) row; the fp16 copy of the codes the prefill reads "
                                   f"({K16_BYTES_PER_ROW} B per row) is overhead, not counted"}
    name = f"fp8_ctx{FP8_CONTEXT}"
    a = alg[name]
    pms, dms = mean[(name, "prefill_fp8_dense")], mean[(name, "fp8_dequant")]
    out[name] = {"tokens": FP8_CONTEXT, "chunks": len(W.chunk_schedule(FP8_CONTEXT)), "ms": round(pms + dms, 4),
                 "tok_s": round(FP8_CONTEXT / ((pms + dms) * 1e-3), 1),
                 "tflops_incl_dequant": round(tf(a["prefill_flops"], pms + dms), 2),
                 "prefill_ms": round(pms, 4), "prefill_tflops": round(tf(a["prefill_flops"], pms), 2),
                 "frac_bf16_peak": round(tf(a["prefill_flops"], pms) / peaks["bf16_tflops"], 4),
                 "dequant_ms": round(dms, 4), "dequant_gbs": round(gb(a["dequant_bytes"], dms), 1),
                 "dequant_frac_hbm": round(gb(a["dequant_bytes"], dms) / peaks["hbm_gbs"], 4)}
    vp, vc = mean[("verify_batch32", "verify_partial")], mean[("verify_batch32", "verify_combine")]
    nb = alg["verify_batch32"]["bytes"]
    out["verify_batch32"] = {"tokens": 32 * T_VERIFY, "sum_seq_len": int(np.sum(st.verify["p"].seq_lens)),
                             "ms": round(vp + vc, 4), "gbs": round(gb(nb, vp + vc), 1),
                             "frac_hbm": round(gb(nb, vp + vc) / peaks["hbm_gbs"], 4), "partial_ms": round(vp, 4),
                             "partial_gbs": round(gb(nb, vp), 1), "combine_ms": round(vc, 4),
                             "split_tokens": st.verify["split"], "algorithmic_bytes": int(nb)}
    return out


def roofline(kernel, by_kernel, alg, peaks, st):
    """roofline of the kernel class with the most time per step: its algorithmic work over all its
    launches in the step divided by their total time (the same as per-launch work over the mean
    launch time)."""
    ms = by_kernel[kernel]
    launches = sum(1 for _, k, _, _, _ in st.items if k == kernel)
    if kernel.startswith("prefill"):
        flops = 0
        for name, a in alg.items():
            kern = {"bigpool": "prefill_bf16", f"fp8_ctx{FP8_CONTEXT}": "prefill_fp8_dense"}.get(name, "prefill_int8")
            if kern == kernel and "prefill_flops" in a:
                flops += a["prefill_flops"]
        achieved = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": load_traffic(kernel), "kernel": kernel,
                "launches_per_step": launches, "flop_per_launch": int(flops / launches),
                "peak_source": peaks["source"] + " (bf16 dense, burst)"}
    nbytes = {"int8_quant": sum(a.get("quant_bytes", 0) for a in alg.values()),
              "fp8_dequant": sum(a.get("dequant_bytes", 0) for a in alg.values()),
              "verify_partial": alg["verify_batch32"]["bytes"]}.get(kernel, 0)
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": load_traffic(kernel), "kernel": kernel,
            "launches_per_step": launches, "peak_source": peaks["source"]}


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
    """dram read + write bytes per launch of `kernel` in the step, from the committed ncu capture
    (profiles/traffic.json), or None when there is none or the kernel source has changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            ent = json.load(f).get(kernel)
        if not ent:
            return None
        for src, sha in ent["sources"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None
        return int(ent["dram_bytes_per_launch"])
    except Exception:
        return None


def run_e2e(torch, pkv, st, args):
    """The same step through the public API with host buffers: every step copies each launch's
    queries in from pinned host memory and its output back, inside the timed region. The copies run
    on their own streams, overlapped with the kernels of the other chunks: a chunk's queries land
    once the previous step's use of its device buffer is done, and its output leaves as soon as it
    is written (the next step's write of that buffer waits for the copy)."""
    items = [(fn, q, out) for _, _, fn, q, out in st.items]
    hq = [None if q is None else q.cpu().pin_memory() for _, q, _ in items]
    ho = [None if o is None else torch.empty_like(o, device="cpu").pin_memory() for _, _, o in items]
    h2d = sum(q.numel() * q.element_size() for q in hq if q is not None)
    d2h = sum(o.numel() * o.element_size() for o in ho if o is not None)
    steps = max(1, args.steps)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n = len(items)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for s in range(steps):
        for i, (fn, q, out) in enumerate(items):
            if q is not None:
                with torch.cuda.stream(s_in):
                    s_in.wait_event(a)
                    if s > 0:
                        s_in.wait_event(ev_comp[i])  # the previous step's kernel has read this buffer
                    q.copy_(hq[i], non_blocking=True)
                    ev_in[i].record(s_in)
                comp.wait_event(ev_in[i])
            if out is not None and s > 0:
                comp.wait_event(ev_out[i])  # the previous step's output has left this buffer
            fn()
            ev_comp[i].record(comp)
            if out is not None:
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[i])
                    ho[i].copy_(out, non_blocking=True)
                    ev_out[i].record(s_out)
    for i in range(n):
        comp.wait_event(ev_out[i])
    b.record(comp)
    b.synchronize()
    ms = a.elapsed_time(b)
    return {"value": round(step_tokens() * steps / (ms * 1e-3), 1), "unit": "tok/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": "per-launch query copies in and output copies out on their own streams, overlapped with "
                        "the kernels of the other chunks",
            "l2": "not flushed between steps (a serving loop), unlike the device-timed step"}


def _time(torch, fn, flush, reps, warm=3):
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def run_extras(torch, pkv, st, flush, args, dev):
    """Measurements outside the step, each launch timed alone with CUDA events, L2 flushed before
    every repetition."""
    from _devsetup import device_meta, device_pool, device_q, device_scale_pool, u16_to_bf16
    peaks = load_peaks()
    reps = max(5, min(args.steps, 20))
    res = {}

    # the big-pool chunk with each launch: one CTA per query tile or the persistent grid; int8 QK
    # reading the fp16 copy of the codes or widening the int8 codes in converter warps
    bp = st.bigpool
    p = bp["p"]
    L = W.BIGPOOL_L
    k8 = torch.zeros((1, L, HKV, D), dtype=torch.int8, device=dev)
    ks = torch.zeros((1, L, HKV), dtype=torch.float32, device=dev)
    k16 = torch.zeros((1, L, HKV, D), dtype=torch.float16, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_int8_stats_quant(bp["k"], bp["bt"], zero, bp["sl"], L, k8, ks, k16=k16)
    out = torch.empty_like(bp["q"])
    flops = prefill_pairs(L, CHUNK) * FLOP_PER_PAIR
    calls = {
        "bf16": lambda ws: pkv.paged_prefill_attn(bp["q"], bp["k"], bp["v"], bp["bt"], bp["sl"], bp["qsl"], CHUNK,
                                                  p.softmax_scale, out, workspace=ws),
        "int8_fp16_copy": lambda ws: pkv.paged_prefill_attn(bp["q"], None, bp["v"], bp["bt"], bp["sl"], bp["qsl"], CHUNK,
                                                            p.softmax_scale, out, qk_mode=pkv.PKV_QK_INT8, k8_scale=ks,
                                                            k16=k16, workspace=ws),
        "int8_converter": lambda ws: pkv.paged_prefill_attn(bp["q"], None, bp["v"], bp["bt"], bp["sl"], bp["qsl"], CHUNK,
                                                            p.softmax_scale, out, qk_mode=pkv.PKV_QK_INT8, k8=k8,
                                                            k8_scale=ks, workspace=ws),
    }
    launches = {}
    for name, fn in calls.items():
        launches[name] = {}
        for kind, ws in (("per_query_tile", None), ("persistent", st.ws)):
            ms = _time(torch, lambda: fn(ws), flush, reps)
            launches[name][kind] = {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 2)}
    res["bigpool_prefill_launches"] = launches
    del k8, ks, k16

    # fp8: the last chunk of the 32,768-token context, dequantize-once dense path vs per-tile dequant
    f = st.fp8
    pf = f["p"]
    sl, qsl = torch.tensor([FP8_CONTEXT], dtype=torch.int32, device=dev), torch.tensor([0, CHUNK], dtype=torch.int32,
                                                                                       device=dev)
    q = f["q"][FP8_CONTEXT - CHUNK:]
    out = torch.empty_like(q)
    fl = prefill_pairs(FP8_CONTEXT, CHUNK) * FLOP_PER_PAIR
    dq = _time(torch, lambda: pkv.kv_fp8_dequant_dense(f["k"], f["v"], f["bt"], sl, f["sc"], f["sc"], f["kd"], f["vd"]),
               flush, reps)
    at = _time(torch, lambda: pkv.paged_prefill_attn(q, f["kd"], f["vd"], f["ident"], sl, qsl, CHUNK, pf.softmax_scale,
                                                     out, workspace=st.ws), flush, reps)
    fu = _time(torch, lambda: pkv.paged_prefill_attn_fp8(q, f["k"], f["v"], f["sc"], f["sc"], f["bt"], sl, qsl, CHUNK,
                                                         pf.softmax_scale, out, workspace=st.ws), flush, reps)
    tfl = lambda ms: round(fl / (ms * 1e-3) / 1e12, 2)
    res["fp8_last_chunk_paths"] = {
        "dense": {"dequant_ms": round(dq, 4), "dequant": _gbs(FP8_CONTEXT * DEQUANT_BYTES_PER_TOKEN, dq, peaks),
                  "attn_ms": round(at, 4), "attn_tflops": tfl(at), "total_ms": round(dq + at, 4),
                  "tflops_incl_dequant": tfl(dq + at)},
        "fused": {"ms": round(fu, 4), "tflops": tfl(fu)}}

    # whole-context quantization (a from-scratch prefill's, 47,104 tokens): with and without the fp16 copy
    c = st.int8[INT8_CONTEXTS[-1]]
    ctx = INT8_CONTEXTS[-1]
    sl = torch.tensor([ctx], dtype=torch.int32, device=dev)
    for name, k16x in (("quant_ctx47104", None), ("quant_ctx47104_with_fp16_copy", c["k16"])):
        ms = _time(torch, lambda: pkv.kv_int8_stats_quant(c["k"], c["bt"], zero, sl, ctx, c["k8"], c["ks"], k16=k16x),
                   flush, reps)
        r = _gbs(ctx * HKV * QUANT_BYTES_PER_ROW, ms, peaks)
        if k16x is not None:
            r["moved_gbs_incl_copy"] = round(ctx * HKV * (QUANT_BYTES_PER_ROW + K16_BYTES_PER_ROW) / (ms * 1e-3) / 1e9, 1)
        res[name] = r

    # verify: the literal 480k-token pool (546 blocks, shared blocks), a T = 1 decode step on the
    # step's cache, and the pages' 24 / 4 heads
    v = st.verify
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def verify_rate(pb, kk, vv, kss, vss, bt, q, seq_lens, T, hq):
        sld = torch.from_numpy(np.asarray(seq_lens, dtype=np.int32)).to(dev)
        split = pick_split(pkv, seq_lens, n_sms, T, hq)
        S = pkv.splits_needed(int(max(seq_lens)), split)
        po = torch.empty((S, q.shape[0], hq, D), dtype=torch.float32, device=dev)
        pl = torch.empty((S, q.shape[0], hq), dtype=torch.float32, device=dev)
        o = torch.empty_like(q)

        def fn():
            pkv.spec_verify_attn_partial(q, kk, vv, kss, vss, bt, sld, T, pb.softmax_scale, split, po, pl)
            pkv.spec_verify_combine(po, pl, sld, T, split, o)
        ms = _time(torch, fn, flush, reps)
        r = _gbs(verify_bytes(seq_lens, T, hq), ms, peaks)
        r.update({"T": T, "q_heads": hq, "split_tokens": split, "sum_seq_len": int(np.sum(seq_lens))})
        return r

    vp = v["p"]
    res["verify_decode_t1"] = verify_rate(vp, v["k"], v["v"], v["ksp"], v["vsp"], v["bt"],
                                          u16_to_bf16(W.bf16_normal(7, (vp.num_reqs, HQ, D))).to(dev),
                                          vp.seq_lens - (T_VERIFY - 1), 1, HQ)
    res["verify_heads_24x4"] = verify_rate(vp, v["k"], v["v"], v["ksp"], v["vsp"], v["bt"],
                                           u16_to_bf16(W.bf16_normal(8, (vp.num_reqs * T_VERIFY, 24, D))).to(dev),
                                           vp.seq_lens, T_VERIFY, 24)
    lit = verify_problem(distinct=False)
    lk, lv = device_pool(lit, "k"), device_pool(lit, "v")
    lks, lvs = device_scale_pool(lit, "k"), device_scale_pool(lit, "v")
    lbt, _, _ = device_meta(lit)
    res["verify_literal_pool546"] = verify_rate(lit, lk, lv, lks, lvs, lbt, device_q(lit), lit.seq_lens, T_VERIFY, HQ)
    res["verify_literal_pool546"]["note"] = ("546 blocks hold 480,480 tokens, fewer than the batch's; requests share "
                                             "blocks, so DRAM bytes fall below the algorithmic bytes (L2 reuse)")
    del lk, lv, lks, lvs

    # cache write of one 2,048-row chunk (the big-pool request's last rows) per cache format
    res["cache_write_chunk2048"] = run_cache_write(torch, pkv, flush, reps, dev, peaks)
    return res


def run_cache_write(torch, pkv, flush, reps, dev, peaks):
    """kv_cache_write of a 2,048-token chunk (K and V rows of 4 heads) into 2,600-block pools at the
    top blocks, per format: bf16 copy, int8 per token-head with scales, e4m3 per tensor."""
    from _devsetup import u16_to_bf16
    p = W.bigpool(top=True, q_len=CHUNK, with_kv=False)
    rows = W.bf16_normal(9, (CHUNK, HKV, D))
    kn, vn = u16_to_bf16(rows).to(dev), u16_to_bf16(W.bf16_normal(10, (CHUNK, HKV, D))).to(dev)
    bt = torch.from_numpy(p.block_table(fill=-1)).to(dev)
    sl = torch.from_numpy(p.seq_lens).to(dev)
    qsl = torch.from_numpy(p.query_start_loc).to(dev)
    shape = (p.num_blocks, BS, HKV, D)
    sc = torch.tensor([0.5], dtype=torch.float32, device=dev)
    res = {}
    for name, dt, tdt, out_b in (("bf16", pkv.PKV_KV_BF16, torch.bfloat16, 2 * D),
                                 ("int8", pkv.PKV_KV_INT8, torch.int8, D + 4),
                                 ("fp8", pkv.PKV_KV_FP8, torch.uint8, D)):
        kc = torch.zeros(shape, dtype=tdt, device=dev)
        vc = torch.zeros_like(kc)
        ksc = torch.zeros(shape[:3], dtype=torch.float32, device=dev) if dt == pkv.PKV_KV_INT8 else None
        vsc = torch.zeros_like(ksc) if ksc is not None else None
        fn = lambda: pkv.kv_cache_write(kn, vn, bt, sl, qsl, CHUNK, kc, vc, kv_dtype=dt, k_scale_cache=ksc,
                                        v_scale_cache=vsc, k_scale=sc if dt == pkv.PKV_KV_FP8 else None,
                                        v_scale=sc if dt == pkv.PKV_KV_FP8 else None)
        ms = _time(torch, fn, flush, reps)
        res[name] = _gbs(2 * CHUNK * HKV * (2 * D + out_b), ms, peaks)
        del kc, vc, ksc, vsc
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------------------------
# CPU oracle (baseline arm)
# ----------------------------------------------------------------------------------------------

class OracleSample:
    """A bounded sample of the step for the CPU oracle: `per` query tokens (all 16 heads) of every
    prefill workload, spread over its chunks, each with its share of its chunk's quantization or
    dequantization (the chunk's rows divided by its queries), and one request of the verify batch.
    Inputs (pools, the int8 codes of earlier positions, the dense fp8 scratch) are prepared once,
    untimed, as the earlier steps of a real prefill would have left them."""

    def __init__(self, per):
        import oracle
        self.oracle = oracle
        self.per = per
        self.bp = bigpool_problem()
        self.bp_pools = (self.bp.pool_numpy("k"), self.bp.pool_numpy("v"), self.bp.block_table(fill=0))
        self.int8 = {}
        for ctx in INT8_CONTEXTS:
            p = int8_problem(ctx)
            kp, vp, bt = p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0)
            k8, ks = oracle.kv_int8_stats_quant(kp, bt, [0], [ctx], BS, ctx)
            self.int8[ctx] = (p, kp, vp, bt, k8, ks)
        p = fp8_problem()
        kp, vp, bt = p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0)
        kd, vd = oracle.kv_fp8_dequant_dense(kp, vp, bt, [FP8_CONTEXT], FP8_CONTEXT, FP8_SCALE, FP8_SCALE)
        self.fp8 = (p, kp, vp, bt, kd.reshape(1, FP8_CONTEXT, HKV, D), vd.reshape(1, FP8_CONTEXT, HKV, D))
        self.vb = verify_problem()
        self.vargs = (self.vb.q, self.vb.pool_numpy("k"), self.vb.pool_numpy("v"), self.vb.scale_pool_numpy("k"),
                      self.vb.scale_pool_numpy("v"), self.vb.block_table(fill=0), self.vb.seq_lens)
        self.calls = 0

    def tasks(self):
        """(kind, fn) work items of one sample step; every prefill item is one query token."""
        o, per = self.oracle, self.per
        shift = self.calls
        self.calls += 1
        t = []
        p = self.bp
        kp, vp, bt = self.bp_pools
        for i in range(per):
            tok = (i * CHUNK) // per + shift % max(1, CHUNK // per)
            t.append(("prefill", lambda tok=tok: o.paged_prefill_attn(p.q, kp, vp, bt, p.seq_lens, p.query_start_loc, HQ,
                                                                      p.softmax_scale, 0, None, None, tok, tok + 1)))
        for ctx, (pi, kpi, vpi, bti, k8, ks) in self.int8.items():
            for i in range(per):
                pos = (i * ctx) // per + shift % max(1, ctx // per)
                L = min(ctx, (pos // CHUNK + 1) * CHUNK)

                def item(pos=pos, L=L, pi=pi, kpi=kpi, vpi=vpi, bti=bti, k8=k8, ks=ks):
                    o.kv_int8_stats_quant(kpi, bti, [pos], [pos + 1], BS, L)  # its row of the chunk's pass
                    return o.paged_prefill_attn(pi.q, kpi, vpi, bti, [L], [0, L], HQ, pi.softmax_scale, 1, k8, ks,
                                                pos, pos + 1)
                t.append(("prefill", item))
        pf, kpf, vpf, btf, kd, vd = self.fp8
        ident = np.zeros((1, 1), np.int32)
        for i in range(per):
            pos = (i * FP8_CONTEXT) // per + shift % max(1, FP8_CONTEXT // per)
            L = (pos // CHUNK + 1) * CHUNK
            share = max(1, L // CHUNK)  # the chunk dequantizes [0, L): L / 2,048 positions per query

            def item(pos=pos, L=L, share=share):
                o.kv_fp8_dequant_dense(kpf, vpf, btf, [share], share, FP8_SCALE, FP8_SCALE)
                return o.paged_prefill_attn(pf.q, kd, vd, ident, [L], [0, L], HQ, pf.softmax_scale, 0, None, None, pos,
                                            pos + 1)
            t.append(("prefill", item))
        r = shift % self.vb.num_reqs
        t.append(("verify", lambda r=r: o.spec_verify_attn(*self.vargs, T_VERIFY, HQ, self.vb.softmax_scale,
                                                           req_begin=r, req_end=r + 1)))
        return t

    def tokens_per_step(self):
        return 4 * self.per + T_VERIFY

    def describe(self):
        return (f"{self.per} query tokens x 16 heads of each of the four prefill workloads (big-pool chunk, int8 24,576 "
                f"and 47,104, fp8 32,768; positions spread over the chunks, each with its share of its chunk's quant "
                f"or dequant) and one 8-token verify request per step; value = those tokens / measured time")


def run_oracle_steps(sample, steps, warmup, cores):
    """Runs warmup untimed and `steps` timed sample steps on a pool of `cores` threads (the C oracle
    releases the GIL); returns the wall seconds of each timed step."""
    from concurrent.futures import ThreadPoolExecutor
    times = []
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for s in range(warmup + steps):
            tasks = sample.tasks()
            t0 = time.perf_counter()
            for f in [pool.submit(fn) for _, fn in tasks]:
                f.result()
            if s >= warmup:
                times.append(time.perf_counter() - t0)
    return times


def cpu_baseline(args):
    """The oracle timed on this machine's host cores on a bounded sample of the step (a few
    seconds per sample step): tok/s of the tokens actually processed."""
    cores = os.cpu_count() or 1
    sample = OracleSample(per=max(1, min(cores, 32)))
    times = run_oracle_steps(sample, steps=max(1, args.cpu_steps), warmup=1, cores=cores)
    s = statistics.mean(times)
    return {"value": round(sample.tokens_per_step() / s, 3), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": sample.describe(), "seconds_per_sample_step": round(s, 3), "sample_steps": len(times)}


def run_reference(args):
    """The reference arm: the CPU oracle on the step's workloads, a bounded sample per step; every
    number is the measured wall time of the work actually run."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    sample = OracleSample(per=max(1, min(cores, 32)))
    times = run_oracle_steps(sample, steps=args.steps, warmup=args.warmup, cores=cores)
    ms = 1e3 * statistics.mean(times)
    value = sample.tokens_per_step() / (ms * 1e-3)
    line = {"metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": "the step's workloads, bounded sample per step: " + sample.describe(),
                       "tokens_per_step": sample.tokens_per_step()},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample.describe(), "value": round(value, 3)},
            "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------------------------------------
# small self-contained cases for profiler capture
# ----------------------------------------------------------------------------------------------

def run_ncu_case(args):
    """One kernel on a small case for profiler capture (not a bench line), launched --warmup +
    --steps times: the big-pool request (20,000 tokens, last 2,048-token chunk) in a 64-block pool
    (its 23 blocks at the top), one 2,048-token chunk of the int8 context, the whole-context quant,
    the fp8 dequant, or the 32-request verify batch."""
    import torch
    from __graft_entry__ import build
    build()
    import paged_kv_cache_int64_gb300 as pkv
    from _devsetup import device_meta, device_pool, device_q, device_scale_pool
    dev = "cuda:0"
    torch.cuda.set_device(0)
    case = args.ncu_case
    L = W.BIGPOOL_L
    if case == "verify":
        p = verify_problem()
        k, v = device_pool(p, "k"), device_pool(p, "v")
        ks, vs = device_scale_pool(p, "k"), device_scale_pool(p, "v")
        bt, sl, _ = device_meta(p)
        q = device_q(p)
        split = pick_split(pkv, p.seq_lens, torch.cuda.get_device_properties(dev).multi_processor_count)
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
            "int8_quant_context": lambda: pkv.kv_int8_stats_quant(k, bt, zero, sl, L, k8, k8s),
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-steps", type=int, default=8, help="sample steps of the oracle for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-extras", action="store_true")
    ap.add_argument("--ncu-case", choices=["prefill_bf16", "prefill_bf16_persistent", "prefill_int8", "int8_quant",
                                           "int8_quant_context", "fp8_dequant", "verify"],
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
