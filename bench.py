"""Benchmark of the tensor-parallel block on B300.

A step is one pass of the whole block (column QKV -> per-shard attention ->
row-parallel O + reduce -> column FFN-up + SwiGLU -> row-parallel FFN-down +
reduce) over one batch of the LLaMA-2-7B-shaped prefill workload
(d_model 4096, 32 heads, d_ffn 11008, tp 4 logical shards, batch 1 x 2048
tokens, causal, bf16), inputs resident in HBM.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs one independent replica per GPU (launched by torchrun); the
block does not shard across GPUs here (its shards are logical partitions of
one GPU), so ranks exchange nothing but the timing.  ``--impl reference``
times the float64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and TFLOP/s (prefill), HBM GB/s (decode) per TP block on 1 B300 vs roofline"
L2_FLUSH_BYTES = 256 << 20  # > 126 MB L2
REF_BUDGET_S = 150.0        # reference arm: warm-up + timed oracle calls


def workload_config(name, wl, world):
    """The `config` object of both arms' lines (the same workload, process
    layout and L2 policy of the timed GPU steps, so the two lines compare)."""
    s = wl.shape
    return {"workload": name, "d_model": s.d_model, "n_heads": s.n_heads, "d_ffn": s.d_ffn, "tp_degree": wl.tp,
            "batch": wl.batch, "seq": wl.seq, "causal": wl.causal, "act": s.act,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": f"GPU steps: L2 flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)"}


def block_flops(wl):
    s = wl.shape
    d, f, B, T = s.d_model, s.d_ffn, wl.batch, wl.seq
    lin = 2.0 * B * T * (4 * d * d + 3 * d * f)
    # QK^T and PV over the visible keys (causal: T(T+1)/2 per head-row sum)
    keys = T * (T + 1) / 2 if wl.causal else T * T
    attn = 4.0 * d * B * keys
    return lin, attn


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons sampled during the
    timed window [mark_start, mark_end]: read-only NVML queries from a
    background thread every ~1 ms (so a window of a few ms still gets
    samples), else nvidia-smi every 100 ms.  Nothing is ever set."""
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_s=0.001):
        self.gpu, self.period = gpu_index, period_s
        self.samples = []  # (time, sm_mhz, max_mhz, power_w, reasons)
        self.t0 = self.t1 = None
        self.proc, self.out, self.thread, self.nvml = None, "", None, None
        self._stop = False

    def start(self):
        try:
            import ctypes
            import threading
            nv = ctypes.CDLL("libnvidia-ml.so.1")  # the driver's NVML, read-only queries below
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            clk_sm = ctypes.c_int(1)  # NVML_CLOCK_SM
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, clk_sm, ctypes.byref(mx))
            # clock-event reason bits of nvml.h
            bits = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nvml = nv

            def loop():
                sm, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop:
                    if (nv.nvmlDeviceGetClockInfo(h, clk_sm, ctypes.byref(sm)) == 0 and
                            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 and
                            reasons_fn(h, ctypes.byref(rs)) == 0):
                        self.samples.append((time.perf_counter(), sm.value, mx.value, pw.value / 1000.0,
                                             [n for n, b in bits.items() if rs.value & b]))
                    time.sleep(self.period)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.nvml = None
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                              "--format=csv,noheader,nounits", "-lms", "100"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
            time.sleep(1.0)  # let nvidia-smi come up before the timed region
        return self

    def mark_start(self):
        self.t0 = (time.perf_counter(), datetime.datetime.now())

    def mark_end(self):
        self.t1 = (time.perf_counter(), datetime.datetime.now())

    def stop(self):
        self._stop = True
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons, power = [], [], set(), []
        if self.t0 is not None and self.t1 is not None:
            for t, c, m, pw, rs in self.samples:
                if self.t0[0] <= t <= self.t1[0]:
                    sm.append(float(c))
                    mx.append(float(m))
                    power.append(pw)
                    reasons.update(rs)
            for line in (self.out or "").splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                    if not (self.t0[1] <= ts <= self.t1[1]):
                        continue
                    sm.append(float(f[2]))
                    mx.append(float(f[3]))
                    power.append(float(f[4]))
                except ValueError:
                    continue
                for n, v in zip(self.NAMES, f[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(power),
                "source": "nvml (read-only, ~1 ms)" if self.nvml else "nvidia-smi (100 ms)"}


def dist_setup(ngpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import datetime

        import torch.distributed as dist
        backend = "nccl" if os.environ.get("TP_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        # a replica that dies ends the others' next barrier or all-reduce with
        # an error after this long, instead of leaving them waiting
        timeout = datetime.timedelta(seconds=float(os.environ.get("TP_BENCH_PG_TIMEOUT_S", "600")))
        dist.init_process_group(backend, timeout=timeout)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(value, pg, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# reference arm: the float64 CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def time_oracle(wl, sample_tokens, steps, warmup=0):
    """Seconds per oracle call on the first `sample_tokens` tokens of the
    workload (causal: those tokens form a self-contained prefix)."""
    import oracle
    from tensor_transformer_layer_03_b300 import inputs as I
    inp = I.make_inputs(wl)
    w = {k: v for k, v in inp.items() if k.startswith("W")}
    w = {k: oracle.to64(v) for k, v in w.items()}
    x = oracle.to64(inp["X"][:1, :sample_tokens])
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        oracle.block_forward(x, w, wl.shape.n_heads, wl.shape.act, wl.causal)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    return times


def time_oracle_seq(wl, b):
    """Seconds of one float64 oracle call on sequence b of the workload
    (sequences are independent)."""
    import torch

    import oracle
    from tensor_transformer_layer_03_b300 import inputs as I
    gen = torch.Generator().manual_seed(0)
    w = {k: oracle.to64(v) for k, v in I.make_weights(wl.shape, wl.dtype, gen).items()}
    x = torch.randn(wl.batch, wl.seq, wl.shape.d_model, generator=gen).to(torch.bfloat16)
    x = oracle.to64(x[b:b + 1])
    t0 = time.perf_counter()
    oracle.block_forward(x, w, wl.shape.n_heads, wl.shape.act, wl.causal)
    return time.perf_counter() - t0


def reference_sample(wl, steps, warmup, per_token_s, budget_s=REF_BUDGET_S):
    """Tokens of sequence 0 that each reference step runs: the whole
    sequence when warm-up + steps fit the time budget, else the longest
    causal prefix (a multiple of 64 tokens, at least 64) that does."""
    fit = int(budget_s / max(1, steps + warmup) / per_token_s)
    if fit >= wl.seq:
        return wl.seq
    return max(64, min(wl.seq, fit // 64 * 64))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0  # the oracle runs once, on rank 0's host cores
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from tensor_transformer_layer_03_b300 import inputs as I
    wl = I.WORKLOADS[args.workload]
    probe_tokens = min(128, wl.seq)
    per_token = time_oracle(wl, probe_tokens, 1)[0] / probe_tokens
    sample = reference_sample(wl, args.steps, args.warmup, per_token)
    times = time_oracle(wl, sample, args.steps, args.warmup)
    total = sum(times)
    value = sample * len(times) / total
    cores = oracle_cores()
    if sample == wl.seq and wl.batch == 1:
        sample_desc = f"the whole workload (1 x {wl.seq} tokens) per step, float64 numpy oracle"
    elif sample == wl.seq:
        sample_desc = (f"sequence 0 of the {wl.batch} ({wl.seq} tokens) per step, float64 numpy oracle "
                       "(the sequences are independent)")
    else:
        sample_desc = (f"first {sample} of the {wl.seq} tokens of sequence 0 per step (causal prefix), "
                       "float64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, wl, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def bench_decode(args, dev, flush=None, batch=1, timeline=False, prenorm=False, with_cpu=False):
    """One-token decode step of the 7B-shaped block (tp 2, 1024 cached
    positions + the new one) for `batch` sequences, captured in a CUDA graph;
    HBM GB/s against the algorithmic bytes (every packed weight once + the
    K/V cache read).  With `timeline`, also the device start/end of every
    kernel of one replay (CUPTI through torch.profiler).  `prenorm`: the
    RMSNorm + RoPE variant of the block (two more launches per step)."""
    import torch

    from tensor_transformer_layer_03_b300 import inputs as I
    from tensor_transformer_layer_03_b300.runtime import TPBlock
    wl = I.WORKLOADS["llama7b_decode"].with_(batch=batch)
    inp = I.make_inputs(wl, seed=0)
    w = {k: v for k, v in inp.items() if k.startswith("W")}
    s = wl.shape
    B, P = wl.batch, wl.cache_len
    cap = P + 1
    norm = {}
    if prenorm:
        w.update(I.make_norm_gains(s, wl.dtype, torch.Generator().manual_seed(1)))
        norm = {"rms_eps": 1e-5, "rope_theta": 10000.0}
    n_launch = 8 if prenorm else 6
    blk = TPBlock(s, wl.tp, wl.dtype, w, device=dev, max_batch=B, max_seq=1, **norm)
    kc = torch.zeros(B, s.n_heads, cap, s.d_head, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:, :, :P] = inp["Kcache"].to(dev)
    vc[:, :, :P] = inp["Vcache"].to(dev)
    x = inp["X"].to(dev)
    y = torch.empty(B, 1, s.d_model, dtype=torch.float32, device=dev)
    del inp, w
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        for _ in range(3):
            blk.forward(x, True, out=y, k_cache=kc, v_cache=vc, cache_pos=P, stream=st)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            blk.forward(x, True, out=y, k_cache=kc, v_cache=vc, cache_pos=P, stream=st)
        st.synchronize()
        n = max(50, args.steps // 2)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(3):
            graph.replay()
        for i in range(n):
            # no flush: a step streams the packed weights (405 MB) and the
            # cache (> 126 MB L2), so nothing it reads survives in L2
            evs[i][0].record(st)
            graph.replay()
            evs[i][1].record(st)
        st.synchronize()
        tl = None
        if timeline:
            from torch.profiler import ProfilerActivity, profile
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                for i in range(3):
                    graph.replay()
                st.synchronize()
            allk = sorted((e.time_range.start, e.time_range.end, e.name) for e in prof.events()
                          if e.device_type.name == "CUDA")
            ks = allk[-(len(allk) // 3):]  # the last of the three replays (memsets included)
            t0 = ks[0][0]
            tl = [{"kernel": n.replace("(anonymous namespace)::", "").replace("void ", "").split("(")[0],
                   "start_us": round(a - t0, 2), "end_us": round(b - t0, 2)} for a, b, n in ks]
    blk.plan.sync_status(st)
    us = [a.elapsed_time(b) * 1000.0 for a, b in evs]
    d, f = s.d_model, s.d_ffn
    weight_bytes = 2 * (4 * d * d + 3 * d * f)
    kv_bytes = 2 * B * s.n_heads * (P + 1) * s.d_head * 2
    algo = weight_bytes + kv_bytes
    med = statistics.median(us)
    gbs = algo / (med * 1e-6) / 1e9
    pk = peaks()
    cpu = None
    if with_cpu:
        # the float64 oracle on the same one-token step (batch B over the
        # same cache), on the host cores
        import oracle
        inp = I.make_inputs(wl, seed=0)
        w64 = {k: oracle.to64(v) for k, v in inp.items() if k.startswith("W")}
        kc64, vc64 = oracle.to64(inp["Kcache"]), oracle.to64(inp["Vcache"])
        x64 = oracle.to64(inp["X"])
        t = []
        for _ in range(3):
            t0 = time.perf_counter()
            oracle.block_forward(x64, w64, s.n_heads, s.act, True, kc64, vc64, P)
            t.append(time.perf_counter() - t0)
        sec = statistics.median(t)
        cpu = {"value": B / sec, "unit": "tokens/s", "gb_s": algo / sec / 1e9, "cores": oracle_cores(), "kind": "oracle",
               "sample": f"the whole step ({B} token(s) over {P} cached positions), float64 numpy oracle, median of 3"}
    return {"workload": "llama7b_decode" + ("_prenorm" if prenorm else ""), "tp_degree": wl.tp, "batch": B, "cache_positions": P + 1,
            "us_per_step_median": med, "us_per_step_p10": sorted(us)[len(us) // 10],
            "algorithmic_bytes": algo, "gb_s": gbs, "hbm_peak_gb_s": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"],
            "tokens_per_s": B / (med * 1e-6), "graph": True, "launches_per_step": n_launch,
            "l2": f"not flushed: each step streams {algo / 1e6:.1f} MB of weights and cache (> 126 MB L2)",
            **({"timeline": tl} if tl else {}), **({"cpu_baseline": cpu} if cpu else {})}


def bench_seq(args, dev, wl_name="llama7b_prefill", steps=50):
    """The block with sequence parallelism (tp_block_forward_seq: x and Y as
    tp slices of the token rows in padded regions) next to the plain block,
    interleaved step by step on one box, L2 flushed between steps."""
    import torch

    from tensor_transformer_layer_03_b300 import inputs as I
    from tensor_transformer_layer_03_b300.runtime import TPBlock
    wl = I.WORKLOADS[wl_name]
    gen = torch.Generator().manual_seed(0)
    w = I.make_weights(wl.shape, wl.dtype, gen)
    blk = TPBlock(wl.shape, wl.tp, wl.dtype, w, device=dev, max_batch=wl.batch, max_seq=wl.seq)
    del w
    B, T, d = wl.batch, wl.seq, wl.shape.d_model
    M = B * T
    x = torch.randn(B, T, d, generator=gen).to(torch.bfloat16).to(dev)
    cap = M // wl.tp + 64
    xs = torch.zeros(wl.tp, cap, d, dtype=torch.bfloat16, device=dev)
    xs[:, :M // wl.tp] = x.reshape(wl.tp, M // wl.tp, d)
    y = torch.empty(B, T, d, dtype=torch.float32, device=dev)
    ys = torch.empty(wl.tp, cap, d, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    times = {"plain": [], "seq": []}
    with torch.cuda.stream(st):
        for i in range(3 + steps):
            for kind in ("plain", "seq"):
                flush.fill_(i & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                if kind == "plain":
                    blk.forward(x, wl.causal, out=y, stream=st)
                else:
                    blk.forward_seq(xs, B, T, wl.causal, out_slices=ys, stream=st)
                e1.record(st)
                if i >= 3:
                    times[kind].append((e0, e1))
        st.synchronize()
    blk.plan.sync_status(st)
    med = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in times.items()}
    lin, attn = block_flops(wl)
    return {"workload": wl.name + "_sequence_parallel", "tp_degree": wl.tp, "batch": B, "seq": T,
            "slice_rows": M // wl.tp, "slice_region_rows": cap, "ms_per_block_seq": med["seq"],
            "ms_per_block_plain": med["plain"], "tokens_per_s_seq": M / (med["seq"] / 1e3),
            "tflops_seq": (lin + attn) / (med["seq"] / 1e3) / 1e12, "steps": steps}


def run_sweep(args):
    """One JSON line per workload of the batch x prompt sweep (7B shape, tp 4)
    and of the tp sweep (13B shape, 4 x 1024 tokens): the whole block through
    tp_block_forward, inputs resident, L2 flushed between steps, CUDA events."""
    import torch

    from tensor_transformer_layer_03_b300 import inputs as I
    from tensor_transformer_layer_03_b300.runtime import TPBlock
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pk = peaks()
    wls = I.sweep_workloads() + [I.WORKLOADS["llama13b_b4t1024"].with_(name=f"llama13b_b4t1024_tp{t}", tp=t)
                                 for t in I.TP_SWEEP]
    # the pre-norm (RMSNorm + RoPE) variant of the 7B prefill block
    wls.append(I.WORKLOADS["llama7b_prefill"].with_(name="llama7b_prefill_prenorm"))
    st = torch.cuda.Stream(device=dev)
    blk, key = None, None
    cpu_done = set()
    # SM clock and throttle reasons per point (read-only NVML sampling; the
    # long points run under the power cap, so their clocks matter)
    clk = ClockSampler(0).start()
    for wl in wls:
        gen = torch.Generator().manual_seed(0)
        pre = wl.name.endswith("_prenorm")
        if key != (wl.shape, wl.tp, pre):  # one set of packed weights per block variant and degree
            blk = None
            torch.cuda.empty_cache()
            w = I.make_weights(wl.shape, wl.dtype, gen)
            norm = {}
            if pre:
                w.update(I.make_norm_gains(wl.shape, wl.dtype, gen))
                norm = {"rms_eps": 1e-5, "rope_theta": 10000.0}
            blk = TPBlock(wl.shape, wl.tp, wl.dtype, w, device=dev, **norm)
            key = (wl.shape, wl.tp, pre)
            del w
        blk.reserve(wl.batch, wl.seq)
        x = torch.randn(wl.batch, wl.seq, wl.shape.d_model, generator=gen).to(torch.bfloat16).to(dev)
        y = torch.empty(wl.batch, wl.seq, wl.shape.d_model, dtype=torch.float32, device=dev)
        n = max(5, min(50, int(2e12 / sum(block_flops(wl)))))  # about 2 TFLOP of work per workload
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(st):
            for i in range(3):
                blk.forward(x, wl.causal, out=y, stream=st)
            st.synchronize()
            clk.mark_start()
            for i in range(n):
                flush.fill_(i & 0xFF)
                evs[i][0].record(st)
                blk.forward(x, wl.causal, out=y, stream=st)
                evs[i][1].record(st)
            st.synchronize()
            clk.mark_end()
        blk.plan.sync_status(st)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        lin, attn = block_flops(wl)
        tf = (lin + attn) / (ms / 1e3) / 1e12
        line = {"clocks": clk.summary() if clk.nvml else None,
                "workload": wl.name, "d_model": wl.shape.d_model, "tp_degree": wl.tp, "batch": wl.batch,
                "seq": wl.seq, "ms_per_block": ms, "tokens_per_s": wl.tokens / (ms / 1e3),
                "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"], "steps": n}
        if not args.no_cpu_baseline and not pre and (wl.shape, wl.batch, wl.seq) not in cpu_done:
            # the float64 oracle (unsharded: the same for every degree) on the
            # first and last sequences, per-sequence time x batch
            cpu_done.add((wl.shape, wl.batch, wl.seq))
            sec = statistics.mean(time_oracle_seq(wl, b) for b in sorted({0, wl.batch - 1}))
            line["cpu_baseline"] = {"value": wl.seq / sec, "unit": "tokens/s", "cores": oracle_cores(),
                                    "kind": "oracle", "sample": f"sequences {sorted({0, wl.batch - 1})} of {wl.batch}"
                                    f" ({wl.seq} tokens each), float64 numpy oracle; tokens/s extrapolated to the"
                                    f" batch as per-sequence time x {wl.batch}"}
        print(json.dumps(line), flush=True)
        del x, y
    blk = None
    torch.cuda.empty_cache()
    # a stack of 4 7B-shaped layers (tp 4), prefill of 1 x 2048 tokens
    from tensor_transformer_layer_03_b300.runtime import TPStack
    wl = I.WORKLOADS["llama7b_prefill"]
    gen = torch.Generator().manual_seed(0)
    stk = TPStack(wl.shape, wl.tp, wl.dtype, [I.make_weights(wl.shape, wl.dtype, gen) for _ in range(4)],
                  device=dev, max_batch=wl.batch, max_seq=wl.seq)
    x = torch.randn(wl.batch, wl.seq, wl.shape.d_model, generator=gen).to(torch.bfloat16).to(dev)
    y = torch.empty(wl.batch, wl.seq, wl.shape.d_model, dtype=torch.float32, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    with torch.cuda.stream(st):
        for i in range(3):
            stk.forward(x, True, out=y, stream=st)
        for i in range(10):
            flush.fill_(i & 0xFF)
            evs[i][0].record(st)
            stk.forward(x, True, out=y, stream=st)
            evs[i][1].record(st)
        st.synchronize()
    stk.plan.sync_status(st)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    lin, attn = block_flops(wl)
    tf = 4 * (lin + attn) / (ms / 1e3) / 1e12
    print(json.dumps({"workload": "llama7b_stack4_b1_t2048", "layers": 4, "tp_degree": wl.tp, "ms_per_stack": ms,
                      "tokens_per_s": wl.tokens / (ms / 1e3), "tflops": tf,
                      "frac_of_bf16_peak": tf / pk["bf16_tflops"]}), flush=True)
    del stk, x, y
    torch.cuda.empty_cache()
    print(json.dumps(bench_seq(args, dev)), flush=True)
    torch.cuda.empty_cache()
    # batched one-token decode at 1024 cached positions (7B shape, tp 2)
    for b in (1, 4, 16, 64):
        r = bench_decode(args, dev, batch=b)
        print(json.dumps({**r, "workload": f"llama7b_decode_b{b}"}), flush=True)
        torch.cuda.empty_cache()
    r = bench_decode(args, dev, batch=1, prenorm=True)
    print(json.dumps({**r, "workload": "llama7b_decode_prenorm_b1"}), flush=True)
    clk.stop()
    return 0


def run_ours(args):
    import torch

    from tensor_transformer_layer_03_b300 import inputs as I
    from tensor_transformer_layer_03_b300 import tp as tpb
    from tensor_transformer_layer_03_b300.runtime import TPBlock

    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = I.WORKLOADS[args.workload]
    inp = I.make_inputs(wl, seed=0)
    w = {k: v for k, v in inp.items() if k.startswith("W")}
    blk = TPBlock(wl.shape, wl.tp, wl.dtype, w, device=dev, max_batch=wl.batch, max_seq=wl.seq)
    plan = blk.plan
    B, T, d = wl.batch, wl.seq, wl.shape.d_model
    M = B * T
    x = inp["X"].to(dev)
    del inp, w
    stream = torch.cuda.Stream(device=dev)
    h = plan.h_l * plan.d_head
    qkv = torch.empty(wl.tp, M, 3 * h, dtype=torch.bfloat16, device=dev)
    att = torch.empty(wl.tp, M, h, dtype=torch.bfloat16, device=dev)
    hf = torch.empty(M, d, dtype=torch.float32, device=dev)
    ha = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    u = torch.empty(wl.tp, M, plan.f_l, dtype=torch.bfloat16, device=dev)
    y = torch.empty(M, d, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # split-tile partials and counters of the linears (contents on entry are ignored)
    gscr = torch.zeros(max(plan.linear_scratch_bytes(M), 16), dtype=torch.uint8, device=dev)
    stages = ["column_qkv", "attention", "row_o_reduce", "column_ffn_up_swiglu", "row_ffn_down_reduce"]

    def step(ev):
        """The five launches of one block step.  `ev` holds 2 events (the
        step's start and end: the launches run back to back, each one's
        set-up overlapping the previous one's tail) or 6 (one between every
        two launches, for the per-stage times; an event between two launches
        keeps the second from starting early)."""
        per_stage = len(ev) == 6
        ev[0].record(stream)
        plan.column_linear(tpb.TP_QKV, x, M, blk.packed, qkv, stream, scratch=gscr)
        if per_stage:
            ev[1].record(stream)
        plan.attention_heads(qkv, B, T, wl.causal, None, None, 0, 0, att, None, stream)
        if per_stage:
            ev[2].record(stream)
        plan.row_linear_reduce(tpb.TP_ATTN_OUT, att, M, blk.packed, x, hf, ha, stream, scratch=gscr)
        if per_stage:
            ev[3].record(stream)
        plan.column_linear(tpb.TP_FFN_UP, ha, M, blk.packed, u, stream, scratch=gscr)
        if per_stage:
            ev[4].record(stream)
        plan.row_linear_reduce(tpb.TP_FFN_DOWN, u, M, blk.packed, hf, y, None, stream, scratch=gscr)
        ev[-1].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps + args.warmup)]
    clk = ClockSampler(local).start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            step(evs[i])
        stream.synchronize()
        plan.sync_status(stream)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)
        clk.mark_start()
        t_wall0 = time.perf_counter()
        for i in range(args.warmup, args.warmup + args.steps):
            flush.fill_(i & 0xFF)  # evicts the previous step's lines from L2 (outside the step's events)
            step(evs[i])
        stream.synchronize()
        t_wall = time.perf_counter() - t_wall0
        clk.mark_end()
        clk.stop()
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        # per-stage times: the same steps again with an event between every
        # two launches (diagnostic; the headline uses the whole-step events)
        n_stage = min(args.steps, 200)
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_stage)]
        for i in range(n_stage):
            flush.fill_(i & 0xFF)
            step(sevs[i])
        stream.synchronize()
    plan.sync_status(stream)
    per_stage = [[sevs[i][j].elapsed_time(sevs[i][j + 1]) for i in range(n_stage)] for j in range(5)]
    step_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.warmup, args.warmup + args.steps)]
    dev_ms_total = sum(step_ms)
    dev_ms_total = max_over_ranks(dev_ms_total, pg, dev)
    ms_per_step = dev_ms_total / args.steps
    tokens = M * args.steps * world
    value = tokens / (dev_ms_total / 1000.0)
    lin, attn = block_flops(wl)
    tflops = (lin + attn) / (ms_per_step / 1000.0) / 1e12

    # dominant kernel: the stage with the largest mean time
    stage_mean = [statistics.mean(s) for s in per_stage]
    dom = max(range(5), key=lambda j: stage_mean[j])
    s = wl.shape
    stage_flops = [2.0 * M * d * 3 * d, attn, 2.0 * M * d * d, 2.0 * M * d * 2 * s.d_ffn, 2.0 * M * s.d_ffn * d]
    pk = peaks()
    achieved = stage_flops[dom] / (stage_mean[dom] / 1000.0) / 1e12
    # DRAM traffic (read + write) per launch of each stage's kernel, from one
    # ncu capture of this workload (profiles/tc_gemm_llama7b_prefill.md)
    traffic = {"column_qkv": 150.30e6, "attention": 50.73e6, "row_o_reduce": 85.17e6,
               "column_ffn_up_swiglu": 230.71e6, "row_ffn_down_reduce": 267.20e6}
    roofline = {"bound": "tensor", "kernel": stages[dom], "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": traffic[stages[dom]],
                "peak_source": f"{pk['source']} bf16 dense burst (cuBLAS)",
                "timing": "per-stage CUDA events over a second timed pass of the same steps"}

    # end to end through the public call: every step copies its input X from
    # pinned host memory and reads its output Y back to pinned host memory.
    # Copy-in, compute and copy-out run on three streams with double-buffered
    # device tensors, so step i's copies overlap steps i-1 / i+1's compute;
    # every step's two copies are inside the timed region.  No L2 flush: the
    # weights and activations a step touches (~0.6 GB) exceed the 126 MB L2.
    e2e = None
    if True:
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        xh = x.cpu().pin_memory()
        yh = [torch.empty(M, d, dtype=torch.float32).pin_memory() for _ in range(2)]
        xd = [torch.empty_like(x) for _ in range(2)]
        yd = [torch.empty(B, T, d, dtype=torch.float32, device=dev) for _ in range(2)]

        def pipelined(n):
            ev = lambda: torch.cuda.Event()
            in_done, comp_done, out_done = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
            for i in range(n):
                k = i & 1
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp_done[i - 2])  # xd[k] consumed
                    xd[k].copy_(xh, non_blocking=True)
                    in_done[i].record(s_in)
                with torch.cuda.stream(stream):
                    stream.wait_event(in_done[i])
                    if i >= 2:
                        stream.wait_event(out_done[i - 2])  # yd[k] read back
                    blk.forward(xd[k], wl.causal, out=yd[k], stream=stream)
                    comp_done[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[i])
                    yh[k].copy_(yd[k].view(M, d), non_blocking=True)
                    out_done[i].record(s_out)
            return out_done[-1]

        pipelined(args.warmup)
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        s_in.wait_event(t_start)
        last = pipelined(args.steps)
        stream.wait_event(last)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        plan.sync_status(stream)
        tot = max_over_ranks(t_start.elapsed_time(t_end), pg, dev)
        e2e = {"value": M * args.steps * world / (tot / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": x.numel() * x.element_size(), "d2h_bytes_per_step": M * d * 4,
               "ms_per_step": tot / args.steps, "pipelined": "copy-in / compute / copy-out streams, double buffers",
               "l2": "no flush; a step touches ~0.6 GB (> 126 MB L2)"}

    decode = (bench_decode(args, dev, with_cpu=(rank == 0 and world == 1 and not args.no_cpu_baseline))
              if not args.no_decode else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times = time_oracle(wl, T, 2)
        cpu = {"value": M * len(times) / sum(times), "unit": "tokens/s", "cores": oracle_cores(), "kind": "oracle",
               "sample": f"the whole workload ({B} x {T} tokens), float64 numpy oracle, 2 calls"}

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload, wl, world),
            "tflops": tflops,
            "tflops_frac_of_peak": tflops / pk["bf16_tflops"],
            "stage_ms": {n: m for n, m in zip(stages, stage_mean)},
            "roofline": roofline,
            "decode": decode,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 5 * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama7b_prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="instead of the headline line: only the decode leg (for profiling its kernels)")
    ap.add_argument("--decode-batch", type=int, default=1)
    ap.add_argument("--timeline", action="store_true", help="with --decode-only: per-kernel device timeline")
    ap.add_argument("--prenorm", action="store_true", help="with --decode-only: the RMSNorm + RoPE block variant")
    ap.add_argument("--seq", action="store_true",
                    help="instead of the headline line: the sequence-parallel block next to the plain one")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the headline line: one line per batch/prompt and tp-sweep workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.seq:
        import torch
        print(json.dumps(bench_seq(args, torch.device("cuda", 0))), flush=True)
        return 0
    if args.decode_only:
        import torch
        print(json.dumps(bench_decode(args, torch.device("cuda", 0), batch=args.decode_batch,
                                      timeline=args.timeline, prenorm=args.prenorm)), flush=True)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
