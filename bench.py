"""Benchmark: causal bf16 attention forward + backward on GB300.

One step = the whole hot path over one batch: attn_fwd_residual (forward with
the output residual), then the backward's preprocess and main kernels. The
default workload is the Llama-3-8B-shaped attention layer (B=2, Hq=32, Hkv=8,
S=4096, D=128, causal). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores, on a bounded sample of the same workload.
Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the path has no exchange step); rank 0 prints the line.
"""
import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal bf16 attention fwd+bwd TFLOP/s at 1 GB300; % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "llama3_8b_s4096"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of each workload's
# roofline kernel per launch, from one ncu capture per workload: workload ->
# (hash of the kernel sources it was taken on, bytes). It reads null once the
# sources change.
DENSE_SOURCES = ("attn_bwd.cu", "attn_common.cuh", "sm100_ptx.cuh")
SPARSE_SOURCES = ("attn_sparse_bwd.cu", "attn_sparse.cuh", "attn_common.cuh", "sm100_ptx.cuh")
TRAFFIC = {
    "llama3_8b_s4096": ("ccfec240ad5645db", 973.71e6),
    "mha_d64_s2048": ("ccfec240ad5645db", 1017.44e6),
    "swa_w128_s4096": ("ccfec240ad5645db", 929.02e6),
    "llama3_70b_s8192": ("ccfec240ad5645db", 3388.44e6),
    "long_s32768": ("ccfec240ad5645db", 12870.36e6),
    "csa_flash_cr4_t8192": ("8ab932384a96e3be", 546.67e6),
    "csa_pro_cr4_t16384": ("8ab932384a96e3be", 2249.29e6),
}


def kernel_source_hash(names=DENSE_SOURCES):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "attention_fwd_bwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(workload, names):
    """Bytes per launch of the workload's roofline kernel, or None if there is
    no capture for the current sources."""
    key, nbytes = TRAFFIC.get(workload, (None, None))
    return nbytes if key is not None and key == kernel_source_hash(names) else None


# Dense bf16 tcgen05 rate per SM and clock: an M128 N256 K16 MMA from shared
# memory (1,048,576 FLOP) completes every 128 cycles (microbenchmarked on a GB300).
TCGEN05_BF16_FLOP_PER_CLK_SM = 8192


def theoretical_tflops(sm_count, sm_max_mhz):
    """SM count x maximum SM clock x the per-SM tcgen05 bf16 rate."""
    return sm_count * sm_max_mhz * 1e6 * TCGEN05_BF16_FLOP_PER_CLK_SM / 1e12


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value, world):
    """Max of a float over ranks (identity on one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank, seconds_max, world):
    """Throughput of the whole job: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / seconds_max


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"attn_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        self.t_begin = datetime.datetime.now()
        return self

    def __exit__(self, *exc):
        self.t_end = datetime.datetime.now()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    rows.append((t, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        # samples taken while the timed steps ran (all of them if none fell inside)
        inside = [r for r in rows if self.t_begin <= r[0] <= self.t_end] or rows
        reasons = {n for r in inside for n, val in zip(names, r[3]) if val.lower().startswith("active")}
        mhz = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": inside[-1][2] if inside else None,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores, on a bounded sample.
# ---------------------------------------------------------------------------
def oracle_sample(w, budget_s=12.0, max_heads=None):
    """Time the oracle's forward + backward on query heads of batch 0, one at a
    time against their kv head, until `budget_s` has passed. Returns
    (convention FLOP/s, sample description, seconds)."""
    import numpy as np
    from attention_fwd_bwd_gb300.inputs import make_inputs
    from oracle import attn_ref_bwd, attn_ref_fwd
    q, k, v, do = make_inputs(1, w.Hq, w.Hkv, w.S, w.D, w.seed, w.qk_std)
    f64 = lambda t: t.double().numpy()
    G = w.Hq // w.Hkv
    heads, t0 = 0, time.perf_counter()
    max_heads = max_heads or w.Hq
    while heads < max_heads:
        h = heads
        g = h // G
        qs, ks, vs, ds = (f64(q[:, :, h:h + 1]), f64(k[:, :, g:g + 1]), f64(v[:, :, g:g + 1]), f64(do[:, :, h:h + 1]))
        attn_ref_fwd(qs, ks, vs, w.causal, w.scale, window=w.window)
        attn_ref_bwd(qs, ks, vs, ds, w.causal, w.scale, window=w.window)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    per_head = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.Hq)
    return per_head * heads / secs, f"{heads} of {w.B * w.Hq} (batch, query head) slices, full S={w.S}", secs


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


# ---------------------------------------------------------------------------
def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    rates, secs = [], 0.0
    sample = ""
    for i in range(args.warmup + args.steps):
        r, sample, s = oracle_sample(w, budget_s=args.ref_budget, max_heads=1)
        if i >= args.warmup:
            rates.append(r)
            secs += s
    value = statistics.mean(rates) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs of the workload's shape)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D,
                   "window": w.window,
                   "causal": w.causal, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"per step: {sample}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w, world, rank, local):
    import torch
    import attention_fwd_bwd_gb300 as attn
    from attention_fwd_bwd_gb300._build import build
    from attention_fwd_bwd_gb300.inputs import workload_inputs

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = attn.lib()
    q_h, k_h, v_h, do_h = workload_inputs(w)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    B, S, Hq, Hkv, D = w.B, w.S, w.Hq, w.Hkv, w.D
    o, o_lo = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(k.shape, **f32)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, Hq, Hkv, S, D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    plain = args.path == "plain"
    if plain:
        o_lo = None

    def step(ev=None):
        # residual path: attn_fwd_residual's kernels, then the backward's
        # preprocess and main kernels. plain path: attn_fwd's kernel, then the
        # preprocess, the Dvec pass and the main kernel (attn_bwd without o_lo).
        if ev is not None:
            ev[0].record(stream)
        attn.attn_fwd_ex(q, k, v, o, lse, w.causal, w.window, w.scale, o_lo=o_lo, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        attn.attn_bwd_preprocess(q, k, o, do, lse, dq, ws, o_lo=o_lo, stream=stream)
        if plain:
            attn.attn_bwd_dvec(q, k, v, do, w.causal, w.scale, ws, window=w.window, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        attn.attn_bwd_main_ex(q, k, v, do, dq, dk, dv, w.causal, w.window, w.scale, ws, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if attn.attn_check_status(ws) != 0:
        raise RuntimeError("kernel pipeline timeout during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if attn.attn_check_status(ws) != 0:
        raise RuntimeError("kernel pipeline timeout during the timed steps")
    total_ms = start.elapsed_time(stop)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    pre_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    main_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    total_ms = reduce_max(total_ms, world)
    ms_per_step = total_ms / args.steps
    flops = w.flops_fwd() + w.flops_bwd()
    value = whole_job_value(flops, ms_per_step / 1e3, world) / 1e12

    # End to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory, runs the forward and the backward
    # (attn_fwd_ex, attn_bwd_ex) and copies its outputs and gradients back.
    # Two steps are in flight, as a training loop would run them: step k's
    # device-to-host reads overlap step k+1's host-to-device copies and kernels
    # (separate copy and compute streams, two device buffer sets, events for
    # the dependencies between them).
    pin = lambda t: t.pin_memory()
    hq_, hk_, hv_, hdo_ = (pin(t) for t in (q_h, k_h, v_h, do_h))
    ho, hlse = pin(torch.empty(o.shape, dtype=o.dtype)), pin(torch.empty(lse.shape, dtype=lse.dtype))
    hdq, hdk, hdv = (pin(torch.empty(t.shape, dtype=t.dtype)) for t in (dq, dk, dv))
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hdo_))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
    sets = [dict(q=q, k=k, v=v, do=do, o=o, o_lo=o_lo, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws)]
    sets.append({n: (None if t is None else torch.empty_like(t)) for n, t in sets[0].items()})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in sets]    # inputs of the set copied in
    ev_done = [torch.cuda.Event() for _ in sets]  # the set's kernels finished
    ev_out = [torch.cuda.Event() for _ in sets]   # the set's results copied out
    used = [False, False]

    def e2e_step(i):
        b = sets[i % 2]
        j = i % 2
        if used[j]:
            s_in.wait_event(ev_done[j])       # the set's previous kernels have read its inputs
            stream.wait_event(ev_out[j])      # the set's previous results have been read back
        with torch.cuda.stream(s_in):
            for n, src in (("q", hq_), ("k", hk_), ("v", hv_), ("do", hdo_)):
                b[n].copy_(src, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        attn.attn_fwd_ex(b["q"], b["k"], b["v"], b["o"], b["lse"], w.causal, w.window, w.scale,
                         o_lo=b["o_lo"], stream=stream)
        # attn_bwd_ex without o_lo runs the Dvec pass itself
        attn.attn_bwd_ex(b["q"], b["k"], b["v"], b["o"], b["do"], b["lse"], b["dq"], b["dk"], b["dv"],
                         w.causal, w.window, w.scale, b["ws"], o_lo=b["o_lo"], stream=stream)
        ev_done[j].record(stream)
        s_out.wait_event(ev_done[j])
        with torch.cuda.stream(s_out):
            for dst, n in ((ho, "o"), (hlse, "lse"), (hdq, "dq"), (hdk, "dk"), (hdv, "dv")):
                dst.copy_(b[n], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(2, min(args.steps, 10))
    e_start.record(s_in)
    for i in range(e_steps):
        e2e_step(i)
    s_out.wait_event(ev_done[(e_steps - 1) % 2])
    e_stop.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e_start.elapsed_time(e_stop), world) / e_steps
    e2e_value = whole_job_value(flops, e2e_ms / 1e3, world) / 1e12
    if attn.attn_check_status(ws) != 0 or attn.attn_check_status(sets[1]["ws"]) != 0:
        raise RuntimeError("kernel pipeline timeout during the end-to-end steps")

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    main_tf = w.flops_bwd() / (main_ms / 1e3) / 1e12
    fwd_tf = w.flops_fwd() / (fwd_ms / 1e3) / 1e12
    # Preprocess bytes as this path moves them: o, dO (and o_lo) read, lse read,
    # the log2-scaled LSE and Dvec rows written, dq zeroed. The algorithmic
    # count leaves out o_lo and the two row vectors: o, dO and lse read, dq
    # zeroed.
    n_rd = 2 if plain else 3
    pre_bytes = (n_rd * B * S * Hq * D * 2 + B * Hq * S * 4 + 2 * B * Hq * S * 4 + B * S * Hq * D * 4)
    pre_bytes_alg = 2 * B * S * Hq * D * 2 + B * Hq * S * 4 + B * S * Hq * D * 4
    traffic = traffic_for(w.name, DENSE_SOURCES)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    theo = theoretical_tflops(sm_count, float(peaks.get("sm_max_mhz", 2070.0)))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q, k, v, dO of the workload's shape)",
            "config": {"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "D": D, "causal": w.causal,
                       "window": w.window,
                       "parallelism": f"replicas x{world}",
                       "l2": f"no flush: q, k, v, dO ({in_bytes / 1e6:.0f} MB) exceed the 129 MB L2",
                       "flops_per_step": flops, "sm_count": sm_count},
            "path": args.path,
            "gpu_launches": (4 if plain else 3) * args.steps,
            "passes": {
                "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak,
                        "frac_of_theoretical": fwd_tf / theo},
                # (plain path: the preprocess and the Dvec pass together)
                "bwd_preprocess": {"ms": pre_ms, "gbs": pre_bytes / (pre_ms / 1e3) / 1e9,
                                   "frac_of_hbm": pre_bytes / (pre_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                                   "frac_of_hbm_algorithmic_bytes":
                                       pre_bytes_alg / (pre_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"])},
                "bwd_main": {"ms": main_ms, "tflops": main_tf, "frac_of_peak": main_tf / peak,
                             "frac_of_theoretical": main_tf / theo},
                "bwd": {"ms": pre_ms + main_ms,
                        "tflops": w.flops_bwd() / ((pre_ms + main_ms) / 1e3) / 1e12,
                        "frac_of_peak": w.flops_bwd() / ((pre_ms + main_ms) / 1e3) / 1e12 / peak},
            },
            "roofline": {"kernel": "attn_bwd_main_kernel", "bound": "tensor", "achieved": main_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": main_tf / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "theoretical_peak": theo, "frac_of_theoretical": main_tf / theo,
                         "theoretical_source": f"{sm_count} SMs x {peaks.get('sm_max_mhz', 2070.0):.0f} MHz x "
                                               f"{TCGEN05_BF16_FLOP_PER_CLK_SM} flop/clk/SM"},
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps_in_flight": 2},
        }
        if not args.no_cpu_baseline:
            rate, sample, secs = oracle_sample(w, budget_s=args.ref_budget)
            line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                    "sample": f"{sample}; {secs:.1f} s"}
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Sparse top-k gather attention (forward), on its own workloads.
# ---------------------------------------------------------------------------
SPARSE_METRIC = "sparse top-k gather attention fwd+bwd TFLOP/s over filled slots at 1 GB300"


def sparse_flops(w, idx):
    """Forward: 2 * H * (DK + DV) per filled (token, slot), the scores and the
    P.V product; the backward counts 2.5 times that (the dense convention)."""
    return 2.0 * w.H * (w.DK + w.DV) * float((idx >= 0).sum())


def sparse_oracle_sample(w, q, kp, vp, idx, do, budget_s=12.0):
    """Time the sparse oracle's forward and backward over tokens of batch 0
    (from the last, the longest lists, down) until `budget_s` has passed."""
    from oracle.sparse import sparse_ref_bwd, sparse_ref_tokens_fwd
    f64 = lambda t: t.double().numpy()
    qn, kn, vn, dn, ix = f64(q[:1]), f64(kp[:1]), f64(vp[:1]), f64(do[:1]), idx[:1].numpy()
    done, flops, t0 = 0, 0.0, time.perf_counter()
    for t in range(w.T - 1, -1, -1):
        sparse_ref_tokens_fwd(qn, kn, vn, ix, w.scale, 0, [t])
        sparse_ref_bwd(qn[:, t:t + 1], kn, vn, ix[:, t:t + 1], dn[:, t:t + 1], w.scale)
        flops += 3.5 * 2.0 * w.H * (w.DK + w.DV) * float((ix[0, t] >= 0).sum())
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    return flops / secs, f"{done} of {w.B * w.T} tokens (the last ones of batch 0, full lists)", secs


def run_sparse(args, w, world, rank, local):
    import torch
    import attention_fwd_bwd_gb300 as attn
    from attention_fwd_bwd_gb300._build import build
    from attention_fwd_bwd_gb300.inputs import make_sparse_inputs

    q_h, kp_h, vp_h, do_h, idx_h = make_sparse_inputs(w)
    fwd_flops = sparse_flops(w, idx_h)
    flops = 3.5 * fwd_flops
    if args.impl == "reference":
        if rank != 0:
            return 0
        rates, secs, sample = [], 0.0, ""
        for i in range(args.warmup + args.steps):
            r, sample, sc = sparse_oracle_sample(w, q_h, kp_h, vp_h, idx_h, do_h, budget_s=args.ref_budget / 4)
            if i >= args.warmup:
                rates.append(r)
                secs += sc
        value = statistics.mean(rates) / 1e12
        print(json.dumps({
            "impl": "reference", "metric": SPARSE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded CSA-shaped top-k lists, N(0,1) bf16 tensors)",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "DK": w.DK, "DV": w.DV, "K": w.K,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"per step: {sample}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return 0

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    attn.lib()
    q, kp, vp, do, idx = (t.to(dev) for t in (q_h, kp_h, vp_h, do_h, idx_h))
    o = torch.empty(w.B, w.T, w.H, w.DV, dtype=torch.bfloat16, device=dev)
    o_lo = torch.empty_like(o)
    lse = torch.empty(w.B, w.H, w.T, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty(w.B, w.T, w.H, w.DK, **f32)
    dkp, dvp = torch.empty(w.B, w.P, w.DK, **f32), torch.empty(w.B, w.P, w.DV, **f32)
    ws = torch.empty(attn.attn_sparse_bwd_workspace_size(w.B, w.T, w.H), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        attn.attn_sparse_fwd(q, kp, vp, idx, o, lse, w.scale, o_lo=o_lo, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        attn.attn_sparse_bwd(q, kp, vp, idx, o, do, lse, dq, dkp, dvp, w.scale, ws, o_lo=o_lo, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if attn.attn_check_status(ws) != 0:
        raise RuntimeError("kernel pipeline timeout during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if attn.attn_check_status(ws) != 0:
        raise RuntimeError("kernel pipeline timeout during the timed steps")
    ms = reduce_max(start.elapsed_time(stop), world) / args.steps
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    value = whole_job_value(flops, ms / 1e3, world) / 1e12

    pin = lambda t: t.pin_memory()
    hq_, hk_, hv_, hd_, hi_ = (pin(t) for t in (q_h, kp_h, vp_h, do_h, idx_h))
    ho, hlse, hdq, hdk, hdv = (pin(torch.empty(t.shape, dtype=t.dtype)) for t in (o, lse, dq, dkp, dvp))
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hd_, hi_))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

    def e2e_step():
        for dst, src in ((q, hq_), (kp, hk_), (vp, hv_), (do, hd_), (idx, hi_)):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in ((ho, o), (hlse, lse), (hdq, dq), (hdk, dkp), (hdv, dvp)):
            dst.copy_(src, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e_steps = max(1, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world) / e_steps

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf = fwd_flops / (fwd_ms / 1e3) / 1e12
    bwd_tf = 2.5 * fwd_flops / (bwd_ms / 1e3) / 1e12
    gathered = w.B * w.T * w.K * (w.DK + w.DV) * 2
    if rank == 0:
        line = {
            "metric": SPARSE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded CSA-shaped top-k lists, N(0,1) bf16 tensors)",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "P": w.P, "K": w.K, "DK": w.DK,
                       "DV": w.DV, "window": w.window, "topk": w.topk, "ratio": w.ratio,
                       "parallelism": f"replicas x{world}",
                       "l2": "no flush: q and o (1 GB and more) exceed the 129 MB L2; the pool is L2-resident",
                       "flops_per_step": flops},
            "gpu_launches": 3 * args.steps,
            "passes": {"sparse_fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak,
                                      "gathered_gbs": gathered / (fwd_ms / 1e3) / 1e9},
                       "sparse_bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak,
                                      "gathered_gbs": gathered / (bwd_ms / 1e3) / 1e9}},
            "roofline": {"kernel": "attn_sparse_bwd_kernel", "bound": "tensor", "achieved": bwd_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": bwd_tf / peak,
                         "traffic": traffic_for(w.name, SPARSE_SOURCES),
                         "peak_source": f"{peak_src} bf16_tflops (burst)"},
            "clocks": clocks.summary(),
            "e2e": {"value": whole_job_value(flops, e2e_ms / 1e3, world) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        }
        if not args.no_cpu_baseline:
            rate, sample, secs = sparse_oracle_sample(w, q_h, kp_h, vp_h, idx_h, do_h, budget_s=args.ref_budget)
            line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                    "sample": f"{sample}; {secs:.1f} s"}
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", choices=["residual", "plain"], default="residual",
                    help="residual: attn_fwd_residual + attn_bwd with o_lo (the training pair); "
                         "plain: attn_fwd + attn_bwd without o_lo (Dvec from the Dvec pass)")
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    from attention_fwd_bwd_gb300.inputs import BY_NAME, SPARSE_BY_NAME
    if args.workload not in BY_NAME and args.workload not in SPARSE_BY_NAME:
        ap.error(f"unknown workload {args.workload!r}; dense: {', '.join(BY_NAME)}; "
                 f"sparse: {', '.join(SPARSE_BY_NAME)}")
    sparse = args.workload in SPARSE_BY_NAME
    w = SPARSE_BY_NAME[args.workload] if sparse else BY_NAME[args.workload]
    world, rank, local = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if sparse:
            return run_sparse(args, w, world, rank, local)
        if args.impl == "reference":
            return run_reference(args, w, world, rank)
        return run_ours(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
