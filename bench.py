"""Benchmark of the KDA token-mixer hot path on GB300.

Main line (value): prefill tokens/s per layer on the single-layer, Ling-shaped workload
(B=1, T=4096, H=64, d=128, bf16 I/O, fp32 state, zero initial state, chunk 64).  One step is
the whole prefill hot path over that batch: kda_prologue (width-4 causal conv + SiLU over the
raw q|k|v projections, beta = sigmoid) then kda_prefill (q/k L2 norm, g clamp at -5, the
chunked recurrence).  Each activation runs once, inside the kernel that consumes it: the
prefill reads the raw log-retention and normalises q and k itself, so the prologue writes
neither a clamped copy of g nor normalised q, k.
Also reported: the prefill kernel alone, the decode workload (256 sequences x 1 token,
H=64, d=128, fp32 state pool ~N(0,0.02), fused conv + decode, 100 consecutive steps) as
state GB/s, the roofline of the dominant kernel against MEASURED_PEAKS.json, an end-to-end
number through the host-buffer call kda_prefill_host (copies in and out inside the timed
region), and the oracle timed on the host cores.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_PREFILL, H, D = 4096, 64, 128
N_DECODE, DECODE_STEPS = 256, 100
METRIC = "KDA prefill tokens/s/layer"
WORKLOAD = ("Single-layer KDA prefill, Ling-shaped: B=1, T=4096, H=64, d_k=d_v=128, bf16 "
            "q/k/v (raw projections ~N(0,1) through the width-4 causal conv+SiLU prologue), "
            "fp32 log-alpha ~U(-5,0) clamped at -5, beta=sigmoid(N(0,1)), fp32 state, zero "
            "initial state, chunk 64")
L2_BYTES = 129 * 2**20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(
            pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


CSRC = os.path.join(ROOT, "hybrid_linear_attention_gb300", "csrc")


def _profiled_traffic(summary, sources):
    """DRAM bytes per launch from a committed ncu summary in profiles/, or None when the
    kernel's sources changed since that capture (hash of the concatenated sources)."""
    import hashlib
    try:
        h = hashlib.sha256()
        for src in sources:
            with open(os.path.join(CSRC, src), "rb") as f:
                h.update(f.read())
        want, traffic = None, None
        with open(os.path.join(ROOT, "profiles", summary)) as f:
            for line in f:
                if line.startswith("source_sha256_16:"):
                    want = line.split()[1]
                elif line.startswith("traffic_bytes_per_launch:"):
                    traffic = int(line.split()[1])
        return traffic if want == h.hexdigest()[:16] else None
    except Exception:
        return None


def _prefill_bytes(T, H, d, with_state_out=True):
    """Algorithmic HBM bytes of one kda_prefill launch: q, k, v, out (bf16), g (fp32),
    beta (fp32), plus the final fp32 state."""
    per_tok = H * d * (2 * 3 + 4 + 2) + H * 4
    return T * per_tok + (H * d * d * 4 if with_state_out else 0)


def _prefill_flops(T, H, d, C=64):
    """Algorithmic tensor FLOPs of the chunked form, each dense contraction counted once per
    64-token chunk and head: A and P (two C x C x d_k), T = (I + A)^-1 (C^3 / 3), X = [K Gamma;
    Q Gamma] S (2C x d_k x d_v), u = T Y (C x C x d_v), O += P' u (C x C x d_v), S += Kbar^T u
    (d_k x C x d_v); 2 flops per multiply-add."""
    per = 2 * (2 * C * C * d + C ** 3 / 3 + 2 * C * d * d + 2 * C * C * d + d * C * d)
    return T / C * H * per


# a triangle-aware count of the prefill's dense work per head and token at d = 128, C = 64:
# 2 (3 d^2 + 2.5 C d) -- the state read, correction and update (3 d^2 multiply-adds) and the
# intra-chunk products on their triangles (2.5 C d)
TRIANGLE_FLOPS_PER_HEAD_TOKEN = 2 * (3 * 128 * 128 + 2.5 * 64 * 128)


def _prefill_bytes_batch(lengths, H, d, *, gate, state_in, state_bytes=4):
    """Algorithmic HBM bytes of one kda_prefill launch over a packed batch: per token q, k, v,
    out (bf16), g (fp32), beta (fp32) and, with the output norm and gate, the gate logits
    (bf16); per sequence the final state and, when given, the initial state."""
    T = int(sum(lengths))
    per_tok = H * d * (2 * 3 + 4 + 2) + H * 4 + (H * d * 2 if gate else 0)
    n = len(lengths)
    st = H * d * d * state_bytes
    return T * per_tok + n * st * (2 if state_in else 1)


def _prologue_bytes(T, H, d):
    """kda_prologue as the step runs it: read raw x (3Hd bf16) + beta logits; write q, k, v
    (bf16) and beta (fp32)."""
    C = 3 * H * d
    return T * (C * 2 * 2 + H * 4 * 2)


def _decode_bytes(n, H, d):
    """One fused decode step for n sequences: state read+write (fp32), conv tail read+write,
    raw x, g, beta, conv weights, out."""
    C = 3 * H * d
    return (2 * n * H * d * d * 4 + 2 * n * 3 * C * 2 + n * C * 2 + n * H * d * 4 + n * H * 4
            + C * 4 * 2 + n * H * d * 2)


class ClockSampler:
    """nvidia-smi samples every 50 ms; the summary keeps the samples whose timestamps fall
    inside the timed window (window() marks its start and end)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def window(self, start):
        import datetime
        if start:
            self.t0 = datetime.datetime.now()
        else:
            self.t1 = datetime.datetime.now()
            time.sleep(0.1)  # the sample in flight at the end

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        import datetime
        rows = []
        try:
            for line in open(self.path):
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 10:
                    try:
                        p[0] = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f")
                    except ValueError:
                        continue
                    rows.append(p)
        except Exception:
            pass
        if self.t0 and self.t1:
            inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
            rows = inside or [r for r in rows if r[0] >= self.t0]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows), "period_ms": 50}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")
        return dist, dist.get_rank(), ws
    return None, 0, 1


def _barrier(dist):
    if dist:
        dist.barrier()


def _max_over_ranks(dist, x):
    if not dist:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# Oracle timing (host cores)
# ---------------------------------------------------------------------------------------

def _oracle_prefill_sample(heads, seed=0):
    """The oracle on the prefill workload restricted to `heads` heads (the whole layer when
    heads == H): prologue (conv+SiLU+L2 on the sampled heads' channels) then recurrence.
    Returns (seconds, threads)."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_gb300 import inputs

    pin = inputs.prologue_inputs([T_PREFILL], heads, D, seed=seed, conv_state=False)
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    pr = oracle.prologue(pin["x"], pin["conv_w"], pin["cu_seqlens"], heads, D,
                         beta_logit=pin["beta_logit"])
    y = pr["y"].reshape(T_PREFILL, 3, heads, D)
    oracle.kda_forward(np.ascontiguousarray(y[:, 0]), np.ascontiguousarray(y[:, 1]),
                       np.ascontiguousarray(y[:, 2]), pin["g_raw"],
                       pr["beta"].astype(np.float32), pin["cu_seqlens"], qk_l2norm=True,
                       n_threads=threads)
    return time.perf_counter() - t0, threads


CPU_SAMPLE_HEADS = 32


CPU_SINGLE_HEADS = 4


def _oracle_single_thread(heads=CPU_SINGLE_HEADS, seed=5):
    """The oracle's fp64 recurrence on one host thread over `heads` heads of the prefill
    workload (T = 4096, post-conv inputs drawn directly); returns seconds."""
    import oracle
    from hybrid_linear_attention_gb300 import inputs

    inp = inputs.kda_inputs([T_PREFILL], heads, D, seed=seed)
    t0 = time.perf_counter()
    oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"],
                       n_threads=1)
    return time.perf_counter() - t0


def _cpu_baseline():
    secs, threads = _oracle_prefill_sample(CPU_SAMPLE_HEADS)
    # tokens/s/layer: the sample covers CPU_SAMPLE_HEADS of the layer's H heads
    value = T_PREFILL * CPU_SAMPLE_HEADS / H / secs
    s1 = _oracle_single_thread()
    v1 = T_PREFILL * CPU_SINGLE_HEADS / H / s1
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"T=4096 tokens x {CPU_SAMPLE_HEADS} of 64 heads (prologue + fp64 "
                      f"recurrence), scaled to one full layer; {secs:.2f} s wall",
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                              "sample": f"T=4096 tokens x {CPU_SINGLE_HEADS} of 64 heads (fp64 "
                                        f"recurrence, one host thread), scaled to one full "
                                        f"layer; {s1:.2f} s wall"}}


def run_reference(args):
    dist, rank, ws = _dist()
    if rank != 0:
        return
    for _ in range(args.warmup):
        _oracle_prefill_sample(CPU_SAMPLE_HEADS, seed=1)
    times = []
    threads = 1
    for s in range(args.steps):
        secs, threads = _oracle_prefill_sample(CPU_SAMPLE_HEADS, seed=2 + s)
        times.append(secs)
    per = sum(times) / len(times)
    value = T_PREFILL * CPU_SAMPLE_HEADS / H / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{CPU_SAMPLE_HEADS} of 64 heads per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"T=4096 x {CPU_SAMPLE_HEADS}/64 heads per step, scaled"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------

class PrefillWorkload:
    def __init__(self, dev, seed=0):
        from hybrid_linear_attention_gb300 import inputs, kda
        self.kda = kda
        self.p = kda.params(H=H, d=D)
        pin = inputs.prologue_inputs([T_PREFILL], H, D, seed=seed, device=dev, conv_state=False)
        self.x, self.w = pin["x"], pin["conv_w"]
        self.beta_logit, self.g_raw = pin["beta_logit"], pin["g_raw"]
        self.cu = pin["cu_seqlens"]
        T = T_PREFILL
        self.q = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
        self.k, self.v = torch.empty_like(self.q), torch.empty_like(self.q)
        self.beta = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
        self.out_q = torch.empty((T, H, D), dtype=torch.uint8, device=dev)
        self.out_scale = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.fin = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)

    def prologue(self, stream=None):
        self.kda.kda_prologue(self.p, self.x, self.w, None, self.cu, self.q, self.k, self.v,
                              l2norm_qk=False, beta_logit=self.beta_logit, beta=self.beta,
                              stream=stream)

    def prefill(self, stream=None):
        # the raw log-retention goes straight in: the kernel clamps it at g_min (and the
        # params' qk_l2norm normalises q, k) as it loads them
        self.kda.kda_prefill(self.p, self.q, self.k, self.v, self.g_raw, self.beta, self.cu,
                             self.out, final_state=self.fin, stream=stream)

    def prefill_fp8(self, stream=None):
        # the same recurrence with the output quantised to FP8 in the epilogue
        self.kda.kda_prefill_fp8(self.p, self.q, self.k, self.v, self.g_raw, self.beta, self.cu,
                                 self.out_q, self.out_scale, final_state=self.fin, stream=stream)


def run_ours(args):
    dist, rank, ws = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from hybrid_linear_attention_gb300 import inputs, kda

    hbm, tflops, tflops_sus, peak_kind = _peaks()
    # the global batch is one T=4096 sequence per rank; each rank owns its share (no
    # collective on the data path)
    from hybrid_linear_attention_gb300.sharding import sequence_shard
    mine = sequence_shard([T_PREFILL] * ws, ws, rank)
    wl = PrefillWorkload(dev, seed=mine[0])
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    for _ in range(max(args.warmup, 3)):
        wl.prologue()
        wl.prefill()
    torch.cuda.synchronize()

    # ---- timed region: K steps (prologue + prefill), L2 flushed between steps ----------
    step_ms, pro_ms, pf_ms = [], [], []
    launches0 = kda.kda_launch_count()
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.window(True)
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()
            e0, e1, e2 = ev(), ev(), ev()
            e0.record(stream)
            wl.prologue()
            e1.record(stream)
            wl.prefill()
            e2.record(stream)
            e2.synchronize()
            pro_ms.append(e0.elapsed_time(e1))
            pf_ms.append(e1.elapsed_time(e2))
            step_ms.append(e0.elapsed_time(e2))
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        clk.window(False)
    _barrier(dist)
    launches = kda.kda_launch_count() - launches0
    kda.kda_check_device_error()
    ms = _max_over_ranks(dist, sum(step_ms) / len(step_ms))
    pf = _max_over_ranks(dist, sum(pf_ms) / len(pf_ms))
    pro = _max_over_ranks(dist, sum(pro_ms) / len(pro_ms))
    value = ws * T_PREFILL / (ms * 1e-3)

    # ---- the prefill with FP8 output (codes + one scale per token and head) ------------
    pf8_ms = []
    for i in range(3 + min(args.steps, 50)):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        wl.prefill_fp8()
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            pf8_ms.append(e0.elapsed_time(e1))
    kda.kda_check_device_error()
    pf8 = _max_over_ranks(dist, sum(pf8_ms) / len(pf8_ms))

    # ---- end to end through the host-buffer call (kda_prefill_host) -----------------
    e2e_line = _e2e(wl, flush, args, dist) if not args.no_e2e else None

    # ---- the other prefill workloads: long-context gated (4 x 32768) and the packed
    #      variable-length batch (~500K tokens; fp32 and bf16 state storage) ----------------
    long_ctx = varlen = None
    if not args.no_configs:
        long_ctx = _long_context_bench(dev, kda, inputs, hbm, tflops, args)
        varlen = None if args.no_varlen else _varlen_bench(dev, kda, inputs, hbm, args)

    # ---- decode: 256 sequences x 100 fused steps --------------------------------------
    dec = dmulti = mla = None
    if not args.no_decode:
        dec = _decode_bench(dev, kda, inputs, hbm, rank, args)
        dmulti = _decode_multi_bench(dev, kda, inputs, hbm, rank)
        mla = _mla_bench(dev, kda, inputs, hbm, rank)

    if rank != 0:
        return
    pf_bytes = _prefill_bytes(T_PREFILL, H, D)
    pf_flops = _prefill_flops(T_PREFILL, H, D)
    achieved = pf_bytes / (pf * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": T_PREFILL, "heads": H, "d": D,
                   "chunk": 64, "parallelism": f"sequence-sharded x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2 (403 MB) and a 258 MB buffer written between "
                         "steps"},
        "breakdown_ms": {"prologue": pro, "prefill": pf},
        "prefill_fp8_output_ms": pf8,
        "prefill_kernel_tokens_per_s": ws * T_PREFILL / (pf * 1e-3),
        "roofline": {"kernel": "kda_prefill", "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "traffic": _profiled_traffic(
                         "kda_prefill_tc_T4096_H64.md",
                         ["kda_prefill_tc.cu", "kda_tc_ptx.cuh", "kda_common.cuh"]),
                     "algorithmic_bytes_per_launch": pf_bytes,
                     # the same launch against the tensor-core peak (the chunked form's dense
                     # contractions, counted once; intensity ~107 flop/B is under the ridge,
                     # so HBM is the binding roofline)
                     "tensor": {"achieved_tflops": pf_flops / (pf * 1e-3) / 1e12,
                                "peak_tflops": tflops,
                                "frac": pf_flops / (pf * 1e-3) / 1e12 / tflops,
                                "peak_kind": f"{peak_kind} bf16_tflops (burst)",
                                "algorithmic_flops_per_launch": pf_flops,
                                # the triangle-aware count, 139,264 flop per head-token
                                "triangle_flops_per_head_token": TRIANGLE_FLOPS_PER_HEAD_TOKEN,
                                "triangle_frac": TRIANGLE_FLOPS_PER_HEAD_TOKEN * T_PREFILL * H
                                               / (pf * 1e-3) / 1e12 / tflops}},
        "gpu_launches": int(launches),
        "gpu_launches_per_step": launches / args.steps,
        "wall_s_timed_region": wall,
        "clocks": clk.summary(),
    }
    if e2e_line:
        line["e2e"] = e2e_line
    if long_ctx:
        line["long_context_gated"] = long_ctx
    if varlen:
        line["varlen_500k"] = varlen
    if dec:
        line["decode"] = dec
    if dmulti:
        line["decode_multi"] = dmulti
        line["mla_decode"] = mla
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = _cpu_baseline()
    print(json.dumps(line), flush=True)


E2E_SEGMENT = 512  # tokens per streamed segment of kda_prefill_host


def _e2e(wl, flush, args, dist):
    """The same step through the public host-buffer call, kda_prefill_host: the step's inputs
    (raw projections, raw log-retention, beta logits) in pinned host memory, the output and
    final state written back to pinned host memory; the call streams the sequence through
    the GPU in chunk-aligned segments, so the copies of neighbouring segments overlap the
    kernels.  Everything from the first copy in to the last copy out is inside the timed
    region (host clock around the call and a device synchronisation)."""
    kda = wl.kda
    ws_ = dist.get_world_size() if dist else 1
    hx = wl.x.cpu().pin_memory()
    hg = wl.g_raw.cpu().pin_memory()
    hb = wl.beta_logit.cpu().pin_memory()
    hcu = wl.cu.cpu().contiguous()
    hout = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()
    hfin = torch.empty(wl.fin.shape, dtype=wl.fin.dtype).pin_memory()
    work = torch.empty(kda.kda_prefill_host_workspace_size(wl.p, 1, E2E_SEGMENT),
                       dtype=torch.uint8, device=wl.x.device)
    h2d = hx.numel() * 2 + hg.numel() * 4 + hb.numel() * 4
    d2h = hout.numel() * 2 + hfin.numel() * 4
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        kda.kda_prefill_host(wl.p, hx, wl.w, None, hcu, hb, hg, hout, workspace=work,
                             segment_tokens=E2E_SEGMENT, final_state=hfin)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = _max_over_ranks(dist, sum(e2e_ms) / len(e2e_ms))
    return {"value": ws_ * T_PREFILL / (e2e * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e,
            "api": "kda_prefill_host", "segment_tokens": E2E_SEGMENT}


def _time_prefill(kda, p, inp, out, fin, *, gate, reps, flush):
    """CUDA-event milliseconds of kda_prefill over a resident batch (L2 flushed between
    launches; 3 untimed launches first)."""
    ts = []
    for i in range(3 + reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kda.kda_prefill(p, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                        inp["cu_seqlens"], out, init_state=inp.get("init_state"),
                        final_state=fin, gate_logit=inp["gate"] if gate else None,
                        norm_w=inp["norm_w"] if gate else None)
        e1.record()
        e1.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1))
    kda.kda_check_device_error()
    return sum(ts) / len(ts)


def _long_context_bench(dev, kda, inputs, hbm, tflops, args):
    """Long-context prefill: 4 sequences x 32768 tokens, H = 64, d = 128, bf16 q, k, v drawn
    N(0,1) as the post-conv streams, fp32 log-retention U(-5,0) and beta, nonzero initial
    state ~N(0,0.02), the output RMSNorm x sigmoid(gate) with gate logits ~N(0,1)."""
    per_seq = args.long_tokens
    lens = [per_seq] * 4
    inp = inputs.kda_inputs(lens, H, D, seed=700, device=dev, init_state="all", gate=True)
    p = kda.params(H=H, d=D)
    T = sum(lens)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((len(lens), H, D, D), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    ms = _time_prefill(kda, p, inp, out, fin, gate=True, reps=min(args.steps, 5), flush=flush)
    b = _prefill_bytes_batch(lens, H, D, gate=True, state_in=True)
    gbs = b / (ms * 1e-3) / 1e9
    tf = TRIANGLE_FLOPS_PER_HEAD_TOKEN * T * H / (ms * 1e-3) / 1e12
    del inp, out, fin
    torch.cuda.empty_cache()
    # DRAM bytes of one launch from the ncu summary of the same kernel on 4 x 8192 tokens,
    # scaled by the tokens (the launch streams its inputs once: traffic grows in proportion)
    traffic = _profiled_traffic("kda_prefill_tc_fused_gated_4x8192_H64.md",
                                ["kda_prefill_tc.cu", "kda_tc_ptx.cuh", "kda_common.cuh"])
    return {"workload": f"4 x {per_seq} tokens, H=64, d=128, bf16 q/k/v, fp32 g/beta/state, "
                        "initial state ~N(0,0.02), output RMSNorm(128) x sigmoid(gate), gate "
                        "logits ~N(0,1) bf16",
            "ms": ms, "tokens_per_s": T / (ms * 1e-3),
            "roofline": {"kernel": "kda_prefill (gated)", "bound": "hbm", "achieved": gbs,
                         "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "traffic": traffic * per_seq / 8192 if traffic else None,
                         "algorithmic_bytes_per_launch": b,
                         "bytes_per_token": 114944,
                         "tensor_frac": tf / tflops}}


def _varlen_bench(dev, kda, inputs, hbm, args):
    """The packed variable-length batch: 32 sequences, lengths log-uniform in [512, 65536]
    (total ~500K tokens), even-indexed sequences from a nonzero initial state; once with fp32
    and once with bf16 state storage."""
    lens, _ = inputs.varlen_lengths(n_seqs=32, seed=0)
    T = sum(lens)
    res = {"workload": f"32 sequences, log-uniform lengths in [512, 65536], {T} tokens packed "
                       f"by cu_seqlens, H=64, d=128, bf16 I/O, even sequences from ~N(0,0.02)",
           "tokens": T}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for name, sd in (("fp32_state", torch.float32), ("bf16_state", torch.bfloat16)):
        inp = inputs.kda_inputs(lens, H, D, seed=710, device=dev, init_state="even",
                                state_dtype=sd)
        p = kda.params(H=H, d=D, state_dtype=sd)
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
        fin = torch.empty((len(lens), H, D, D), dtype=sd, device=dev)
        ms = _time_prefill(kda, p, inp, out, fin, gate=False, reps=min(args.steps, 3),
                           flush=flush)
        b = _prefill_bytes_batch(lens, H, D, gate=False, state_in=True,
                                 state_bytes=2 if sd == torch.bfloat16 else 4)
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3),
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                  "frac": gbs / hbm, "algorithmic_bytes_per_launch": b}}
        del inp, out, fin
        torch.cuda.empty_cache()
    return res


def _decode_bench(dev, kda, inputs, hbm, rank, args):
    n, C = N_DECODE, 3 * H * D
    p = kda.params(H=H, d=D)
    state = inputs.normal((n, H, D, D), seed=300 + rank, device=dev, dtype=torch.float32,
                          std=0.02)
    cs = inputs.normal((n, 3, C), seed=301 + rank, device=dev)
    w = inputs.normal((C, 4), seed=302 + rank, device=dev, std=0.5)
    K = DECODE_STEPS
    x = inputs.normal((K, n, C), seed=303 + rank, device=dev)
    g = inputs.uniform((K, n, H, D), -5.0, 0.0, seed=304 + rank, device=dev)
    beta = inputs.beta_draw((K, n, H), seed=305 + rank, device=dev)
    out = torch.empty((K, n, H, D), dtype=torch.bfloat16, device=dev)
    for t in range(3):
        kda.kda_decode_step_fused(p, x[t], w, cs, g[t], beta[t], state, out[t])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(K):
        kda.kda_decode_step_fused(p, x[t], w, cs, g[t], beta[t], state, out[t])
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / K
    b = _decode_bytes(n, H, D)
    gbs = b / (ms * 1e-3) / 1e9
    # the same steps with the output quantised to FP8 in the epilogue (codes + one fp32
    # scale per sequence and head instead of bf16 values)
    q8 = torch.empty((K, n, H, D), dtype=torch.uint8, device=dev)
    sc8 = torch.empty((K, n, H), dtype=torch.float32, device=dev)
    for t in range(3):
        kda.kda_decode_step_fused_fp8(p, x[t], w, cs, g[t], beta[t], state, q8[t], sc8[t])
    torch.cuda.synchronize()
    e0.record()
    for t in range(K):
        kda.kda_decode_step_fused_fp8(p, x[t], w, cs, g[t], beta[t], state, q8[t], sc8[t])
    e1.record()
    e1.synchronize()
    ms8 = e0.elapsed_time(e1) / K
    b8 = b - n * H * D * 2 + n * H * D + n * H * 4
    fp8 = {"kernel": "kda_decode_step_fused_fp8", "ms_per_step": ms8,
           "achieved_gbs": b8 / (ms8 * 1e-3) / 1e9, "frac": b8 / (ms8 * 1e-3) / 1e9 / hbm,
           "algorithmic_bytes_per_launch": b8}
    return {"metric": "KDA decode state GB/s", "value": gbs, "unit": "GB/s", "fp8_output": fp8,
            "workload": "256 sequences x 1 token, H=64, d=128, fp32 state pool [256,64,128,128]"
                        " ~N(0,0.02) (1 GiB, > L2), bf16 conv tails, fused conv+decode, 100 "
                        "consecutive steps",
            "ms_per_step": ms, "tokens_per_s": n / (ms * 1e-3),
            "roofline": {"kernel": "kda_decode_step_fused", "bound": "hbm", "achieved": gbs,
                         "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "traffic": _profiled_traffic("kda_decode_fused_N256_H64.md",
                                                      ["kda_decode.cu", "kda_common.cuh"]),
                         "algorithmic_bytes_per_launch": b}}


N_MLA, L_MLA = 256, 4096


def _mla_bench(dev, kda, inputs, hbm, rank):
    """Absorbed gated-MLA decode: 256 sequences x 4096 cached positions, 64 heads, 576-wide
    bf16 latent cache (1.21 GB, > L2), one query token each; the latent attention streams the
    cache once.  Also the whole step (absorption + attention + up-projection + gate)."""
    B, L = N_MLA, L_MLA
    cache = inputs.normal((B, L, 576), seed=600 + rank, device=dev)
    q_nope = inputs.normal((B, 64, 128), seed=601 + rank, device=dev)
    q_rope = inputs.normal((B, 64, 64), seed=602 + rank, device=dev)
    w_uk = inputs.normal((64, 128, 512), seed=603 + rank, device=dev, std=0.05)
    w_uv = inputs.normal((64, 128, 512), seed=604 + rank, device=dev, std=0.05)
    gate = inputs.normal((B, 64), seed=605 + rank, device=dev)
    lengths = torch.full((B,), L, dtype=torch.int32, device=dev)
    q_cat = torch.empty((B, 64, 576), dtype=torch.bfloat16, device=dev)
    z = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
    out = torch.empty((B, 64, 128), dtype=torch.bfloat16, device=dev)
    # the workspace the library asks for (none at 256 sequences: no split pays)
    ws_n = kda.mla_decode_workspace_size(B, L)
    ws = torch.empty(max(ws_n // 4, 1), dtype=torch.float32, device=dev) if ws_n else None
    step = lambda: kda.mla_decode(q_nope, q_rope, w_uk, w_uv, cache, lengths, gate, q_cat, z, out,
                                  workspace=ws)
    lat = lambda: kda.mla_decode_latent(q_cat, cache, lengths, z, workspace=ws)
    reps = 20
    res = {}
    step()  # the absorbed queries the latent attention reads alone come from the step
    for name, fn in (("latent", lat), ("step", step)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        e1.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
    kda.kda_check_device_error()
    b = B * L * 576 * 2 + B * 64 * 576 * 2 + B * 64 * 512 * 4  # cache + query + z
    gbs = b / (res["latent"] * 1e-3) / 1e9
    del cache
    small = _mla_small_batch(dev, kda, inputs, hbm, rank)
    return {"metric": "MLA decode latent-cache GB/s", "value": gbs, "unit": "GB/s",
            "workload": "256 sequences x 4096 cached positions, 64 heads, 576-wide bf16 latent "
                        "cache (512 latent + 64 positional key; 1.21 GB, > L2), one query token "
                        "each, synthetic weights",
            "ms_latent": res["latent"], "ms_step": res["step"], "workspace_bytes": ws_n,
            "tokens_per_s": B / (res["step"] * 1e-3),
            "roofline": {"kernel": "mla_decode_latent", "bound": "hbm", "achieved": gbs,
                         "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "traffic": _profiled_traffic(
                             "mla_latent_B256_L4096.md",
                             ["mla_decode.cu", "kda_tc_ptx.cuh", "kda_common.cuh"]),
                         "algorithmic_bytes_per_launch": b},
            "small_batch": small}


def _mla_small_batch(dev, kda, inputs, hbm, rank):
    """4 sequences x 65536 cached positions (302 MB, > L2): one CTA per sequence leaves most
    SMs idle; with the workspace each sequence's positions are split across CTAs and merged."""
    B, L, reps = 4, 65536, 20
    cache = inputs.normal((B, L, 576), seed=610 + rank, device=dev)
    q_cat = inputs.normal((B, 64, 576), seed=611 + rank, device=dev)
    lengths = torch.full((B,), L, dtype=torch.int32, device=dev)
    z = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
    ws_bytes = kda.mla_decode_workspace_size(B, L)
    ws = torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=dev)
    res = {}
    for name, w in (("split", ws), ("one_cta_per_sequence", None)):
        fn = lambda: kda.mla_decode_latent(q_cat, cache, lengths, z, workspace=w)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        e1.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
    kda.kda_check_device_error()
    b = B * L * 576 * 2 + B * 64 * 576 * 2 + B * 64 * 512 * 4
    gbs = b / (res["split"] * 1e-3) / 1e9
    return {"workload": "4 sequences x 65536 cached positions (302 MB latent cache)",
            "workspace_bytes": ws_bytes, "ms_latent_split": res["split"],
            "ms_latent_one_cta_per_sequence": res["one_cta_per_sequence"],
            "gbs": gbs, "frac": gbs / hbm}


def _decode_multi_bench(dev, kda, inputs, hbm, rank):
    """Speculative draft: 256 sequences x K=3 tokens, state after every token kept (fp32),
    then the commit of the accepted steps."""
    n, K, reps = N_DECODE, 3, 20
    p = kda.params(H=H, d=D)
    rows = n * K
    pool = inputs.normal((n, H, D, D), seed=400 + rank, device=dev, dtype=torch.float32,
                         std=0.02)
    q = inputs.normal((rows, H, D), seed=401 + rank, device=dev)
    k = inputs.normal((rows, H, D), seed=402 + rank, device=dev)
    v = inputs.normal((rows, H, D), seed=403 + rank, device=dev)
    g = inputs.uniform((rows, H, D), -5.0, 0.0, seed=404 + rank, device=dev)
    beta = inputs.beta_draw((rows, H), seed=405 + rank, device=dev)
    out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    steps = torch.empty((rows, H, D, D), dtype=torch.float32, device=dev)
    acc = (torch.arange(n, device=dev, dtype=torch.int32) % (K + 1)).contiguous()
    for _ in range(3):
        kda.kda_decode_multi(p, q, k, v, g, beta, pool, out, K, step_states=steps)
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record()
    for _ in range(reps):
        kda.kda_decode_multi(p, q, k, v, g, beta, pool, out, K, step_states=steps)
    e1.record()
    for _ in range(reps):
        kda.kda_state_accept(p, steps, acc, pool, K)
    e2.record()
    e2.synchronize()
    ms = e0.elapsed_time(e1) / reps
    ms_acc = e1.elapsed_time(e2) / reps
    st = n * H * D * D * 4
    b = st * (1 + K) + rows * H * (3 * D * 2 + D * 4 + 4 + D * 2)
    acc_bytes = 2 * st * int((acc > 0).sum().item()) // n
    gbs = b / (ms * 1e-3) / 1e9
    return {"metric": "KDA speculative draft GB/s", "value": gbs, "unit": "GB/s",
            "workload": "256 sequences x K=3 draft tokens, H=64, d=128, fp32 state pool (1 GiB) "
                        "read once, fp32 state after every token written (3 GiB)",
            "ms_per_call": ms, "tokens_per_s": rows / (ms * 1e-3),
            "roofline": {"kernel": "kda_decode_multi", "bound": "hbm", "achieved": gbs,
                         "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "algorithmic_bytes_per_launch": b},
            "accept": {"ms_per_call": ms_acc, "bytes": acc_bytes,
                       "gbs": acc_bytes / (ms_acc * 1e-3) / 1e9}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    # tokens per sequence of the long-context gated workload (4 sequences): 32768; a smaller
    # value serves the profiler's capture of the same kernel
    ap.add_argument("--long-tokens", type=int, default=32768)
    ap.add_argument("--no-varlen", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
