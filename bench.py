#!/usr/bin/env python3
"""Benchmark of the batch-invariant selected-token logprob on GB300.

Workload (one "step" = one pass of the whole path over one batch):
  Qwen3-8B-shaped LM head, training recompute: T = 4096 rows (8 packed
  sequences of 512), H = 4096, V = 151936, RMS-normalised bf16 hidden states,
  W ~ N(0, 0.02) bf16, uniform int32 targets, inv_temp = 1.0, 10% of the
  tokens masked out of the acceptance statistics.  Synthetic and seeded: no
  model weights or datasets exist here.
  Step = rlk_logprob_partials (fused tcgen05 GEMM + vocabulary-tile epilogue)
       -> rlk_lse_merge (fixed-tree merge)
       -> rlk_consistency_stats_async against a stored "rollout" logprob
          vector (the acceptance check of every step, stream-ordered into
          device memory; every step's statistics are read and checked after
          the timed region).
  W alone is 1.245 GB, ten times L2 (129 MB), so inputs are larger than L2 and
  no flush is needed between steps.

Printed (rank 0, one JSON line): device-timed tokens/s over the whole job,
e2e tokens/s through rlk_logprob + rlk_consistency_stats_async with pinned
host buffers (H2D of h and targets, D2H of logp/lse/argmax and the 8
statistics inside the timed region; W stays resident as model weights do), the dominant kernel's roofline from live CUDA events, SM
clocks sampled during the timed region, the CPU oracle's throughput on a
bounded sample, decode-regime points (T = 1..256: HBM-bound at small T), the
backward (rlk_logprob_backward on the same batch), the FP8 (W8A8) variants
(per-row and block-scaled scales), the entropy path and the vocabulary-sharded phases (R = 2, 3, 6 shards emulated on
one GPU).

--workload picks the batch a step runs over: train4096 (the default above),
prefill16384 (4 x 4096 = 16384 rows, H = 4096, inv_temp = fp32(1/0.7), no
mask) or packed32768 (32768 rows, H = 5120, 1% outlier rows x8, 10% masked).
Each prints the same JSON line (roofline, clocks, e2e, CPU baseline); the
other regimes (decode, backward, fp8, entropy, shards) run with the default
workload only.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores, each step a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_CFG, H_CFG, V_CFG = 4096, 4096, 151936
# --workload: the training-recompute batch (the default, the headline line) and
# the two larger tensor-bound workloads, timed the same way.
WORKLOADS = {
    "train4096": dict(T=4096, H=4096, inv_temp=1.0, outlier_frac=0.0, mask_zero_frac=0.1,
                      name="Qwen3-8B LM head, training recompute: T=4096 (8 packed x 512), "
                           "H=4096, V=151936"),
    "prefill16384": dict(T=16384, H=4096, inv_temp=float(__import__("numpy").float32(1 / 0.7)),
                         outlier_frac=0.0, mask_zero_frac=0.0,
                         name="prefill vs decode phase consistency: 4 sequences x 4096 = "
                              "T=16384, H=4096, V=151936, inv_temp=fp32(1/0.7)"),
    "packed32768": dict(T=32768, H=5120, inv_temp=1.0, outlier_frac=0.01, mask_zero_frac=0.1,
                        name="large packed batch: T=32768, H=5120, V=151936, 1% outlier rows "
                             "x8, 10% of tokens masked out of the statistics"),
}
METRIC = "tokens/s of batch-invariant logprob (H=4096,V=151936); % of TC/HBM roofline"
KERNEL_SOURCES = ["invariant_token_logprob_gb300/csrc/rlk_lmhead.cu",
                  "invariant_token_logprob_gb300/csrc/rlk_sm103.cuh",
                  "invariant_token_logprob_gb300/csrc/rlk_lse.cuh",
                  "invariant_token_logprob_gb300/csrc/rlk_fp8_quant.cuh",
                  "invariant_token_logprob_gb300/csrc/rlk_internal.h"]
def traffic_file(T, H, V):
    return os.path.join(ROOT, "profiles", f"lmhead_partials_T{T}_H{H}_V{V}.md")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="train4096", choices=sorted(WORKLOADS),
                   help="train4096 (default): T=4096, H=4096; prefill16384: T=16384, "
                        "inv_temp=fp32(1/0.7); packed32768: T=32768, H=5120 (the other regimes "
                        "-- decode, backward, fp8, entropy, shards -- run with the default only)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-fp8", action="store_true")
    p.add_argument("--no-entropy", action="store_true")
    p.add_argument("--no-shard", action="store_true")
    p.add_argument("--decode-only", action="store_true",
                   help="time only the decode regime at T = --decode-T (for profiling)")
    p.add_argument("--decode-T", type=int, default=1)
    p.add_argument("--fp8", action="store_true", help="decode-only: the FP8 (e4m3 W) variant")
    p.add_argument("--backward-only", action="store_true",
                   help="time only rlk_logprob_backward (T=4096, H=4096, V=--bwd-V) per product "
                        "(for profiling)")
    p.add_argument("--bwd-V", type=int, default=V_CFG)
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def kernel_hash():
    """Hash of the LM-head kernel's code: comments and whitespace are dropped, so
    only a change that can change the compiled kernel invalidates recorded
    counters."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        src = open(os.path.join(ROOT, rel), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(T, H, V):
    """DRAM bytes per launch of the LM-head kernel from the committed ncu summary
    of this workload, if that capture was taken of the kernel sources as they are
    now."""
    path = traffic_file(T, H, V)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    mh = re.search(r"^kernel_hash:\s*([0-9a-f]+)\s*$", text, re.M)
    mt = re.search(r"^traffic_bytes_per_launch:\s*([0-9]+)\s*$", text, re.M)
    if not mh or not mt or mh.group(1) != kernel_hash():
        return None
    return dict(bytes_per_launch=int(mt.group(1)), source=os.path.relpath(path, ROOT))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.samples:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(t=t, sm=float(f[1]), smax=float(f[2]), active=f[4],
                                 hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        inwin = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r["t"] <= self.t_stop]
        window = "timed"
        if len(inwin) < 3:  # very short timed region: fall back to all samples under load
            inwin = [r for r in rows if r["sm"] > 0.5 * r["smax"]] or rows
            window = "warmup+timed"
        reasons = set()
        for r in inwin:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return dict(sm_mhz=statistics.median(r["sm"] for r in inwin),
                    sm_max_mhz=max(r["smax"] for r in inwin), reasons=sorted(reasons),
                    samples=len(inwin), window=window)


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(d, wl, rows_per_thread=8):
    """Time the oracle as it stands on a bounded sample of rows of the workload."""
    import numpy as np
    import oracle
    lib = oracle.load()
    threads = oracle.num_threads(lib)
    n = max(1, rows_per_thread * threads)
    g = np.random.default_rng(1234)
    rows = np.sort(g.choice(d["h"].shape[0], size=min(n, d["h"].shape[0]), replace=False))
    h = d["h"].cpu()
    W = d["W"].cpu()
    tg = d["targets"].cpu()
    t0 = time.perf_counter()
    oracle.logprob(h, W, tg, wl["inv_temp"], rows=rows, lib=lib)
    dt = time.perf_counter() - t0
    return dict(value=len(rows) / dt, unit="tokens/s", cores=threads, kind="oracle",
                sample=f"{len(rows)} seeded rows of the T={wl['T']} batch (full V={V_CFG}, "
                       f"H={wl['H']}), fp64 oracle, OpenMP over rows, {dt:.1f} s")


def run_reference(args):
    world, rank, local = dist_init()
    if rank != 0:
        return 0
    import torch
    import oracle
    from invariant_token_logprob_gb300.inputs import lm_head_inputs
    lib = oracle.load()
    threads = oracle.num_threads(lib)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = WORKLOADS[args.workload]
    d = lm_head_inputs(wl["T"], wl["H"], V_CFG, seed=1000, device=dev, hidden="rms",
                       outlier_frac=wl["outlier_frac"], mask_zero_frac=wl["mask_zero_frac"])
    h, W, tg = d["h"].cpu(), d["W"].cpu(), d["targets"].cpu()
    rows_per_step = threads  # one row per core per step: about a second a step
    import numpy as np
    g = np.random.default_rng(7)
    times = []
    for i in range(args.warmup + args.steps):
        rows = np.sort(g.choice(wl["T"], size=rows_per_step, replace=False))
        t0 = time.perf_counter()
        oracle.logprob(h, W, tg, wl["inv_temp"], rows=rows, lib=lib)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = rows_per_step * len(times) / total
    line = dict(impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * total / len(times),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic",
                config=dict(workload=wl["name"], T=wl["T"], H=wl["H"], V=V_CFG,
                            inv_temp=wl["inv_temp"],
                            step=f"oracle over {rows_per_step} seeded rows of the batch"),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=threads, kind="oracle",
                                  sample=f"{rows_per_step} rows per step, full V and H"),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def time_decode(rlk, torch, W, Ts, reps, rounds, stream):
    """Device time per call of the whole path at small T (weight streaming).
    The T values are interleaved over `rounds` rounds and the median per-call
    time of each T is kept, so no T is measured only in one clock state."""
    cases = {}
    for T in Ts:
        h = torch.randn(T, H_CFG, device=W.device).to(torch.bfloat16)
        tg = torch.randint(0, V_CFG, (T,), device=W.device, dtype=torch.int32)
        out = [torch.empty(T, device=W.device, dtype=dt)
               for dt in (torch.float32, torch.float32, torch.int32)]
        cases[T] = (h, tg, out)
        for _ in range(3):
            rlk.logprob(h, W, tg, 1.0, out=out)
    times = {T: [] for T in Ts}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(rounds):
        for T in Ts:
            h, tg, out = cases[T]
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                rlk.logprob(h, W, tg, 1.0, out=out)
            e1.record(stream)
            e1.synchronize()
            times[T].append(e0.elapsed_time(e1) / reps * 1e-3)
    return {T: statistics.median(v) for T, v in times.items()}


def graph_time(torch, call, k=20, replays=5):
    """Seconds per call of `call(stream)` replayed from a CUDA graph of k calls,
    as a decode loop captured in a graph runs it (no per-launch host work)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        call(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            for _ in range(k):
                call(side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / (replays * k) * 1e-3


def decode_points(rlk, torch, W, stream, pk, Ts=(1, 2, 4, 8, 16, 32, 64, 128, 256), reps=50,
                  rounds=3, graph_Ts=(1, 16)):
    """Eager calls back to back (T{T}) and, for graph_Ts, the same call replayed
    from a CUDA graph (T{T}_graph); explicit workspaces, so nothing allocates
    during capture."""
    wbytes = V_CFG * H_CFG * 2
    res = {}
    for T, s in time_decode(rlk, torch, W, Ts, reps, rounds, stream).items():
        res[f"T{T}"] = dict(tokens_per_s=T / s, us_per_call=s * 1e6, hbm_gbs=wbytes / s / 1e9,
                            hbm_frac=wbytes / s / 1e9 / pk["hbm_gbs"])
    for T in graph_Ts:
        h = torch.randn(T, H_CFG, device=W.device).to(torch.bfloat16)
        tg = torch.randint(0, V_CFG, (T,), device=W.device, dtype=torch.int32)
        out = [torch.empty(T, device=W.device, dtype=dt)
               for dt in (torch.float32, torch.float32, torch.int32)]
        ws = torch.empty(rlk.workspace_size(T, H_CFG, V_CFG), dtype=torch.uint8, device=W.device)
        s = graph_time(torch, lambda st: rlk.logprob_ws(h, W, tg, ws, 1.0, out=out, stream=st))
        res[f"T{T}_graph"] = dict(tokens_per_s=T / s, us_per_call=s * 1e6,
                                  hbm_gbs=wbytes / s / 1e9, hbm_frac=wbytes / s / 1e9 / pk["hbm_gbs"])
    return res


def backward_point(rlk, torch, h, W, tg, pk, reps=10):
    """Backward of the same workload (T=4096): rlk_logprob_backward producing both
    fp32 gradients (recompute GEMM + dz epilogue, then the two library GEMMs),
    and the fused recompute/dz kernel alone (both outputs NULL)."""
    T, H = h.shape
    V = W.shape[0]
    lp, lse, am = rlk.logprob(h, W, tg, 1.0)
    grad = torch.ones(T, device=h.device)
    ws = torch.empty(rlk.backward_workspace_size(T, H, V), dtype=torch.uint8, device=h.device)
    gW = torch.empty((V, H), dtype=torch.float32, device=h.device)
    stream = torch.cuda.current_stream()

    def timed(need_h, need_W):
        for _ in range(2):
            rlk.logprob_backward(h, W, tg, lse, grad, 1.0, need_h=need_h, need_W=need_W,
                                 workspace=ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            rlk.logprob_backward(h, W, tg, lse, grad, 1.0, need_h=need_h, need_W=need_W,
                                 workspace=ws)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps * 1e-3

    t_all = timed(True, True)
    t_dz = timed(False, False)
    rlk.check_device_error()
    gemm = 2.0 * T * H * V
    del gW
    return dict(tokens_per_s=T / t_all, ms_per_call=t_all * 1e3,
                tflops=3 * gemm / t_all / 1e12, frac=3 * gemm / t_all / 1e12 / pk["bf16_tflops"],
                grad_logits_kernel_ms=t_dz * 1e3,
                grad_logits_kernel_frac=gemm / t_dz / 1e12 / pk["bf16_tflops"],
                gemms_ms=(t_all - t_dz) * 1e3,
                note="flops = 3 x 2*T*H*V (recompute, dz.W, dz^T.h); peak = bf16 burst")


def entropy_point(rlk, torch, h, W, tg, pk, reps=10):
    """rlk_logprob_entropy on the same batch (T=4096): the forward kernel with the
    entropy epilogue plus the entropy merge, against the bf16 peak; its logp / lse
    / argmax must be the forward's bits."""
    T, H = h.shape
    V = W.shape[0]
    ws = torch.empty(rlk.entropy_workspace_size(T, H, V), dtype=torch.uint8, device=h.device)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        res = rlk.logprob_entropy(h, W, tg, 1.0, workspace=ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        res = rlk.logprob_entropy(h, W, tg, 1.0, workspace=ws)
    e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / reps * 1e-3
    fwd = rlk.logprob(h, W, tg, 1.0)
    same = all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(res[:3], fwd))
    rlk.check_device_error()
    fl = 2.0 * T * H * V
    return dict(tokens_per_s=T / t, ms_per_call=t * 1e3, tflops=fl / t / 1e12,
                frac=fl / t / 1e12 / pk["bf16_tflops"], logp_bits_equal_forward=bool(same),
                mean_entropy=float(res[3].mean().item()))


def shard_points(rlk, torch, h, W, tg, pk, Rs=(2, 3, 6), reps=10):
    """Vocabulary-sharded (tensor-parallel) phases emulated on one GPU at T=4096:
    R shards of whole 256-column tiles (594 = R x tiles per shard for R = 2, 3, 6),
    each shard's partials on its own W slice, then the shard-count-invariant merge
    over the stacked records (what an all-gather would deliver).  Per R: one
    shard's partials (the per-rank work of an R-way split) against the bf16 peak,
    the merge, and whether the merged bits equal the unsharded call."""
    T, H = h.shape
    V = W.shape[0]
    bn = rlk.vocab_tile()
    nvt = (V + bn - 1) // bn
    stream = torch.cuda.current_stream()
    full = rlk.logprob(h, W, tg, 1.0)

    def timed(fn, n):
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e-3

    res = {}
    for R in Rs:
        if nvt % R:
            continue
        nvt_s = nvt // R
        bounds = [(r * nvt_s * bn, min((r + 1) * nvt_s * bn, V)) for r in range(R)]
        slices = [W[lo:hi].contiguous() for lo, hi in bounds]
        buf = torch.empty((R, T, nvt_s, 4), dtype=torch.float32, device=h.device)

        def shard(r):
            rlk.logprob_partials_shard(h, slices[r], tg, V, bounds[r][0], 1.0, out=buf[r])

        t_shard = timed(lambda: shard(0), reps)
        for r in range(R):
            shard(r)
        t_merge = timed(lambda: rlk.lse_merge_sharded(buf, tg, V), reps)
        got = rlk.lse_merge_sharded(buf, tg, V)
        same = all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(got, full))
        rows = bounds[0][1] - bounds[0][0]
        fl = 2.0 * T * H * rows
        res[f"R{R}"] = dict(shard_partials_ms=t_shard * 1e3, shard_tflops=fl / t_shard / 1e12,
                            shard_frac=fl / t_shard / 1e12 / pk["bf16_tflops"],
                            merge_ms=t_merge * 1e3, bitwise_equal_unsharded=bool(same))
        del slices, buf
    rlk.check_device_error()
    return res


def fp8_points(rlk, torch, h, W, tg, pk, reps=20):
    """The FP8 (W8A8) variant on the same batch: whole rlk_logprob_fp8 call
    (per-token quantisation of h, e4m3 LM-head kernel, merge) at T=4096 against
    the fp8 tensor peak (measured bf16 burst x the nominal fp8/bf16 ratio 2), and
    decode calls streaming the e4m3 weight (V*H bytes) against measured HBM.
    Returns the results and a function that adds the T=4096 point."""
    T, H = h.shape
    V = W.shape[0]
    wq, wsc = rlk.quantize_fp8_weight(W)
    stream = torch.cuda.current_stream()
    res = {}
    # the weight quantisation a training step repeats whenever W changes; the
    # untimed calls let the clock settle after the GEMM loops timed before it
    for _ in range(10):
        rlk.quantize_fp8_weight(W, out=(wq, wsc))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(20):
        rlk.quantize_fp8_weight(W, out=(wq, wsc))
    e1.record(stream)
    e1.synchronize()
    tq = e0.elapsed_time(e1) / 20 * 1e-3
    qbytes = V * H * 2 + wq.numel() + V * 4
    res["quantize_weight"] = dict(ms_per_call=tq * 1e3, hbm_gbs=qbytes / tq / 1e9,
                                  hbm_frac=qbytes / tq / 1e9 / pk["hbm_gbs"])

    def timed(hh, tt, n, warm=3):
        buf = torch.empty(rlk.fp8_workspace_size(hh.shape[0], H, V), dtype=torch.uint8,
                          device=h.device)
        out = [torch.empty(hh.shape[0], device=h.device, dtype=dt)
               for dt in (torch.float32, torch.float32, torch.int32)]
        for _ in range(warm):
            rlk.logprob_fp8(hh, wq, wsc, tt, 1.0, workspace=buf, out=out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            rlk.logprob_fp8(hh, wq, wsc, tt, 1.0, workspace=buf, out=out)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e-3

    for Td in (1, 16):
        hh, tt = h[:Td].contiguous(), tg[:Td].contiguous()
        td = timed(hh, tt, 200, warm=100)  # the untimed calls let the clock settle
        res[f"decode_T{Td}"] = dict(tokens_per_s=Td / td, us_per_call=td * 1e6,
                                     hbm_gbs=V * H / td / 1e9, hbm_frac=V * H / td / 1e9 / pk["hbm_gbs"])
        buf = torch.empty(rlk.fp8_workspace_size(Td, H, V), dtype=torch.uint8, device=h.device)
        out = [torch.empty(Td, device=h.device, dtype=dt)
               for dt in (torch.float32, torch.float32, torch.int32)]
        tg_ = graph_time(torch, lambda st: rlk.logprob_fp8(hh, wq, wsc, tt, 1.0, workspace=buf,
                                                           out=out, stream=st))
        res[f"decode_T{Td}_graph"] = dict(tokens_per_s=Td / tg_, us_per_call=tg_ * 1e6,
                                           hbm_gbs=V * H / tg_ / 1e9,
                                           hbm_frac=V * H / tg_ / 1e9 / pk["hbm_gbs"])
    rlk.check_device_error()

    def forward():  # the tensor-bound point, timed after every lighter one
        t = timed(h, tg, reps)
        peak8 = 2.0 * pk["bf16_tflops"]
        fl = 2.0 * T * H * V
        res["forward_T4096"] = dict(tokens_per_s=T / t, ms_per_call=t * 1e3, tflops=fl / t / 1e12,
                                    peak_tflops=peak8, frac=fl / t / 1e12 / peak8,
                                    peak_note="fp8 peak = measured bf16 burst x 2 (nominal ratio)")
        rlk.check_device_error()
    return res, forward


def fp8_block_points(rlk, torch, h, W, tg, pk, reps=20):
    """The block-scaled FP8 variant (1 x 128 activation blocks, 128 x 128 weight
    blocks) on the same batch: weight block quantisation, the whole
    rlk_logprob_fp8_block call at T=4096 against the fp8 tensor peak (measured
    bf16 burst x 2), and decode calls streaming the e4m3 weight against HBM.
    Returns the results and a function that adds the T=4096 point."""
    T, H = h.shape
    V = W.shape[0]
    wq, wsc = rlk.quantize_fp8_weight_blocks(W)
    stream = torch.cuda.current_stream()
    res = {}
    for _ in range(10):
        rlk.quantize_fp8_weight_blocks(W, out=(wq, wsc))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(20):
        rlk.quantize_fp8_weight_blocks(W, out=(wq, wsc))
    e1.record(stream)
    e1.synchronize()
    tq = e0.elapsed_time(e1) / 20 * 1e-3
    qbytes = V * H * 2 + wq.numel() + wsc.numel() * 4
    res["quantize_weight"] = dict(ms_per_call=tq * 1e3, hbm_gbs=qbytes / tq / 1e9,
                                  hbm_frac=qbytes / tq / 1e9 / pk["hbm_gbs"])

    def timed(hh, tt, n, warm=3):
        buf = torch.empty(rlk.fp8_block_workspace_size(hh.shape[0], H, V), dtype=torch.uint8,
                          device=h.device)
        out = [torch.empty(hh.shape[0], device=h.device, dtype=dt)
               for dt in (torch.float32, torch.float32, torch.int32)]
        for _ in range(warm):
            rlk.logprob_fp8_block(hh, wq, wsc, tt, V, 1.0, workspace=buf, out=out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            rlk.logprob_fp8_block(hh, wq, wsc, tt, V, 1.0, workspace=buf, out=out)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e-3

    for Td in (1, 16):
        td = timed(h[:Td].contiguous(), tg[:Td].contiguous(), 200, warm=100)
        wb = V * H + wsc.numel() * 4
        res[f"decode_T{Td}"] = dict(tokens_per_s=Td / td, us_per_call=td * 1e6,
                                     hbm_gbs=wb / td / 1e9, hbm_frac=wb / td / 1e9 / pk["hbm_gbs"])
    rlk.check_device_error()

    def forward():  # the tensor-bound point, timed after every lighter one
        t = timed(h, tg, reps)
        peak8 = 2.0 * pk["bf16_tflops"]
        fl = 2.0 * T * H * V
        res["forward_T4096"] = dict(tokens_per_s=T / t, ms_per_call=t * 1e3, tflops=fl / t / 1e12,
                                    peak_tflops=peak8, frac=fl / t / 1e12 / peak8,
                                    peak_note="fp8 peak = measured bf16 burst x 2 (nominal ratio)")
        rlk.check_device_error()
    return res, forward


def run_decode_only(args):
    """Decode regime alone (T = --decode-T rows per call, H=4096, V=151936): used
    for profiling the weight-streaming regime; prints one JSON line."""
    import torch
    import invariant_token_logprob_gb300 as rlk
    torch.cuda.set_device(0)
    pk = peaks()
    g = torch.Generator(device="cuda").manual_seed(1000)
    W = (torch.randn(V_CFG, H_CFG, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    if args.fp8:
        T = args.decode_T
        wq, wsc = rlk.quantize_fp8_weight(W)
        h = torch.randn(T, H_CFG, device="cuda").to(torch.bfloat16)
        tg = torch.randint(0, V_CFG, (T,), device="cuda", dtype=torch.int32)
        buf = torch.empty(rlk.fp8_workspace_size(T, H_CFG, V_CFG), dtype=torch.uint8, device="cuda")
        out = [torch.empty(T, device="cuda", dtype=dt) for dt in (torch.float32, torch.float32, torch.int32)]
        for _ in range(3):
            rlk.logprob_fp8(h, wq, wsc, tg, 1.0, workspace=buf, out=out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            rlk.logprob_fp8(h, wq, wsc, tg, 1.0, workspace=buf, out=out)
        e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / args.steps * 1e-3
        res = {f"T{T}_fp8": dict(us_per_call=t * 1e6, hbm_gbs=V_CFG * H_CFG / t / 1e9,
                                  hbm_frac=V_CFG * H_CFG / t / 1e9 / pk["hbm_gbs"])}
    else:
        res = decode_points(rlk, torch, W, stream, pk, Ts=(args.decode_T,), reps=args.steps,
                            rounds=1, graph_Ts=())
    rlk.check_device_error()
    print(json.dumps(dict(mode="decode-only", H=H_CFG, V=V_CFG, **res)), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    world, rank, local = dist_init()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (ours) needs a CUDA device: the library has no CPU path")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import invariant_token_logprob_gb300 as rlk
    from invariant_token_logprob_gb300.inputs import lm_head_inputs
    rlk.lib()
    pk = peaks()

    # ---------------------------------------------------------------- inputs
    wl = WORKLOADS[args.workload]
    default_wl = args.workload == "train4096"
    d = lm_head_inputs(wl["T"], wl["H"], V_CFG, seed=1000 + rank, device=dev, hidden="rms",
                       outlier_frac=wl["outlier_frac"], mask_zero_frac=wl["mask_zero_frac"])
    h, W, tg, mask = d["h"], d["W"], d["targets"], d["mask"]
    T, H, V = wl["T"], wl["H"], V_CFG
    it = wl["inv_temp"]
    nvt = (V + rlk.vocab_tile() - 1) // rlk.vocab_tile()
    partials = torch.empty((T, nvt, 4), dtype=torch.float32, device=dev)
    out = [torch.empty(T, device=dev, dtype=dt) for dt in (torch.float32, torch.float32, torch.int32)]
    stream = torch.cuda.current_stream(dev)
    # the "rollout" logprobs the acceptance statistics compare against
    rollout = rlk.logprob(h, W, tg, it)[0].clone()

    # each step's 8 statistics land in its own row, stream-ordered (no host sync
    # inside the loop); they are read and checked once the timed region is over
    stats_rows = torch.empty((max(args.steps, 3, args.warmup), 8), dtype=torch.float64, device=dev)
    stats_ws = torch.empty(max(16, rlk.stats_workspace_size(T)), dtype=torch.uint8, device=dev)

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        rlk.logprob_partials(h, W, tg, it, out=partials)
        if ev is not None:
            ev[1].record(stream)
        rlk.lse_merge(partials, tg, V, out=out)
        rlk.consistency_stats_async(out[0], rollout, mask, out=stats_rows[i], workspace=stats_ws)

    for i in range(max(3, args.warmup)):
        step(i)
    st = rlk.stats_dict(stats_rows[max(3, args.warmup) - 1])
    assert st["n_bit_mismatch"] == 0, "step outputs drifted from the first call"
    rlk.check_device_error()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("start")
    t_start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark("stop")
    barrier(world)
    clocks.stop()
    rlk.check_device_error()
    mism = int(stats_rows[:args.steps, 6].sum().item())
    elapsed = t_start.elapsed_time(t_end) * 1e-3
    elapsed = max_over_ranks(elapsed, world, dev)
    gemm_s = [a.elapsed_time(b) * 1e-3 for a, b in evs]
    gemm_avg = sum(gemm_s) / len(gemm_s)
    tokens = T * args.steps * world
    value = tokens / elapsed

    # ---------------------------------------------------------------- e2e
    # Through the public calls (rlk_logprob + rlk_consistency_stats_async), run
    # the way a training or serving loop runs them: step i+1's inputs are copied
    # from pinned host memory on a copy stream while step i computes, and step
    # i's results (logp, lse, argmax and the 8 statistics) are copied back on
    # the copy stream and read on the host during step i+1.  Every step moves its
    # own bytes both ways inside the timed region; the last step's results are
    # waited for before the clock stops.
    f32, i32 = torch.float32, torch.int32
    h_host = h.cpu().pin_memory()
    tg_host = tg.cpu().pin_memory()
    NB = 2  # double-buffered device inputs / outputs
    h_dev = [torch.empty_like(h) for _ in range(NB)]
    tg_dev = [torch.empty_like(tg) for _ in range(NB)]
    outs_dev = [[torch.empty(T, device=dev, dtype=dt) for dt in (f32, f32, i32)] for _ in range(NB)]
    st_dev = [torch.empty(8, dtype=torch.float64, device=dev) for _ in range(NB)]
    outs_host = [[torch.empty(T, dtype=dt).pin_memory() for dt in (f32, f32, i32)]
                 for _ in range(NB)]
    st_host = [torch.empty(8, dtype=torch.float64).pin_memory() for _ in range(NB)]
    copy_stream = torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(NB)]
    computed = [torch.cuda.Event() for _ in range(NB)]
    d2h_done = [torch.cuda.Event() for _ in range(NB)]
    e2e_mism = [0]

    def h2d(b):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(computed[b])  # the step that last used buffer b
            h_dev[b].copy_(h_host, non_blocking=True)
            tg_dev[b].copy_(tg_host, non_blocking=True)
            h2d_done[b].record(copy_stream)

    def compute_and_d2h(b):
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])  # its previous results have left the device
        lp, lse, am = rlk.logprob(h_dev[b], W, tg_dev[b], it, out=outs_dev[b])
        rlk.consistency_stats_async(lp, rollout, mask, out=st_dev[b], workspace=stats_ws)
        computed[b].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(computed[b])
            for o, oh in zip(outs_dev[b], outs_host[b]):
                oh.copy_(o, non_blocking=True)
            st_host[b].copy_(st_dev[b], non_blocking=True)
            d2h_done[b].record(copy_stream)

    def read_host(b):
        d2h_done[b].synchronize()
        e2e_mism[0] += int(st_host[b][6].item())

    def e2e_run(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d((i + 1) % NB)
            compute_and_d2h(i % NB)
            if i >= 1:
                read_host((i - 1) % NB)
        read_host((n - 1) % NB)

    e2e_steps = max(3, min(args.steps, 100))
    e2e_run(3)
    barrier(world)
    torch.cuda.synchronize()
    e2e_mism[0] = 0
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_el = max_over_ranks(time.perf_counter() - t0, world, dev)
    last = (e2e_steps - 1) % NB
    assert np.array_equal(outs_host[last][0].numpy().view(np.uint32),
                          out[0].cpu().numpy().view(np.uint32))
    assert e2e_mism[0] == 0, "e2e outputs drifted from the device-timed steps"
    e2e = dict(value=T * e2e_steps * world / e2e_el, unit="tokens/s",
               h2d_bytes_per_step=int(h.numel() * 2 + tg.numel() * 4),
               d2h_bytes_per_step=int(T * 12 + 8 * 8),
               pipeline="inputs of step i+1 copied while step i computes; results of step i "
                        "read on the host during step i+1")

    # ---------------------------------------------------------------- regimes
    # the other regimes are measured on the default workload's batch only
    # Order: the weight-streaming and quantisation measurements (issue- or
    # latency-sensitive, so clock-sensitive) come before the long tensor-bound
    # loops of other regimes, whose heat would otherwise still hold the clock
    # down while they run; each regime's own heavy part comes last in it.
    decode = None
    if not args.no_decode and default_wl:
        decode = decode_points(rlk, torch, W, stream, pk)
    fp8 = fp8_block = None
    if not args.no_fp8 and default_wl:
        # both formats' weight quantisers and decode calls, then both forwards
        fp8, fp8_forward = fp8_points(rlk, torch, h, W, tg, pk)
        fp8_block, fp8_block_forward = fp8_block_points(rlk, torch, h, W, tg, pk)
        fp8_forward()
        fp8_block_forward()
    backward = None
    if not args.no_backward and default_wl:
        backward = backward_point(rlk, torch, h, W, tg, pk)
    entropy = None if (args.no_entropy or not default_wl) else entropy_point(rlk, torch, h, W, tg, pk)
    sharded = None if (args.no_shard or not default_wl) else shard_points(rlk, torch, h, W, tg, pk)

    if rank != 0:
        return 0

    flops = 2.0 * T * H * V
    achieved = flops / gemm_avg / 1e12
    tr = recorded_traffic(T, H, V)
    roofline = dict(bound="tensor", achieved=achieved, peak=pk["bf16_tflops"], unit="TFLOP/s",
                    frac=achieved / pk["bf16_tflops"],
                    frac_of_sustained=achieved / pk["bf16_tflops_sustained"],
                    peak_source=f"bf16_tflops burst, {pk['source']} (MEASURED_PEAKS.json)"
                    if pk["source"] == "measured" else "fallback 1.9 PFLOP/s",
                    traffic=(tr["bytes_per_launch"] if tr else None),
                    algorithmic_flops_per_launch=flops,
                    kernel="lmhead_kernel<0, false, true, false> (bf16 forward partials, CTA pair)", launch_avg_us=gemm_avg * 1e6,
                    step_share=gemm_avg * args.steps / (elapsed if world == 1 else elapsed))
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample(d, wl)
    clk = clocks.summary()
    line = dict(metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * elapsed / args.steps,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
                data="synthetic",
                config=dict(workload=wl["name"], T=T, H=H, V=V, inv_temp=it,
                            masked_frac=wl["mask_zero_frac"], outlier_frac=wl["outlier_frac"],
                            l2="inputs larger than L2 (W 1.245 GB vs 129 MB L2): no flush",
                            step="partials (fused GEMM+epilogue) -> merge -> consistency stats",
                            parallelism=f"dp{world} (rows; no collective)"),
                roofline=roofline, cpu_baseline=cpu, e2e=e2e,
                gpu_launches=4 * args.steps,
                clocks=dict(sm_mhz=clk["sm_mhz"], sm_max_mhz=clk["sm_max_mhz"],
                            reasons=clk["reasons"], samples=clk["samples"],
                            window=clk.get("window")),
                decode=decode, backward=backward, fp8=fp8, fp8_block=fp8_block,
                entropy=entropy, sharded=sharded,
                bitwise_mismatch_vs_first_call=mism)
    print(json.dumps(line), flush=True)
    return 0


def run_backward_only(args):
    """rlk_logprob_backward alone on T=4096, H=4096, V=--bwd-V: per call the dz
    kernel alone, dz + grad_W, dz + grad_h and dz + both, interleaved over
    rounds (CUDA events, median per case); prints one JSON line.  Used for
    profiling the backward's kernels."""
    import torch
    import invariant_token_logprob_gb300 as rlk
    from invariant_token_logprob_gb300.inputs import lm_head_inputs
    torch.cuda.set_device(0)
    pk = peaks()
    T, H, V = T_CFG, H_CFG, args.bwd_V
    d = lm_head_inputs(T, H, V, seed=1000, device="cuda", hidden="rms")
    h, W, tg = d["h"], d["W"], d["targets"]
    lp, lse, am = rlk.logprob(h, W, tg, 1.0)
    grad = torch.ones(T, device="cuda")
    ws = torch.empty(rlk.backward_workspace_size(T, H, V), dtype=torch.uint8, device="cuda")
    gh = torch.empty((T, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    L = rlk.lib()
    import ctypes

    def call(need_h, need_W):
        st = L.rlk_logprob_backward(
            ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()),
            ctypes.c_void_p(tg.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
            ctypes.c_void_p(grad.data_ptr()), T, H, V, ctypes.c_float(1.0),
            ctypes.c_void_p(gh.data_ptr()) if need_h else None,
            ctypes.c_void_p(gW.data_ptr()) if need_W else None, 0,
            ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, st

    cases = {"dz": (False, False), "dz+grad_W": (False, True), "dz+grad_h": (True, False),
             "all": (True, True)}
    for c in cases.values():
        for _ in range(args.warmup):
            call(*c)
    times = {k: [] for k in cases}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        for k, c in cases.items():
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                call(*c)
            e1.record(stream)
            e1.synchronize()
            times[k].append(e0.elapsed_time(e1) / args.steps)
    rlk.check_device_error()
    med = {k: statistics.median(v) for k, v in times.items()}
    fl = 2.0 * T * H * V
    res = dict(mode="backward-only", T=T, H=H, V=V, ms=med,
               grad_W_ms=med["dz+grad_W"] - med["dz"], grad_h_ms=med["dz+grad_h"] - med["dz"])
    res["grad_W_frac"] = fl / (res["grad_W_ms"] * 1e-3) / 1e12 / pk["bf16_tflops"]
    res["grad_h_frac"] = fl / (res["grad_h_ms"] * 1e-3) / 1e12 / pk["bf16_tflops"]
    print(json.dumps(res), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.decode_only:
        return run_decode_only(args)
    if args.backward_only:
        return run_backward_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
