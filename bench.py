"""Benchmark: causal linear-attention forward (phi = elu + 1) tokens/s on GB300.

One step = one la_causal_fwd call (every kernel of the causal path) over one
batch of the long-context causal workload B=2 H=8 N=65536 D=64 bf16 (k scaled
by 1/8), the largest causal configuration, inputs resident in device memory.
Input sets rotate so that the bytes touched between two reads of one set
exceed the L2 cache. `--workload image` times the B=8 H=8 N=3072 shape (a
32x32x3 pixel-channel sequence) instead; it is also reported under `also`.

Prints ONE JSON line (rank 0). `--impl reference` times the float64 CPU
oracle on the same workload instead (a deliberately slow baseline).
Multi-GPU (torchrun): every rank runs its own batch (heads are independent,
no collective on the data path), timing is the max over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, make_workload, to_f64  # noqa: E402

METRIC = "causal linear-attn fwd tokens/s (B·H·N/s) & % of HBM/tensor roofline, 1 GB300"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long", choices=["image", "long"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--also-only", default=None,
                   help="comma-separated names of the secondary measurements to run")
    p.add_argument("--no-also", action="store_true",
                   help="skip the secondary non-causal and decode measurements")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(rank, r):
    """Seed of input set r on rank `rank`: every rank draws its own batch (weak scaling)."""
    return rank * 1000 + r


def job_ms(ms, dist, device):
    """Whole-job time of a timed region: the maximum over ranks (no-op on one rank)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Aggregate throughput: the units all ranks processed over the whole-job time."""
    return units_per_rank * world / (ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor TFLOP/s: the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:  # noqa: BLE001
        return 1900.0


def alg_bytes(w):
    """Algorithmic bytes of one forward: read q, k, v and write o once."""
    elem = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * w.N * (3 * w.D + w.D) * elem


# Sources that make up the causal tensor-core kernel: a recorded DRAM traffic
# figure is trusted only while these are unchanged.
# The files that compile into the causal kernel's device code (host launcher
# declarations elsewhere do not change it).
CAUSAL_SOURCES = ("causal_tc.cu", "tc_common.cuh", "tc_util.cuh", "common.cuh")


def csrc_digest(files=CAUSAL_SOURCES):
    h = hashlib.sha256()
    for name in sorted(files):
        with open(os.path.join(ROOT, "linear_attention_elu_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch from an ncu capture, if taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(key)
        if rec and rec.get("csrc_digest") == csrc_digest():
            return rec["bytes_per_launch"]
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return None
        self.out.flush()
        with open(self.out.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def host_numa(device_index, host_ptr):
    """NUMA placement of the e2e path: the GPU's node (from its PCI device) and the
    nodes holding the pages of a pinned host buffer (from /proc/self/numa_maps)."""
    out = {"cpus": len(os.sched_getaffinity(0))}
    try:
        props = torch.cuda.get_device_properties(device_index)
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            out["gpu_numa_node"] = int(f.read().strip())
        out["gpu_pci"] = bus
    except Exception:  # noqa: BLE001
        out["gpu_numa_node"] = None
    try:
        with open("/proc/self/numa_maps") as f:
            for line in f:
                addr = int(line.split()[0], 16)
                # numa_maps lists each mapping by its start address; the buffer's
                # mapping is the last one that starts at or below it.
                if addr <= host_ptr:
                    best = line
                else:
                    break
        nodes = {}
        for tok in best.split()[1:]:
            if tok.startswith("N") and "=" in tok:
                n, c = tok[1:].split("=")
                nodes[int(n)] = int(c)
        out["pinned_buffer_pages_by_node"] = nodes
    except Exception:  # noqa: BLE001
        out["pinned_buffer_pages_by_node"] = None
    return out


def cpu_baseline(w, budget_s=10.0):
    """Times the float64 oracle (recurrent form) on whole heads of the workload."""
    import oracle
    q, k, v = make_workload(w, seed=0)
    BH = w.B * w.H
    qf, kf, vf = (to_f64(t).reshape(BH, w.N, w.D) for t in (q, k, v))
    threads = oracle.default_threads()
    heads, elapsed, n = 0, 0.0, 1
    while elapsed < budget_s and heads < BH:
        n = min(n, BH - heads)
        t0 = time.perf_counter()
        oracle.recurrent(qf[heads:heads + n], kf[heads:heads + n], vf[heads:heads + n], True,
                         nthreads=threads)
        elapsed += time.perf_counter() - t0
        heads += n
        n *= 2
    return {"value": heads * w.N / elapsed, "unit": UNIT, "cores": min(threads, BH),
            "kind": "oracle",
            "sample": f"{heads} of {BH} heads x {w.N} tokens, float64 recurrent form, "
                      f"{elapsed:.2f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    q, k, v = make_workload(w, seed=0)
    BH = w.B * w.H
    qf, kf, vf = (to_f64(t).reshape(BH, w.N, w.D) for t in (q, k, v))
    threads = oracle.default_threads()
    sample_heads = max(1, min(BH, threads))  # one head per core per step

    def step(i):
        h0 = (i * sample_heads) % BH
        idx = [(h0 + j) % BH for j in range(sample_heads)]
        oracle.recurrent(qf[idx], kf[idx], vf[idx], True, nthreads=threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * sample_heads * w.N / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, sample_heads),
                         "kind": "oracle",
                         "sample": f"each step: {sample_heads} of {BH} heads x {w.N} tokens, "
                                   "float64 recurrent form"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# Multiply-adds the fp32 backward executes per token at Dk = Dv = 64 with
# 64-token chunks (32.5 in-chunk keys on average, 32.5 x 64 = 2,080 for a masked
# in-chunk product). Causal: the chunk states phi(k) [v | 1] (4,160); the rows
# pass (12,513: A 2,080, den 64 + 32.5, num 2,080 + 4,096, the chunk's reverse
# sum 4,160); the gradient pass (24,832: W 2,080, G 2,080, dq 4,096 + 2,080 + 64,
# dk 4,096 + 2,080, dv 4,096 + 2,080). Non-causal, no in-chunk terms: states
# 4,160; rows 8,320 (den 64, num 4,096, reverse sum 4,160); gradients 12,352
# (dq 4,096 + 64, dk 4,096, dv 4,096).
BWD_MACS_PER_TOKEN_D64 = 4160 + 12513 + 24832
# Multiply-adds the tensor-core backward issues per token (bf16, Dk = Dv = 64,
# 128-token chunks, MMA shapes as executed). Causal: chunk state [V | 1]^T phi(K)
# 64 x 128 = 8,192; rows pass: phi(Q) phi(K)^T 128 x 64 = 8,192, P [V | 1]
# 80 x 128 = 10,240, phi(Q) [S^T | z] 80 x 64 = 5,120, [dnum | dd]^T phi(Q)
# 64 x 128 = 8,192; gradient pass: G and W 2 x 8,192, and each of dphi(q),
# dphi(k), dv 64 x 64 + 64 x 128 = 12,288. Non-causal: state 8,192; rows 5,120 +
# 8,192; gradients 3 x 4,096.
TC_BWD_MACS_PER_TOKEN_D64 = 8192 + 8192 + 10240 + 5120 + 8192 + 2 * 8192 + 3 * 12288
TC_NC_BWD_MACS_PER_TOKEN_D64 = 8192 + 5120 + 8192 + 3 * 4096
# Bytes a backward pass must move per token at D = 64 bf16: q, k, v, dout read,
# dq, dk, dv written.
BWD_ALG_BYTES_PER_TOKEN_D64 = 7 * 64 * 2
# The fp32 causal forward per token at Dk = Dv = 64: chunk state 4,160; output
# A 2,080, den 64, A V 2,080, phi(q) S_prev 4,096.
FWD_F32_MACS_PER_TOKEN_D64 = 4160 + 2080 + 64 + 2080 + 4096
# The fp32 non-causal forward per token: partial state 4,160; den 64, phi(q) S 4,096.
NC_F32_MACS_PER_TOKEN_D64 = 4160 + 64 + 4096
NC_BWD_MACS_PER_TOKEN_D64 = 4160 + 8320 + 12352
# fp32 FMA peak from the unit counts and clock: 152 SMs x 128 lanes x 2 flop x 2.07 GHz.
FP32_FMA_PEAK = 152 * 128 * 2 * 2.07e9


def causal_also(la, w, dev, stream, calls=100):
    """The causal forward on another workload: rotating input sets larger than L2,
    one graph of `calls` consecutive calls, CUDA events around its replay."""
    hbm, _ = peaks()
    per_set = alg_bytes(w)
    R = max(2, -(-3 * L2_BYTES // per_set) + 1)
    sets = []
    for r in range(R):
        q, k, v = make_workload(w, seed=r)
        sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(v, device=dev)))
    ws = la.workspace(la.LA_OP_CAUSAL, w.B, w.H, w.N, w.D, w.D, sets[0][0].dtype, dev)
    for i in range(3):
        q, k, v, o = sets[i % R]
        la.la_causal_fwd(q, k, v, o=o, ws=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(calls):
            q, k, v, o = sets[i % R]
            la.la_causal_fwd(q, k, v, o=o, ws=ws)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / calls
    gbps = alg_bytes(w) / (ms * 1e-3) / 1e9
    return {"workload": w.name, "value": w.tokens / (ms * 1e-3), "unit": "tokens/s",
            "ms_per_call": ms,
            "roofline": {"bound": "hbm", "achieved": gbps, "peak": hbm, "unit": "GB/s",
                         "frac": gbps / hbm},
            "l2": f"{R} rotating input sets of {per_set / 1e6:.1f} MB",
            "status": la.la_query_status(ws)}


def other_paths(la, dev, stream, main_workload, only=None):
    """Secondary measurements: the other causal shape and the other operations of
    the path (`only`: the names of the entries to measure, all when None)."""
    hbm, _ = peaks()
    out = {}

    def want(name):
        return only is None or name in only

    gen = torch.Generator(device=dev)
    gen.manual_seed(123)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    us = None                               # decode step time, for the layer entry
    other = "image" if main_workload == "long" else "long"
    if want(other):
        out[other] = causal_also(la, WORKLOADS[other], dev, stream,
                                 calls=200 if other == "image" else 20)
    if want("noncausal"):
        # Non-causal, B=16 H=8 N=8192 D=128 bf16 (one 1.07 GB input set, larger than L2).
        w = WORKLOADS["bidir"]
        q, k, v = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen).bfloat16()
                   for _ in range(3))
        o = torch.empty_like(v)
        ws = la.workspace(la.LA_OP_NONCAUSAL, w.B, w.H, w.N, w.D, w.D, q.dtype, dev)
        for _ in range(3):
            la.la_noncausal_fwd(q, k, v, o=o, ws=ws)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            la.la_noncausal_fwd(q, k, v, o=o, ws=ws)
        g.replay()
        torch.cuda.synchronize()
        reps = 10
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        alg = w.tokens * 4 * w.D * 2
        out["noncausal"] = {"workload": w.name, "value": w.tokens / (ms * 1e-3), "unit": "tokens/s",
                            "ms_per_call": ms, "alg_GBps": alg / (ms * 1e-3) / 1e9,
                            "frac_of_hbm": alg / (ms * 1e-3) / 1e9 / hbm,
                            "status": la.la_query_status(ws)}
        del q, k, v, o, ws, g
    if want("causal_d128"):
        # Causal at D = 128 on the bidirectional workload's shape (B=16 H=8 N=8192 bf16):
        # run sums, seed scan and output pass; one 1.07 GB input set, larger than L2.
        w = WORKLOADS["bidir"]
        q, k, v = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen).bfloat16()
                   for _ in range(3))
        o = torch.empty_like(v)
        ws = la.workspace(la.LA_OP_CAUSAL, w.B, w.H, w.N, w.D, w.D, q.dtype, dev)
        for _ in range(3):
            la.la_causal_fwd(q, k, v, o=o, ws=ws)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            la.la_causal_fwd(q, k, v, o=o, ws=ws)
        g.replay()
        torch.cuda.synchronize()
        reps = 10
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        alg = w.tokens * 4 * w.D * 2
        out["causal_d128"] = {"workload": w.name.replace("non-causal", "causal"),
                              "value": w.tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms,
                              "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9,
                                           "peak": hbm, "unit": "GB/s",
                                           "frac": alg / (ms * 1e-3) / 1e9 / hbm},
                              "launches_per_call": la.la_launch_count(la.LA_OP_CAUSAL, w.B, w.H, w.N,
                                                                      w.D, w.D, la.LA_BF16),
                              "status": la.la_query_status(ws)}
        del q, k, v, o, ws, g
    if want("noncausal_d64"):
        # Non-causal at D = 64 on the image shape (B=8 H=8 N=3072 bf16): 100.7 MB per call,
        # six rotating input sets so that each use finds its inputs outside L2.
        w = WORKLOADS["image"]
        sets = []
        for r in range(6):
            q, k, v = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen).bfloat16()
                       for _ in range(3))
            sets.append((q, k, v, torch.empty_like(v)))
        ws = la.workspace(la.LA_OP_NONCAUSAL, w.B, w.H, w.N, w.D, w.D, torch.bfloat16, dev)
        for i in range(6):
            q, k, v, o = sets[i]
            la.la_noncausal_fwd(q, k, v, o=o, ws=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        reps = 60
        with torch.cuda.graph(g):
            for i in range(reps):
                q, k, v, o = sets[i % 6]
                la.la_noncausal_fwd(q, k, v, o=o, ws=ws)
        g.replay()
        torch.cuda.synchronize()
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        alg = w.tokens * 4 * w.D * 2
        out["noncausal_d64"] = {"workload": w.name.replace("causal", "non-causal"),
                                "value": w.tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms,
                                "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9,
                                             "peak": hbm, "unit": "GB/s",
                                             "frac": alg / (ms * 1e-3) / 1e9 / hbm},
                                "status": la.la_query_status(ws)}
        del sets, ws, g
    if want("decode") or want("decode_2048") or want("l2_peak"):
        # L2 reference for the decode step, whose fp32 state stays in L2 between steps:
        # an in-place scale of a 64 MB fp32 buffer (each byte read and written at the
        # same address, as the decode step does with S and z), 200 launches in one graph.
        x = torch.ones(16 * 2 ** 20, device=dev)
        g = torch.cuda.CUDAGraph()
        x.mul_(1.0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(200):
                x.mul_(1.0)
        best = None
        for _ in range(3):
            g.replay()
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            t = a.elapsed_time(b) / 200
            best = t if best is None else min(best, t)
        l2_gbps = 2 * x.numel() * 4 / (best * 1e-3) / 1e9
        out["l2_peak"] = {"GBps": l2_gbps, "how": "torch in-place x.mul_(1.0) over a 64 MB fp32 "
                          "buffer (read + write, L2-resident), 200 launches in one CUDA graph, best of 3"}
        del x, g

        def decode_run(B, T):
            """us per step of T consecutive decode steps in one graph (B sequences x 8 heads)."""
            w = WORKLOADS["decode"]
            q, k, v = (torch.randn(T, B, w.H, w.D, device=dev, generator=gen).bfloat16()
                       for _ in range(3))
            o = torch.empty_like(v)
            S = torch.zeros(B, w.H, w.D, w.D, device=dev)
            z = torch.zeros(B, w.H, w.D, device=dev)

            def steps():
                for t in range(T):
                    la.la_decode_step(q[t], k[t], v[t], S, z, o=o[t])

            steps()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                steps()
            g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / T * 1e3

        # Decode, 512 sequences x 8 heads, D=64: all 3072 steps of the configuration in one
        # graph. The 68 MB fp32 state stays in the 129 MB L2 between steps, so its
        # roofline is the L2 read+write rate above.
        w = WORKLOADS["decode"]
        us = decode_run(w.B, w.N)
        per_step = 33792 * w.B * w.H
        gbps = per_step / (us * 1e-6) / 1e9
        out["decode"] = {"workload": w.name + ", all steps timed", "value": 1e6 / us,
                         "unit": "steps/s", "us_per_step": us, "alg_GBps": gbps,
                         "roofline": {"bound": "l2", "achieved": gbps, "peak": l2_gbps,
                                      "unit": "GB/s", "frac": gbps / l2_gbps,
                                      "peak_source": "l2_peak (measured in this run)"},
                         "frac_of_hbm": gbps / hbm,
                         "note": "the 68 MB fp32 state stays resident in the 129 MB L2 across steps"}
        # The same step with 2048 sequences x 8 heads: 272 MB of fp32 state, larger than
        # L2, so every step streams it from and to HBM.
        Bbig, Tbig = 2048, 256
        us_big = decode_run(Bbig, Tbig)
        per_big = 33792 * Bbig * w.H
        gbps_big = per_big / (us_big * 1e-6) / 1e9
        out["decode_2048"] = {"workload": f"decode {Bbig} seq x H=8 D=64 bf16, fp32 state 272 MB, "
                                          f"{Tbig} steps timed",
                              "value": 1e6 / us_big, "unit": "steps/s", "us_per_step": us_big,
                              "alg_GBps": gbps_big,
                              "roofline": {"bound": "hbm", "achieved": gbps_big, "peak": hbm,
                                           "unit": "GB/s", "frac": gbps_big / hbm}}
    if want("layer_decode"):
        # Layer decode step at the same batch (512 sequences, d_model = 8 x 64, bf16,
        # synthetic weights): QKV projection, the decode step, output projection.
        w = WORKLOADS["decode"]
        T = 256
        dm = w.H * w.D
        Wqkv = (torch.randn(dm, 3 * dm, device=dev, generator=gen) * dm ** -0.5).bfloat16()
        Wo = (torch.randn(dm, dm, device=dev, generator=gen) * dm ** -0.5).bfloat16()
        xs = torch.randn(T, w.B, dm, device=dev, generator=gen).bfloat16()
        ys = torch.empty_like(xs)
        S = torch.zeros(w.B, w.H, w.D, w.D, device=dev)
        z = torch.zeros(w.B, w.H, w.D, device=dev)
        ws = la.workspace(la.LA_OP_LAYER_DECODE, w.B, w.H, 1, w.D, w.D, xs.dtype, dev)

        def layer_steps():
            for t in range(T):
                la.la_layer_decode_step(xs[t], Wqkv, Wo, S, z, w.H, y=ys[t], ws=ws)

        layer_steps()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer_steps()
        g.replay()
        torch.cuda.synchronize()
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        lus = a.elapsed_time(b) / T * 1e3
        gemm_flops = 2 * w.B * dm * 4 * dm
        out["layer_decode"] = {
            "workload": f"layer decode step, {w.B} sequences, d_model {dm} = {w.H} x {w.D}, bf16, "
                        f"synthetic weights, {T} steps timed",
            "value": 1e6 / lus, "unit": "steps/s", "us_per_step": lus,
            "attention_share_est": us / lus if us else None,
            "projection_tflops_if_rest": gemm_flops / max(lus - us, 1e-3) / 1e6 if us else None,
            "note": "projections: the library's tcgen05 bf16 products (128 x 64 tiles); "
                    "the decode step between them is the library's decode kernel"}
        del Wqkv, Wo, xs, ys, S, z, ws, g
    if want("causal_f32") or want("noncausal_f32"):
        # Causal and non-causal forward on fp32 inputs (the fp32 SIMT path) at the
        # image shape B=8 H=8 N=3072 D=64; 151 MB of inputs, larger than L2.
        w = WORKLOADS["image"]
        q, k, v = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen) for _ in range(3))
        o = torch.empty_like(v)
        for key, fn, op, macs, name in (
                ("causal_f32", la.la_causal_fwd, la.LA_OP_CAUSAL, FWD_F32_MACS_PER_TOKEN_D64,
                 w.name.replace("bf16", "f32")),
                ("noncausal_f32", la.la_noncausal_fwd, la.LA_OP_NONCAUSAL, NC_F32_MACS_PER_TOKEN_D64,
                 w.name.replace("bf16", "f32").replace("causal", "non-causal"))):
            ws = la.workspace(op, w.B, w.H, w.N, w.D, w.D, q.dtype, dev)
            fn(q, k, v, o=o, ws=ws)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(q, k, v, o=o, ws=ws)
            g.replay()
            torch.cuda.synchronize()
            reps = 10
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            flops = w.tokens * 2 * macs
            out[key] = {"workload": name, "value": w.tokens / (ms * 1e-3), "unit": "tokens/s",
                        "ms_per_call": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                        "frac_of_fp32_fma": flops / (ms * 1e-3) / FP32_FMA_PEAK,
                        "bound": "alu (fp32 FMA)"}
            del ws, g
        del q, k, v, o
    if want("causal_bwd") or want("noncausal_bwd"):
        # Causal and non-causal backward (tensor-core kernels for bf16 D = 64) at the
        # image shape B=8 H=8 N=3072 D=64 bf16.
        w = WORKLOADS["image"]
        q, k, v, dout = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen).bfloat16()
                         for _ in range(4))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for key, fn, op, macs, name in (
                ("causal_bwd", la.la_causal_bwd, la.LA_OP_CAUSAL_BWD, TC_BWD_MACS_PER_TOKEN_D64,
                 w.name.replace("causal", "causal backward")),
                ("noncausal_bwd", la.la_noncausal_bwd, la.LA_OP_NONCAUSAL_BWD,
                 TC_NC_BWD_MACS_PER_TOKEN_D64, w.name.replace("causal", "non-causal backward"))):
            ws = la.workspace(op, w.B, w.H, w.N, w.D, w.D, q.dtype, dev)
            fn(q, k, v, dout, dq, dk, dv, ws=ws)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(q, k, v, dout, dq, dk, dv, ws=ws)
            g.replay()
            torch.cuda.synchronize()
            reps = 5
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            flops = w.tokens * 2 * macs
            gbps = w.tokens * BWD_ALG_BYTES_PER_TOKEN_D64 / (ms * 1e-3) / 1e9
            out[key] = {"workload": name, "value": w.tokens / (ms * 1e-3), "unit": "tokens/s",
                        "ms_per_call": ms, "tflops_executed": flops / (ms * 1e-3) / 1e12,
                        "frac_of_bf16_dense": flops / (ms * 1e-3) / 1e12 / bf16_peak(),
                        "alg_GBps": gbps, "frac_of_hbm": gbps / hbm,
                        "bound": "latency: one CTA per 128-token chunk runs load, MMAs and "
                                 "epilogue in sequence (neither pipe nor DRAM saturated)"}
            del ws, g
    if want("random_features_causal"):
        # Positive random features (R = 64, x scaled by D^-1/4) of q and k, then the
        # identity-map causal forward on the tensor-core path, at the image shape.
        w = WORKLOADS["image"]
        q, k, v = (torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=gen).bfloat16()
                   for _ in range(3))
        R = 64
        W = torch.randn(R, w.D, device=dev, generator=gen).bfloat16()
        qs, ks = (q.float() * w.D ** -0.25).bfloat16(), (k.float() * w.D ** -0.25).bfloat16()
        fq = torch.empty(w.B, w.H, w.N, R, device=dev, dtype=torch.bfloat16)
        fk = torch.empty_like(fq)
        o = torch.empty_like(v)
        ws = la.workspace(la.LA_OP_CAUSAL, w.B, w.H, w.N, R, w.D, q.dtype, dev)

        def features():
            la.la_positive_random_features(qs, W, out=fq)
            la.la_positive_random_features(ks, W, out=fk)

        def chain():
            features()
            la.la_causal_fwd(fq, fk, v, o=o, ws=ws, phi=la.LA_PHI_IDENTITY)

        res = {}
        for name, fn in (("features_ms", features), ("chain_ms", chain)):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            torch.cuda.synchronize()
            reps = 10
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) / reps
            del g
        rows = 2 * w.tokens
        feat_bytes = rows * (w.D + R) * 2          # x read and features written once, bf16
        out["random_features_causal"] = {
            "workload": w.name.replace("causal", "random features (R=64) + identity-map causal"),
            "value": w.tokens / (res["chain_ms"] * 1e-3), "unit": "tokens/s", **res,
            "features_alg_GBps": feat_bytes / (res["features_ms"] * 1e-3) / 1e9,
            "features_frac_of_hbm": feat_bytes / (res["features_ms"] * 1e-3) / 1e9 / hbm,
            "bound": "features: hbm (tcgen05 projection, exp epilogue); attention: as the causal path"}
    return out


def main():
    args = parse()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import linear_attention_elu_gb300 as la

    # Inputs: R independent sets so the sets touched between two uses of one set exceed L2.
    per_set = alg_bytes(w)
    R = max(2, -(-3 * L2_BYTES // per_set) + 1)
    sets = []
    for r in range(R):
        q, k, v = make_workload(w, seed=replica_seed(rank, r))
        sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(v, device=dev)))
    ws = la.workspace(la.LA_OP_CAUSAL, w.B, w.H, w.N, w.D, w.D, sets[0][0].dtype, dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = la.la_launch_count(la.LA_OP_CAUSAL, w.B, w.H, w.N, w.D, w.D,
                                           sets[0][0].dtype)

    def step(i):
        q, k, v, o = sets[i % R]
        la.la_causal_fwd(q, k, v, o=o, ws=ws)

    # One CUDA graph per input set, each holding exactly one step (the launches
    # of one la_causal_fwd call), for per-call timing; and one graph holding the
    # K timed steps in order (input sets rotating), replayed once: consecutive
    # calls then overlap launch and set-up as they would on a stream.
    graphs = []
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for r in range(R):
            step(r)
    stream.wait_stream(side)
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(r)
        graphs.append(g)
    g_warm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm):
        for i in range(max(3, args.warmup)):
            step(i)
    g_timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_timed):
        for i in range(args.steps):
            step(i)

    g_warm.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ev0.record(stream)
        g_timed.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(ev0.elapsed_time(ev1), dist, dev)
    if dist:
        dist.barrier()
    status = la.la_query_status(ws)
    if status != 0:
        raise RuntimeError(f"device status after timed region: {la.la_status_string(status)}")
    ms_per_step = ms / args.steps
    tokens = w.tokens * world
    value = job_rate(w.tokens, world, ms_per_step)

    # Per-call device time: events around each replay (one call each).
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        evs[i][0].record(stream)
        graphs[i % R].replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)

    # The same steps submitted eagerly through the binding (host cost included).
    torch.cuda.synchronize()
    ea = torch.cuda.Event(enable_timing=True)
    eb = torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for i in range(args.steps):
        step(i)
    eb.record(stream)
    torch.cuda.synchronize()
    eager_ms = ea.elapsed_time(eb) / args.steps

    # End to end: pinned host inputs -> device, forward, result -> pinned host,
    # through the host-buffer entry (head groups stream through two device
    # buffers; copies in, compute and copies out overlap).
    hq, hk, hv = (t.cpu().pin_memory() for t in make_workload(w, seed=replica_seed(rank, 77)))
    ho = torch.empty_like(hv).pin_memory()
    staging = la.host_staging(w.B, w.H, w.N, w.D, w.D, hq.dtype, dev)

    def e2e_step():
        la.la_causal_fwd_host(hq, hk, hv, o=ho, staging=staging, ws=ws, device=dev)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = job_ms(e0.elapsed_time(e1) / args.e2e_steps, dist, dev)
    numa = host_numa(local, hq.data_ptr())
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    del sets, graphs, g_warm, g_timed

    only = set(args.also_only.split(",")) if args.also_only else None
    also = {} if args.no_also else other_paths(la, dev, stream, args.workload, only)

    hbm, src = peaks()
    # Average launch duration over the timed region (events around the K steps);
    # every launch of a step processes the whole batch, so bytes per launch are
    # the step's algorithmic bytes divided by the launches per step.
    launch_ms = ms_per_step / launches_per_step
    achieved = alg_bytes(w) / launches_per_step / (launch_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Dk": w.D, "Dv": w.D,
                   "eps": 1e-6, "state_dtype": "f32",
                   "l2": f"{R} rotating input sets of {per_set / 1e6:.1f} MB (> L2 between reuses)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                     if src == "measured" else "fallback 6.8 TB/s",
                     "traffic": recorded_traffic(f"causal:{args.workload}"),
                     "kernel": f"la_causal_fwd ({launches_per_step} launches per call)",
                     "alg_bytes_per_launch": alg_bytes(w) / launches_per_step,
                     "avg_launch_ms_timed": launch_ms,
                     "isolated_call_ms": call_ms},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "host_numa": numa},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "submission": {"timed": "one CUDA graph of the K steps, replayed once",
                       "eager_ms_per_step": eager_ms},
        "also": also,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
