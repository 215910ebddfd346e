"""Benchmark: GDN chunk forward throughput on B4 H16 T4096 K=V=128 bf16.

One step = one chunked forward (cumulative gate, UT transform, state
recurrence, output: gdn_chunk_fwd) over one batch of the synthetic BSND
workload ``gdn_bsnd_bf16`` (B=4, T=4096, H=16, K=V=128, chunk 64, scalar
gate, scale K^-1/2). Inputs are resident in HBM before the timed region and
rotate over 4 copies (4 x 65.5 MB, above the 129 MB L2) so that no step reads
its inputs from L2. N > 1 (torchrun) runs one independent replica per GPU:
heads are independent, there is no collective on the data path (weak scaling).

``--impl reference`` times the CPU oracle (fp64 token recurrence, all host
cores) on a bounded sample of the same workload and prints the same line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunk fwd tokens/s & TFLOP/s (B4 H16 T4096 K=V=128 bf16), % roofline"
WORKLOAD = dict(workload="gdn_bsnd_bf16", B=4, T=4096, H=16, K=128, V=128, chunk=64,
                layout="BSND", gate="scalar per head", dtype_in="bf16", state="fp32")
# algorithmic work per (token, head): flops of the chunk algorithm (KK^T, QK^T and w:
# 3*2C^2K; u and A_qk v_new: 2*2C^2V; w h, kg^T v_new, q h: 3*2CKV, per 64 tokens)
FLOP_PER_TOKEN_HEAD = 180224
# bytes per (token, head): q, k, v, o bf16 (4 x 256) + g fp32 (4) + beta bf16 (2)
BYTES_PER_TOKEN_HEAD = 1030
STATE_BYTES = 128 * 128 * 4  # final state per head, fp32
ROTATE = 4


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except Exception:
                ts = None
            rows.append((ts, parts))
        inside = [p for ts, p in rows if ts is not None and self.t0 is not None
                  and self.t0 - 1 <= ts <= self.t1 + 1]
        use = inside or [p for _, p in rows]
        sm = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for p in use if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if "Active" in p[6 + i]
                          and "Not" not in p[6 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


class NvmlClockSampler:
    """SM clock and clock-event reasons read from NVML (the driver's libnvidia-ml, through
    ctypes; reads only) every millisecond on a background thread, so that even a timed
    region of a few milliseconds holds several samples. Same report as ClockSampler."""

    # clock-event reason bits of the NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading
        import torch
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        pr = torch.cuda.get_device_properties(device)
        bus = f"{pr.pci_domain_id:x}:{pr.pci_bus_id:x}:{pr.pci_device_id:x}.0".encode()
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + bus.decode())
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # 1: SM clock
        self.max_mhz = float(mx.value)
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:  # the older name of the same query
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.t0 = self.t1 = None
        self.run = False
        self.thread = threading.Thread(target=self._loop, daemon=True)

    def _read(self):
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c))
        self.reasons_fn(self.h, self.ct.byref(r))
        return time.perf_counter(), float(c.value), int(r.value)

    def _loop(self):
        while self.run:
            self.samples.append(self._read())
            time.sleep(0.001)

    def start(self):
        self.run = True
        self.thread.start()

    def mark(self, which):
        setattr(self, which, time.perf_counter())

    def stop(self):
        self.run = False
        self.thread.join()
        inside = [s for s in self.samples if self.t0 is not None and self.t0 <= s[0] <= self.t1]
        use = inside or self.samples
        sm = [s[1] for s in use]
        reasons = sorted({name for s in use for bit, name in self.REASONS.items() if s[2] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "source": "NVML, 1 ms period"}


def clock_sampler(device):
    try:
        return NvmlClockSampler(device)
    except Exception:
        return ClockSampler(device.index)


FWD_SOURCES = ("ut_fwd.cu", "fwd_ws.cu", "tile_ops.cuh", "tc.cuh")


def fwd_source_sha256():
    """Digest of the forward kernels' code (the UT transform and the state kernel): the
    sources without // comments and blank lines, so that an edit of comments alone keeps
    the recorded counters valid while any change of code voids them."""
    import hashlib
    import re
    d = hashlib.sha256()
    for f in FWD_SOURCES:
        text = open(os.path.join(ROOT, "gated_delta_rule_28_gb300", "csrc", f)).read()
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        d.update("\n".join(ln for ln in lines if ln).encode())
    return d.hexdigest()


def _recorded_traffic():
    """DRAM bytes per forward call (both kernels) from the committed ncu summary, only while
    the kernel sources are the ones those counters were taken on (else None)."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["gdn_bsnd_bf16_fwd"]
        if fwd_source_sha256() == rec["kernel_source_sha256"]:
            return rec["bytes_per_launch"]
    except Exception:
        pass
    return None


def max_over_ranks(seconds, device=None):
    """The largest of the ranks' times, on every rank (the whole job ends with the slowest
    rank); the local time when no process group is initialised. ``device`` is where the
    reduction runs: the rank's GPU under NCCL, None (host) under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(seconds)
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, steps, seconds):
    """Whole-job throughput: every rank processes its own copy of the workload (weak scaling)."""
    return world * tokens_per_rank * steps / seconds


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(inp, n_pairs, first=0):
    """``n_pairs`` (batch, head) pairs of the BSND workload, from pair ``first`` on (modulo
    all pairs), as the heads of one batch row [1, T, n_pairs, D]: independent problems that
    the oracle runs one thread each."""
    B, _, H = inp.q.shape[:3]
    sel = [((first + j) % (B * H)) // H for j in range(n_pairs)], \
          [((first + j) % (B * H)) % H for j in range(n_pairs)]
    take = lambda x: np.ascontiguousarray(x[sel[0], :, sel[1]].swapaxes(0, 1)[None])  # noqa: E731
    return [take(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]


def time_oracle(inp, n_pairs, threads, first=0):
    """Seconds the oracle takes for ``n_pairs`` pairs of 4096 tokens on ``threads`` threads
    (the sample is cut out before the clock starts)."""
    from oracle import recurrence as R
    q, k, v, g, beta = oracle_sample(inp, n_pairs, first)
    t0 = time.perf_counter()
    R.forward(q, k, v, g, beta, n_threads=threads)
    return time.perf_counter() - t0


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from gated_delta_rule_28_gb300 import workloads
    from oracle import recurrence as R
    inp = workloads.make(2)
    cores = os.cpu_count() or 1
    R.build()
    # each step: one (batch, head) pair of 4096 tokens per host core (at most all 64),
    # one oracle thread per pair, so every core is busy
    per_step = min(cores, 64)
    for i in range(args.warmup):
        time_oracle(inp, per_step, cores, first=i * per_step)
    t = sum(time_oracle(inp, per_step, cores, first=(args.warmup + i) * per_step)
            for i in range(args.steps))
    token_heads = args.steps * per_step * 4096
    value = token_heads / 16 / t  # full-forward tokens/s equivalent (16 heads per token)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": WORKLOAD,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} of 64 (batch, head) pairs x 4096 tokens per step, "
                                   f"fp64 token recurrence, one thread per pair on {cores} host "
                                   "cores, tokens/s scaled to 16 heads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _time_ms(fn, reps, warmup, stream):
    """Mean device time of fn() over reps launches on `stream` (CUDA events)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


ROWS = ("packed_fwd", "kda_split_fwd", "train_fwd_bwd", "frame_scan", "aux_paths")


def secondary_rows(dev, hbm_peak, only=None, reps=None, kda_tokens=65536, train_tokens=8192,
                   frame_positions=4096):
    """The other scope rows, each on its own workload at full size (device-generated
    seeded inputs with the workloads' distributions; timing only, parity is in tests).
    ``only`` restricts the run to one row; ``reps`` overrides the timed repetitions
    (a profiler capture wants few); ``kda_tokens`` shrinks the per-key workload for a
    profiler capture (same distributions and segment length), ``train_tokens`` the training
    workload's tokens per batch row, ``frame_positions`` the transition scan's positions per
    sequence."""
    import torch
    from gated_delta_rule_28_gb300 import api, binding as Bd
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    stream = torch.cuda.Stream(device=dev)
    out = {}

    def unit(shape):
        x = torch.randn(shape, device=dev, generator=g)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    def common(shape, gshape, gscale):
        q, k = unit(shape), unit(shape)
        v = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        beta = torch.sigmoid(torch.randn(shape[:-1], device=dev, generator=g)).to(torch.bfloat16)
        gg = -gscale * torch.nn.functional.softplus(torch.randn(gshape, device=dev, generator=g))
        return q, k, v, gg, beta

    want = lambda name: only is None or only == name  # noqa: E731
    R = (lambda n: n) if reps is None else (lambda n: reps)  # noqa: E731
    with torch.cuda.stream(stream):
        from gated_delta_rule_28_gb300 import workloads
        if want("packed_fwd"):  # packed documents: 32768 tokens, H=32, lengths U[37, 8192]
            lens = workloads.doc_lengths(np.random.default_rng(2), 32768)
            cu = np.concatenate([[0], np.cumsum(lens)])
            q, k, v, gg, beta = common((32768, 32, 128), (32768, 32), 0.1)
            vl = api.Varlen(cu, 32768, dev)
            ms = _time_ms(lambda: api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, varlen=vl,
                                                                 stream=stream.cuda_stream), R(5), 2, stream)
            byts = 32768 * 32 * BYTES_PER_TOKEN_HEAD + len(lens) * 32 * STATE_BYTES
            out["packed_fwd"] = {"workload": "gdn_packed_bf16", "ms": ms, "tokens_per_s": 32768 / ms * 1e3,
                                 "hbm_frac": byts / (ms * 1e-3) / 1e9 / hbm_peak, "docs": int(len(lens))}
            del q, k, v, gg, beta
        if want("kda_split_fwd"):  # KDA long context: per-key base-2 gates, 16 segments of 4096
            TK = kda_tokens
            q, k, v, gg, beta = common((1, TK, 8, 128), (1, TK, 8, 128), 0.05)
            ms_split = _time_ms(lambda: api.split_forward(q, k, v, gg, beta, 4096, use_exp2=True,
                                                          stream=stream.cuda_stream), R(5), 2, stream)
            ms_whole = _time_ms(lambda: api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, use_exp2=True,
                                                                       stream=stream.cuda_stream), R(5), 2, stream)
            # algorithmic bytes of the scan: q, k, v, o bf16, per-key g fp32, beta bf16, final state
            kda_bytes = TK * 8 * (4 * 256 + 512 + 2) + 8 * STATE_BYTES
            out["kda_split_fwd"] = {"workload": "kda_long_bf16", "ms_split": ms_split, "ms_unsplit": ms_whole,
                                    "tokens_per_s_split": TK / ms_split * 1e3, "tokens": TK,
                                    "hbm_frac_split": kda_bytes / (ms_split * 1e-3) / 1e9 / hbm_peak}
            del q, k, v, gg, beta
        if want("train_fwd_bwd"):  # training step: forward with saved slots + backward, B8 H16 T8192
            TT = train_tokens
            q, k, v, gg, beta = common((8, TT, 16, 128), (8, TT, 16), 0.1)
            h0 = 0.1 * torch.randn((8, 16, 128, 128), device=dev, generator=g)
            dO = torch.randn((8, TT, 16, 128), device=dev, generator=g).to(torch.bfloat16)
            f = api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, h0=h0, return_g_cumsum=True,
                                               return_A=True, stream=stream.cuda_stream)
            ms_f = _time_ms(lambda: api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, h0=h0, return_g_cumsum=True,
                                                                   return_A=True, stream=stream.cuda_stream),
                            R(2), 1, stream)
            ms_b = _time_ms(lambda: api.chunk_gated_delta_rule_bwd(q, k, v, f["g_cumsum"], beta, f["A"], dO,
                                                                   h0=h0, stream=stream.cuda_stream), R(2), 1, stream)
            out["train_fwd_bwd"] = {"workload": "gdn_train_bf16", "ms_fwd": ms_f, "ms_bwd": ms_b,
                                    "tokens_per_s": 8 * TT / (ms_f + ms_b) * 1e3, "tokens": TT}
            del q, k, v, gg, beta, h0, dO, f
        if want("frame_scan"):  # dense per-token transition scan: 16 sequences x 4096 positions, D = 64
            BH, TF, D = 16, frame_positions, 64
            eye = torch.eye(D, device=dev)

            def trans():
                return 0.9 * eye + (0.05 / D ** 0.5) * torch.randn((BH, TF, D, D), device=dev, generator=g)

            W_kv = trans()
            U_kv = torch.randn((BH, TF, D, D), device=dev, generator=g) / D ** 0.5
            W_z = trans()
            u_z = torch.randn((BH, TF, D), device=dev, generator=g) / D ** 0.5
            S0 = torch.randn((BH, D, D), device=dev, generator=g)
            s0 = torch.randn((BH, D), device=dev, generator=g)
            # algorithmic bytes: W_kv, U_kv, W_z, u_z in and every position's two states out
            fbytes = BH * TF * (4 * D * D + 2 * D) * 4
            sweep = {}
            for seg in (128, 256, 512, 0):
                sweep[seg] = _time_ms(lambda: api.frame_scan(W_kv, U_kv, W_z, u_z, S0_kv=S0, s0_z=s0,
                                                             segment_len=seg, stream=stream.cuda_stream),
                                      R(3), 1, stream)
            ms = sweep[0]
            out["frame_scan"] = {"workload": "frame_scan_f32", "BH": BH, "T": TF, "D": D, "segment_len": 0,
                                 "ms": ms, "positions_per_s": BH * TF / ms * 1e3,
                                 "hbm_frac": fbytes / (ms * 1e-3) / 1e9 / hbm_peak,
                                 "ms_by_segment_len": {str(k2): v2 for k2, v2 in sweep.items()}}
            del W_kv, U_kv, W_z, u_z
        if only == "aux_paths":  # the other kernels, for their profiles (not part of the default run)
            aux = {}
            # fp32 scalar gate: the FMA forward and backward kernels
            q, k, v, gg, beta = common((2, 2048, 8, 128), (2, 2048, 8), 0.1)
            q, k, v, beta = q.float(), k.float(), v.float(), beta.float()
            dO = torch.randn((2, 2048, 8, 128), device=dev, generator=g)
            f = api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, return_g_cumsum=True, return_A=True,
                                               stream=stream.cuda_stream)
            aux["f32_fwd_ms"] = _time_ms(lambda: api.chunk_gated_delta_rule_fwd(
                q, k, v, gg, beta, stream=stream.cuda_stream), R(3), 1, stream)
            aux["f32_bwd_ms"] = _time_ms(lambda: api.chunk_gated_delta_rule_bwd(
                q, k, v, f["g_cumsum"], beta, f["A"], dO, stream=stream.cuda_stream), R(3), 1, stream)
            # bf16 per-key gate backward (recompute on the per-key kernels, FMA reverse recurrence
            # and local gradients)
            q, k, v, gg, beta = common((1, 4096, 8, 128), (1, 4096, 8, 128), 0.05)
            dO = torch.randn((1, 4096, 8, 128), device=dev, generator=g).to(torch.bfloat16)
            f = api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, use_exp2=True, return_g_cumsum=True,
                                               return_A=True, stream=stream.cuda_stream)
            aux["kda_bwd_ms"] = _time_ms(lambda: api.chunk_gated_delta_rule_bwd(
                q, k, v, f["g_cumsum"], beta, f["A"], dO, use_exp2=True, stream=stream.cuda_stream),
                R(3), 1, stream)
            # bf16 scalar gate with the in-kernel input maps (L2 norm of q, k; beta sigmoid)
            q, k, v, gg, beta = common((1, 4096, 16, 128), (1, 4096, 16), 0.1)
            dO = torch.randn((1, 4096, 16, 128), device=dev, generator=g).to(torch.bfloat16)
            kw = dict(use_qk_l2norm=True, use_beta_sigmoid=True, stream=stream.cuda_stream)
            f = api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, return_g_cumsum=True, return_A=True, **kw)
            aux["maps_fwd_ms"] = _time_ms(lambda: api.chunk_gated_delta_rule_fwd(q, k, v, gg, beta, **kw),
                                          R(3), 1, stream)
            aux["maps_bwd_ms"] = _time_ms(lambda: api.chunk_gated_delta_rule_bwd(
                q, k, v, f["g_cumsum"], beta, f["A"], dO, **kw), R(3), 1, stream)
            out["aux_paths"] = aux
    Bd.gdn_device_status(stream.cuda_stream)
    return out


def run_ours(args):
    import torch
    from gated_delta_rule_28_gb300 import binding as Bd, build as gbuild, workloads

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    gbuild.build()
    Bd.load()

    inp = workloads.make(2)
    Bsz, T, H, K, V = 4, 4096, 16, 128, 128
    tokens = Bsz * T
    t = lambda x, dt=torch.bfloat16: torch.from_numpy(np.ascontiguousarray(x)).to(dev, dt)  # noqa: E731
    sets = []
    for r in range(ROTATE):
        sets.append(dict(q=t(inp.q), k=t(inp.k), v=t(inp.v), g=t(inp.g, torch.float32),
                         beta=t(inp.beta), o=torch.empty((Bsz, T, H, V), device=dev, dtype=torch.bfloat16),
                         ht=torch.empty((Bsz, H, K, V), device=dev, dtype=torch.float32)))
    p = Bd.make_problem(Bsz, T, H, K, V, dtype=Bd.GDN_DTYPE_BF16)
    nws = Bd.gdn_chunk_fwd_workspace(p)
    ws = torch.empty(max(nws, 1), device=dev, dtype=torch.uint8)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def launch(i):
        s = sets[i % ROTATE]
        Bd.gdn_chunk_fwd(p, s["q"], s["k"], s["v"], s["g"], s["beta"], None, s["o"], s["ht"],
                         None, None, None, ws, nws, sp)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(i)
    stream.synchronize()
    Bd.gdn_device_status(sp)

    sampler = clock_sampler(dev)
    sampler.start()
    time.sleep(0.05)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark("t0")
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            launch(args.warmup + i)
            ev[i][1].record(stream)
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler.mark("t1")
    clocks = sampler.stop()
    Bd.gdn_device_status(sp)
    elapsed = start.elapsed_time(end) / 1e3
    kern = [a.elapsed_time(b) / 1e3 for a, b in ev]
    elapsed = max_over_ranks(elapsed, dev)
    value = job_tokens_per_s(world, tokens, args.steps, elapsed)
    kavg = sum(kern) / len(kern)

    # end to end with host buffers: every step copies its inputs in from pinned host memory
    # and o and ht back out, through api.HostPipeline (the copies of one call overlap the
    # kernels of its neighbours; the host link, about 0.2 TB/s each way, is the bound)
    from gated_delta_rule_28_gb300 import api as A
    hq, hk, hv = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (inp.q, inp.k, inp.v))
    hg = torch.from_numpy(inp.g).pin_memory()
    hb = torch.from_numpy(inp.beta).to(torch.bfloat16).pin_memory()
    ho = torch.empty((Bsz, T, H, V), dtype=torch.bfloat16).pin_memory()
    hht = torch.empty((Bsz, H, K, V), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hg, hb))
    d2h = ho.numel() * ho.element_size() + hht.numel() * hht.element_size()
    del sets
    torch.cuda.empty_cache()
    pipe = A.HostPipeline(Bsz, T, H, K, V, dev, depth=2, h2d_streams=1)
    for _ in range(max(1, args.warmup)):
        pipe.submit(hq, hk, hv, hg, hb, ho, hht)
    pipe.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in[0])
    for st in pipe.streams():
        st.wait_event(e0)
    for _ in range(args.steps):
        pipe.submit(hq, hk, hv, hg, hb, ho, hht)
    e1.record(pipe.s_out)  # after the last call's copies out, which follow all of its work
    pipe.synchronize()
    torch.cuda.synchronize()
    e2e_t = e0.elapsed_time(e1) / 1e3
    Bd.gdn_device_status(pipe.s_comp.cuda_stream)
    e2e_t = max_over_ranks(e2e_t, dev)
    e2e_value = job_tokens_per_s(world, tokens, args.steps, e2e_t)

    hbm, tc, src = _peaks()
    alg_bytes = Bsz * T * H * BYTES_PER_TOKEN_HEAD + Bsz * H * STATE_BYTES
    flops = Bsz * T * H * FLOP_PER_TOKEN_HEAD
    achieved = alg_bytes / kavg / 1e9
    traffic = _recorded_traffic()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import recurrence as R
        R.build()
        cores = os.cpu_count() or 1
        # bounded sample: two (batch, head) pairs per host core (at most all 64), one oracle
        # thread per pair on every core
        n_pairs = min(2 * cores, 64)
        ct = time_oracle(inp, n_pairs, cores)
        cpu = {"value": n_pairs * T / 16 / ct, "unit": "tokens/s", "cores": cores,
               "kind": "oracle",
               "sample": f"{n_pairs} of 64 (batch, head) pairs x 4096 tokens, fp64 token "
                         f"recurrence, one thread per pair on {cores} host cores, tokens/s "
                         "scaled to 16 heads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {**WORKLOAD, "l2": f"inputs larger than L2: {ROTATE} rotating input sets"},
            "tflops": flops / kavg / 1e12,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic, "peak_source": src,
                         "kernel": "gdn_chunk_fwd: ut_kernel + tc_fwd_ws_kernel",
                         "launches_per_step": 2, "alg_bytes_per_launch": alg_bytes,
                         "kernel_ms": 1e3 * kavg,
                         "tensor_frac": flops / kavg / 1e12 / tc},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks,
            "step_ms": {"median": 1e3 * statistics.median(kern), "min": 1e3 * min(kern),
                        "max": 1e3 * max(kern), "mean": 1e3 * kavg,
                        "method": "CUDA events around every step on the launching stream; "
                                  f"{ROTATE} rotating input sets larger than L2 in place of an "
                                  "L2 flush"},
            "gpu_launches": 2 * args.steps,
        }
        if not args.no_rows and world == 1:
            try:
                line["rows"] = secondary_rows(dev, hbm)
            except Exception as exc:  # reported, never hidden
                line["rows"] = {"error": repr(exc)}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the other scope rows' timings")
    ap.add_argument("--row", choices=ROWS, help="time only this secondary row and print it (profiling)")
    ap.add_argument("--reps", type=int, default=None, help="timed repetitions of --row")
    ap.add_argument("--kda-tokens", type=int, default=65536, help="tokens of the per-key row (profiling)")
    ap.add_argument("--train-tokens", type=int, default=8192, help="tokens per batch row of the training row")
    ap.add_argument("--frame-positions", type=int, default=4096,
                    help="positions per sequence of the transition-scan row (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.row:
        import torch
        from gated_delta_rule_28_gb300 import build as gbuild
        gbuild.build()
        torch.cuda.set_device(0)
        hbm, _, _ = _peaks()
        print(json.dumps(secondary_rows(torch.device("cuda", 0), hbm, only=args.row, reps=args.reps,
                                        kda_tokens=args.kda_tokens, train_tokens=args.train_tokens,
                                        frame_positions=args.frame_positions)),
              flush=True)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
