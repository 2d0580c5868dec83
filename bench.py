"""Benchmark of the DeepSeekMoE layer forward (+ balancing-bias update) on B300.

One step = moe_forward (route -> dispatch -> gate/up grouped GEMM + SwiGLU ->
down grouped GEMM -> combine) + moe_update_bias over one batch of synthetic
tokens, on the V3-shaped prefill layer by default (T=8192, d=7168, 256 routed
experts top-8 + 1 shared, intermediate 2048, bf16).

    python bench.py [--gpus N --steps K --warmup W] [--config NAME] [--impl reference]
                    [--train]   (training step: forward with saved state + backward)

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
of the layer on its own batch (replicas, weak scaling); times are the max over
ranks.  --impl reference times the CPU oracle on a bounded token sample of
the same workload instead.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_inputs import get_config, make_inputs  # noqa: E402

METRIC = "MoE-layer tokens/s (256e top-8, T=8192, bf16) + grouped-GEMM % of tensor peak"
UNIT = "tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """SM clock and clock-event reasons of this process's GPU, read through NVML
    (the driver's libnvidia-ml via ctypes; queries only) every `period_s` on a
    background thread.  window() marks a timed region; summary() reports the
    samples that fell inside the marked windows, so a short region still gets
    its own samples.  Falls back to an nvidia-smi query loop (whole-run
    samples) when NVML cannot be loaded."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device: torch.device, period_s: float = 0.005):
        self.device = device
        self.period = period_s
        self.samples = []          # (monotonic time, sm MHz, reasons bitmask, power W)
        self.windows = []
        self.sm_max = None
        self._stop = None
        self._thread = None
        self._smi = None
        self.nvml_error = None

    @staticmethod
    def _nvml():
        """NVML through ctypes (the driver's libnvidia-ml; queries only)."""
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        return lib

    def _handle(self, lib):
        import ctypes
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.device)
        uuid = str(getattr(props, "uuid", ""))
        for u in ([uuid, "GPU-" + uuid] if uuid else []):
            if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                return h
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            pci = (f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:"
                   f"{getattr(props, 'pci_device_id', 0):02x}.0")
            if lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(h)) == 0:
                return h
        if lib.nvmlDeviceGetHandleByIndex_v2(self.device.index or 0, ctypes.byref(h)) == 0:
            return h
        raise RuntimeError("no NVML handle for the device")

    def __enter__(self):
        import ctypes
        import threading
        try:
            lib = self._nvml()
            h = self._handle(lib)
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
                self.sm_max = float(mx.value)
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # noqa: BLE001
            self.nvml_error = f"{type(e).__name__}: {e}"
            self._start_smi()
            return self
        self._stop = threading.Event()

        def loop():
            clk = ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            mw = ctypes.c_uint()
            while not self._stop.is_set():
                if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                        reasons_fn(h, ctypes.byref(rs)) == 0):
                    pw = (mw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0
                          else None)
                    self.samples.append((time.monotonic(), float(clk.value), int(rs.value), pw))
                self._stop.wait(self.period)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._smi is not None:
            self._smi[0].terminate()
            try:
                self._smi[0].wait(timeout=5)
            except Exception:
                self._smi[0].kill()
            self._smi[1].close()

    def window(self):
        """Context manager marking one timed region."""
        sampler = self

        class _W:
            def __enter__(self):
                self.t0 = time.monotonic()
                return self

            def __exit__(self, *a):
                sampler.windows.append((self.t0, time.monotonic()))
        return _W()

    def _start_smi(self):
        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            fd, path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            fh = open(path, "w")
            proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device.index or 0),
                                     f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                                     "-lms", "20"], stdout=fh, stderr=subprocess.DEVNULL)
            self._smi = (proc, fh, path)
        except Exception:
            self._smi = None

    def summary(self, windows=None):
        """Median SM clock and the reasons seen in `windows` (default: every
        marked window)."""
        if self._smi is not None:
            return self._smi_summary()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["unavailable"],
                    "samples": 0}
        wins = self.windows if windows is None else windows
        inside = [x for x in self.samples if any(a <= x[0] <= b for a, b in wins)]
        known = 0
        for bit in self.REASONS:
            known |= bit
        share = {}
        for x in inside:
            names = [n for bit, n in self.REASONS.items() if x[2] & bit]
            if x[2] & ~known:
                names.append(hex(x[2] & ~known))
            for n in names:
                share[n] = share.get(n, 0) + 1
        power = [x[3] for x in inside if x[3] is not None]
        return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None,
                "sm_max_mhz": self.sm_max, "reasons": sorted(share),
                "reason_share": {n: round(c / len(inside), 3) for n, c in sorted(share.items())},
                "power_w": round(statistics.median(power), 1) if power else None,
                "samples": len(inside),
                "source": f"NVML every {self.period * 1e3:.0f} ms inside the timed region"}

    def _smi_summary(self):
        proc, fh, path = self._smi
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        fh.flush()
        with open(path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 6:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax = float(parts[1])
                except ValueError:
                    continue
                for n, v in zip(names, parts[2:6]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi every 20 ms over the whole run",
                "nvml_error": self.nvml_error}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, 0, 1, 0


def _max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist, device):
    if dist is not None:
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# FP8 tensor-core peak = the measured bf16 peak x the nominal fp8 : bf16
# ratio of B300 (4.5 : 2.25 dense PFLOP/s)
FP8_OVER_BF16 = 2.0


def kernel_roofline(cfg, traces, peaks):
    """Per-kernel algorithmic work / measured average launch time."""
    T, d, E, K, S, I = cfg.T, cfg.d, cfg.E, cfg.K, cfg.S, cfg.I
    R = T * K + S * T
    es = 4 if cfg.act == "f32" else 2
    work = {
        # flops
        "gemm_gateup_swiglu": ("TFLOP/s", 2.0 * R * d * 2 * I),
        "gemm_down": ("TFLOP/s", 2.0 * R * I * d),
        "gemm_fp8_gateup_swiglu": ("TFLOP/s fp8", 2.0 * R * d * 2 * I),
        "gemm_fp8_down": ("TFLOP/s fp8", 2.0 * R * I * d),
        # e4m3 weights dequantised in shared memory, bf16 tensor cores
        "gemm_w8_gateup_swiglu": ("TFLOP/s", 2.0 * R * d * 2 * I),
        "gemm_w8_down": ("TFLOP/s", 2.0 * R * I * d),
        # bytes: algorithmic traffic (inputs read once, outputs written once)
        "gemm_router": ("GB/s", es * (T * d + E * d) + 4.0 * T * E),
        "router_topk": ("GB/s", 4.0 * T * E + 8.0 * T * K),
        # fused router: tokens and centroids read once, idx and gates written
        "router_fused": ("GB/s", es * (T * d + E * d) + 8.0 * T * K),
        "dispatch_scatter": ("GB/s", es * (T * d + T * K * d) + 4.0 * T * K),
        # bf16 tokens in, e4m3 rows + fp32 1x128 scales out (K routed + S>0 shared copies)
        "dispatch_scatter_fp8": ("GB/s", es * T * d + (T * K + (T if S else 0)) *
                                 (d + 4.0 * d / 128) + 4.0 * T * K),
        "combine": ("GB/s", es * (R * d + 2 * T * d) + 8.0 * T * K),
        # x read once, xn written once, the weight row
        "rmsnorm": ("GB/s", es * 2.0 * T * d + 4.0 * d),
        # behind the RMSNorm: centroids read and their weighted copy written
        "fold_centroids": ("GB/s", 2.0 * es * E * d + 4.0 * d),
        # x read once, normalised rows written to K routed rows and the shared row
        "dispatch_scatter_norm": ("GB/s", es * (T * d + T * K * d + (T * d if S else 0)) +
                                  4.0 * T * K + 4.0 * T),
        "dispatch_scatter_fp8_norm": ("GB/s", es * T * d + (T * K + (T if S else 0)) *
                                      (d + 4.0 * d / 128) + 4.0 * T * K + 4.0 * T),
    }
    out = {}
    for name, launches, ms in traces:
        if name in work and launches > 0:
            unit, amount = work[name]
            avg_s = ms / launches / 1e3
            if unit.startswith("TFLOP/s"):
                ach = amount / avg_s / 1e12
                peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if "fp8" in unit else 1)
            else:
                ach = amount / avg_s / 1e9
                peak = peaks["hbm_gbs"]
            out[name] = {"unit": unit, "achieved": round(ach, 2), "peak": peak,
                         "frac": round(ach / peak, 4), "avg_ms": round(avg_s * 1e3, 4),
                         "launches": launches, "work": amount}
    return out


def dram_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload`, from the
    ncu capture recorded in profiles/dram_traffic.json, or None when there is
    none or the kernel's source file changed since (sha256 recorded with it)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(workload, {}).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "mixture_experts_layer_88_b300", "csrc", rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
            return None
    return rec["bytes_per_launch"]


def cpu_oracle_tokens_per_s(cfg, inp, n_tokens: int, seed: int = 7, prenorm: bool = False):
    """Times the CPU oracle on n_tokens tokens of the workload (weights of the
    experts those tokens use are copied to host first, untimed)."""
    from oracle import moe_oracle as O
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.choice(cfg.T, n_tokens, replace=False))
    x_host = inp["x"][torch.as_tensor(tok, device=inp["x"].device)].cpu()
    norm_w = inp["norm_w"].cpu() if prenorm else None
    u = (O.round_act(O.rmsnorm(x_host, norm_w, NORM_EPS)[0], cfg.act) if prenorm else x_host)
    idx, _, _, _ = O.route(u, inp["centroids"].cpu(), inp["bias"].cpu(), cfg.K,
                           cfg.score_func, cfg.normalize, cfg.n_groups, cfg.topk_groups)
    used = sorted(set(int(e) for e in idx.reshape(-1)))

    class _Experts:
        def __init__(self, src, ids):
            self.shape = src.shape
            self.d = {e: src[e].cpu() for e in ids}

        def __getitem__(self, e):
            return self.d[int(e)]

    host = {"x": x_host, "centroids": inp["centroids"].cpu(), "bias": inp["bias"].cpu(),
            "w13": _Experts(inp["w13"], used), "w2": _Experts(inp["w2"], used),
            "ws13": inp["ws13"].cpu(), "ws2": inp["ws2"].cpu()}
    for k in ("w13", "w2"):
        if k + "_scale" in inp:                       # FP8 layer: block scales too
            host[k + "_scale"] = _Experts(inp[k + "_scale"], used)
            host["s" + k + "_scale"] = inp["s" + k + "_scale"].cpu()
    t0 = time.perf_counter()
    O.moe_layer(host, cfg.K, cfg.normalize, cfg.score_func, cfg.add_residual,
                n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, norm_w=norm_w,
                norm_eps=NORM_EPS, act=cfg.act)
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    return n_tokens / dt, dt, cores


def _one_core_oracle(cfg, inp, args):
    try:
        from threadpoolctl import threadpool_limits
        with threadpool_limits(limits=1):
            rate, secs, _ = cpu_oracle_tokens_per_s(cfg, inp, args.cpu_tokens,
                                                    prenorm=args.prenorm)
        how = "BLAS pool limited to one thread"
    except ImportError:
        if not hasattr(os, "sched_setaffinity"):
            return None
        cpus = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(cpus)})
        try:
            rate, secs, _ = cpu_oracle_tokens_per_s(cfg, inp, args.cpu_tokens,
                                                    prenorm=args.prenorm)
        finally:
            os.sched_setaffinity(0, cpus)
        how = "process pinned to one CPU"
    return {"value": round(rate, 4), "unit": UNIT, "seconds": round(secs, 1), "how": how}


def run_reference(args, cfg, dist, rank, ws, device):
    """Reference arm: the CPU oracle timed on bounded token samples."""
    if rank != 0:
        return
    inp = make_inputs(cfg, device if device.type == "cuda" else "cpu")
    per_step = max(1, args.ref_tokens)
    rates = []
    cores = None
    if args.train:
        from moe_inputs import make_dout
        dout = make_dout(cfg, device if device.type == "cuda" else "cpu")
        cores = os.cpu_count()
    for i in range(args.warmup + args.steps):
        if args.train:
            _, dt = cpu_oracle_train_tokens_per_s(cfg, inp, dout, per_step, seed=100 + i)
        else:
            _, dt, cores = cpu_oracle_tokens_per_s(cfg, inp, per_step, seed=100 + i,
                                                   prenorm=args.prenorm)
        if i >= args.warmup:
            rates.append((per_step, dt))
    tok = sum(t for t, _ in rates)
    secs = sum(s for _, s in rates)
    value = tok / secs
    line = {"impl": "reference", "metric": TRAIN_METRIC if args.train else METRIC,
            "value": round(value, 4), "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / len(rates) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload(cfg, args) + ("+train" if args.train else ""),
                       "T": cfg.T, "d": cfg.d, "E": cfg.E,
                       "K": cfg.K, "S": cfg.S, "I": cfg.I, "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": f"{per_step} random tokens of the {cfg.name} batch per "
                                       f"step through the fp64 oracle" +
                                       (", forward and backward" if args.train else "") +
                                       (f"; rank 0 of {ws} alone" if ws > 1 else "")},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# eps of the RMSNorm in front of the layer (V3 walk-through, section 4.1)
NORM_EPS = 1e-6


TRAIN_METRIC = ("MoE-layer training tokens/s (forward + backward + bias update, 256e top-8, "
                "T=8192, bf16)")


def train_roofline(cfg, traces, peaks):
    """Algorithmic work of the training step's kernels / measured launch time."""
    T, d, E, K, S, I = cfg.T, cfg.d, cfg.E, cfg.K, cfg.S, cfg.I
    R = T * K + S * T
    es = 2
    work = {
        "gemm_gateup_h": ("TFLOP/s", 2.0 * R * d * 2 * I),
        "gemm_down": ("TFLOP/s", 2.0 * R * I * d),
        "gemm_dgrad_down": ("TFLOP/s", 2.0 * R * d * I),
        "gemm_dgrad_gateup": ("TFLOP/s", 2.0 * R * 2 * I * d),
        "gemm_wgrad_down": ("TFLOP/s", 2.0 * R * d * I),
        "gemm_wgrad_gateup": ("TFLOP/s", 2.0 * R * 2 * I * d),
        # bytes: each operand read once, each result written once
        "swiglu_fwd": ("GB/s", es * 3.0 * R * I),
        "combine_bwd": ("GB/s", es * (T * d + T * K * d + R * d) + 4.0 * T * K),
        "swiglu_bwd": ("GB/s", es * 5.0 * R * I),
        "dx_gather": ("GB/s", es * (R * d + 2.0 * T * d)),
        "dcent_partial": ("GB/s", es * T * K * d + 4.0 * T * K),
        "combine": ("GB/s", es * (R * d + 2 * T * d) + 8.0 * T * K),
        "dispatch_scatter": ("GB/s", es * (T * d + T * K * d) + 4.0 * T * K),
    }
    out = {}
    for name, launches, ms in traces:
        if name in work and launches > 0:
            unit, amount = work[name]
            avg_s = ms / launches / 1e3
            if unit == "TFLOP/s":
                ach, peak = amount / avg_s / 1e12, peaks["bf16_tflops"]
            else:
                ach, peak = amount / avg_s / 1e9, peaks["hbm_gbs"]
            out[name] = {"unit": unit, "achieved": round(ach, 2), "peak": peak,
                         "frac": round(ach / peak, 4), "avg_ms": round(avg_s * 1e3, 4),
                         "launches": launches, "total_ms": round(ms, 3), "work": amount}
    return out


def cpu_oracle_train_tokens_per_s(cfg, inp, dout, n_tokens: int, seed: int = 7):
    """The oracle's forward and backward of a few tokens of the full layer
    (route, their K experts and the shared experts forward and backward, the
    router's backward): tokens/s and seconds.  The whole-batch oracle
    backward is not timed: its weight gradients alone are 68 GB in fp64."""
    from oracle import moe_oracle as O
    rng = np.random.default_rng(seed)
    toks = rng.choice(cfg.T, n_tokens, replace=False)
    host = {k: inp[k] for k in ("centroids", "bias")}
    t0 = time.perf_counter()
    for t in toks:
        u = O._f64(inp["x"][int(t):int(t) + 1])
        go = O._f64(dout[int(t):int(t) + 1])
        idx, gates, _, s = O.route(u, host["centroids"], host["bias"], cfg.K, cfg.score_func,
                                   cfg.normalize, cfg.n_groups, cfg.topk_groups)
        dg = np.zeros((1, cfg.K))
        for k in range(cfg.K):
            e = int(idx[0, k])
            w13, w2 = inp["w13"][e].cpu(), inp["w2"][e].cpu()
            dg[0, k] = float(np.sum(go * O.swiglu_ffn(u, w13, w2)))
            O.swiglu_ffn_backward(u, w13, w2, gates[:, k:k + 1] * go)
        for sx in range(cfg.S):
            O.swiglu_ffn_backward(u, inp["ws13"][sx].cpu(), inp["ws2"][sx].cpu(), go)
        O.router_backward(u, host["centroids"], s, idx, gates, dg, cfg.normalize,
                          cfg.score_func)
    secs = time.perf_counter() - t0
    return n_tokens / secs, secs


def run_train(args, cfg, dist, rank, ws, device, peaks):
    """Training step: moe_forward_train + moe_backward + moe_update_bias."""
    import mixture_experts_layer_88_b300 as m
    from moe_inputs import make_dout
    inp = make_inputs(cfg, device, seed=rank)
    dout = make_dout(cfg, device, seed=rank)
    mc = m.cfg_from_layer(cfg)
    state = m.alloc_train_state(mc, device)
    grads = m.alloc_grads(mc, device)
    ws_f = m.alloc_workspace(mc, m.MOE_WS_FORWARD_TRAIN, device)
    ws_b = m.alloc_workspace(mc, m.MOE_WS_BACKWARD, device)
    x = inp["x"]
    out = torch.empty_like(x)
    bias = inp["bias"].clone()
    sh = cfg.S > 0
    stream = torch.cuda.current_stream()

    from mixture_experts_layer_88_b300 import parallel

    def step(xx=x, dd=dout):
        m.forward_train(mc, xx, inp["centroids"], bias, inp["w13"], inp["w2"],
                        inp["ws13"] if sh else None, inp["ws2"] if sh else None, state, out, ws_f)
        m.backward(mc, dd, xx, inp["centroids"], inp["w13"], inp["w2"],
                   inp["ws13"] if sh else None, inp["ws2"] if sh else None, state, grads, ws_b)
        # data parallel (N > 1): parameter gradients and load counts summed over
        # the ranks before the bias update; one rank: no exchange
        parallel.allreduce_grads(grads)
        parallel.balance_step(mc, state["counts"], bias,
                              lambda cfg, c, b: m.update_bias(cfg, c, b), T_global=mc.T * ws)

    clk = ClockSampler(device).__enter__()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert m.get_status() == 0, "device error during warm-up"
    m.trace_enable(True)
    m.trace_read_all()
    _barrier(dist, device)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clk.window():
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    _barrier(dist, device)
    traces = m.trace_read_all()
    m.trace_enable(False)
    st = m.get_status()
    ms_step = _max_over_ranks(dist, ev0.elapsed_time(ev1), device) / args.steps
    value = ws * cfg.T / (ms_step / 1e3)

    # end to end: tokens and output gradients in from pinned host memory, the
    # layer output and the input gradients back, every step
    x_h = x.cpu().pin_memory()
    d_h = dout.cpu().pin_memory()
    o_h = torch.empty_like(x_h).pin_memory()
    dx_h = torch.empty_like(x_h).pin_memory()
    xd, dd = torch.empty_like(x), torch.empty_like(dout)

    def e2e_step():
        xd.copy_(x_h, non_blocking=True)
        dd.copy_(d_h, non_blocking=True)
        step(xd, dd)
        o_h.copy_(out, non_blocking=True)
        dx_h.copy_(grads["dx"], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    _barrier(dist, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(dist, e0.elapsed_time(e1), device) / args.steps
    if rank != 0:
        return
    roof = train_roofline(cfg, traces, peaks)
    gemms = [k for k in roof if k.startswith("gemm_")]
    top = max(gemms, key=lambda k: roof[k]["total_ms"]) if gemms else None
    R = cfg.T * cfg.K + cfg.S * cfg.T
    flops = 6.0 * R * cfg.d * 2 * cfg.I          # forward 3 GEMM-halves, backward 6
    gemm_ms = sum(roof[k]["total_ms"] for k in gemms) / args.steps
    line = {
        "metric": TRAIN_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random tokens, output gradients and random-init weights)",
        "config": {"workload": cfg.name + "+train", "T": cfg.T, "d": cfg.d, "E": cfg.E,
                   "K": cfg.K, "S": cfg.S, "I": cfg.I, "renormalize": bool(cfg.normalize),
                   "parallelism": ("one replica" if ws == 1 else
                                   f"data parallel x{ws}: parameter gradients and load "
                                   f"counts all-reduced every step"),
                   "launch": "eager stream launches",
                   "l2": "inputs larger than L2 (weights, their gradients and the saved rows)"},
        "grouped_gemm": {"tflops": round(flops / (gemm_ms / 1e3) / 1e12, 1),
                         "frac_of_peak": round(flops / (gemm_ms / 1e3) / 1e12 /
                                               peaks["bf16_tflops"], 4),
                         "peak_kind": f"bf16 burst, {peaks['source']}",
                         "frac_of_sustained": round(flops / (gemm_ms / 1e3) / 1e12 /
                                                    peaks["bf16_tflops_sustained"], 4),
                         "kernels": gemms, "ms_per_step": round(gemm_ms, 4)},
        "roofline": ({"kernel": top, "bound": "tensor", "achieved": roof[top]["achieved"],
                      "peak": roof[top]["peak"], "unit": "TFLOP/s", "frac": roof[top]["frac"],
                      "traffic": dram_traffic(cfg.name + "+train", top),
                      "flop_per_launch": roof[top]["work"],
                      "avg_launch_ms": roof[top]["avg_ms"],
                      "peak_kind": f"bf16 burst, {peaks['source']}",
                      "frac_of_sustained": round(roof[top]["achieved"] /
                                                 peaks["bf16_tflops_sustained"], 4)}
                     if top else None),
        "kernels": roof,
        "gpu_launches": sum(t[1] for t in traces),
        "device_status": st,
        "clocks": clk.summary(),
        "e2e": {"value": round(ws * cfg.T / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(2 * x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(2 * out.numel() * out.element_size()),
                "ms_per_step": round(e2e_ms, 4)},
    }
    if not args.no_cpu_baseline:
        n = max(1, args.cpu_tokens // 4)
        rate, secs = cpu_oracle_train_tokens_per_s(cfg, inp, dout, n)
        line["cpu_baseline"] = {"value": round(rate, 4), "unit": UNIT,
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{n} random tokens of the {cfg.name} batch, forward "
                                          f"and backward through the fp64 oracle ({secs:.1f} s)"}
    print(json.dumps(line), flush=True)


def time_layer(m, layer, x, out, steps, warmup, clk, dist=None, device=None, graph=False):
    """W warm-up steps, then exactly `steps` timed steps of layer.step (forward
    + bias update) between CUDA events on the launching stream, inside a clock
    window, with a barrier and a synchronise on both sides.  Returns
    (ms per step, max over ranks), the per-kernel traces of the timed steps
    and the device status word."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        layer.step(x, out)
    torch.cuda.synchronize()
    assert m.get_status() == 0, "device error during warm-up"
    run_step = lambda: layer.step(x, out)  # noqa: E731
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.step(x, out)
        g.replay()
        torch.cuda.synchronize()
        run_step = g.replay
    m.trace_enable(True)
    m.trace_read_all()
    if dist is not None:
        _barrier(dist, device)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clk.window():
        ev0.record(stream)
        for _ in range(steps):
            run_step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        _barrier(dist, device)
    traces = m.trace_read_all()
    if graph:
        # replayed launches bypass the library's per-launch events: take the
        # per-kernel figures from the same number of traced eager steps
        for _ in range(steps):
            layer.step(x, out)
        torch.cuda.synchronize()
        traces = m.trace_read_all()
    m.trace_enable(False)
    st = m.get_status()
    ms = _max_over_ranks(dist, ev0.elapsed_time(ev1), device) if dist is not None else \
        ev0.elapsed_time(ev1)
    return ms / steps, traces, st


def decode_record(m, cfg_prefill, inp, device, peaks, clk, steps, warmup, graph=False):
    """The V3 decode batch (T = 128) on the same layer weights as the prefill
    run: weight streaming.  ms per step, tokens/s and the touched expert
    weights (every expert at least one token chose, plus the shared experts,
    read once per step) per second of the two expert GEMMs, against the
    measured HBM copy bandwidth."""
    from moe_inputs import make_tokens
    cfg = get_config("v3_decode")
    assert (cfg.d, cfg.E, cfg.K, cfg.S, cfg.I) == (cfg_prefill.d, cfg_prefill.E,
                                                    cfg_prefill.K, cfg_prefill.S, cfg_prefill.I)
    w = dict(inp)
    w["bias"] = inp["bias"].clone()
    layer = m.MoeLayer(m.cfg_from_layer(cfg), w, device=device)
    x = make_tokens(cfg, device)
    out = torch.empty_like(x)
    n0 = len(clk.windows)
    ms, traces, st = time_layer(m, layer, x, out, steps, warmup, clk, graph=graph)
    touched = int((layer.counts > 0).sum().item()) + cfg.S
    wbytes = touched * 3.0 * cfg.I * cfg.d * 2 + cfg.E * cfg.d * 2
    gemm_ms = sum(t[2] for t in traces if t[0] in ("gemm_gateup_swiglu", "gemm_down")) / steps
    return {"workload": cfg.name, "T": cfg.T, "steps": steps, "warmup": warmup,
            "launch": _launch(graph),
            "ms_per_step": round(ms, 4), "tokens_per_s": round(cfg.T / (ms / 1e3), 1),
            "touched_experts": touched, "weight_bytes_per_step": int(wbytes),
            "weight_stream": {"achieved_gbs": round(wbytes / (gemm_ms / 1e3) / 1e9, 1),
                              "peak_gbs": peaks["hbm_gbs"],
                              "frac": round(wbytes / (gemm_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                            4),
                              "over": "the gate/up + down GEMMs' event time",
                              "gemm_ms_per_step": round(gemm_ms, 4)},
            "step_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
            "kernels": kernel_roofline(cfg, traces, peaks),
            "gpu_launches": sum(t[1] for t in traces), "device_status": st,
            "clocks": clk.summary(clk.windows[n0:])}


def fp8_record(m, device, peaks, clk, steps, warmup, balance_steps, graph=False):
    """The Zipf-skewed V3 layer (T = 16384) with e4m3 128x128 block-scaled
    expert weights: ms per step, tokens/s, the e4m3 expert GEMMs' TFLOP/s
    against the fp8 peak (2 x the measured bf16 burst peak), and the max /
    mean expert load over `balance_steps` bias-update steps from bias 0."""
    from moe_inputs import make_tokens
    cfg = get_config("v3_skewed_fp8")
    inp = make_inputs(cfg, device)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), inp, device=device, fp8_path="e4m3")
    x = inp["x"]
    out = torch.empty_like(x)
    n0 = len(clk.windows)
    ms, traces, st = time_layer(m, layer, x, out, steps, warmup, clk, graph=graph)
    names = ("gemm_fp8_gateup_swiglu", "gemm_fp8_down")
    gemm_ms = sum(t[2] for t in traces if t[0] in names) / steps
    tf = cfg.gemm_flops() / (gemm_ms / 1e3) / 1e12
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    layer.bias.zero_()
    loads = []
    for step in range(balance_steps):
        layer.forward(make_tokens(cfg, device, step=step + 1), out)
        loads.append(round(float(layer.update_bias()[0].item()), 3))
    rec = {"workload": cfg.name + "+e4m3", "T": cfg.T, "steps": steps, "warmup": warmup,
           "launch": _launch(graph),
           "ms_per_step": round(ms, 4), "tokens_per_s": round(cfg.T / (ms / 1e3), 1),
           "grouped_gemm": {"tflops": round(tf, 1), "peak_tflops": fp8_peak,
                            "frac": round(tf / fp8_peak, 4),
                            "peak_kind": f"fp8 = 2 x bf16 burst, {peaks['source']}",
                            "ms_per_step": round(gemm_ms, 4), "kernels": list(names)},
           "balance": {"steps": balance_steps, "gamma": cfg.gamma,
                       "max_over_mean_load": loads},
           "kernels": kernel_roofline(cfg, traces, peaks),
           "gpu_launches": sum(t[1] for t in traces), "device_status": st,
           "clocks": clk.summary(clk.windows[n0:])}
    del layer, inp
    torch.cuda.empty_cache()
    return rec


def dsmoe16b_record(m, device, peaks, clk, steps, warmup, graph=False):
    """The 16B-shape layer (T = 32768, d = 2048, 64 routed experts top-6 with
    Softmax scores and no renormalisation, 2 shared experts, I = 1408): ms per
    step, tokens/s and the bf16 expert GEMMs' TFLOP/s against the measured
    bf16 peaks."""
    cfg = get_config("dsmoe16b")
    inp = make_inputs(cfg, device)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), inp, device=device)
    x = inp["x"]
    out = torch.empty_like(x)
    n0 = len(clk.windows)
    ms, traces, st = time_layer(m, layer, x, out, steps, warmup, clk, graph=graph)
    names = ("gemm_gateup_swiglu", "gemm_down")
    gemm_ms = sum(t[2] for t in traces if t[0] in names) / steps
    tf = cfg.gemm_flops() / (gemm_ms / 1e3) / 1e12
    rec = {"workload": cfg.name, "T": cfg.T, "steps": steps, "warmup": warmup,
           "launch": _launch(graph),
           "ms_per_step": round(ms, 4), "tokens_per_s": round(cfg.T / (ms / 1e3), 1),
           "grouped_gemm": {"tflops": round(tf, 1), "peak_tflops": peaks["bf16_tflops"],
                            "frac": round(tf / peaks["bf16_tflops"], 4),
                            "peak_kind": f"bf16 burst, {peaks['source']}",
                            "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                            "ms_per_step": round(gemm_ms, 4), "kernels": list(names)},
           "kernels": kernel_roofline(cfg, traces, peaks),
           "gpu_launches": sum(t[1] for t in traces), "device_status": st,
           "clocks": clk.summary(clk.windows[n0:])}
    del layer, inp
    torch.cuda.empty_cache()
    return rec


def _launch(graph: bool) -> str:
    return "CUDA graph replay" if graph else "eager stream launches"


def _workload(cfg, args) -> str:
    w = cfg.name + ("+rmsnorm" if args.prenorm else "")
    if cfg.wgt == "e4m3":
        w += "+" + args.fp8_path
    return w


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="v3_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=24,
                    help="tokens of the oracle CPU-baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=1,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--balance-steps", type=int, default=20,
                    help="skewed layers: bias-update steps of the balancing run")
    ap.add_argument("--fp8-path", default="e4m3", choices=["e4m3", "w8a16"],
                    help="FP8 layers: e4m3 x e4m3 with fp32 promotion every 128 K (e4m3) or "
                         "e4m3 weights dequantised to bf16 on the fly (w8a16)")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step from a CUDA graph captured after the warm-up (the "
                         "per-kernel figures then come from traced eager steps after the "
                         "timed region, so the default times eager launches)")
    ap.add_argument("--prenorm", action="store_true",
                    help="the layer behind its RMSNorm: h = x + MoE(RMSNorm(x))")
    ap.add_argument("--train", action="store_true",
                    help="training step: forward with saved state + backward + bias update")
    ap.add_argument("--no-subconfigs", action="store_true",
                    help="skip the decode, FP8 and 16B-shape sub-records of the default V3 prefill run")
    ap.add_argument("--sub-steps", type=int, default=20,
                    help="timed steps of each sub-record")
    ap.add_argument("--override", default="",
                    help="comma-separated shape overrides, e.g. T=1024,E=32 (profiling cases)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    dist, rank, ws, local = _dist()
    if ws > 1:
        args.graph = False    # the count all-reduce is not captured into a graph
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    if device.type == "cuda":
        torch.cuda.set_device(device)
    cfg = get_config(args.config)
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        cfg = cfg.with_(name=f"{cfg.name}[{args.override}]", **{k: int(v) for k, v in kv.items()})

    if args.impl == "reference":
        run_reference(args, cfg, dist, rank, ws, device)
        if dist is not None:
            dist.destroy_process_group()
        return

    import mixture_experts_layer_88_b300 as m
    peaks = _peaks()
    if args.train:
        run_train(args, cfg, dist, rank, ws, device, peaks)
        if dist is not None:
            dist.destroy_process_group()
        return
    inp = make_inputs(cfg, device, seed=rank)
    mc = m.cfg_from_layer(cfg)
    layer = m.MoeLayer(mc, inp, device=device,
                       norm_w=inp["norm_w"] if args.prenorm else None, norm_eps=NORM_EPS,
                       fp8_path=args.fp8_path)
    layer.T_global = cfg.T * ws          # every rank runs the same batch size
    x = inp["x"]
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    # ---- device-resident timed region
    clk = ClockSampler(device).__enter__()
    ms_step, traces, st = time_layer(m, layer, x, out, args.steps, args.warmup, clk, dist,
                                     device, graph=args.graph)
    value = ws * cfg.T / (ms_step / 1e3)
    main_window = list(clk.windows)

    # ---- end to end: every step copies its tokens in from pinned host memory
    # and its output back to pinned host memory (HostPipeline overlaps the
    # copies of neighbouring steps with the compute)
    x_host = x.cpu().pin_memory()
    out_hosts = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    pipe = m.HostPipeline(layer, x)
    pipe.run([x_host] * args.warmup, [out_hosts[i & 1] for i in range(args.warmup)])
    torch.cuda.synchronize()
    _barrier(dist, device)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run([x_host] * args.steps, [out_hosts[i & 1] for i in range(args.steps)], stream)
    e1.record(pipe.d2h)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(dist, e0.elapsed_time(e1), device) / args.steps
    e2e_value = ws * cfg.T / (e2e_ms / 1e3)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    roof = kernel_roofline(cfg, traces, peaks)
    w8 = layer.w8a16                        # FP8 weights on the bf16 tensor cores
    fp8 = cfg.wgt == "e4m3" and not w8      # e4m3 x e4m3 tensor cores
    pre = "gemm_w8_" if w8 else "gemm_fp8_" if fp8 else "gemm_"
    top_name = pre + "gateup_swiglu"
    top = roof.get(top_name)
    gemm_flops = cfg.gemm_flops()
    gemm_names = (top_name, pre + "down")
    gemm_ms = sum(t[2] for t in traces if t[0] in gemm_names)
    gemm_ms_step = gemm_ms / args.steps if gemm_ms else None
    gemm_tflops = gemm_flops / (gemm_ms_step / 1e3) / 1e12 if gemm_ms_step else None
    launches = sum(t[1] for t in traces)
    traffic = dram_traffic(cfg.name, top_name)

    # The timed region lasts well under a second, so the tensor-core roofline
    # is the measured burst bf16 peak (x 2 for e4m3); the sustained figure,
    # measured under seconds of dense load at the power cap, is given beside it.
    mult = FP8_OVER_BF16 if fp8 else 1
    gemm_peak = peaks["bf16_tflops"] * mult
    gemm_peak_sus = peaks["bf16_tflops_sustained"] * mult
    kind = (f"fp8 = 2 x bf16 burst, {peaks['source']}" if fp8 else
            f"bf16 burst, {peaks['source']}")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 x e4m3 (fp32 promotion), bf16 tokens" if fp8 else
                  "e4m3 weights dequantised to bf16, bf16 x bf16 (fp32 accumulate)" if w8
                  else "bf16"),
        "data": "synthetic (seeded random tokens and random-init weights of the layer's shape)",
        "config": {"workload": _workload(cfg, args), "T": cfg.T, "d": cfg.d, "E": cfg.E,
                   "K": cfg.K, "S": cfg.S, "I": cfg.I, "renormalize": bool(cfg.normalize),
                   "parallelism": (f"data parallel x{ws}, load counts all-reduced for the "
                                   f"bias update" if ws > 1 else "one replica"),
                   "launch": _launch(args.graph),
                   "l2": (f"inputs larger than L2: "
                          f"{(cfg.E + cfg.S) * 3 * cfg.I * cfg.d * {'e4m3': 1, 'bf16': 2}.get(cfg.wgt, 4) / 1e9:.1f} GB "
                          f"of expert weights streamed per step")},
        "grouped_gemm": {"tflops": round(gemm_tflops, 1) if gemm_tflops else None,
                         "frac_of_peak": round(gemm_tflops / gemm_peak, 4)
                         if gemm_tflops else None,
                         "peak_tflops": gemm_peak, "peak_kind": kind,
                         "frac_of_sustained": round(gemm_tflops / gemm_peak_sus, 4)
                         if gemm_tflops else None,
                         "sustained_peak_tflops": gemm_peak_sus,
                         "kernels": list(gemm_names),
                         "ms_per_step": round(gemm_ms_step, 4) if gemm_ms_step else None},
        "roofline": ({"kernel": top_name, "bound": "tensor",
                      "achieved": top["achieved"], "peak": gemm_peak, "unit": "TFLOP/s",
                      "frac": round(top["achieved"] / gemm_peak, 4), "traffic": traffic,
                      "flop_per_launch": top["work"], "avg_launch_ms": top["avg_ms"],
                      "peak_kind": kind,
                      "frac_of_sustained": round(top["achieved"] / gemm_peak_sus, 4),
                      "sustained_peak": gemm_peak_sus}
                     if top else None),
        "kernels": roof,
        "gpu_launches": launches,
        "device_status": st,
        "clocks": clk.summary(main_window),
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                "h2d_bytes_per_step": int(x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "ms_per_step": round(e2e_ms, 4)},
    }
    if cfg.zipf_s > 0:
        # balancing run of the skewed layer: fresh tokens every step, bias
        # from 0, one sign update per step; max / mean expert load per step
        from moe_inputs import make_tokens
        layer.bias.zero_()
        loads = []
        for step in range(args.balance_steps):
            xb = make_tokens(cfg, device, seed=rank, step=step + 1)
            layer.forward(xb, out)
            loads.append(round(float(layer.update_bias()[0].item()), 3))
        line["balance"] = {"steps": args.balance_steps, "gamma": cfg.gamma,
                           "max_over_mean_load": loads}
    sub = (ws == 1 and not args.no_subconfigs and not args.override and not args.prenorm
           and args.config == "v3_prefill")
    if sub:
        # the other V3 configurations, each with its own timed region and clocks
        line["subconfigs"] = {"v3_decode": decode_record(m, cfg, inp, device, peaks, clk,
                                                         args.sub_steps, args.warmup,
                                                         args.graph)}
    if not args.no_cpu_baseline:
        rate, secs, cores = cpu_oracle_tokens_per_s(cfg, inp, args.cpu_tokens,
                                                    prenorm=args.prenorm)
        line["cpu_baseline"] = {"value": round(rate, 4), "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"{args.cpu_tokens} random tokens of the {cfg.name} "
                                          f"batch through the fp64 oracle ({secs:.1f} s)"}
        # the same sample on one core: numpy's BLAS pool limited to one thread,
        # or (without threadpoolctl) the process pinned to one CPU meanwhile
        one = _one_core_oracle(cfg, inp, args)
        if one is not None:
            line["cpu_baseline"]["one_core"] = one
    if sub:
        del layer, pipe, inp, x, out
        torch.cuda.empty_cache()
        line["subconfigs"]["v3_skewed_fp8"] = fp8_record(m, device, peaks, clk, args.sub_steps,
                                                         args.warmup, args.balance_steps,
                                                         args.graph)
        line["subconfigs"]["dsmoe16b"] = dsmoe16b_record(m, device, peaks, clk, args.sub_steps,
                                                         args.warmup, args.graph)
    clk.__exit__(None, None, None)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
