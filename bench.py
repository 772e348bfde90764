"""Benchmark of the OAL hot path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Step (default workload, Llama-3.2-1B-shaped prefill: B=4, Hq=32, Hkv=8, d=64,
T=8192, G=6, bf16 inputs, packed fp32 states): coefficient expansion, chunked
causal prefill of 8192 tokens per sequence, then one decode token for every
sequence continuing from the prefill state -- every step of the method in one
pass.  Inputs are resident in HBM; L2 is flushed (256 MiB write) before every
timed step and each step is timed with CUDA events on the launching stream.
The timed steps replay the step captured once as a CUDA graph (the host's
per-call Python and tensor-map setup is then off the device timeline); the
e2e leg calls the API directly every step.

The JSON line also carries:
  roofline      the dominant kernel (the contraction with the largest device
                time per prefill call; a kernel launched twice per call is
                summed): its algorithmic FLOPs per call / its device time,
                against the measured peak in MEASURED_PEAKS.json;
  e2e           the same step through the C ABI with host buffers: pinned
                host->device copies of the inputs and device->host copies of
                the outputs inside the timed region, pipelined per sequence
                (the last one in groups of 4 KV heads) on two copy streams
                beside two compute streams;
  config1       the Qwen2.5-0.5B-shaped prefill (B=1, Hq=14, Hkv=2, T=4096,
                G=4) measured the same way;
  config4       the long-context prefill (B=1, Hq=14, Hkv=2, T=65536, G=4) at
                chunk sizes 64, 128 and 256;
  backward      the prefill backward (dQ, dK, dV, dL) on the Qwen-shaped
                workload;
  group_counts  prefill time per head on the Qwen shape for one global group
                (G = 1), five groups, and heads of 1 to 5 groups in one launch;
  decode        the decode workload (B=64, Hq=14, Hkv=2, 1024 steps after a
                2048-token prefill): steps/s and achieved HBM bandwidth for the
                full fp32 state (4161 x 65 per KV head) and the packed one;
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the same
                workload on this host's cores (rank 0, N = 1 only);
  clocks        SM clocks and throttle reasons sampled during the timed region.

Under torchrun (N > 1) every rank runs its own copy of the workload on its
own GPU (independent sequences, no data exchange): weak scaling, value =
tokens of all ranks / max over ranks of the timed region.

--impl reference times the fp64 CPU oracle (the only reference there is:
the pages publish no code) on bounded samples of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "OAL prefill tokens/s & decode steps/s (1×GB300), % of tensor/HBM roofline"
D = 64
F_PACKED = 1 + D + D * (D + 1) // 2      # 2145
F_FULL = 1 + D + D * D                   # 4161
U = D + 1
FP32_SIMT_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # CUDA-core fp32 FMA at 2070 MHz
CSRC = os.path.join(ROOT, "grouped_quadratic_gb300", "csrc")

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of a
# kernel from one ncu capture, with the SHA-256 of the kernel's source file at
# the time of the capture.  A record is reported only while that source file
# is unchanged (otherwise the traffic is null: the counters are stale).
TRAFFIC = [
    # (kernel, source file, workload key (B, Hq, Hkv, T, G, layout, chunk), bytes per
    #  launch, source sha256)
    ("tc_readout_kernel", "prefill_tc.cu", (4, 32, 8, 8192, 6, "packed", 128),
     1103470848 + 120884224, "a14fccb057ced4be7cd21ff10807f399b2b408d6b5682ae689f41066d1fed96f"),
    ("decode_stream_kernel", "decode.cu", (64, 14, 2, "full"),
     138927872 + 81893888, "0147d4d17b168bad5f1527d1d50dd9e605973467cd8f82b2714e8ac749a363fe"),
]


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(kernel, key):
    for k, src, wkey, nbytes, sha in TRAFFIC:
        if k == kernel and wkey == key and _sha(os.path.join(CSRC, src)) == sha:
            return nbytes
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "samples": len(sms), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, target_s, max_rows=None):
    """Time the fp64 oracle on a stride sample of query rows; returns dict."""
    import oracle
    total_rows = w.B * w.Hq * w.T_prefill
    probe = np.arange(0, total_rows, max(1, total_rows // 64))
    oracle.direct(w.Q[:, :, :w.T_prefill], w.K[:, :, :w.T_prefill], w.V[:, :, :w.T_prefill],
                  w.L, w.group, w.eps, rows=probe[:4])   # load and thread start-up, untimed
    t0 = time.perf_counter()
    oracle.direct(w.Q[:, :, :w.T_prefill], w.K[:, :, :w.T_prefill], w.V[:, :, :w.T_prefill],
                  w.L, w.group, w.eps, rows=probe)
    per_row = (time.perf_counter() - t0) / probe.size
    n = int(min(total_rows, max(probe.size, target_s / max(per_row, 1e-9))))
    if max_rows:
        n = min(n, max_rows)
    rows = np.unique(np.linspace(0, total_rows - 1, n).astype(np.int64))
    t0 = time.perf_counter()
    oracle.direct(w.Q[:, :, :w.T_prefill], w.K[:, :, :w.T_prefill], w.V[:, :, :w.T_prefill],
                  w.L, w.group, w.eps, rows=rows)
    dt = time.perf_counter() - t0
    tokens_per_s = rows.size / w.Hq / dt
    return {"value": tokens_per_s, "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": "%d of %d query rows (uniform stride over batch x heads x tokens) of "
                      "the %s prefill; tokens/s = rows / Hq / time"
                      % (rows.size, total_rows, workload_label(w))}


def run_reference(args, world, rank):
    if rank != 0:
        return
    from grouped_quadratic_gb300 import inputs
    w = inputs.config(args.config, decode_steps=1, T=inputs.CONFIGS[args.config]["T"] + 1)
    per_step = max(2.0, min(20.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    vals, secs = [], 0.0
    last = None
    for _ in range(args.steps):
        last = oracle_sample(w, per_step)
        vals.append(last["value"])
        secs += last["seconds"]
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * secs / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.layout, args.chunk),
            "cpu_baseline": {"kind": "oracle", "cores": last["cores"], "value": value,
                             "unit": "tokens/s", "sample": last["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_label(w):
    """e.g. "llama-3.2-1b-prefill+1-decode B4 Hq32 Hkv8 T8192+1 d64 G6"."""
    return ("%s+1-decode B%d Hq%d Hkv%d T%d+1 d64 G%d"
            % (w.name.split()[0], w.B, w.Hq, w.Hkv, w.T_prefill, w.G))


def workload_config(w, layout, chunk):
    return {"workload": workload_label(w),
            "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T_prefill, "decode_tokens": 1,
            "d": 64, "dv": 64, "G": w.G, "state_layout": layout, "chunk": chunk,
            "l2": "flushed (256 MiB write) before every timed step",
            "seed": w.seed}


# ----------------------------------------------------------------- GPU legs
def algorithmic_flops(B, Hq, Hkv, T, chunk):
    """Algorithmic FLOPs of one prefill call, per step of the method (packed
    state, F_p = 2145 features; MMA padding and repeated passes not credited)."""
    readout = 2.0 * B * T * Hq * F_PACKED * U            # Phi~(Q) S_{c-1}
    intra = float(B) * T * Hq * chunk * (D + U)          # causal half of the C x C tile
    update = 2.0 * B * T * Hkv * F_PACKED * U            # phi(K)^T [V | 1]
    return {"readout": readout, "intra": intra, "update": update,
            "total": readout + intra + update}


def kernel_work(name, fl):
    """(algorithmic FLOPs per prefill call, tensor-core?) credited to a kernel."""
    if "readout" in name:
        return fl["readout"] if "tc_" in name else fl["readout"] + fl["intra"], "tc_" in name
    if "intra" in name:
        return fl["intra"], True
    if "state" in name or "delta" in name or "scan" in name:
        return fl["update"], "tc_" in name
    return 0.0, False


def e2e_pieces(B, Hkv):
    """The end-to-end pipeline's pieces (sequence, first KV head, KV heads):
    whole sequences, the last one split into groups of 4 KV heads (a multiple
    of 4 keeps every state slice 16-byte aligned) so that the work left after
    the last input lands is small."""
    split = 4 if Hkv % 4 == 0 and Hkv > 4 else Hkv
    return [(bb, 0, Hkv) for bb in range(B - 1)] + \
        [(B - 1, g, split) for g in range(0, Hkv, split)]


class PrefillBench:
    """One prefill workload on the device: inputs resident in HBM, the step
    (expand + prefill + one decode token) callable directly or from a graph."""

    def __init__(self, cfg_idx, chunk, layout_name, dev, stream):
        import torch
        from grouped_quadratic_gb300 import inputs, oal
        self.oal = oal
        self.dev, self.stream = dev, stream
        self.layout_name = layout_name
        self.layout = oal.OAL_STATE_PACKED if layout_name == "packed" else oal.OAL_STATE_FULL
        cfg = inputs.CONFIGS[cfg_idx]
        w = inputs.config(cfg_idx, T=cfg["T"] + 1, decode_steps=1)
        self.w = w
        Tp = w.T_prefill
        self.Tp = Tp
        self.chunk = chunk
        Qh, Kh, Vh = w.torch_inputs("cpu")
        self.host = (Qh, Kh, Vh)
        self.Q = Qh[:, :, :Tp].contiguous().to(dev)
        self.K = Kh[:, :, :Tp].contiguous().to(dev)
        self.V = Vh[:, :, :Tp].contiguous().to(dev)
        self.q1 = Qh[:, :, Tp].contiguous().to(dev)
        self.k1 = Kh[:, :, Tp].contiguous().to(dev)
        self.v1 = Vh[:, :, Tp].contiguous().to(dev)
        self.L = torch.from_numpy(w.L).to(dev)
        self.group = torch.from_numpy(w.group).to(dev)
        self.dt = oal.OAL_BF16 if w.dtype == "bf16" else oal.OAL_F32
        B, Hq, Hkv = w.B, w.Hq, w.Hkv
        self.a = torch.empty(Hq, device=dev)
        self.b = torch.empty(Hq, D, device=dev)
        self.C = torch.empty(Hq, oal.oal_coeff_table_elems(D, self.layout), device=dev)
        self.state = torch.empty(B, Hkv, oal.oal_state_rows(D, self.layout), U, device=dev)
        self.Y = torch.empty(B, Hq, Tp, D, dtype=self.Q.dtype, device=dev)
        self.y1 = torch.empty(B, Hq, D, dtype=self.Q.dtype, device=dev)
        self.ws_p = torch.empty(max(256, oal.oal_prefill_workspace_bytes(
            B, Hq, Hkv, Tp, D, D, self.dt, self.layout, chunk)), dtype=torch.uint8, device=dev)
        self.pieces = e2e_pieces(B, Hkv)
        self.ws_e2e = [torch.empty(max(256, oal.oal_prefill_workspace_bytes(
            1, Hq, Hkv, Tp, D, D, self.dt, self.layout, chunk)),
            dtype=torch.uint8, device=dev) for _ in range(2)]
        self.ws_d = torch.empty(max(256, oal.oal_decode_workspace_bytes(B, Hq, Hkv, D, D,
                                                                        self.layout)),
                                dtype=torch.uint8, device=dev)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    @property
    def tokens_per_step(self):
        return self.w.B * (self.Tp + 1)

    def step(self, st=None):
        oal, w = self.oal, self.w
        st = self.stream if st is None else st
        oal.oal_expand_coeffs(self.L, self.group, w.eps, self.layout, self.a, self.b, self.C,
                              stream=st)
        oal.oal_prefill(self.Q, self.K, self.V, self.L, self.group, w.eps, self.a, self.b,
                        self.C, self.layout, state=self.state, Y=self.Y, chunk=self.chunk,
                        workspace=self.ws_p, stream=st)
        oal.oal_decode_step(self.q1, self.k1, self.v1, self.a, self.b, self.C, self.state,
                            self.layout, y=self.y1, workspace=self.ws_d, stream=st)

    def timed(self, steps, warmup, lib, world=1, clocks=None):
        """Graph-replayed timed steps; returns (ms per step list, launches per step)."""
        import torch
        stream = self.stream
        for _ in range(warmup):
            self.flush.zero_()
            self.step()
        self.oal.oal_sync_status()
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        c0 = lib.oal_launch_counter()
        with torch.cuda.graph(graph):
            self.step(torch.cuda.current_stream())
        launches_per_step = lib.oal_launch_counter() - c0
        for _ in range(warmup):
            self.flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        self.oal.oal_sync_status()
        barrier(world)
        torch.cuda.synchronize()
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for s in range(steps):
            self.flush.zero_()
            ev0[s].record(stream)
            graph.replay()
            ev1[s].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        self.oal.oal_sync_status()
        del graph
        return [ev0[s].elapsed_time(ev1[s]) for s in range(steps)], launches_per_step

    def per_kernel(self, steps, lib):
        """Per-kernel device ms per prefill call: a second pass with CUDA
        events recorded between the prefill's launches (the C ABI's timing
        hook, on the launching stream).  The events serialise the launches,
        so these are upper bounds of the times inside the graph-replayed steps."""
        import ctypes

        import torch
        oal, w, stream = self.oal, self.w, self.stream
        n_ev = 12
        kev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
        for evs in kev:
            for e in evs:
                e.record(stream)
        torch.cuda.synchronize()
        ev_arrays = [(ctypes.c_void_p * n_ev)(*[e.cuda_event for e in evs]) for evs in kev]
        names = None
        for s in range(steps):
            self.flush.zero_()
            oal.oal_expand_coeffs(self.L, self.group, w.eps, self.layout, self.a, self.b,
                                  self.C, stream=stream)
            lib.oal_set_launch_events(ev_arrays[s], n_ev)
            oal.oal_prefill(self.Q, self.K, self.V, self.L, self.group, w.eps, self.a, self.b,
                            self.C, self.layout, state=self.state, Y=self.Y, chunk=self.chunk,
                            workspace=self.ws_p, stream=stream)
            nk = lib.oal_last_call_launches()
            names = [lib.oal_last_call_launch_name(i).decode() for i in range(nk)]
            lib.oal_set_launch_events(None, 0)
        torch.cuda.synchronize()
        oal.oal_sync_status()
        nk = min(len(names), n_ev - 1)
        per_call, launches = {}, {}
        for k in range(nk):
            launches[names[k]] = launches.get(names[k], 0) + 1
        for s in range(steps):
            acc = {}
            for k in range(nk):
                acc[names[k]] = acc.get(names[k], 0.0) + kev[s][k].elapsed_time(kev[s][k + 1])
            for k, v in acc.items():
                per_call.setdefault(k, []).append(v)
        return {k: statistics.mean(v) for k, v in per_call.items()}, launches

    def roofline(self, pk, launches, step_ms, pks):
        w = self.w
        chunk = self.chunk if self.chunk else (128 if self.dt == self.oal.OAL_BF16 else 64)
        fl = algorithmic_flops(w.B, w.Hq, w.Hkv, self.Tp, chunk)
        cands = [k for k in pk if kernel_work(k, fl)[0] > 0]
        dom = max(cands, key=pk.get)
        work, tensor = kernel_work(dom, fl)
        achieved = work / (pk[dom] / 1000.0) / 1e12
        peak = pks["bf16_tflops"] if tensor else FP32_SIMT_PEAK_TFLOPS
        key = (w.B, w.Hq, w.Hkv, self.Tp, w.G, self.layout_name, chunk)
        nbytes = traffic_for(dom, key)
        kernel_ms = pk[dom] / launches[dom]
        return {"bound": "tensor" if tensor else "alu", "kernel": dom,
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": nbytes,
                "traffic_unit": "DRAM bytes per launch (ncu dram__bytes_read.sum + "
                                "dram__bytes_write.sum, cold cache)",
                "peak_source": ("measured bf16 burst (MEASURED_PEAKS.json)" if tensor else
                                "fp32 CUDA-core FMA peak: 152 SMs x 128 lanes x 2 x 2.07 GHz"),
                "kernel_ms_per_call": pk[dom],
                "kernel_ms_per_launch": kernel_ms,
                "kernel_launches_per_call": launches[dom],
                "kernel_share": pk[dom] / statistics.mean(step_ms),
                "per_kernel_timing": "second pass, CUDA events between launches",
                "per_kernel_ms_per_call": pk,
                "launches_per_call": launches,
                "algorithmic_flops_per_call": work,
                "prefill_total": {"algorithmic_flops": fl["total"],
                                  "device_ms": sum(pk.values()),
                                  "achieved_tflops": fl["total"] / (sum(pk.values()) / 1e3) / 1e12,
                                  "frac": fl["total"] / (sum(pk.values()) / 1e3) / 1e12 /
                                          pks["bf16_tflops"]}}

    def e2e(self, steps, warmup, world):
        """Step through the C ABI with host buffers: pinned host->device copies
        of every input and device->host copies of the outputs inside the timed
        region.  The prefill runs one call per piece (self.pieces: a sequence's
        KV heads with their query heads; pieces are independent), on two
        compute streams in turn, so later pieces' inputs copy in on one stream
        and earlier pieces' outputs copy out on another while pieces compute.
        The host link is the bound; the small last pieces shorten the compute
        and copy-out left after the last input lands."""
        import torch
        oal, w = self.oal, self.w
        stream, Tp, B = self.stream, self.Tp, w.B
        Qh, Kh, Vh = self.host
        Qp, Kp, Vp = (t[:, :, :Tp].contiguous().pin_memory() for t in (Qh, Kh, Vh))
        q1p, k1p, v1p = (t[:, :, Tp].contiguous().pin_memory() for t in (Qh, Kh, Vh))
        Lp = torch.from_numpy(w.L).pin_memory()
        gp = torch.from_numpy(w.group).pin_memory()
        Yp = torch.empty(self.Y.shape, dtype=self.Y.dtype).pin_memory()
        y1p = torch.empty(self.y1.shape, dtype=self.y1.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (Qp, Kp, Vp, q1p, k1p, v1p, Lp, gp))
        d2h = Yp.numel() * Yp.element_size() + y1p.numel() * y1p.element_size()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        sc = [torch.cuda.Stream(), torch.cuda.Stream()]
        rho = w.Hq // w.Hkv
        pieces = self.pieces

        def e2e_step(ev_start):
            cin.wait_event(ev_start)
            with torch.cuda.stream(cin):
                self.L.copy_(Lp, non_blocking=True)
                self.group.copy_(gp, non_blocking=True)
                e_par = torch.cuda.Event()
                e_par.record(cin)
                e_in = []
                for bb, k0, nk in pieces:
                    hs, ks = slice(k0 * rho, (k0 + nk) * rho), slice(k0, k0 + nk)
                    self.Q[bb, hs].copy_(Qp[bb, hs], non_blocking=True)
                    self.K[bb, ks].copy_(Kp[bb, ks], non_blocking=True)
                    self.V[bb, ks].copy_(Vp[bb, ks], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(cin)
                    e_in.append(e)
                for dst, src in ((self.q1, q1p), (self.k1, k1p), (self.v1, v1p)):
                    dst.copy_(src, non_blocking=True)
                e_tok = torch.cuda.Event()
                e_tok.record(cin)
            stream.wait_event(e_par)
            oal.oal_expand_coeffs(self.L, self.group, w.eps, self.layout, self.a, self.b,
                                  self.C, stream=stream)
            e_coef = torch.cuda.Event()
            e_coef.record(stream)
            e_done = []
            for i, (bb, k0, nk) in enumerate(pieces):
                s2 = sc[i % 2]
                hs, ks = slice(k0 * rho, (k0 + nk) * rho), slice(k0, k0 + nk)
                s2.wait_event(e_coef)
                s2.wait_event(e_in[i])
                oal.oal_prefill(self.Q[bb:bb + 1, hs], self.K[bb:bb + 1, ks],
                                self.V[bb:bb + 1, ks], self.L[hs], self.group[hs], w.eps,
                                self.a[hs], self.b[hs], self.C[hs], self.layout,
                                state=self.state[bb:bb + 1, ks], Y=self.Y[bb:bb + 1, hs],
                                chunk=self.chunk, workspace=self.ws_e2e[i % 2], stream=s2)
                e = torch.cuda.Event()
                e.record(s2)
                e_done.append(e)
                cout.wait_event(e)
                with torch.cuda.stream(cout):
                    Yp[bb, hs].copy_(self.Y[bb, hs], non_blocking=True)
            for e in e_done[-2:]:
                stream.wait_event(e)
            stream.wait_event(e_tok)
            oal.oal_decode_step(self.q1, self.k1, self.v1, self.a, self.b, self.C, self.state,
                                self.layout, y=self.y1, workspace=self.ws_d, stream=stream)
            e = torch.cuda.Event()
            e.record(stream)
            cout.wait_event(e)
            with torch.cuda.stream(cout):
                y1p.copy_(self.y1, non_blocking=True)
            e_out = torch.cuda.Event()
            e_out.record(cout)
            stream.wait_event(e_out)

        for _ in range(warmup):
            e = torch.cuda.Event()
            e.record(stream)
            e2e_step(e)
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world)
        for s in range(steps):
            self.flush.zero_()
            es[s].record(stream)
            e2e_step(es[s])
            ee[s].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_s = max_over_ranks(sum(es[s].elapsed_time(ee[s]) for s in range(steps)) / 1e3,
                               world)
        return {"value": self.tokens_per_step * world * steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1e3 * e2e_s / steps,
                "pipeline": "one prefill call per piece on two compute streams in turn, "
                            "copies in and out on two more streams; pieces: %s" % ", ".join(
                                "(seq %d, KV heads %d..%d)" % (bb, k0, k0 + nk - 1)
                                for bb, k0, nk in self.pieces)}


def measure_prefill(cfg_idx, chunk, layout, steps, warmup, dev, stream, lib, pks, world=1,
                    with_e2e=False):
    import torch
    pb = PrefillBench(cfg_idx, chunk, layout, dev, stream)
    step_ms, launches_per_step = pb.timed(steps, warmup, lib, world)
    total_s = max_over_ranks(sum(step_ms) / 1000.0, world)
    pk, launches = pb.per_kernel(steps, lib)
    out = {"workload": workload_label(pb.w), "config": workload_config(pb.w, layout, chunk),
           "value": pb.tokens_per_step * world * steps / total_s, "unit": "tokens/s",
           "ms_per_step": 1e3 * total_s / steps,
           "step_ms": step_ms,
           "roofline": pb.roofline(pk, launches, step_ms, pks),
           "gpu_launches": int(launches_per_step * steps),
           "launches_per_step": int(launches_per_step)}
    if with_e2e:
        out["e2e"] = pb.e2e(steps, warmup, world)
    out["_w"] = pb.w
    del pb
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import torch
    from grouped_quadratic_gb300 import build as gq_build
    from grouped_quadratic_gb300 import oal

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    gq_build.build()
    lib = oal.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    pks = peaks()
    gpu_id = "GPU-%s" % torch.cuda.get_device_properties(dev).uuid

    with ClockSampler(gpu_id) as clk:
        head = measure_prefill(args.config, args.chunk, args.layout, args.steps, args.warmup,
                               dev, stream, lib, pks, world, with_e2e=not args.no_e2e)
    w = head.pop("_w")

    subs = {}
    if not args.no_sub:
        with ClockSampler(gpu_id) as clk_sub:
            if args.config != 1:
                r = measure_prefill(1, 0, args.layout, args.steps, args.warmup, dev, stream,
                                    lib, pks, world)
                r.pop("_w")
                subs["config1"] = r
            sweep = {}
            for ch in (64, 128, 256):
                r = measure_prefill(4, ch, args.layout, max(3, args.steps // 2), args.warmup,
                                    dev, stream, lib, pks, world)
                r.pop("_w")
                sweep[str(ch)] = r
            subs["config4"] = {"chunk_sweep": sweep}
        subs["clocks"] = clk_sub.summary()

    decode = None
    if not args.no_decode:
        decode = {lay: run_decode(args, world, dev, stream, lib, pks, lay)
                  for lay in ("full", "packed")}
    calib = run_contribution(args, world, dev, stream, lib, pks) if args.contribution else None
    backward = None if args.no_backward else run_backward(args, world, dev, stream, lib, pks)
    groups = None if args.no_sub else run_group_counts(args, world, dev, stream, lib, pks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, args.cpu_seconds)

    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu,
            "e2e": head.get("e2e"), "gpu_launches": head["gpu_launches"],
            "clocks": clk.summary(), "decode": decode, "peaks_source": pks["source"]}
    line.update(subs)
    if backward is not None:
        line["backward"] = backward
    if groups is not None:
        line["group_counts"] = groups
    if calib is not None:
        line["calibration"] = calib
    line["config"]["launch"] = "one step captured as a CUDA graph, replayed per timed step"
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_contribution(args, world, dev, stream, lib, pks):
    """Contribution scores (the calibration step before the path) on 40
    prompts of 4096 tokens, Qwen-shaped heads: one pass over Q and K."""
    import torch
    from grouped_quadratic_gb300 import oal
    P, Hq, Hkv, T = 40, 14, 2, 4096
    g = torch.Generator(device="cpu").manual_seed(20261005)
    Q = torch.randn(P, Hq, T, D, generator=g).to(torch.bfloat16).to(dev)
    K = torch.randn(P, Hkv, T, D, generator=g).to(torch.bfloat16).to(dev)
    chi = torch.empty(P, Hq, D, dtype=torch.float32, device=dev)
    ws = torch.empty(oal.oal_contribution_workspace_bytes(P, Hq, Hkv, T), dtype=torch.uint8,
                     device=dev)

    def call():
        oal.oal_contribution_scores(Q, K, chi=chi, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        call()
    oal.oal_sync_status()
    n = 20
    c0 = lib.oal_launch_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = lib.oal_launch_counter() - c0
    oal.oal_sync_status()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world) / n
    nbytes = (Q.numel() + K.numel()) * 2 + chi.numel() * 4
    gbs = nbytes / secs / 1e9
    return {"workload": "contribution scores P%d Hq%d Hkv%d T%d d64 bf16 (inputs %.0f MB > L2)"
                        % (P, Hq, Hkv, T, nbytes / 1e6),
            "ms_per_call": 1e3 * secs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pks["hbm_gbs"], "algorithmic_bytes_per_call": nbytes},
            "gpu_launches": int(launches)}


def run_group_counts(args, world, dev, stream, lib, pks):
    """Prefill time per head on the Qwen2.5-0.5B shape (B=1, Hq=14, Hkv=2,
    T=4096, bf16) for one global group (G = 1), the grouped kernel at G = 5, and
    a launch of G = 5 where heads keep 1 to 5 groups (the others empty)."""
    import torch
    from grouped_quadratic_gb300 import inputs, oal
    out = {}
    for name, G, mixed in (("G1", 1, False), ("G5", 5, False), ("G5_mixed_1_to_5", 5, True)):
        w = inputs.make_workload("qwen-shape G%d" % G, B=1, Hq=14, Hkv=2, T=4096, G=G,
                                 seed=inputs.SEED_BASE + 20 + G)
        if mixed:
            for h in range(w.Hq):
                w.group[h][w.group[h] > 1 + h % 5] = 1
        Q, K, V = w.torch_inputs(dev)
        L = torch.from_numpy(w.L).to(dev)
        group = torch.from_numpy(w.group).to(dev)
        layout = oal.OAL_STATE_PACKED
        a, b, C = oal.oal_expand_coeffs(L, group, w.eps, layout)
        state = torch.empty(w.B, w.Hkv, oal.oal_state_rows(D, layout), U, device=dev)
        Y = torch.empty_like(Q)
        ws = torch.empty(oal.oal_prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.T, layout=layout),
                         dtype=torch.uint8, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def call():
            oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout, state=state, Y=Y,
                            workspace=ws, stream=stream)

        for _ in range(3):
            call()
        oal.oal_sync_status()
        n = max(3, args.steps)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        barrier(world)
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        oal.oal_sync_status()
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        out[name] = {"ms_per_call": ms, "us_per_head": 1e3 * ms / w.Hq,
                     "tokens_per_s": w.B * w.T / (ms / 1e3)}
        del Q, K, V, ws, flush
        torch.cuda.empty_cache()
    out["workload"] = "qwen2.5-0.5b-shaped prefill B1 Hq14 Hkv2 T4096 bf16, packed state"
    return out


def run_backward(args, world, dev, stream, lib, pks):
    """Prefill backward (dQ, dK, dV, dL) on the Qwen2.5-0.5B-shaped workload."""
    import torch
    from grouped_quadratic_gb300 import inputs, oal
    w = inputs.config(1)
    Q, K, V = w.torch_inputs(dev)
    g = torch.Generator(device="cpu").manual_seed(20261011)
    dY = torch.randn(Q.shape, generator=g).to(Q.dtype).to(dev)
    L = torch.from_numpy(w.L).to(dev)
    group = torch.from_numpy(w.group).to(dev)
    dQ = torch.empty(Q.shape, dtype=torch.float32, device=dev)
    dK = torch.empty(K.shape, dtype=torch.float32, device=dev)
    dV = torch.empty(V.shape, dtype=torch.float32, device=dev)
    dL = torch.empty(w.L.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(oal.oal_prefill_backward_workspace_bytes(w.B, w.Hq, w.Hkv, w.T),
                     dtype=torch.uint8, device=dev)

    def call():
        oal.oal_prefill_backward(Q, K, V, dY, L, group, w.eps, dQ, dK, dV, dL, workspace=ws,
                                 stream=stream)

    for _ in range(2):
        call()
    oal.oal_sync_status()
    n = 3
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    c0 = lib.oal_launch_counter()
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = lib.oal_launch_counter() - c0
    oal.oal_sync_status()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world) / n
    pairs = w.B * w.Hq * w.T * (w.T + 1) / 2
    # per causal pair: the group sums, dY . v, dQ, dK and dV (5 x 64 multiply-adds) and
    # the recomputed forward numerator and group sums (2 x 64): 7 x 128 FLOPs
    flops = pairs * 7 * 128
    achieved = flops / secs / 1e12
    return {"workload": "qwen2.5-0.5b-prefill backward B%d Hq%d Hkv%d T%d d64 G%d bf16 "
                        "(dQ, dK, dV, dL)" % (w.B, w.Hq, w.Hkv, w.T, w.G),
            "ms_per_call": 1e3 * secs, "tokens_per_s": world * w.B * w.T / secs,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": FP32_SIMT_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / FP32_SIMT_PEAK_TFLOPS,
                         "peak_source": "fp32 CUDA-core FMA peak: 152 SMs x 128 lanes x 2 x "
                                        "2.07 GHz",
                         "algorithmic_flops_per_call": flops},
            "gpu_launches": int(launches)}


def run_decode(args, world, dev, stream, lib, pks, layout_name):
    """Decode workload: B=64, Hq=14, Hkv=2, 2048-token prefill then decode steps."""
    import torch
    from grouped_quadratic_gb300 import inputs, oal
    n_steps = args.decode_steps
    w = inputs.config(3, T=2048 + n_steps, decode_steps=n_steps)
    layout = oal.OAL_STATE_FULL if layout_name == "full" else oal.OAL_STATE_PACKED
    Tp = w.T_prefill
    Qh, Kh, Vh = w.torch_inputs("cpu")
    Q = Qh[:, :, :Tp].contiguous().to(dev)
    K = Kh[:, :, :Tp].contiguous().to(dev)
    V = Vh[:, :, :Tp].contiguous().to(dev)
    qd = Qh[:, :, Tp:].permute(2, 0, 1, 3).contiguous().to(dev)   # [steps, B, Hq, 64]
    kd = Kh[:, :, Tp:].permute(2, 0, 1, 3).contiguous().to(dev)
    vd = Vh[:, :, Tp:].permute(2, 0, 1, 3).contiguous().to(dev)
    L = torch.from_numpy(w.L).to(dev)
    group = torch.from_numpy(w.group).to(dev)
    a, b, C = oal.oal_expand_coeffs(L, group, w.eps, layout)
    _, state = oal.oal_prefill(Q, K, V, L, group, w.eps, a, b, C, layout)
    del Q, K, V
    y = torch.empty(n_steps, w.B, w.Hq, D, dtype=qd.dtype, device=dev)
    ws = torch.empty(oal.oal_decode_workspace_bytes(w.B, w.Hq, w.Hkv, D, D, layout),
                     dtype=torch.uint8, device=dev)
    for t in range(min(3, n_steps)):     # warm-up on a copy of the state
        s2 = state.clone()
        oal.oal_decode_step(qd[t], kd[t], vd[t], a, b, C, s2, layout, y=y[t], workspace=ws)
    del s2
    oal.oal_sync_status()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    c0 = lib.oal_launch_counter()
    e0.record(stream)
    for t in range(n_steps):
        oal.oal_decode_step(qd[t], kd[t], vd[t], a, b, C, state, layout, y=y[t], workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = lib.oal_launch_counter() - c0
    oal.oal_sync_status()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    F = F_FULL if layout == oal.OAL_STATE_FULL else F_PACKED
    state_bytes = w.B * w.Hkv * F * U * 4
    io_bytes = (w.B * w.Hq * D * 2 + 2 * w.B * w.Hkv * D) * qd.element_size()
    bytes_per_step = 2 * state_bytes + io_bytes
    gbs = bytes_per_step * n_steps / secs / 1e9
    key = (w.B, w.Hq, w.Hkv, layout_name)
    dk = "decode_stream_kernel"
    nbytes = traffic_for(dk, key)
    out = {"workload": "qwen2.5-0.5b-decode B%d Hq%d Hkv%d prefill %d then %d steps, %s state"
                       % (w.B, w.Hq, w.Hkv, Tp, n_steps, layout_name),
           "steps_per_s": world * n_steps / secs, "ms_per_step": 1e3 * secs / n_steps,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pks["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / pks["hbm_gbs"],
                        "traffic": nbytes, "traffic_kernel": dk,
                        "traffic_unit": "DRAM bytes per launch (ncu, cold cache)",
                        "algorithmic_bytes_per_step": bytes_per_step},
           "gpu_launches": int(launches),
           "l2": "state set %.0f MB vs 126 MB L2" % (state_bytes / 1e6)}
    if nbytes:
        out["roofline"]["dram_frac"] = nbytes / (secs / n_steps) / 1e9 / pks["hbm_gbs"]
    del state, qd, kd, vd
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 4])
    ap.add_argument("--layout", choices=["packed", "full"], default="packed")
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the config-1 and config-4 sub-lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--contribution", action="store_true",
                    help="also time the contribution scores (calibration step)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
