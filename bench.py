"""Benchmark of the NF4 quantize + fused NF4-dequant matmul path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
for the default workload (a Qwen2.5-7B-shaped decoder layer, seven linear
weights) it quantizes every fp32 weight (NF4, blocksize 64, double quant),
runs the fused forward of every projection at M = 1, 64 and 2048 tokens and
the fused input gradient at M = 2048. The printed `value` is the step's
matmul FLOP divided by the device time of the step (quantization included in
the time); per-kernel-class numbers, their roofline fractions and the
quantize bandwidth are in `parts`.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

`--impl reference` times the CPU oracle (the plain fp64 reference the kernels
are checked against) on a bounded sample of the same workload on this host's
cores. Under torchrun each rank runs its own replica (weak scaling) and rank 0
prints one JSON line with the max time over ranks.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dequant_gemm_gb300 import workloads as wl  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def traffic_per_launch(workload, category):
    """Mean DRAM bytes (read + write) per launch of a kernel class, from the
    committed ncu capture for this workload, or None when there is none or the
    CUDA sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals, stamp, files = [], None, []
    for line in open(path):
        if line.startswith("# sources_sha256"):
            # "# sources_sha256 <digest> <file> ...": the files that define
            # the captured kernel, relative to the CUDA source folder
            f = line.split()
            stamp, files = f[2], f[3:]
        elif line.strip() and not line.startswith("#"):
            f = line.split()
            if f[0] == category:
                vals.append(int(f[2]) + int(f[3]))
    if stamp is None or not files or not vals:
        return None
    if stamp != sources_digest(files):
        return None
    return sum(vals) / len(vals)


def sources_digest(files):
    """sha256 over the named CUDA source files, in the order given."""
    import hashlib
    d = os.path.join(ROOT, "dequant_gemm_gb300", "csrc")
    return hashlib.sha256(b"".join(open(os.path.join(d, f), "rb").read() for f in files)).hexdigest()


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


# ----------------------------------------------------------- work accounting --
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


def packed_bytes(rows, cols, wdtype="nf4"):
    """Stored bytes of a quantized weight: 4-bit codes + uint8 absmax codes +
    fp32 group scales, or int8 values + fp32 block absmax."""
    n = rows * cols
    nb = n // 64
    if wdtype == "int8":
        return n + 4 * nb
    return n // 2 + nb + 4 * ((nb + 255) // 256)


SMALL_M = 16    # forwards up to this many tokens take the streaming small-M kernel
GROUP_SMALL_M = True   # projections sharing an input take one grouped small-M launch
PARALLEL_TC = True     # tensor-core calls of projections sharing an input on parallel streams


def fwd_work(p, M, w=None):
    """(flop, algorithmic bytes) of Y = X W^T: packed W + X in + Y out."""
    wd, a, o = (w.wdtype, w.act, w.out) if w else ("nf4", "bf16", "f32")
    return 2 * M * p.rows * p.cols, (packed_bytes(p.rows, p.cols, wd) + ELEM_BYTES[a] * M * p.cols
                                     + ELEM_BYTES[o] * M * p.rows)


def dx_work(p, M, w=None):
    wd, a, o = (w.wdtype, w.act, w.out) if w else ("nf4", "bf16", "f32")
    return 2 * M * p.rows * p.cols, (packed_bytes(p.rows, p.cols, wd) + ELEM_BYTES[a] * M * p.rows
                                     + ELEM_BYTES[o] * M * p.cols)


def quant_bytes(p, w=None):
    wd, wi = (w.wdtype, w.w_in) if w else ("nf4", "f32")
    return ELEM_BYTES[wi] * p.rows * p.cols + packed_bytes(p.rows, p.cols, wd)


# --------------------------------------------------------------------- clocks --
class NvmlClockSampler:
    """SM clock and clock-event reasons, read through NVML (the driver's
    libnvidia-ml, read-only queries) every ~1 ms from a thread, so that a timed
    region of a few tens of milliseconds still gets samples of its own."""

    # clock-event (throttle) reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.samples = []
        self.window = None
        self.stop_flag = False
        self.thread = None

    def _poll(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            t = time.perf_counter()
            if (self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ct.byref(clk)) == 0
                    and self.reason_fn(self.handle, ct.byref(rs)) == 0):
                self.samples.append((t, float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        import threading
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        time.sleep(0.01)   # polling before the timed region begins

    def mark(self, t0, t1):
        """The host-side bounds of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        self.stop_flag = True
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()
        t0, t1 = self.window if self.window else (-1e30, 1e30)
        inside = [(c, r) for (t, c, r) in self.samples if t0 <= t <= t1]
        if not inside:
            return None
        reasons = sorted({name for _, r in inside for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "source": "nvml, ~1 ms"}


class ClockSampler:
    """nvidia-smi sampling every 200 ms (fallback when NVML cannot be loaded)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"nf4_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0, t1):
        pass

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax = max(smax, float(f[2]))
                except ValueError:
                    continue
                for name, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
            os.unlink(self.path)
        except OSError:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms"}


def clock_sampler(index):
    try:
        return NvmlClockSampler(index)
    except (OSError, AttributeError):
        return ClockSampler(index)


# -------------------------------------------------------------- our workload --
class Step:
    """Device buffers and the call list of one step of a workload."""

    def __init__(self, name, device, rotate=1):
        import dequant_gemm_gb300 as nf4
        self.nf4 = nf4
        self.w = wl.WORKLOADS[name]
        self.dev = device
        self.rotate = rotate
        self.weights = []       # fp32 weights (inputs of quantize)
        self.q = []             # quantized weights, one set per rotation copy
        self.x = {}             # (K, M) -> bf16 activations
        self.dy = {}            # (N, M) -> bf16 output gradients
        self.y = {}             # (proj index, M) -> fp32 outputs
        self.dx = {}
        w = self.w
        act_dt, out_dt = TORCH_DT[w.act], TORCH_DT[w.out]
        for i, p in enumerate(self.w.projections):
            W = p.make_weight().to(TORCH_DT[w.w_in]).to(device)
            self.weights.append(W)
        # with rotation, every copy of the quantized weight has its own copy of
        # the input weight, so that quantize also reads from HBM
        self.wcopies = [self.weights] + [[W.clone() for W in self.weights] for _ in range(rotate - 1)]
        for r in range(rotate):
            self.q.append([nf4.nf4_quantize(W, dtype=w.wdtype) for W in self.wcopies[r]])
        for i, p in enumerate(self.w.projections):
            for M in self.w.fwd_m:
                if (p.cols, M) not in self.x:
                    self.x[(p.cols, M)] = wl.activations(M, p.cols, std=self.w.x_std,
                                                         seed=wl.SEED_X + M, dtype=act_dt).to(device)
                self.y[(i, M)] = torch.empty(M, p.rows, dtype=out_dt, device=device)
            for M in self.w.dx_m:
                if (p.rows, M) not in self.dy:
                    self.dy[(p.rows, M)] = wl.activations(M, p.rows, std=self.w.dy_std,
                                                          seed=wl.SEED_X + 7 + M,
                                                          dtype=act_dt).to(device)
                self.dx[(i, M)] = torch.empty(M, p.cols, dtype=out_dt, device=device)
        self.quantize_in_step = True
        self.group_small_m = GROUP_SMALL_M
        self.parallel_tc = PARALLEL_TC
        self.calls = self._calls()
        self.side = []
        self.graphs = None

    def parallel(self, M):
        """Whether the calls of one input group at M tokens go out on
        parallel streams: the small-M kernel's separate launches (when not
        grouped) and the tensor-core launches (measured faster than one after
        another at 64 and 2048 tokens: the small projections' grids overlap)."""
        return (M <= SMALL_M and not self.group_small_m) or (M > SMALL_M and self.parallel_tc)

    def _calls(self):
        """List of (category, flop, bytes, launches, fn, group, projection) in
        step order.
        Calls with the same group are independent and may be issued together
        (the projections of the layer that share an input); groups run in
        order. With rotating weight copies, one step walks every copy once."""
        nf4 = self.nf4
        calls = []
        P = self.w.projections
        groups = self.w.issue_groups()
        for r in range(self.rotate):
            for i, p in enumerate(P):
                calls.append(("quantize", 0, quant_bytes(p, self.w), 1,
                              lambda r=r, i=i: nf4.nf4_quantize(self.wcopies[r][i], out=self.q[r][i],
                                                                dtype=self.w.wdtype),
                              ("quantize", r), i))
        for M in sorted(self.w.fwd_m, reverse=True):
            for r in range(self.rotate):
                for gi, g in enumerate(groups):
                    if M <= SMALL_M and len(g) > 1 and self.group_small_m:
                        # projections sharing their input: one grouped launch;
                        # X counted once in the algorithmic bytes
                        ps = [P[i] for i in g]
                        f = sum(fwd_work(p, M, self.w)[0] for p in ps)
                        b = sum(fwd_work(p, M, self.w)[1] for p in ps) - \
                            (len(ps) - 1) * ELEM_BYTES[self.w.act] * M * ps[0].cols
                        calls.append((f"fwd_M{M}", f, b, 1,
                                      lambda r=r, g=g, M=M, K=ps[0].cols: nf4.nf4_matmul_fwd_group(
                                          self.x[(K, M)], [self.q[r][i] for i in g],
                                          outs=[self.y[(i, M)] for i in g]),
                                      (f"fwd_M{M}", r, gi), tuple(g)))
                        continue
                    for i in g:
                        p = P[i]
                        f, b = fwd_work(p, M, self.w)
                        tag = (f"fwd_M{M}", r, gi) if self.parallel(M) else (f"fwd_M{M}", r, gi, i)
                        calls.append((f"fwd_M{M}", f, b, 1,
                                      lambda r=r, i=i, M=M, p=p: nf4.nf4_matmul_fwd(
                                          self.x[(p.cols, M)], self.q[r][i], out=self.y[(i, M)]),
                                      tag, i))
        for M in self.w.dx_m:
            for r in range(self.rotate):
                for gi, g in enumerate(groups):
                    for i in g:
                        p = P[i]
                        f, b = dx_work(p, M, self.w)
                        tag = (f"dx_M{M}", r, gi) if self.parallel(M) else (f"dx_M{M}", r, gi, i)
                        calls.append((f"dx_M{M}", f, b, 1,
                                      lambda r=r, i=i, M=M, p=p: nf4.nf4_matmul_bwd_dx(
                                          self.dy[(p.rows, M)], self.q[r][i], out=self.dx[(i, M)]),
                                      tag, i))
        return calls

    def issue(self, idx):
        """Launch calls idx in order; the members of a group go out on
        parallel streams forked from and joined back to the current one, so
        the tail wave of one can share the SMs with the next."""
        main = torch.cuda.current_stream(self.dev)
        runs = []
        for k in idx:
            if runs and runs[-1][0] == self.calls[k][5]:
                runs[-1][1].append(k)
            else:
                runs.append((self.calls[k][5], [k]))
        for _, ks in runs:
            if len(ks) == 1:
                self.calls[ks[0]][4]()
                continue
            while len(self.side) < len(ks):
                self.side.append(torch.cuda.Stream(self.dev))
            for s, k in zip(self.side, ks):
                s.wait_stream(main)
                with torch.cuda.stream(s):
                    self.calls[k][4]()
            for s in self.side[:len(ks)]:
                main.wait_stream(s)

    def blocks(self):
        """Contiguous runs of one category: (category, [call indices])."""
        out = []
        for k, c in enumerate(self.calls):
            if out and out[-1][0] == c[0]:
                out[-1][1].append(k)
            else:
                out.append((c[0], [k]))
        return out

    def capture(self):
        """One CUDA graph per category run, replayed in step order: the timed
        region then measures the kernels, not the Python launch path."""
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            self.run_eager()
        torch.cuda.current_stream(self.dev).wait_stream(side)
        torch.cuda.synchronize(self.dev)
        self.graphs = []
        for cat, idx in self.blocks():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.issue(idx)
            self.graphs.append((cat, idx, g))
        torch.cuda.synchronize(self.dev)

    def flop(self):
        return sum(c[1] for c in self.calls)

    def launches(self):
        return sum(c[3] for c in self.calls)

    def run_eager(self):
        self.issue(range(len(self.calls)))

    def run(self, events=None):
        """Replay the captured step; events[j] brackets graph j."""
        for j, (cat, idx, g) in enumerate(self.graphs):
            if events is not None:
                events[j][0].record()
            g.replay()
            if events is not None:
                events[j][1].record()

    # end to end: host inputs -> device, step, outputs -> host
    def host_buffers(self):
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        self.h_w = [pin(W) for W in self.weights] if self.quantize_in_step else []
        self.h_x = {k: pin(v) for k, v in self.x.items()}
        self.h_dy = {k: pin(v) for k, v in self.dy.items()}
        self.h_y = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in self.y.items()}
        self.h_dx = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in self.dx.items()}
        h2d = sum(t.numel() * t.element_size() for t in
                  self.h_w + list(self.h_x.values()) + list(self.h_dy.values()))
        d2h = sum(t.numel() * t.element_size() for t in
                  list(self.h_y.values()) + list(self.h_dx.values()))
        return h2d, d2h

    def e2e_schedule(self, order):
        """For weights landing in `order`: the turn (index into order) at
        which each call runs, once every weight it reads has landed (a
        grouped call reads several), and the turn at which each output
        ("fwd" or "dx", projection, M) goes back: right after the call that
        writes it."""
        pos = {i: n for n, i in enumerate(order)}
        projs = [c[6] if isinstance(c[6], tuple) else (c[6],) for c in self.calls]
        turn = [max(pos[j] for j in js) for js in projs]
        out_turn = {}
        for c, js, t in zip(self.calls, projs, turn):
            for kind in ("fwd", "dx"):
                if c[0].startswith(kind + "_M"):
                    M = int(c[0][len(kind) + 2:])
                    for j in js:
                        out_turn[(kind, j, M)] = t
        return turn, out_turn

    def run_e2e(self):
        """One step from host inputs to host outputs, streamed by projection:
        the activations and then each weight go in on a copy stream; a
        projection's quantize, forwards and input gradient run as soon as its
        weight has landed, and its outputs go back on a second copy stream
        while later weights are still arriving. The largest weights go first,
        so that what is left after the last copy-in is small. Same work as
        run(); only the order (by projection) and the overlap differ."""
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "cin"):
            self.cin, self.cout = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        cin, cout = self.cin, self.cout
        cin.wait_stream(main)        # the previous step's kernels have read their inputs
        P = self.w.projections
        order = sorted(range(len(P)), key=lambda i: -P[i].rows * P[i].cols)
        with torch.cuda.stream(cin):
            for k, v in self.x.items():
                v.copy_(self.h_x[k], non_blocking=True)
            for k, v in self.dy.items():
                v.copy_(self.h_dy[k], non_blocking=True)
            ev_act = torch.cuda.Event()
            ev_act.record(cin)
            ev_w = {}
            if self.h_w:
                for i in order:
                    self.weights[i].copy_(self.h_w[i], non_blocking=True)
                    ev_w[i] = torch.cuda.Event()
                    ev_w[i].record(cin)
        main.wait_event(ev_act)
        turn, out_turn = self.e2e_schedule(order)
        for n, i in enumerate(order):
            if ev_w:
                main.wait_event(ev_w[i])
            for c, t in zip(self.calls, turn):
                if t == n:
                    c[4]()
            done = torch.cuda.Event()
            done.record(main)
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                for (j, M), v in self.y.items():
                    if out_turn.get(("fwd", j, M)) == n:
                        self.h_y[(j, M)].copy_(v, non_blocking=True)
                for (j, M), v in self.dx.items():
                    if out_turn.get(("dx", j, M)) == n:
                        self.h_dx[(j, M)].copy_(v, non_blocking=True)
        main.wait_stream(cout)


# ------------------------------------------------------------ oracle sample --
_ORACLE_CACHE = {}


def oracle_sample(name, budget_s=15.0):
    """Time the CPU oracle on a bounded sample of the workload: repeated
    passes over the projections; each pass quantizes + dequantizes whole
    16384-weight groups covering a few rows and multiplies those rows in fp64
    against the activations of every forward and dX token count. Stops once
    `budget_s` seconds of oracle work have run.
    Returns (matmul flop/s, description, cores, seconds)."""
    from oracle import nf4_oracle as o
    w = wl.WORKLOADS[name]
    if name not in _ORACLE_CACHE:
        data = []
        for p in w.projections:
            W = p.make_weight().numpy()
            xs = [wl.activations(M, p.cols, std=w.x_std, seed=wl.SEED_X + M).float().numpy()
                  for M in w.fwd_m]
            dys = [wl.activations(M, p.rows, std=w.dy_std).float().numpy() for M in w.dx_m]
            data.append((p, W, xs, dys))
        _ORACLE_CACHE[name] = data
    g = np.random.default_rng(0)
    per_proj = 8
    t_total, flop_total, rows_total, passes = 0.0, 0, 0, 0
    while t_total < budget_s:
        for p, W, xs, dys in _ORACLE_CACHE[name]:
            K = p.cols
            r0 = int(g.integers(0, max(1, p.rows - per_proj)))
            lo = (r0 * K) // 16384 * 16384
            hi = min(((r0 + per_proj) * K + 16383) // 16384 * 16384, p.rows * K)
            t0 = time.perf_counter()
            packed, a8, s2 = o.quantize_flat(W.reshape(-1)[lo:hi])
            what = o.dequantize_flat(packed, a8, s2)
            rows = what[(r0 * K - lo):(r0 * K - lo) + per_proj * K].reshape(per_proj, K)
            for X in xs:
                o.matmul_fwd(X, rows)
                flop_total += 2 * X.shape[0] * per_proj * K
            for dY in dys:
                o.matmul_bwd_dx(dY[:, r0:r0 + per_proj], rows)
                flop_total += 2 * dY.shape[0] * per_proj * K
            t_total += time.perf_counter() - t0
            rows_total += per_proj
        passes += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"{passes} passes, {rows_total} weight rows in all ({per_proj} consecutive rows per "
            f"projection per pass; the whole 16384-weight groups under them quantized + "
            f"dequantized) x every forward and dX token count of {name}; numpy fp64 "
            "(matmuls on the BLAS thread pool = host cores)")
    return flop_total / t_total, desc, cores, t_total


# ------------------------------------------------------------------- helpers --
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    vals, descs, cores = [], None, None
    for _ in range(args.warmup):
        oracle_sample(args.workload, budget_s=1.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, descs, cores, _ = oracle_sample(args.workload, budget_s=5.0)
        vals.append(v)
    dt = time.perf_counter() - t0
    value = statistics.median(vals) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": descs},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = ("fused NF4 matmul TFLOP/s and HBM GB/s vs roofline; nf4_quantize GB/s "
          "(value: matmul FLOP of one layer step / device time of the step, quantization included)")


# The single-GPU workloads beside the default one, each measured into a record
# of its own in the same JSON line (the tiny 256x256 case is a parity case).
CONFIG_WORKLOADS = ("decode_4096", "prefill_up_11008x4096", "bwd_down_4096x11008",
                    "prefill_up_11008x4096_bf16", "bwd_down_4096x11008_f16",
                    "decode_4096_fp4", "decode_4096_int8", "prefill_up_11008x4096_fp4",
                    "prefill_up_11008x4096_int8")


def class_record(flop, nbytes, seconds, pk):
    """Throughput of one kernel class over `seconds` of device time and its
    place under the roofline: the HBM fraction, the tensor fractions against
    the burst and the sustained bf16 peaks, and the fraction of the larger of
    the two roofline times (bytes / copy bandwidth, FLOP / burst peak)."""
    tf = flop / seconds / 1e12
    gbs = nbytes / seconds / 1e9
    t_mem = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tensor = flop / (pk["bf16_tflops"] * 1e12)
    return {"TFLOP/s": tf, "GB/s": gbs, "hbm_frac": gbs / pk["hbm_gbs"],
            "tensor_frac_burst": tf / pk["bf16_tflops"],
            "tensor_frac_sustained": tf / pk["bf16_tflops_sustained"],
            "bound": "tensor" if t_tensor > t_mem else "hbm",
            "roofline_frac": max(t_mem, t_tensor) / seconds}


def measure_workload(name, dev, steps, warmup, world, clocks=False):
    """Build a workload's step, capture it, warm up, and time `steps` steps
    with CUDA events around every kernel-class graph. Inputs larger than L2
    are read once per step; smaller weight sets rotate over enough quantized
    copies to exceed 3x L2."""
    import dequant_gemm_gb300 as nf4
    work = wl.WORKLOADS[name]
    ws_bytes = sum(ELEM_BYTES[work.w_in] * p.rows * p.cols for p in work.projections)
    rotate = 1 if ws_bytes > L2_BYTES else max(2, int(np.ceil(3 * L2_BYTES / sum(
        packed_bytes(p.rows, p.cols, work.wdtype) for p in work.projections))))
    step = Step(name, dev, rotate=rotate)
    stream = torch.cuda.current_stream(dev)
    step.capture()
    for _ in range(warmup):
        step.run()
    status, site = nf4.nf4_poll_device_status_site(dev)
    if status != 0:
        raise SystemExit(f"{name}: device status {status} after warm-up ({nf4.describe_site(site)})")

    ngraphs = len(step.graphs)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(ngraphs * steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = clock_sampler(dev.index) if clocks else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    h0 = time.perf_counter()
    t_start.record(stream)
    for s in range(steps):
        step.run(events[s * ngraphs:(s + 1) * ngraphs])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark(h0, time.perf_counter())
    barrier(world)
    clk = sampler.stop() if sampler else None
    status, site = nf4.nf4_poll_device_status_site(dev)
    if status != 0:
        raise SystemExit(f"{name}: device status {status} after the timed steps ({nf4.describe_site(site)})")

    cat_ms, cat_flop, cat_bytes, cat_n = {}, {}, {}, {}
    for s in range(steps):
        for j, (cat, idx, _) in enumerate(step.graphs):
            e0, e1 = events[s * ngraphs + j]
            cat_ms[cat] = cat_ms.get(cat, 0.0) + e0.elapsed_time(e1)
            for k in idx:
                _, f, b, n, _, _, _ = step.calls[k]
                cat_flop[cat] = cat_flop.get(cat, 0) + f
                cat_bytes[cat] = cat_bytes.get(cat, 0) + b
                cat_n[cat] = cat_n.get(cat, 0) + n
    pk, _ = peaks()
    parts = {}
    for cat in cat_ms:
        rec = {"ms_per_step": cat_ms[cat] / steps, "launches_per_step": cat_n[cat] // steps}
        rec.update(class_record(cat_flop[cat], cat_bytes[cat], cat_ms[cat] * 1e-3, pk))
        parts[cat] = rec

    # the same calls launched one by one from Python, without graphs
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step.run_eager()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = e0.elapsed_time(e1) / steps
    l2 = (("inputs larger than L2: %.2f GB of weights read per step" % (ws_bytes / 1e9))
          if rotate == 1 else f"one step walks {rotate} quantized copies (> 3x L2)")
    return {"work": work, "step": step, "elapsed_ms": t_start.elapsed_time(t_end), "parts": parts,
            "clocks": clk, "l2": l2, "rotate": rotate, "eager_ms_per_step": eager_ms,
            "steps": steps}


def config_record(r):
    """The record of one workload measured beside the default one."""
    work, step = r["work"], r["step"]
    steps_ms = r["elapsed_ms"]
    rec = {"workload": work.name,
           "projections": [f"{p.name} {p.rows}x{p.cols}" for p in work.projections],
           "weight_format": work.wdtype, "weight_in": work.w_in, "activations": work.act,
           "outputs": work.out,
           "fwd_m": list(work.fwd_m), "dx_m": list(work.dx_m), "l2": r["l2"],
           "timing": "CUDA graph per kernel class, CUDA events between graphs",
           "graph_ms_per_step": steps_ms / r["steps"],
           "eager_ms_per_step": r["eager_ms_per_step"],
           "launches_per_step": step.launches(), "classes": {}}
    for cat, p in r["parts"].items():
        c = dict(p)
        n = max(1, p["launches_per_step"])
        c["us_per_launch"] = 1e3 * p["ms_per_step"] / n
        bound = p["bound"]
        c["roofline"] = ({"bound": "hbm", "achieved": p["GB/s"], "unit": "GB/s",
                          "frac": p["hbm_frac"]} if bound == "hbm" else
                         {"bound": "tensor", "achieved": p["TFLOP/s"], "unit": "TFLOP/s",
                          "frac": p["tensor_frac_burst"],
                          "frac_sustained": p["tensor_frac_sustained"]})
        rec["classes"][cat] = c
    if r["clocks"]:
        rec["clocks"] = r["clocks"]
    return rec


def run_naive(args, dev):
    """The fused NF4 forward against the naive path that the pages' speed claim
    compares with: dequantize the whole weight to fp32 in HBM, cast it to bf16,
    then a cuBLAS bf16 matmul (torch.matmul) widened to fp32; and against the
    leaner form that dequantizes straight to bf16 (nf4_dequantize_ex). Same
    inputs, same output shape and dtype. All timed with CUDA events on the
    current stream after 3 warm-ups, without an L2 flush (a weight smaller
    than L2 stays warm for all). One JSON line for the workload."""
    import dequant_gemm_gb300 as nf4
    work = wl.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)

    def time_ms(fn, reps):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    rows = []
    for p in work.projections:
        W = p.make_weight().to(dev)
        q = nf4.nf4_quantize(W)
        del W
        for M in work.fwd_m:
            X = wl.activations(M, p.cols, std=work.x_std, seed=1 + M).to(dev)
            t_fused = time_ms(lambda: nf4.nf4_matmul_fwd(X, q), args.steps)
            t_naive = time_ms(
                lambda: torch.matmul(X, nf4.nf4_dequantize(q).to(torch.bfloat16).t()).float(),
                args.steps)
            t_bf16 = time_ms(
                lambda: torch.matmul(X, nf4.nf4_dequantize(q, out_dtype=torch.bfloat16).t()).float(),
                args.steps)
            rows.append({"projection": f"{p.name} {p.rows}x{p.cols}", "M": M,
                         "fused_ms": t_fused, "naive_ms": t_naive, "speedup": t_naive / t_fused,
                         "naive_bf16_ms": t_bf16, "speedup_bf16": t_bf16 / t_fused})
    status = nf4.nf4_poll_device_status(dev)
    if status != 0:
        raise SystemExit(f"device status {status}")
    print(json.dumps({"metric": "fused NF4 forward vs dequantize-to-HBM + cuBLAS bf16 matmul",
                      "config": {"workload": args.workload}, "steps": args.steps, "rows": rows}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen2.5_7b_layer", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload records (decode, prefill + quantize, dX)")
    ap.add_argument("--naive", action="store_true",
                    help="time the fused forward against dequantize + cuBLAS instead")
    ap.add_argument("--serial-tc", action="store_true",
                    help="tensor-core calls of projections sharing an input one after another "
                         "instead of on parallel streams")
    ap.add_argument("--no-group", action="store_true",
                    help="small-M forwards of projections sharing an input as separate launches "
                         "on parallel streams instead of one grouped launch")
    args = ap.parse_args()
    global GROUP_SMALL_M, PARALLEL_TC
    GROUP_SMALL_M = not args.no_group
    PARALLEL_TC = not args.serial_tc
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the NF4 kernels have no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import dequant_gemm_gb300 as nf4
    nf4.lib()
    if args.naive:
        return run_naive(args, dev)

    stream = torch.cuda.current_stream(dev)
    main_run = measure_workload(args.workload, dev, args.steps, args.warmup, world, clocks=True)
    work, step = main_run["work"], main_run["step"]
    elapsed_ms = max_over_ranks(main_run["elapsed_ms"], world, dev)
    ms_per_step = elapsed_ms / args.steps
    flop_step = step.flop()
    value = world * flop_step * args.steps / (elapsed_ms * 1e-3) / 1e12

    pk, pk_kind = peaks()
    parts = main_run["parts"]
    dom = max(parts, key=lambda c: parts[c]["ms_per_step"])
    d = parts[dom]
    if d["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": d["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": d["hbm_frac"]}
    else:
        roof = {"bound": "tensor", "achieved": d["TFLOP/s"], "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": d["tensor_frac_burst"],
                "frac_sustained": d["tensor_frac_sustained"],
                "peak_sustained": pk["bf16_tflops_sustained"]}
    roof.update({"kernel": dom, "traffic": traffic_per_launch(work.name, dom),
                 "traffic_unit": "bytes per launch (ncu dram read+write)",
                 "achieved_per": "launch-average over the class",
                 "peak_kind": f"{pk_kind} " + (
                     "burst bf16 (the class runs for well under a second at full clock); "
                     "frac_sustained divides by the power-capped sustained figure"
                     if roof["bound"] == "tensor" else "copy bandwidth")})

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": work.name,
                   "projections": [f"{p.name} {p.rows}x{p.cols}" for p in work.projections],
                   "fwd_m": list(work.fwd_m), "dx_m": list(work.dx_m),
                   "quantize_in_step": step.quantize_in_step,
                   "l2": main_run["l2"],
                   "timing": "CUDA graph per kernel class, CUDA events between graphs",
                   "issue": ("projections sharing an input: "
                             + ("one grouped launch at M <= 16" if GROUP_SMALL_M else
                                "parallel graph branches at M <= 16")
                             + (", parallel graph branches above" if PARALLEL_TC else
                                ", one after another above")),
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": step.launches() * args.steps,
        "roofline": roof,
        "parts": parts,
    }
    if main_run["clocks"]:
        line["clocks"] = main_run["clocks"]
    line["peaks"] = {k: pk.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}
    line["peaks"]["kind"] = pk_kind
    line["peaks"]["sustained_sm_mhz_median"] = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")

    if not args.no_e2e:
        h2d, d2h = step.host_buffers()
        for i in range(2):
            step.run_e2e()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        for s in range(args.steps):
            step.run_e2e()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        line["e2e"] = {"value": world * flop_step * args.steps / (e2e_ms * 1e-3) / 1e12,
                       "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms / args.steps}

    if not args.no_configs:
        del step
        main_run.clear()
        torch.cuda.empty_cache()
        line["configs"] = {}
        for name in CONFIG_WORKLOADS:
            if name == args.workload:
                continue
            r = measure_workload(name, dev, args.steps, args.warmup, world, clocks=True)
            line["configs"][name] = config_record(r)
            r.clear()
            torch.cuda.empty_cache()

    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores, secs = oracle_sample(args.workload, budget_s=20.0)
        line["cpu_baseline"] = {"value": v / 1e12, "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
