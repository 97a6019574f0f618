"""Benchmark of the block-swizzled tile GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--configs 0|1] [--lite]

A step is one call of the GEMM entry point on one batch of synthetic input.
The default workload is the fp16 GEMM M=N=1024, K=2048 (A row-major, B
column-major, entries N(0,1)/sqrt(K), fp32 accumulate, fp16 out) -- the one
the metric "GEMM TFLOP/s at 1 GB300 and % of the dtype's dense tensor peak"
is quoted on.  The default run also measures the other four configurations
the metric is quoted on (the fp16 500x380x256 tail, MXFP8 1024x2048x4096,
grouped bf16 slice-M and int8 8192^3 with per-token dequant) and reports each
under "configs" with its own timing, roofline, clocks, end-to-end figure and
oracle baseline.  Other workloads (--workload fp16_tail | mxfp8 | ...) print
the line for their own shape alone.

Timing: W untimed steps, then exactly K steps replayed from CUDA graphs on one
stream, bracketed by a barrier and a device synchronise, timed with CUDA
events; the graphs are queued behind an untimed device-side wait so that the
host's submission latency is not in the timed region; inputs rotate over
enough independent copies that the bytes touched between two uses of one copy
exceed the 129 MB L2.  The extra configurations time min(K, about one second
of steps).  With N > 1 (torchrun) every rank runs an independent replica on
its own GPU (the path shards by whole problems, no collective on the data
path) and rank 0 prints the total over ranks divided by the slowest rank's
time.

--impl reference times the CPU oracle (the plain fp64 definition in oracle/)
on the host cores on a bounded sample of rows of the same workload.
--lite skips the CPU baseline, the clock sampler, the end-to-end leg and the
extra configurations (for profiler runs).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the oracle's BLAS gets every host core; say so in the output
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "GEMM TFLOP/s at 1 GB300 and % of dtype dense tensor peak"
PROFILE_DIR = os.path.join(ROOT, "profiles")


def code_text(src):
    """C/C++ source with its comments removed and its whitespace collapsed."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


# host-only source (argument checks, tile and split choice, launches): not
# part of the device-code hash
HOST_ONLY_SOURCES = ("api.cu",)


def csrc_hash():
    """Hash of the device code (every CUDA source but the host-only ones, with
    comments and whitespace removed), so stored profiler counters are only
    used for the kernels they were taken from, and an edit of a comment or of
    host code does not discard them."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_swizzled_tile_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def stored_traffic(kernel_key, setting=None):
    """DRAM bytes per step recorded from ncu captures of this step's
    kernels, if they were taken from the current device sources: the entry
    of this swizzle setting (key@Zn4 and the like) where the traffic depends
    on it, else the entry of the kernel alone."""
    p = os.path.join(PROFILE_DIR, "traffic.txt")
    if not os.path.exists(p):
        return None
    cur = csrc_hash()
    found = {}
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not parts[0].startswith("#") and parts[1] == cur:
                found[parts[0]] = float(parts[2])
    if setting and "%s@%s" % (kernel_key, setting) in found:
        return found["%s@%s" % (kernel_key, setting)]
    return found.get(kernel_key)


# ------------------------------------------------------------- workloads --

class Workload:
    """Inputs on the device (``copies`` independent sets), the call that
    runs one step on set i, and the work per step."""

    def __init__(self, name, copies=None, seed=0):
        import block_swizzled_tile_gb300 as bst
        from block_swizzled_tile_gb300 import workloads as wl
        self.bst = bst
        self.name = name
        if name in ("fp16_square", "fp16_tail"):
            w = wl.fp16_square(seed) if name == "fp16_square" else wl.fp16_tail(seed)
            self.w = w
            M, N, K = w["M"], w["N"], w["K"]
            self.flops = 2.0 * M * N * K
            self.in_bytes = (w["a"].nbytes + w["b"].nbytes)
            self.out_bytes = M * N * 2
            self.dtype = "f16"
            self.desc = ("fp16 GEMM M=%d N=%d K=%d, A %s-major, B %s-major, fp32 accumulate, fp16 out"
                         % (M, N, K, "col" if w["a_col_major"] else "row", "col" if w["b_col_major"] else "row"))
            self.kernel_key = "gemm_f16_%dx%dx%d" % (M, N, K)
        elif name == "mxfp8":
            w = wl.mxfp8(seed=seed)
            self.w = w
            M, N, K = w["M"], w["N"], w["K"]
            self.flops = 2.0 * M * N * K
            self.in_bytes = w["a"].nbytes + w["b"].nbytes + w["sa"].nbytes + w["sb"].nbytes
            self.out_bytes = M * N * 2
            self.dtype = "e4m3"
            self.desc = "MXFP8 GEMM M=%d N=%d K=%d, e4m3 A and B, E8M0 scale per 32 K, bf16 out" % (M, N, K)
            self.kernel_key = "gemm_mxf8_%dx%dx%d" % (M, N, K)
        elif name == "grouped_bf16":
            w = wl.grouped_bf16(seed=seed)
            self.w = w
            gm, N, K = w["group_m"], w["N"], w["K"]
            self.flops = 2.0 * sum(gm) * N * K
            self.in_bytes = w["x"].nbytes + sum(K * N * 2 for m in gm if m)
            self.out_bytes = sum(gm) * N * 2
            self.dtype = "bf16"
            self.desc = "grouped bf16 GEMM slice-M, G=%d sizes %s, K=%d N=%d, bf16 out" % (len(gm), gm, K, N)
            self.kernel_key = "gemm_grouped_bf16_%dx%dx%d" % (sum(gm), N, K)
        elif name == "int8_per_token":
            w = wl.int8_per_token(seed=seed)
            self.w = w
            M, N, K = w["M"], w["N"], w["K"]
            self.flops = 2.0 * M * N * K
            self.in_bytes = w["a"].nbytes + w["b"].nbytes + w["sa"].nbytes + w["sb"].nbytes
            self.out_bytes = M * N * 2
            self.dtype = "s8"
            self.desc = "int8 GEMM M=%d N=%d K=%d, int32 accumulate, per-token dequant, bf16 out" % (M, N, K)
            self.kernel_key = "gemm_int8_dequant_%dx%dx%d" % (M, N, K)
        elif name == "grouped_int8_per_token":
            w = wl.grouped_int8_per_token(seed=seed)
            self.w = w
            gm, N, K = w["group_m"], w["N"], w["K"]
            self.flops = 2.0 * sum(gm) * N * K
            self.in_bytes = w["x"].nbytes + sum(N * K for m in gm if m) + w["sa"].nbytes + w["sb"].nbytes
            self.out_bytes = sum(gm) * N * 2
            self.dtype = "s8"
            self.desc = ("grouped int8 GEMM slice-M with per-token dequant, G=%d sizes %s, K=%d N=%d, int32 "
                         "accumulate, bf16 out" % (len(gm), gm, K, N))
            self.kernel_key = "gemm_grouped_int8_dequant_%dx%dx%d" % (sum(gm), N, K)
        elif name == "grouped_slice_k_bf16":
            w = wl.grouped_slice_k_bf16(seed=seed)
            self.w = w
            gk, M, N = w["group_k"], w["M"], w["N"]
            self.flops = 2.0 * M * N * sum(gk)
            self.in_bytes = w["x"].nbytes + w["dy"].nbytes
            self.out_bytes = len(gk) * M * N * 2
            self.dtype = "bf16"
            self.desc = ("grouped bf16 GEMM slice-K (C_g = X_g^T dY_g), G=%d K sizes %s, M=%d N=%d, A and B "
                         "MN-major, bf16 out" % (len(gk), gk, M, N))
            self.kernel_key = "gemm_slice_k_bf16_%dx%dx%dx%d" % (len(gk), M, N, sum(gk))
        elif name == "grouped_slice_k_int8":
            w = wl.grouped_slice_k_int8(seed=seed)
            self.w = w
            gk, M, N = w["group_k"], w["M"], w["N"]
            self.flops = 2.0 * M * N * sum(gk)
            self.in_bytes = w["a"].nbytes + w["b"].nbytes + w["sa"].nbytes + w["sb"].nbytes
            self.out_bytes = len(gk) * M * N * 2
            self.dtype = "s8"
            self.desc = ("grouped int8 GEMM slice-K with per-token dequant, G=%d K sizes %s, M=%d N=%d, A^T [K,M] "
                         "and B [K,N] (MN-contiguous), int32 accumulate, bf16 out" % (len(gk), gk, M, N))
            self.kernel_key = "gemm_slice_k_int8_%dx%dx%dx%d" % (len(gk), M, N, sum(gk))
        else:
            raise SystemExit("unknown workload " + name)
        per_set = self.in_bytes + self.out_bytes
        # enough copies that the bytes between two uses of one copy exceed L2,
        # and at least the sets the end-to-end leg alternates
        self.copies = copies or max(E2E_SETS, min(4096, math.ceil(2 * L2_BYTES / per_set)))
        self.sched = bst.sched(1, 0)
        # kernels per call: int8 widens both operands in one bulk-copy launch
        # before its GEMM; slice-K rewrites its per-group maps in a prep launch
        self.launches_per_step = {"int8_per_token": 2, "grouped_int8_per_token": 2, "grouped_slice_k_bf16": 2,
                                  "grouped_slice_k_int8": 3}.get(name, 1)
        self._alloc()

    def _alloc(self):
        w = self.w

        def to_dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1).copy()).cuda()

        self.sets = []
        for _ in range(self.copies):
            s = {}
            if self.name in ("fp16_square", "fp16_tail"):
                s["A"], s["B"] = to_dev(w["a"]), to_dev(w["b"])
                s["C"] = torch.empty(w["M"] * w["N"], dtype=torch.int16, device="cuda")
            elif self.name == "mxfp8":
                s["A"], s["B"], s["SA"], s["SB"] = (to_dev(w["a"]), to_dev(w["b"]), to_dev(w["sa"]), to_dev(w["sb"]))
                s["C"] = torch.empty(w["M"] * w["N"], dtype=torch.int16, device="cuda")
            elif self.name == "grouped_bf16":
                s["X"], s["W"] = to_dev(w["x"]), to_dev(w["w"])
                s["G"] = torch.tensor(w["group_m"], dtype=torch.int32, device="cuda")
                s["C"] = torch.empty(sum(w["group_m"]) * w["N"], dtype=torch.int16, device="cuda")
            elif self.name == "grouped_int8_per_token":
                gm = w["group_m"]
                s["X"], s["W"] = to_dev(w["x"]), to_dev(w["w"])
                s["SA"], s["SB"] = to_dev(w["sa"]), to_dev(w["sb"])
                s["G"] = torch.tensor(gm, dtype=torch.int32, device="cuda")
                s["C"] = torch.empty(sum(gm) * w["N"], dtype=torch.int16, device="cuda")
                nb = self.bst.gemm_grouped_quant_per_token_workspace_size(len(gm), sum(gm), w["N"], w["K"])
                s["WS"] = torch.empty(nb, dtype=torch.uint8, device="cuda")
                s["WSB"] = nb
            elif self.name == "grouped_slice_k_bf16":
                gk = w["group_k"]
                s["X"], s["DY"] = to_dev(w["x"]), to_dev(w["dy"])
                s["G"] = torch.tensor(gk, dtype=torch.int32, device="cuda")
                s["C"] = torch.empty(len(gk) * w["M"] * w["N"], dtype=torch.int16, device="cuda")
                nb = self.bst.gemm_grouped_slice_k_workspace_size(len(gk))
                s["WS"] = torch.empty(nb, dtype=torch.uint8, device="cuda")
                s["WSB"] = nb
            elif self.name == "grouped_slice_k_int8":
                gk = w["group_k"]
                # the weight-gradient layout: A^T [sum K, M] and B [sum K, N] (any group sizes)
                s["A"], s["B"] = to_dev(np.ascontiguousarray(w["a"].T)), to_dev(w["b"])
                s["SA"], s["SB"] = to_dev(w["sa"]), to_dev(w["sb"])
                s["G"] = torch.tensor(gk, dtype=torch.int32, device="cuda")
                s["C"] = torch.empty(len(gk) * w["M"] * w["N"], dtype=torch.int16, device="cuda")
                nb = self.bst.gemm_grouped_slice_k_quant_per_token_workspace_size(len(gk), w["M"], w["N"], sum(gk))
                s["WS"] = torch.empty(nb, dtype=torch.uint8, device="cuda")
                s["WSB"] = nb
            else:
                s["A"], s["B"] = to_dev(w["a"]), to_dev(w["b"])
                s["SA"], s["SB"] = to_dev(w["sa"]), to_dev(w["sb"])
                s["C"] = torch.empty(w["M"] * w["N"], dtype=torch.int16, device="cuda")
                nb = self.bst.gemm_quant_per_token_workspace_size(w["M"], w["N"], w["K"])
                s["WS"] = torch.empty(nb, dtype=torch.uint8, device="cuda")
                s["WSB"] = nb
            self.sets.append(s)

    def step(self, i, sched=None):
        bst, w, s = self.bst, self.w, self.sets[i % self.copies]
        sched = sched or self.sched
        if self.name in ("fp16_square", "fp16_tail"):
            bst.gemm(w["M"], w["N"], w["K"], s["A"], bst.F16, bst.COL_MAJOR if w["a_col_major"] else bst.ROW_MAJOR,
                     w["lda"], s["B"], bst.F16, bst.COL_MAJOR if w["b_col_major"] else bst.ROW_MAJOR, w["ldb"],
                     s["C"], bst.F16, w["N"], sched=sched)
        elif self.name == "mxfp8":
            bst.gemm(w["M"], w["N"], w["K"], s["A"], bst.E4M3, bst.ROW_MAJOR, w["K"], s["B"], bst.E4M3,
                     bst.COL_MAJOR, w["K"], s["C"], bst.BF16, w["N"], scale_a=s["SA"], scale_b=s["SB"], sched=sched)
        elif self.name == "grouped_bf16":
            gm = w["group_m"]
            bst.gemm_grouped(len(gm), s["G"], sum(gm), w["N"], w["K"], s["X"], w["K"], s["W"], bst.ROW_MAJOR,
                             w["N"], w["K"] * w["N"], s["C"], w["N"], bst.BF16, bst.BF16, sched=sched)
        elif self.name == "grouped_int8_per_token":
            gm, N, K = w["group_m"], w["N"], w["K"]
            bst.gemm_grouped_quant_per_token(len(gm), s["G"], sum(gm), N, K, s["X"], K, s["W"], bst.COL_MAJOR, K,
                                             N * K, s["SA"], s["SB"], N, s["C"], N, None, s["WS"], s["WSB"],
                                             sched=sched)
        elif self.name == "grouped_slice_k_bf16":
            gk, M, N = w["group_k"], w["M"], w["N"]
            bst.gemm_grouped_slice_k(len(gk), s["G"], M, N, sum(gk), s["X"], bst.COL_MAJOR, M, s["DY"], bst.ROW_MAJOR,
                                     N, s["C"], N, M * N, bst.BF16, bst.BF16, s["WS"], s["WSB"], sched=sched)
        elif self.name == "grouped_slice_k_int8":
            gk, M, N = w["group_k"], w["M"], w["N"]
            K = sum(gk)
            bst.gemm_grouped_slice_k_quant_per_token(len(gk), s["G"], M, N, K, s["A"], bst.COL_MAJOR, M, s["B"],
                                                     bst.ROW_MAJOR, N, s["SA"], M, s["SB"], N, s["C"], N, M * N,
                                                     None, s["WS"], s["WSB"], sched=sched)
        else:
            bst.gemm_quant_per_token(w["M"], w["N"], w["K"], s["A"], w["K"], s["B"], bst.COL_MAJOR, w["K"],
                                     s["SA"], s["SB"], s["C"], w["N"], None, s["WS"], s["WSB"], sched=sched)

    def host_inputs(self):
        """Pinned host copies of one input set (for the end-to-end leg)."""
        s = self.sets[0]
        keys = [k for k in s if k not in ("C", "WS", "WSB")]
        return {k: s[k].cpu().pin_memory() for k in keys}


# ------------------------------------------------------------- timing ----

def graph_of(work, steps, offset):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            work.step(offset + i)
    return g


def timed_steps(work, K, stream):
    """Replays exactly K steps from CUDA graphs; returns (ms, graphs)."""
    per = min(K, work.copies * max(1, 32 // work.copies) if work.copies < 32 else work.copies)
    full = graph_of(work, per, 0) if per > 0 else None
    rem = K % per if per else 0
    tail = graph_of(work, rem, 0) if rem else None
    reps = K // per if per else 0
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # an untimed device wait ahead of the first event keeps the GPU busy while
    # the host submits the graphs, so the timed region holds the K steps'
    # device time and not the host's submission latency
    device_wait(stream)
    t0.record(stream)
    for _ in range(reps):
        full.replay()
    if tail is not None:
        tail.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def device_wait(stream, us=50.0):
    """Queues a device-side spin of about ``us`` microseconds on ``stream``
    (untimed; it precedes the first timing event)."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2100))


E2E_SETS = 3                   # buffer sets the end-to-end leg alternates


def e2e_pipelined(work, hin, steps, warm, sets=None):
    """End-to-end steps through the public API: every step copies its inputs
    from pinned host memory to the device (one stream per input tensor, so
    the copies run on several copy engines), runs the GEMM, and copies the
    result back to pinned host memory.  Three device input sets and host
    outputs alternate, so step i+1's inputs go in while step i computes and
    step i-1's result comes out; events keep every reuse ordered (with two
    sets the int8 8192^3 steps took 0.97-1.01 ms, with three 0.88).  The steps are
    captured in a CUDA graph (as the device-timed steps are) and replayed,
    so the host's launch cost does not pace them.  Returns the milliseconds of
    `steps` steps (rounded up to whole graphs; the caller divides by the
    count it gets back), after `warm` untimed replays."""
    nb = min(sets or E2E_SETS, work.copies)
    keys = list(hin)
    cap = torch.cuda.Stream()
    h2d = [torch.cuda.Stream() for _ in keys]
    cs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    hout = [torch.empty(work.sets[j]["C"].numel(), dtype=work.sets[j]["C"].dtype).pin_memory() for j in range(nb)]
    per = 10 * nb                                  # steps per graph, a multiple of the set count
    # one eager pass first: lazy initialisation must not happen under capture
    for j in range(nb):
        for k in keys:
            work.sets[j][k].copy_(hin[k], non_blocking=True)
        work.step(j)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fork = torch.cuda.Event()
        fork.record(cap)
        for st in h2d + [cs, ds]:
            st.wait_event(fork)
        ev_done = [None] * nb
        ev_out = [None] * nb
        for i in range(per):
            j = i % nb
            s = work.sets[j]
            ev_in = []
            for n, k in enumerate(keys):
                st = h2d[n]
                if ev_done[j] is not None:
                    st.wait_event(ev_done[j])
                with torch.cuda.stream(st):
                    s[k].copy_(hin[k], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(st)
                    ev_in.append(e)
            for e in ev_in:
                cs.wait_event(e)
            if ev_out[j] is not None:
                cs.wait_event(ev_out[j])
            with torch.cuda.stream(cs):
                work.step(j)
                ev_done[j] = torch.cuda.Event()
                ev_done[j].record(cs)
            ds.wait_event(ev_done[j])
            with torch.cuda.stream(ds):
                hout[j].copy_(s["C"], non_blocking=True)
                ev_out[j] = torch.cuda.Event()
                ev_out[j].record(ds)
        for st in h2d + [cs, ds]:
            join = torch.cuda.Event()
            join.record(st)
            cap.wait_event(join)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    reps = -(-steps // per)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    device_wait(cap)
    e0.record(cap)
    for _ in range(reps):
        with torch.cuda.stream(cap):
            g.replay()
    e1.record(cap)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), reps * per


def barrier():
    if torch.distributed.is_initialized():
        torch.distributed.barrier()


def whole_job_tflops(world, flops_per_step, steps, ms):
    """Aggregate throughput of ``world`` replicas that each ran ``steps`` steps
    of ``flops_per_step``, over the slowest rank's time ``ms``."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def max_over_ranks(x):
    """Largest value of ``x`` over all ranks (the slowest rank's time)."""
    if not torch.distributed.is_initialized():
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t_begin, t_end):
        win = [s for t, s in self.samples if t_begin <= t <= t_end]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        mhz = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if len(s) > 5 + i and s[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win),
                "power_w_max": max(float(s[3]) for s in win if s[3].replace(".", "").isdigit()) if win else None}


# ---------------------------------------------------------- cpu oracle ---

def oracle_rows(work, rows):
    """The oracle (test-infrastructure, CPU) computing ``rows`` whole output
    rows of the workload; returns the flops it did."""
    from oracle import gemm as og
    w = work.w
    if work.name in ("fp16_square", "fp16_tail"):
        M, N, K = w["M"], w["N"], w["K"]
        a = og.as_logical(og.decode(w["a"], "f16"), M, K, w["lda"], w["a_col_major"])[:rows]
        b = og.as_logical(og.decode(w["b"], "f16"), K, N, w["ldb"], w["b_col_major"])
        og.gemm(a, b, "f16")
        return 2.0 * rows * N * K
    if work.name == "mxfp8":
        og.gemm_mxfp8(w["a"][:rows], w["sa"][:rows], w["b"], w["sb"])
        return 2.0 * rows * w["N"] * w["K"]
    if work.name == "grouped_bf16":
        gm = w["group_m"]
        g = next(i for i, m in enumerate(gm) if m)
        take = min(rows, gm[g])
        off = sum(gm[:g])
        x = og.decode(w["x"][off:off + take], "bf16")
        og.gemm(x, og.decode(w["w"][g], "bf16"), "bf16")
        return 2.0 * take * w["N"] * w["K"]
    if work.name == "grouped_slice_k_bf16":
        take = min(rows, w["M"])
        a = og.decode(np.ascontiguousarray(w["x"][:, :take].T), "bf16")
        og.gemm_grouped_slice_k(a, og.decode(w["dy"], "bf16"), w["group_k"], "bf16")
        return 2.0 * take * w["N"] * sum(w["group_k"])
    if work.name == "grouped_slice_k_int8":
        take = min(rows, w["M"])
        og.gemm_grouped_slice_k_quant_per_token(w["a"][:take], w["b"], w["group_k"], w["sa"][:, :take], w["sb"])
        return 2.0 * take * w["N"] * sum(w["group_k"])
    if work.name == "grouped_int8_per_token":
        gm = w["group_m"]
        g = next(i for i, m in enumerate(gm) if m)
        take = min(rows, gm[g])
        off = sum(gm[:g])
        og.gemm_grouped_quant_per_token(w["x"][off:off + take], [w["w"][g].T], [take], w["sa"][off:off + take],
                                        w["sb"][g:g + 1])
        return 2.0 * take * w["N"] * w["K"]
    og.gemm_quant_per_token(w["a"][:rows], w["b"].T, w["sa"][:rows], w["sb"])
    return 2.0 * rows * w["N"] * w["K"]


def total_rows(work):
    return sum(work.w["group_m"]) if work.name in ("grouped_bf16", "grouped_int8_per_token") else work.w["M"]


def cpu_rate(work, budget_s):
    """Oracle throughput on a sample of whole output rows sized to about
    budget_s of CPU time (the whole problem, repeated, when that is smaller).
    Each oracle call decodes its operands, so the calibration run uses all
    rows.  Returns (TFLOP/s, sample description, seconds)."""
    total = total_rows(work)
    t = time.perf_counter()
    oracle_rows(work, total)
    dt_full = max(time.perf_counter() - t, 1e-6)
    if dt_full >= budget_s:
        rows, reps = max(8, int(total * budget_s / dt_full)), 1
    else:
        rows, reps = total, max(1, int(round(budget_s / dt_full)))
    t = time.perf_counter()
    fl = sum(oracle_rows(work, rows) for _ in range(reps))
    dt = time.perf_counter() - t
    sample = "%d of %d output rows%s (whole rows, %.1f s)" % (rows, total, " x%d" % reps if reps > 1 else "", dt)
    return fl / dt / 1e12, sample, dt


def reference_arm(args, work_name):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    work = Workload.__new__(Workload)          # inputs only, no device memory
    from block_swizzled_tile_gb300 import workloads as wl
    work.name = work_name
    work.w = {"fp16_square": wl.fp16_square, "fp16_tail": wl.fp16_tail, "mxfp8": wl.mxfp8,
              "grouped_bf16": wl.grouped_bf16, "int8_per_token": wl.int8_per_token,
              "grouped_int8_per_token": wl.grouped_int8_per_token,
              "grouped_slice_k_bf16": wl.grouped_slice_k_bf16,
              "grouped_slice_k_int8": wl.grouped_slice_k_int8}[work_name]()
    desc = {"fp16_square": "fp16 GEMM M=1024 N=1024 K=2048, A row-major, B col-major, fp32 accumulate, fp16 out"}
    # size the per-step sample so that warmup + steps take about two minutes
    budget = min(20.0, 120.0 / max(1, args.steps + args.warmup))
    rows = 8
    t = time.perf_counter()
    oracle_rows(work, rows)
    dt = max(time.perf_counter() - t, 1e-6)
    rows = int(max(8, min(total_rows(work), rows * budget / dt)))
    for _ in range(args.warmup):
        oracle_rows(work, rows)
    t = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += oracle_rows(work, rows)
    el = time.perf_counter() - t
    value = fl / el / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": desc.get(work_name, work_name), "sample": "%d whole output rows per step" % rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
                             "kind": "oracle", "sample": "%d of %d output rows per step, fp64 BLAS matmul + one "
                             "rounding" % (rows, total_rows(work))},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main --

# the configurations the metric is quoted on; the first is the headline line
CONFIGS = [("c2", "fp16_square"), ("c1", "fp16_tail"), ("c3", "mxfp8"), ("c4", "grouped_bf16"),
           ("c5", "int8_per_token")]


def sched_opts(args):
    return dict(tile_n=args.tile_n, tile_m=args.tile_m, split_k=args.split_k, dynamic=args.dynamic,
                shuffle_k=args.shuffle_k)


def choose_swizzle(work, args, stream, opts):
    """Untimed sweep of SwizzleOffset {1,2,4,8} x {Zn,Nz}: two passes in
    opposite orders, averaged, after a warm-up of the same work, so a GPU
    that heats up (or cools down) during the sweep favours no setting by its
    position in the order.  Returns ({setting: TFLOP/s}, ms per step of the
    warm-up)."""
    n = max(8, min(200, args.steps))
    order = [(S, d) for S in (1, 2, 4, 8) for d in (0, 1)]
    times = {}
    work.sched = work.bst.sched(1, 0, **opts)
    warm_ms = timed_steps(work, n, stream) / n
    for seq in (order, order[::-1]):
        for S, d in seq:
            work.sched = work.bst.sched(S, d, **opts)
            for i in range(3):
                work.step(i)
            times.setdefault((S, d), []).append(timed_steps(work, n, stream))
    sweep = {}
    for (S, d), ts in times.items():
        ms = sum(ts) / len(ts)
        sweep["%s%d" % ("Zn" if d == 0 else "Nz", S)] = round(work.flops * n / (ms * 1e-3) / 1e12, 2)
    best = max(sweep, key=sweep.get)
    work.sched = work.bst.sched(int(best[2:]), 0 if best.startswith("Zn") else 1, **opts)
    return sweep, warm_ms


def roofline_of(work, per_step_ms, clocks, peaks, src, setting=None):
    """The dominant kernel's roofline entry: tensor-bound GEMMs against the
    dtype's dense peak; a GEMM whose arithmetic intensity is below the ridge
    of the measured peaks (the fp16 tail) against the measured HBM copy rate,
    with its tensor fraction alongside."""
    capped = bool(clocks and "sw_power_cap" in clocks.get("reasons", []))
    kind = "bf16_tflops_sustained" if capped and "bf16_tflops_sustained" in peaks else "bf16_tflops"
    how = "sustained, power cap active" if kind.endswith("sustained") else "burst"
    if work.dtype == "e4m3":
        peak = peaks[kind] * 2.0
        peak_note = "%s bf16 %s x 2 (nominal fp8/bf16 ratio)" % (src, how)
    else:
        peak = peaks[kind]
        peak_note = "%s bf16 %s (%s)" % (src, how, "fp16 runs at the bf16 rate" if work.dtype == "f16" else
                                         "int8 is multiplied on the bf16 pipe" if work.dtype == "s8" else "bf16")
    sec = per_step_ms * 1e-3
    tflops = work.flops / sec / 1e12
    alg_bytes = work.in_bytes + work.out_bytes
    ai = work.flops / alg_bytes
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    entry = {"achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak, "bound": "tensor",
             "traffic": stored_traffic(work.kernel_key, setting), "peak_source": peak_note, "kernel": work.kernel_key,
             "launches_covered": work.launches_per_step, "per_launch_us": per_step_ms * 1e3,
             "algorithmic_bytes": alg_bytes, "arithmetic_intensity": round(ai, 1), "ridge": round(ridge, 1)}
    if ai < ridge:
        gbs = alg_bytes / sec / 1e9
        entry.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": gbs / peaks["hbm_gbs"], "peak_source": "%s HBM copy rate" % src,
                      "tensor_tflops": tflops, "tensor_frac": tflops / peak})
    return entry


TIMELINE_CTAS = 8192          # rows of 64 stamps in the --timeline buffer


def timeline_rows(stamps):
    """Per stamp slot that any CTA wrote: (slot, min, median, max) in us from
    the first CTA's entry (slot 0), over the CTAs that wrote it.  `stamps` is
    [CTAs, 64] of %globaltimer ns, 0 where nothing was written."""
    t = np.asarray(stamps, dtype=np.int64)
    t = t[t[:, 0] > 0]
    if not len(t):
        return []
    t0 = t[:, 0].min()
    rows = []
    for c in range(t.shape[1]):
        v = t[:, c]
        v = v[v > 0]
        if len(v):
            us = (v - t0) / 1e3
            rows.append((c, float(us.min()), float(np.median(us)), float(us.max())))
    return rows


def timeline_report(args):
    """--timeline N: N launches of the workload back to back (schedule from
    --swizzle, default Zn1), then one more whose kernel writes its
    %globaltimer stamps (the `timeline` field of bst_sched; the slots are
    listed in include/bst.h); three rounds.  Prints the CUDA-event time of
    the stamped launch and, per slot, min / median / max over the CTAs."""
    torch.cuda.set_device(0)
    work = Workload(args.workload)
    opts = sched_opts(args)
    S, d = (int(args.swizzle[2:]), 0 if args.swizzle.startswith("Zn") else 1) if args.swizzle else (1, 0)
    buf = torch.zeros(TIMELINE_CTAS * 64, dtype=torch.int64, device="cuda")
    plain = work.bst.sched(S, d, **opts)
    stamped = work.bst.sched(S, d, timeline=buf, **opts)
    for _ in range(3):
        for i in range(args.timeline):
            work.step(i, plain)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        work.step(args.timeline, stamped)
        e1.record()
        torch.cuda.synchronize()
    work.bst.check_async()
    rows = timeline_rows(buf.view(TIMELINE_CTAS, 64).cpu().numpy())
    ctas = int((buf.view(TIMELINE_CTAS, 64)[:, 0] > 0).sum())
    print("%s %s%d, after %d launches: stamped launch %.2f us (CUDA events), %d CTAs"
          % (args.workload, "Zn" if d == 0 else "Nz", S, args.timeline, e0.elapsed_time(e1) * 1e3, ctas))
    print("slot      min   median      max  (us from the first CTA's entry)")
    for c, lo, med, hi in rows:
        print("%4d %8.2f %8.2f %8.2f" % (c, lo, med, hi))


def measure(name, args, world, rank, stream, sampler, cpu_budget, steps):
    """One workload: swizzle choice, warm-up, clock-sampled soak and exactly
    `steps` timed steps, the end-to-end leg and the oracle on the host.
    Returns the fields of its JSON line and frees its device memory."""
    work = Workload(name)
    opts = sched_opts(args)
    sweep = {}
    work.sched = work.bst.sched(1, 0, **opts)
    est_ms = None
    if args.swizzle:
        work.sched = work.bst.sched(int(args.swizzle[2:]), 0 if args.swizzle.startswith("Zn") else 1, **opts)
    elif not args.lite:
        sweep, est_ms = choose_swizzle(work, args, stream, opts)
    for i in range(args.warmup):
        work.step(i)
    torch.cuda.synchronize()
    if est_ms is None:
        est_ms = timed_steps(work, 8, stream) / 8

    clocks = None
    t_soak = time.time()
    if sampler:
        # untimed soak of the same work so the clock samples see the load
        per_soak = max(1, int(args.soak_seconds / max(1e-6, est_ms * 1e-3)))
        timed_steps(work, min(per_soak, 400000), stream)
    ms = timed_steps(work, steps, stream)
    t_end = time.time()
    if sampler:
        time.sleep(0.2)
        clocks = sampler.summary(t_soak, t_end)
        clocks["window"] = "soak+timed"
    ms = max_over_ranks(ms)

    e2e = None
    if not args.lite:
        # end to end: pinned host inputs -> device, GEMM, result -> host, every step
        hin = work.host_inputs()
        ems, ke = e2e_pipelined(work, hin, max(10, min(steps, 500)), 3)
        ems = max_over_ranks(ems)
        e2e = {"value": whole_job_tflops(world, work.flops, ke, ems), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(v.numel() * v.element_size() for v in hin.values())),
               "d2h_bytes_per_step": int(work.sets[0]["C"].numel() * work.sets[0]["C"].element_size()),
               "steps": ke, "pipeline": "3 buffer sets: inputs of step i+1 copied in while step i computes and step i-1 copies out; one "
                                         "copy stream per input tensor; steps replayed from CUDA graphs"}
        del hin

    cpu = None
    if rank == 0 and world == 1 and not args.lite and cpu_budget > 0:
        rate, sample, dt = cpu_rate(work, cpu_budget)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": int(os.environ["OPENBLAS_NUM_THREADS"]), "kind": "oracle",
               "sample": sample + ", fp64 BLAS matmul + one rounding"}

    peaks, src = measured_peaks()
    per_step_ms = ms / steps
    out = {
        "value": whole_job_tflops(world, work.flops, steps, ms), "unit": "TFLOP/s", "steps": steps,
        "ms_per_step": per_step_ms, "dtype": work.dtype,
        "config": {"workload": work.desc,
                   "swizzle": {"offset": work.sched.swizzle_offset,
                               "direction": "Zn" if work.sched.swizzle_direction == 0 else "Nz"},
                   "l2": "inputs rotate over %d copies (%.0f MB %s 129 MB L2)"
                         % (work.copies, work.copies * (work.in_bytes + work.out_bytes) / 1e6,
                            ">" if work.copies * (work.in_bytes + work.out_bytes) > L2_BYTES else "<="),
                   "tile_n": work.sched.tile_n or "auto", "tile_m": work.sched.tile_m or "auto",
                   "split_k": work.sched.split_k or "auto",
                   "tasks": "dynamic (cluster launch control)" if work.sched.dynamic else "static stride",
                   "shuffle_k": bool(work.sched.shuffle_k),
                   "launch": "CUDA graphs, one stream, queued behind an untimed device wait so that the host's "
                             "graph submission is outside the timed region",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline_of(work, per_step_ms, clocks, peaks, src,
                                setting=None if any(opts.values()) else "%s%d" % ("Zn" if work.sched.swizzle_direction == 0 else "Nz",
                                                                    work.sched.swizzle_offset)),
        "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e,
        "gpu_launches": steps * work.launches_per_step,
    }
    if sweep:
        out["swizzle_sweep_tflops"] = sweep
    for s in work.sets:
        s.clear()
    del work
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fp16_square",
                    choices=["fp16_square", "fp16_tail", "mxfp8", "grouped_bf16", "int8_per_token",
                             "grouped_int8_per_token", "grouped_slice_k_bf16", "grouped_slice_k_int8"])
    ap.add_argument("--configs", type=int, default=1, choices=[0, 1],
                    help="1 (default, headline workload only): also measure the other four configurations")
    ap.add_argument("--lite", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.0)
    ap.add_argument("--tile-n", type=int, default=0, help="force the tile width (64/128/256); 0 = automatic")
    ap.add_argument("--tile-m", type=int, default=0, help="force 128 (one CTA) or 256 (CTA pair); 0 = automatic")
    ap.add_argument("--split-k", type=int, default=0, help="0 automatic, 1 off, 2 or 4 split-K CTA pairs")
    ap.add_argument("--swizzle", default="", help="force the schedule, e.g. Zn3 or Nz1; default: sweep")
    ap.add_argument("--dynamic", type=int, default=0, choices=[0, 1],
                    help="1: tasks claimed at run time through cluster launch control (CTA-pair tiles)")
    ap.add_argument("--shuffle-k", type=int, default=0, choices=[0, 1], help="1: ShuffleK (rotated K start per task)")
    ap.add_argument("--timeline", type=int, default=0,
                    help="N > 0: print the kernel's pipeline stamps of one launch after N plain launches, no JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        reference_arm(args, args.workload)
        return
    if args.timeline > 0:
        timeline_report(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)

    from block_swizzled_tile_gb300 import _build
    if _build.stale():
        if rank == 0:
            _build.build()
        barrier()

    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local) if not args.lite else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    try:
        head = measure(args.workload, args, world, rank, stream, sampler, 12.0, args.steps)
        extra = {}
        forced = args.tile_n or args.tile_m or args.split_k or args.swizzle or args.dynamic or args.shuffle_k
        if args.configs and args.workload == "fp16_square" and not args.lite and not forced:
            for tag, name in CONFIGS[1:]:
                # each timed window held to about a second of device time
                probe = extra_steps(name, args.steps)
                extra[tag] = dict(measure(name, args, world, rank, stream, sampler, 6.0, probe),
                                  workload_name=name)
    finally:
        if sampler:
            sampler.stop()

    if rank != 0:
        return
    line = {"metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
            "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"], "clocks": head["clocks"],
            "e2e": head["e2e"], "gpu_launches": head["gpu_launches"]}
    if "swizzle_sweep_tflops" in head:
        line["swizzle_sweep_tflops"] = head["swizzle_sweep_tflops"]
    if extra:
        line["configs"] = extra
    print(json.dumps(line), flush=True)


# device time of one step of each extra configuration, for sizing its timed
# window (the K of the command line when that is shorter)
STEP_US = {"fp16_tail": 10.0, "mxfp8": 15.0, "grouped_bf16": 220.0, "int8_per_token": 800.0}


def extra_steps(name, k):
    return max(3, min(k, int(1e6 / STEP_US[name])))


if __name__ == "__main__":
    main()
