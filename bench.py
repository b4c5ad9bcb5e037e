"""Throughput of the tensor-parallel MLP block, forward + backward, on GB300.

One step = one pass of the whole hot path over one batch: the column-
parallel GEMM with bias + GeLU, the row-parallel GEMM with the in-device
g-operator sum + b2 + residual, the db2 column sums, the dZ GEMM with GeLU'
and the fused db1 partials, the dX GEMM with the in-device f-operator sum,
and the dA / dB weight-gradient GEMMs -- every one a call through the C ABI.

Metric: TFLOPS of fwd+bwd = 12 T h F algorithmic flops per step / time,
also given as % of the measured dense bf16 peak.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores
    python bench.py --sweep                 # one line per sweep point (not the headline)
    python bench.py --all-configs           # one line per workload family and shard count
    python bench.py --call dB --shape T,h,F,t [--repeat N] [--vs-cublas]   # one entry point alone

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (weak scaling, no collective on the data path); rank 0 prints
the line with the max time over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TFLOPS fwd+bwd of TP-sharded MLP block on 1 GB300; % of dense BF16 peak"
UNIT = "TFLOPS"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_mtnlg_full.md")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


CALLS = ("column_gelu", "column_gelu_h_only", "row_sum", "row_sum_dropout", "dgelu", "dx", "dA",
         "dB", "dA_kmajor", "dB_kmajor", "transpose", "dropout_grad", "bias_grad", "ln_forward",
         "ln_backward")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="mt-nlg-530b")
    p.add_argument("--tokens", type=int, default=None)
    p.add_argument("--shards", type=int, default=None)
    p.add_argument("--sweep", action="store_true")
    p.add_argument("--all-configs", action="store_true",
                   help="one line per workload family x shard count (tiny, GPT-2-medium, 8.3B, "
                        "MT-NLG, every sweep point)")
    p.add_argument("--recompute", action="store_true",
                   help="activation recompute: save only X, rebuild Z and H in the backward pass")
    p.add_argument("--dropout", type=float, default=0.0,
                   help="dropout rate before the residual add (0: the block without dropout)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--layernorm", action="store_true",
                   help="time the residual add + LayerNorm kernels instead (GB/s)")
    p.add_argument("--attention", action="store_true",
                   help="time the head-parallel attention block instead (TFLOPS fwd+bwd)")
    p.add_argument("--attn-workload", default="attn-gpt2-8.3b")
    p.add_argument("--pair-mode", type=int, default=None,
                   help="GEMM kernel: 0 single CTA, 1 auto (default), 2 CTA pairs")
    p.add_argument("--tile-scheduler", type=int, default=None,
                   help="GEMM tile assignment: 0 static persistent, 1 dynamic (cluster launch control)")
    p.add_argument("--wide-tiles", type=int, default=None,
                   help="1: 256 x 512 tiles per CTA pair for the K-major plain-store GEMMs (default 0)")
    p.add_argument("--call", choices=CALLS, default=None,
                   help="run ONE entry point --repeat times at --shape, holding only its operands "
                        "on the device (the command a profiler wraps to capture one kernel)")
    p.add_argument("--shape", default="2048,4096,16384,8",
                   help="T,h,F,t of --call (default: a sweep point under 1 GB on the device)")
    p.add_argument("--repeat", type=int, default=4)
    p.add_argument("--vs-cublas", action="store_true",
                   help="with --call: alternate the call with torch.matmul of the same shapes")
    p.add_argument("--rounds", type=int, default=8)
    return p.parse_args(argv)


def workload(args):
    from tensor_transformer_mlp_forward_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if args.tokens or args.shards:
        w = w.with_shape(T=args.tokens or w.T, t=args.shards or w.t)
    return w


def describe(w, n_gpus):
    seq = {"tiny": 64, "gpt2-medium": 1024, "megatron-8.3b": 1024, "mt-nlg-530b": 2048}.get(w.name)
    cfg = {"workload": f"{w.name} MLP block (T={w.T}, h={w.h}, F={w.F}, t={w.t})",
           "tokens": w.T, "hidden": w.h, "ffn": w.F, "shards": w.t}
    if seq and w.T % seq == 0:
        cfg["batch"], cfg["seq_len"] = w.T // seq, seq
    big = 2 * w.h * w.F > 129e6
    cfg["l2"] = ("inputs larger than L2; " if big else "") + "L2 flushed between timed steps (256 MiB write)"
    cfg["parallelism"] = f"t={w.t} shards in-device; {n_gpus} replica(s)"
    return cfg


# ------------------------------------------------------------------ peaks

def peaks():
    try:
        with open(PEAKS_FILE) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


# The sources the GEMM kernels and their host-side tile schedule are built
# from: a recorded DRAM-traffic figure holds while none of their code
# changes (comments and blank lines do not count).
GEMM_SOURCES = ("capi.cu", "gemm.cuh", "gemm_backward_data.cu", "gemm_backward_weight.cu",
                "gemm_forward.cu", "kernels.h", "philox.cuh", "ptx.cuh")


def code_only(text: str) -> str:
    """C/C++ source without its comments, trailing blanks and blank lines
    (string and character literals are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    d = os.path.join(ROOT, "tensor_transformer_mlp_forward_gb300", "csrc")
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        h.update(f.encode())
        h.update(code_only(open(os.path.join(d, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, wname: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    src = kernel_source_hash()
    for m in re.finditer(r"traffic: kernel=(\S+) workload=(\S+) src_sha=(\S+) bytes_per_launch=(\d+)", text):
        if m.group(1) == kernel and m.group(2) == wname and m.group(3) == src:
            return int(m.group(4))
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons;
    summary() keeps only the samples taken inside the marked window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.tmp = None
        self.window = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            deadline = time.time() + 5.0  # let the sampler start before timing begins
            while time.time() < deadline and os.path.getsize(self.tmp.name) == 0:
                time.sleep(0.05)
        except Exception:
            self.proc = None
        return self

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def _when(stamp: str):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.tmp.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    rows.append((self._when(parts[0]), float(parts[1]), float(parts[2]),
                                 float(parts[3]), parts[4:8]))
                except ValueError:
                    continue
        os.unlink(self.tmp.name)
        if self.window and rows:
            lo, hi = self.window
            inside = [r for r in rows if r[0] is not None and lo - 0.05 <= r[0] <= hi + 0.05]
            rows = inside or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = sorted({self.NAMES[i] for r in rows for i, f in enumerate(r[4])
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "power_w_median": statistics.median(r[3] for r in rows), "samples": len(rows),
                "reasons": reasons}


# -------------------------------------------------------------- our step

# On large blocks dA and dB read K-major operands (X, dZ, H and dY
# transposed first), as tp_mlp_backward does
STEP_CALLS = ("column_gelu", "row_sum", "db2", "dgelu", "dx", "dA", "dB")
KMAJOR_CALLS = ("t_X", "t_dZ", "dA", "t_H", "t_dY", "dB")
GEMM_CALLS = ("column_gelu", "row_sum", "dx", "dA", "dB")  # one kernel each


class Step:
    """All buffers of one replica, resident in HBM; run() issues one step."""

    def __init__(self, w, device, p_drop=0.0, seed=0x5EED, recompute=False):
        import torch

        from tensor_transformer_mlp_forward_gb300 import binding, inputs

        self.b = binding
        self.w = w
        T, h, F = w.T, w.h, w.F
        self.cpu = inputs.make_inputs(w)
        self.inp = {k: v.to(device) for k, v in self.cpu.items()}
        e = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        self.Y, self.Z, self.H, self.dZ = e(T, h), e(T, F), e(T, F), e(T, F)
        self.dX, self.dA, self.dB = e(T, h), e(h, F), e(F, h)
        self.db1, self.db2 = e(F, dt=torch.float32), e(h, dt=torch.float32)
        self.p_db1 = e(max(1, int(binding.lib().tp_mlp_dgelu_partial_floats(T, F))), dt=torch.float32)
        self.p_db2 = e(max(1, int(binding.lib().tp_mlp_bias_grad_workspace_floats(T, h))), dt=torch.float32)
        self.ws_split = e(max(16, binding.split_workspace_bytes(T, h, F, w.t)), dt=torch.uint8)
        self.kmajor = binding.weight_grad_kmajor(h, F // w.t)
        if self.kmajor:
            ldT = binding.pitch(T)
            self.Xt, self.dYt, self.dZt, self.Ht = e(h, ldT), e(h, ldT), e(F, ldT), e(F, ldT)
        self.launches = 0
        # dropout before the residual add: a fresh pattern every step (the
        # element counter advances by T*h, rounded up to a Philox block)
        self.p_drop, self.seed, self.offset = p_drop, seed, 0
        self.dP = e(T, h) if p_drop > 0 else None
        # activation recompute: the forward pass writes only H (transient),
        # the backward pass rebuilds Z and H from X before a4
        self.recompute = recompute
        self.names = (("column_gelu", "row_sum") + (("dropout_grad",) if p_drop > 0 else ())
                      + (("recompute",) if recompute else ()) + STEP_CALLS[2:5]
                      + (KMAJOR_CALLS if self.kmajor else STEP_CALLS[5:]))

    def run(self, events=None):
        """One fwd+bwd step.  `events`: a list of one more event than the
        calls, recorded between every two calls on the current stream, or a
        dict {boundary: event} recorded at those boundaries only (boundary k
        is just before call k; len(calls) is after the last)."""
        b, i, t = self.b, self.inp, self.w.t
        rec = self.recompute
        calls = (lambda: b.tp_mlp_column_gelu(i["X"], i["A"], i["b1"], t, Z=None if rec else self.Z,
                                              H=self.H, want_z=not rec),)
        if self.p_drop <= 0:
            dP = i["dY"]
            calls += (lambda: b.tp_mlp_row_sum(self.H, i["B"], i["b2"], i["residual"], t, Y=self.Y,
                                               workspace=self.ws_split),)
        else:
            dP, p, sd, off = self.dP, self.p_drop, self.seed, self.offset
            self.offset += (self.w.T * self.w.h + 3) // 4 * 4
            calls += (
                lambda: b.tp_mlp_row_sum_dropout(self.H, i["B"], i["b2"], i["residual"], t, p, sd,
                                                 off, Y=self.Y, workspace=self.ws_split),
                lambda: b.tp_mlp_dropout_grad(i["dY"], p, sd, off, dP=dP),
            )
        if rec:
            calls += (lambda: b.tp_mlp_column_gelu(i["X"], i["A"], i["b1"], t, Z=self.Z, H=self.H),)
        calls = calls + (
            lambda: b.tp_mlp_bias_grad(dP, db=self.db2, partial=self.p_db2),
            lambda: b.tp_mlp_dgelu(dP, i["B"], self.Z, t, dZ=self.dZ, db1=self.db1, partial=self.p_db1),
            lambda: b.tp_mlp_dx(self.dZ, i["A"], t, dX=self.dX, workspace=self.ws_split),
        )
        if self.kmajor:
            calls += (
                lambda: b.tp_transpose(i["X"], out=self.Xt),
                lambda: b.tp_transpose(self.dZ, out=self.dZt),
                lambda: b.tp_mlp_dA_kmajor(self.Xt, self.dZt, self.w.T, t, dA=self.dA),
                lambda: b.tp_transpose(self.H, out=self.Ht),
                lambda: b.tp_transpose(dP, out=self.dYt),
                lambda: b.tp_mlp_dB_kmajor(self.Ht, self.dYt, self.w.T, t, dB=self.dB),
            )
        else:
            calls += (
                lambda: b.tp_mlp_dA(i["X"], self.dZ, t, dA=self.dA),
                lambda: b.tp_mlp_dB(self.H, dP, t, dB=self.dB),
            )
        marks = events if isinstance(events, dict) else dict(enumerate(events or ()))
        if 0 in marks:
            marks[0].record()
        for k, c in enumerate(calls):
            c()
            self.launches += b.last_launch_count()
            if k + 1 in marks:
                marks[k + 1].record()


def init_distributed(n_gpus):
    import torch
    import torch.distributed as dist

    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def reduce_max_sum(elapsed_s: float, units: float):
    """Max of the elapsed time and sum of the units over all ranks (host
    bookkeeping only; identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def time_ours(w, steps, warmup, local, p_drop=0.0, recompute=False):
    """Two timed passes of `steps` steps each, L2 flushed between steps
    outside the events.  The headline pass records events only at the step's
    start, between the forward and the backward pass and at its end, so that
    a kernel may begin its launch while the one before it finishes, as in a
    training step; it gives the step time, the forward / backward split and
    the launch count.  The breakdown pass records an event between every two
    calls; it gives each call's time (the roofline's kernel duration)."""
    import torch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    step = Step(w, dev, p_drop, recompute=recompute)
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    assert step.b.device_status() == 0, "device wait timed out during warm-up"
    step.launches = 0

    ncalls = len(step.names)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    head = [{0: ev(), 2: ev(), ncalls: ev()} for _ in range(steps)]
    evs = [[ev() for _ in range(ncalls + 1)] for _ in range(steps)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        t0 = time.perf_counter()
        w0 = time.time()
        for k in range(steps):
            flush.fill_(k & 0xFF)  # evict L2 between steps (outside the events)
            step.run(head[k])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        launches = step.launches
        for k in range(steps):
            flush.fill_(k & 0xFF)
            step.run(evs[k])
        torch.cuda.synchronize()
        clocks.mark(w0, time.time())
    barrier()
    assert step.b.device_status() == 0, "device wait timed out"
    dev_ms = sum(head[k][0].elapsed_time(head[k][ncalls]) for k in range(steps))
    per_call = {name: [evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(steps)]
                for j, name in enumerate(step.names)}
    # the forward pass is a2 + a3 (calls 0 and 1), the backward pass the rest
    split = {"fwd_ms": statistics.mean(head[k][0].elapsed_time(head[k][2]) for k in range(steps)),
             "bwd_ms": statistics.mean(head[k][2].elapsed_time(head[k][ncalls]) for k in range(steps)),
             "breakdown_ms_per_step": statistics.mean(evs[k][0].elapsed_time(evs[k][ncalls])
                                                      for k in range(steps))}
    return step, dev_ms / 1e3, wall, per_call, clocks.summary(), launches, split


def time_graph(step, steps, warmup):
    """Seconds of `steps` replays of one step captured as a CUDA graph (the
    library's calls on the capturing stream, workspaces and outputs fixed),
    L2 flushed between replays outside the events."""
    import torch

    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=torch.cuda.current_device())
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    total = 0.0
    for k in range(steps):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    assert step.b.device_status() == 0, "device wait timed out in a graph replay"
    del graph
    return total


def time_e2e(step, steps, warmup):
    """Same step through the public API with the batch tensors (X, residual,
    dY) copied in from pinned host memory and the activation outputs (Y, dX)
    copied back every step; weights and weight gradients stay resident.

    The copies run on a second stream, double-buffered as a training loop
    would run them: step k's outputs go back and step k + 2's inputs come in
    while steps k + 1 computes.  Every copy of every timed step is inside the
    timed region, which ends when the last output has reached the host."""
    import torch

    names_in, names_out = ("X", "residual", "dY"), ("Y", "dX")
    host_in = {k: step.cpu[k].pin_memory() for k in names_in}
    host_out = {k: torch.empty_like(getattr(step, k), device="cpu").pin_memory() for k in names_out}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    inps = [dict(step.inp), {k: (torch.empty_like(v) if k in names_in else v) for k, v in step.inp.items()}]
    outs = [{k: getattr(step, k) for k in names_out}, {k: torch.empty_like(getattr(step, k)) for k in names_out}]
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=compute.device)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]

    def stage_in(slot):
        with torch.cuda.stream(copy):
            for k in names_in:
                inps[slot][k].copy_(host_in[k], non_blocking=True)
            ev_in[slot].record(copy)

    def run(n):
        stage_in(0)
        if n > 1:
            stage_in(1)
        for k in range(n):
            slot = k & 1
            compute.wait_event(ev_in[slot])
            step.inp = inps[slot]
            for name in names_out:
                setattr(step, name, outs[slot][name])
            step.run()
            ev_done[slot].record(compute)
            copy.wait_event(ev_done[slot])
            with torch.cuda.stream(copy):
                for name in names_out:
                    host_out[name].copy_(outs[slot][name], non_blocking=True)
            if k + 2 < n:
                stage_in(slot)
        end = torch.cuda.Event()
        end.record(copy)
        compute.wait_event(end)

    run(max(2, warmup))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(compute)
    run(steps)
    b.record(compute)
    torch.cuda.synchronize()
    step.inp = inps[0]
    for name in names_out:
        setattr(step, name, outs[0][name])
    return a.elapsed_time(b) / 1e3, h2d, d2h


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, cpu, budget_s=20.0, max_rows=64, first=0):
    """The fp64 oracle, as it stands, on whole token rows of forward +
    backward (Y row and dX row); returns (flops, seconds, rows, threads)."""
    import oracle
    from tensor_transformer_mlp_forward_gb300 import inputs

    rows_all = inputs.sample_indices(w.T, min(w.T, first + max_rows), w.seed + 7).tolist()[first:]
    per_row = 10 * w.h * w.F  # Z row, Y row, dH row, recomputed Z row, dX row: 5 x 2hF
    done, spent = 0, 0.0
    while done < len(rows_all) and (done == 0 or spent < budget_s):
        r = rows_all[done:done + 1]
        t0 = time.perf_counter()
        oracle.forward_rows(cpu, w.t, r)
        oracle.backward_rows(cpu, w.t, r)
        spent += time.perf_counter() - t0
        done += 1
    return per_row * done, spent, done, oracle.num_threads()


def cpu_baseline(w, cpu, budget_s=20.0):
    flops, secs, rows, threads = oracle_sample(w, cpu, budget_s)
    rate = flops / secs
    return {"value": rate / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} token row(s) of Y and dX (forward + backward, 10*h*F flops each) "
                      f"of the {w.name} block, fp64, {secs:.1f} s",
            # an extrapolation, not a measurement: the whole step's 12*T*h*F
            # flops at the sample's fp64 rate
            "extrapolated_full_step_s": round(w.flops_fwd_bwd() / rate, 1)}


# ------------------------------------------------------------------ main

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from tensor_transformer_mlp_forward_gb300 import inputs

    w = workload(args)
    cpu = inputs.make_inputs(w)
    total_flops, total_s, rows, threads = 0, 0.0, 0, 1
    for k in range(args.warmup + args.steps):
        f, s, r, threads = oracle_sample(w, cpu, budget_s=0.0, max_rows=1, first=k % w.T)
        if k >= args.warmup:
            total_flops += f
            total_s += s
            rows += r
    value = total_flops / total_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": describe(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"each step: 1 token row of Y and dX (forward + backward) of the "
                                   f"{w.name} block in fp64 ({rows} rows timed)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args, w):
    import torch

    from tensor_transformer_mlp_forward_gb300 import binding

    if args.pair_mode is not None:
        binding.set_cta_pair_mode(args.pair_mode)
    if args.tile_scheduler is not None:
        binding.set_tile_scheduler(args.tile_scheduler)
    if args.wide_tiles is not None:
        binding.set_wide_tiles(args.wide_tiles)
    rank, world, local = init_distributed(args.gpus)
    step, dev_s, wall, per_call, clocks, launches, split = time_ours(
        w, args.steps, args.warmup, local, args.dropout, args.recompute)
    flops = w.flops_fwd_bwd()
    max_s, units = reduce_max_sum(dev_s, flops * args.steps)
    value = units / max_s / 1e12

    e2e = None
    if not args.no_e2e:
        e_s, h2d, d2h = time_e2e(step, args.steps, args.warmup)
        e_max, e_units = reduce_max_sum(e_s, flops * args.steps)
        e2e = {"value": e_units / e_max / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}
    graph_s = time_graph(step, args.steps, args.warmup)

    burst, sustained, src = peaks()
    gemm_flops = 2 * w.T * w.h * w.F
    avg_ms = {k: statistics.mean(v) for k, v in per_call.items()}
    dominant = max(GEMM_CALLS, key=lambda k: avg_ms[k])
    achieved = gemm_flops / (avg_ms[dominant] / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": f"tcgen05_gemm ({dominant})", "achieved": achieved,
                "peak": sustained, "unit": "TFLOP/s", "frac": achieved / sustained,
                "peak_source": f"{src} bf16 sustained (MEASURED_PEAKS.json)" if src == "measured"
                               else "fallback 1.7 PFLOP/s sustained",
                "traffic": recorded_traffic(dominant, w.name)}
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(describe(w, world), **({"dropout": args.dropout} if args.dropout > 0 else {}),
                       **({"activation_recompute": "Z, H rebuilt by a2 in the backward pass; "
                           "value counts the 12*T*h*F model flops only"} if args.recompute else {})),
        "pct_of_peak": {"burst": 100 * value / world / burst, "sustained": 100 * value / world / sustained,
                        "source": src},
        "fwd_ms": round(split["fwd_ms"], 4), "bwd_ms": round(split["bwd_ms"], 4),
        # the per-call pass (an event between every two calls) takes this long a step
        "breakdown_ms_per_step": round(split["breakdown_ms_per_step"], 4),
        "per_call_ms": {k: round(v, 4) for k, v in avg_ms.items()},
        # db2: the column sums of dY, HBM-bound: 2 T h bytes read, 4 h written
        "db2_gbs": round((2 * w.T * w.h + 4 * w.h) / (avg_ms["db2"] / 1e3) / 1e9, 1),
        "roofline": roofline,
        "e2e": e2e,
        # the same step captured once as a CUDA graph and replayed: the device
        # time without the host's per-call launch work between kernels
        "graph": {"ms_per_step": 1e3 * graph_s / args.steps,
                  "value": flops * args.steps / graph_s / 1e12},
        "clocks": clocks,
        "gpu_launches": launches,
        "gemm_kernel": {0: "single CTA", 1: "auto", 2: "CTA pairs"}[
            args.pair_mode if args.pair_mode is not None else 1],
    }
    if args.wide_tiles:
        line["gemm_kernel"] += ", 256 x 512 tiles for dX"
    if args.recompute:  # the rebuilt a2 is a seventh GEMM of 2*T*h*F flops
        line["hardware_tflops"] = value * 14 / 12
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, step.cpu)
    print(json.dumps(line))
    return 0


def run_layernorm(args, w):
    """Residual add + LayerNorm on the workload's activations [T, h]: HBM GB/s
    of the forward and backward calls against the measured copy bandwidth."""
    import torch

    from tensor_transformer_mlp_forward_gb300 import binding

    dev = torch.device("cuda", 0)
    T, h = w.T, w.h
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    bf = lambda *sh: torch.randn(*sh, generator=gen, device=dev).to(torch.bfloat16)  # noqa: E731
    a, r, dX, dres = bf(T, h), bf(T, h), bf(T, h), bf(T, h)
    gam, bet = bf(h), bf(h)
    X, s = torch.empty_like(a), torch.empty_like(a)
    ds = torch.empty_like(a)
    mean = torch.empty(T, device=dev)
    rstd = torch.empty(T, device=dev)
    dg, db = torch.empty(h, device=dev), torch.empty(h, device=dev)
    part = torch.empty(max(1, int(binding.lib().tp_ln_residual_backward_workspace_floats(T, h))),
                       device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    fwd = lambda: binding.tp_ln_residual_forward(a, r, gam, bet, 1e-5, X=X, s=s, mean=mean, rstd=rstd)  # noqa: E731
    bwd = lambda: binding.tp_ln_residual_backward(dX, dres, a, r, gam, mean, rstd, ds=ds,  # noqa: E731
                                                  dgamma=dg, dbeta=db, partial=part)
    out = {}
    for name, fn, algo in (("forward", fwd, 8 * T * h), ("backward", bwd, 10 * T * h)):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.mean(ts)
        out[name] = {"ms": round(ms, 4), "algorithmic_bytes": algo,
                     "gbs": round(algo / (ms / 1e3) / 1e9, 1)}
    try:
        peak = float(json.load(open(PEAKS_FILE))["hbm_gbs"])
        src = "measured"
    except Exception:
        peak, src = 6800.0, "fallback"
    for v in out.values():
        v["frac_of_hbm"] = round(v["gbs"] / peak, 3)
    print(json.dumps({"metric": "GB/s of residual add + LayerNorm (fwd, bwd) on 1 GB300",
                      "unit": "GB/s", "config": {"workload": f"{w.name} activations (T={w.T}, h={w.h})"},
                      "hbm_peak_gbs": peak, "peak_source": src, "steps": args.steps,
                      "l2": "L2 flushed between timed calls", **out}))
    return 0


# -------------------------------------------------------- attention block

ATTN_CALLS = ("qkv", "core_fwd", "out_proj", "dbo", "dWo", "dO", "core_bwd", "dbqkv", "dWqkv",
              "dX")


class AttnStep:
    """All buffers of the attention block, resident in HBM; run() issues one
    forward + backward step as the library's calls (tp_attn_forward and
    tp_attn_backward issue the same calls in the same order)."""

    def __init__(self, w, device):
        import torch

        from tensor_transformer_mlp_forward_gb300 import binding, inputs

        self.b, self.w = binding, w
        T, h, nh = w.T, w.h, w.nh
        self.cpu = inputs.make_attn_inputs(w)
        self.inp = {k: v.to(device) for k, v in self.cpu.items()}
        e = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        self.QKV, self.O, self.Y = e(T, 3 * h), e(T, h), e(T, h)
        self.lse, self.delta = e(nh, T, dt=torch.float32), e(nh, T, dt=torch.float32)
        self.dO, self.dQKV, self.dX = e(T, h), e(T, 3 * h), e(T, h)
        self.dWqkv, self.dWo = e(h, 3 * h), e(h, h)
        self.dbqkv, self.dbo = e(3 * h, dt=torch.float32), e(h, dt=torch.float32)
        lib = binding.lib()
        self.p_sum = e(max(1, int(lib.tp_mlp_bias_grad_workspace_floats(T, 3 * h)),
                           int(lib.tp_mlp_bias_grad_workspace_floats(T, h))), dt=torch.float32)
        # the weight gradients in K-major form where tp_attn_backward takes it
        self.kmajor_o = binding.weight_grad_kmajor(h, h)
        self.kmajor_qkv = binding.weight_grad_kmajor(h, 3 * h)
        # split reductions: the row-parallel GEMMs', and the MN-major weight
        # gradients' where their few output tiles leave SM pairs idle
        self.ws = e(max(16, binding.split_workspace_bytes(T, h, 3 * h, 1),
                        binding.split_workspace_bytes(T, h, h, w.t),
                        0 if self.kmajor_o else binding.weight_grad_workspace_bytes(T, h, h),
                        0 if self.kmajor_qkv else binding.weight_grad_workspace_bytes(T, h, 3 * h)),
                    dt=torch.uint8)
        self.ws_core = e(max(16, int(lib.tp_attn_core_workspace_bytes(w.nb, w.s, h, nh))),
                         dt=torch.uint8)
        self.launches = 0
        ldT = binding.pitch(T)
        if self.kmajor_o:
            self.Ot, self.dYt = e(h, ldT), e(h, ldT)
        if self.kmajor_qkv:
            self.Xt, self.dQKVt = e(h, ldT), e(3 * h, ldT)
        self.names = (ATTN_CALLS[:4] + (("t_O", "t_dY") if self.kmajor_o else ()) + ATTN_CALLS[4:8]
                      + (("t_X", "t_dQKV") if self.kmajor_qkv else ()) + ATTN_CALLS[8:])

    def run(self, events=None):
        b, i, w = self.b, self.inp, self.w
        calls = (
            lambda: b.tp_attn_qkv(i["X"], i["Wqkv"], i["bqkv"], QKV=self.QKV),
            lambda: b.tp_attn_core_forward(self.QKV, w.nb, w.nh, O=self.O, lse=self.lse,
                                           workspace=self.ws_core),
            lambda: b.tp_mlp_row_sum(self.O, i["Wo"], i["bo"], i["residual"], w.t, Y=self.Y,
                                     workspace=self.ws),
            lambda: b.tp_mlp_bias_grad(i["dY"], db=self.dbo, partial=self.p_sum),
        )
        if self.kmajor_o:
            calls += (
                lambda: b.tp_transpose(self.O, out=self.Ot),
                lambda: b.tp_transpose(i["dY"], out=self.dYt),
                lambda: b.tp_mlp_dB_kmajor(self.Ot, self.dYt, w.T, 1, dB=self.dWo),
            )
        else:
            calls += (lambda: b.tp_mlp_dB_ws(self.O, i["dY"], 1, dB=self.dWo, workspace=self.ws),)
        calls += (
            lambda: b.tp_mlp_dx(i["dY"], i["Wo"], 1, dX=self.dO, workspace=self.ws),
            lambda: b.tp_attn_core_backward(self.QKV, self.O, self.lse, self.dO, w.nb, w.nh,
                                            dQKV=self.dQKV, delta=self.delta,
                                            workspace=self.ws_core),
            lambda: b.tp_mlp_bias_grad(self.dQKV, db=self.dbqkv, partial=self.p_sum),
        )
        if self.kmajor_qkv:
            calls += (
                lambda: b.tp_transpose(i["X"], out=self.Xt),
                lambda: b.tp_transpose(self.dQKV, out=self.dQKVt),
                lambda: b.tp_mlp_dA_kmajor(self.Xt, self.dQKVt, w.T, 1, dA=self.dWqkv),
            )
        else:
            calls += (lambda: b.tp_mlp_dA_ws(i["X"], self.dQKV, 1, dA=self.dWqkv, workspace=self.ws),)
        calls += (lambda: b.tp_mlp_dx(self.dQKV, i["Wqkv"], 1, dX=self.dX, workspace=self.ws),)
        if events is not None:
            events[0].record()
        for k, c in enumerate(calls):
            c()
            self.launches += b.last_launch_count()
            if events is not None:
                events[k + 1].record()


def attn_cpu_baseline(w, cpu, budget_s=20.0):
    """The oracle's per-head entry points, as they stand, on whole heads
    (forward output and every parameter gradient of the head)."""
    import oracle

    pairs = w.nb * w.s * (w.s + 1) // 2
    d, T, h = w.d, w.T, w.h
    per_head = (3 * (2 * T * h * 3 * d + 2 * T * d * h) + 12 * pairs * d)
    done, spent = 0, 0.0
    while done < w.nh and (done == 0 or spent < budget_s):
        t0 = time.perf_counter()
        oracle.attn_head(cpu, w.nb, w.nh, done)
        oracle.attn_head_grads(cpu, w.nb, w.nh, done)
        spent += time.perf_counter() - t0
        done += 1
    return {"value": per_head * done / spent / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done} head(s) of the {w.name} block: O_j and dWqkv_j, dbqkv_j, dWo_j "
                      f"(forward + backward of the head's share), fp64, {spent:.1f} s"}


def run_attention(args):
    import torch

    from tensor_transformer_mlp_forward_gb300 import inputs

    w = inputs.ATTN_WORKLOADS[args.attn_workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    step = AttnStep(w, dev)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    assert step.b.device_status() == 0, "device wait timed out during warm-up"
    step.launches = 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(step.names) + 1)]
           for _ in range(args.steps)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        w0 = time.time()
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            step.run(evs[k])
        torch.cuda.synchronize()
        clocks.mark(w0, time.time())
    assert step.b.device_status() == 0, "device wait timed out"
    dev_s = sum(evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)) / 1e3
    per_call = {n: statistics.mean(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps))
                for j, n in enumerate(step.names)}
    flops = w.flops_fwd_bwd()
    value = flops * args.steps / dev_s / 1e12
    burst, sustained, src = peaks()
    pairs = w.nb * w.s * (w.s + 1) // 2
    core = {"core_fwd": 4 * pairs * w.h, "core_bwd": 8 * pairs * w.h}
    core_tf = {k: v / (per_call[k] / 1e3) / 1e12 for k, v in core.items()}
    dominant = max(core, key=lambda k: per_call[k])
    roofline = {"bound": "tensor", "kernel": "attn_fwd_kernel" if dominant == "core_fwd"
                else "attn_bwd_dq_kernel + attn_bwd_dkdv_kernel",
                "achieved": core_tf[dominant], "peak": burst, "unit": "TFLOP/s",
                "frac": core_tf[dominant] / burst,
                "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json)", "traffic": None,
                "algorithmic_flops": {"core_fwd": "4 d per visible (query, key) pair per head",
                                      "core_bwd": "8 d per visible pair per head (dP, dV, dQ, dK; "
                                                  "the recomputed S is not counted)"}}
    e2e = None
    if not args.no_e2e:
        e_s, h2d, d2h = time_e2e(step, args.steps, args.warmup)
        e2e = {"value": flops * args.steps / e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}
    line = {
        "metric": "TFLOPS fwd+bwd of the head-parallel causal attention block on 1 GB300",
        "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dev_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name} attention block (nb={w.nb}, s={w.s}, h={w.h}, nh={w.nh}, "
                               f"d={w.d}, t={w.t}, causal)",
                   "l2": "L2 flushed between timed steps (256 MiB write)",
                   "flops": "projections 3 x (2 T h 3h + 2 T h h) + 12 d per visible pair per head"},
        "pct_of_peak": {"burst": 100 * value / burst, "sustained": 100 * value / sustained,
                        "source": src},
        "per_call_ms": {k: round(v, 4) for k, v in per_call.items()},
        "core_tflops": {k: round(v, 1) for k, v in core_tf.items()},
        "roofline": roofline, "e2e": e2e, "clocks": clocks.summary(),
        "gpu_launches": step.launches,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = attn_cpu_baseline(w, step.cpu)
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------- one call

def run_call(a) -> int:
    """One entry point of the library, --repeat times at --shape, with only
    that call's operands on the device (seeded device-side normals: a profile
    depends on the shapes, not the values).  Prints one JSON line with the
    CUDA-event time of each call.  With --vs-cublas (column_gelu, dx,
    dA_kmajor, dB_kmajor) the call and the plain cuBLAS product of the same
    shapes (torch.matmul, bf16, no epilogue) alternate in rounds of 5 calls,
    and the line gives both medians."""
    import torch

    from tensor_transformer_mlp_forward_gb300 import binding as b

    T, h, F, t = (int(v) for v in a.shape.split(","))
    p_drop = a.dropout if a.dropout > 0 else 0.1
    if a.tile_scheduler is not None:
        b.set_tile_scheduler(a.tile_scheduler)
    if a.wide_tiles is not None:
        b.set_wide_tiles(a.wide_tiles)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(1234)

    def bf(*shape, std=1.0):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)

    c = a.call
    ref = None  # the plain cuBLAS product of the call's shapes (--vs-cublas)
    if c in ("column_gelu", "column_gelu_h_only"):
        X, A, b1 = bf(T, h), bf(h, F, std=0.02), bf(F, std=0.02)
        Z = None if c == "column_gelu_h_only" else bf(T, F)
        H = bf(T, F)
        fn = lambda: b.tp_mlp_column_gelu(X, A, b1, t, Z=Z, H=H, want_z=Z is not None)  # noqa: E731
        C = torch.empty(T, F, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(X, A, out=C)  # noqa: E731
    elif c in ("row_sum", "row_sum_dropout"):
        H, B, b2, R, Y = bf(T, F), bf(F, h, std=0.02), bf(h, std=0.02), bf(T, h), bf(T, h)
        ws = torch.empty(max(16, b.split_workspace_bytes(T, h, F, t)), dtype=torch.uint8, device=dev)
        if c == "row_sum":
            fn = lambda: b.tp_mlp_row_sum(H, B, b2, R, t, Y=Y, workspace=ws)  # noqa: E731
        else:
            fn = lambda: b.tp_mlp_row_sum_dropout(H, B, b2, R, t, p_drop, 7, 0, Y=Y,  # noqa: E731
                                                  workspace=ws)
    elif c == "dgelu":
        dY, B, Z, dZ = bf(T, h), bf(F, h, std=0.02), bf(T, F), bf(T, F)
        db1 = torch.empty(F, device=dev)
        part = torch.empty(max(1, int(b.lib().tp_mlp_dgelu_partial_floats(T, F))), device=dev)
        fn = lambda: b.tp_mlp_dgelu(dY, B, Z, t, dZ=dZ, db1=db1, partial=part)  # noqa: E731
    elif c == "dx":
        dZ, A, dX = bf(T, F), bf(h, F, std=0.02), bf(T, h)
        ws = torch.empty(max(16, b.split_workspace_bytes(T, h, F, t)), dtype=torch.uint8, device=dev)
        fn = lambda: b.tp_mlp_dx(dZ, A, t, dX=dX, workspace=ws)  # noqa: E731
        C = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(dZ, A.t(), out=C)  # noqa: E731
    elif c == "dA":
        X, dZ, dA = bf(T, h), bf(T, F), bf(h, F)
        fn = lambda: b.tp_mlp_dA(X, dZ, t, dA=dA)  # noqa: E731
    elif c == "dB":
        H, dY, dB = bf(T, F), bf(T, h), bf(F, h)
        fn = lambda: b.tp_mlp_dB(H, dY, t, dB=dB)  # noqa: E731
    elif c == "dA_kmajor":  # from X^T [h, ldT] and dZ^T [F, ldT]
        ld = b.pitch(T)
        Xt, dZt, dA = bf(h, ld), bf(F, ld), bf(h, F)
        fn = lambda: b.tp_mlp_dA_kmajor(Xt, dZt, T, t, dA=dA)  # noqa: E731
        C = torch.empty(h, F, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(Xt[:, :T], dZt[:, :T].t(), out=C)  # noqa: E731
    elif c == "dB_kmajor":  # from H^T [F, ldT] and dY^T [h, ldT]
        ld = b.pitch(T)
        Ht, dYt, dB = bf(F, ld), bf(h, ld), bf(F, h)
        fn = lambda: b.tp_mlp_dB_kmajor(Ht, dYt, T, t, dB=dB)  # noqa: E731
        C = torch.empty(F, h, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(Ht[:, :T], dYt[:, :T].t(), out=C)  # noqa: E731
    elif c == "transpose":  # dZ [T, F] -> dZ^T [F, ldT]
        dZ = bf(T, F)
        dZt = torch.empty(F, b.pitch(T), dtype=torch.bfloat16, device=dev)
        fn = lambda: b.tp_transpose(dZ, out=dZt)  # noqa: E731
    elif c == "dropout_grad":
        dY, dP = bf(T, h), bf(T, h)
        fn = lambda: b.tp_mlp_dropout_grad(dY, p_drop, 7, 0, dP=dP)  # noqa: E731
    elif c == "bias_grad":  # db2 = column sums of dY [T, h]
        dY, db = bf(T, h), torch.empty(h, device=dev)
        part = torch.empty(max(1, int(b.lib().tp_mlp_bias_grad_workspace_floats(T, h))), device=dev)
        fn = lambda: b.tp_mlp_bias_grad(dY, db=db, partial=part)  # noqa: E731
    else:
        x, r, gam, bet = bf(T, h), bf(T, h), bf(h, std=0.1), bf(h, std=0.1)
        X, s = torch.empty_like(x), torch.empty_like(x)
        mean, rstd = torch.empty(T, device=dev), torch.empty(T, device=dev)
        b.tp_ln_residual_forward(x, r, gam, bet, 1e-5, X=X, s=s, mean=mean, rstd=rstd)
        if c == "ln_forward":
            fn = lambda: b.tp_ln_residual_forward(x, r, gam, bet, 1e-5, X=X, s=s,  # noqa: E731
                                                  mean=mean, rstd=rstd)
        else:
            dX, dres, ds = bf(T, h), bf(T, h), torch.empty_like(x)
            dg, dbt = torch.empty(h, device=dev), torch.empty(h, device=dev)
            part = torch.empty(max(1, int(b.lib().tp_ln_residual_backward_workspace_floats(T, h))),
                               device=dev)
            fn = lambda: b.tp_ln_residual_backward(dX, dres, x, r, gam, mean, rstd, ds=ds,  # noqa: E731
                                                   dgamma=dg, dbeta=dbt, partial=part)
    if a.vs_cublas:
        if ref is None:
            raise SystemExit(f"--vs-cublas is not defined for {c}")
        return compare_cublas(c, fn, ref, a, 2.0 * T * h * F)
    ms = []
    for _ in range(a.repeat):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    status = b.device_status()
    print(json.dumps({"call": c, "T": T, "h": h, "F": F, "t": t, "repeat": a.repeat,
                      "launches_per_call": b.last_launch_count(),
                      "ms_mean_after_first": sum(ms[1:]) / max(1, len(ms) - 1), "ms": ms,
                      "device_status": status}))
    return 0 if status == 0 else 1


def compare_cublas(call, fn, ref, a, flops) -> int:
    """The call and cuBLAS alternating in rounds (the order flips each round),
    5 calls a round, the first of each round dropped; medians of the rest."""
    import torch

    from tensor_transformer_mlp_forward_gb300 import binding as b

    for f in (fn, ref, fn, ref):
        f()
    torch.cuda.synchronize()
    res = {"ours": [], "cublas": []}
    for rnd in range(a.rounds):
        order = (("ours", fn), ("cublas", ref)) if rnd % 2 == 0 else (("cublas", ref), ("ours", fn))
        for tag, f in order:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            ev[0].record()
            for k in range(5):
                f()
                ev[k + 1].record()
            torch.cuda.synchronize()
            res[tag] += [ev[k].elapsed_time(ev[k + 1]) for k in range(1, 5)]
    mo, mc = statistics.median(res["ours"]), statistics.median(res["cublas"])
    status = b.device_status()
    print(json.dumps({"call": call, "ours_ms": mo, "cublas_ms": mc, "ours_over_cublas": mo / mc,
                      "ours_tflops": flops / mo / 1e9, "cublas_tflops": flops / mc / 1e9,
                      "samples": len(res["ours"]), "device_status": status}))
    return 0 if status == 0 else 1


def main(argv=None):
    args = parse_args(argv)
    if args.call:
        return run_call(args)
    if args.attention and args.impl == "ours":
        return run_attention(args)
    if args.layernorm:
        return run_layernorm(args, workload(args))
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep or args.all_configs:
        from tensor_transformer_mlp_forward_gb300 import inputs

        points = [("sweep-h4096", T, t) for T in inputs.SWEEP_TOKENS for t in inputs.SWEEP_SHARDS]
        if args.all_configs:
            points = [("tiny", 128, 2), ("gpt2-medium", 8192, 1), ("gpt2-medium", 8192, 2)] + [
                ("megatron-8.3b", 8192, t) for t in (8, 1, 2, 4)] + [
                ("mt-nlg-530b", 2048, 8)] + points
        for name, T, t in points:
            a = parse_args(["--workload", name, "--tokens", str(T), "--shards", str(t),
                            "--steps", str(args.steps), "--warmup", str(args.warmup),
                            "--no-cpu-baseline", "--no-e2e"])
            run_ours(a, workload(a))
        return 0
    return run_ours(args, workload(args))


if __name__ == "__main__":
    sys.exit(main())
