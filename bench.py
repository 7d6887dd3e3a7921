#!/usr/bin/env python
"""Benchmark of the INT8 mixed-precision linear-layer hot path on GB300.

One step = forward + backward (grad-input and grad-weight) of the seven
linear layers of one Llama2-1B-shaped decoder layer (q, k, v, o 2048x2048;
gate, up 5632x2048; down 2048x5632) over 16 x 2048 = 32768 tokens, every
matmul in INT8 with dynamic row-wise quantization along its contraction axis
("Quantized model training" README, INT8 mixed precision training; LM head
excluded).  Activations N(0,1), weights N(0,0.02), output gradients
N(0,1e-3), round to nearest even.  Inputs are resident in HBM before the
timed region; every step touches about 5 GB, far more than the 129 MB L2.
Under torchrun with N ranks (one GPU each) the step is data parallel over
tokens: every rank runs its own 16 x 2048 tokens (weak scaling), and the
grad-weight pass forms fp32 partials that one NCCL all-reduce per linear sums
(started when the part is formed, running while the later linears compute)
before a single bf16 rounding (int8_mixed_precision_row_gb300/dp.py).

Output: one JSON line (rank 0).  `value` is whole-job tokens/s; `e2e` is the
same metric through the layer API (int8mp_linear_fwd_save /
int8mp_linear_bwd_saved) with inputs copied from pinned
host memory and dW copied back inside the timed region; `roofline` describes
the dominant kernel (the tensor-core GEMM); `cpu_baseline` times the plain-C
oracle on a bounded token sample on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quant+INT8 scaled-mm TOPS; fwd+bwd linear tok/s at Llama2-1B shapes"
WORKLOAD = ("llama2-1b decoder-layer linears (q,k,v,o 2048x2048; gate,up 5632x2048; "
            "down 2048x5632) fwd+grad_in+grad_w, all INT8, T=16x2048 tokens")
ORACLE_SAMPLE_TOKENS = 512


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", action="store_true",
                    help="short run for a profiler: no extras, no e2e, no CPU baseline")
    ap.add_argument("--tokens", type=int, default=None,
                    help="profiling cases only: tokens per step instead of 16x2048")
    ap.add_argument("--linears", default=None,
                    help="profiling cases only: comma-separated subset of q,k,v,o,gate,up,down")
    ap.add_argument("--rounding", choices=["rne", "sr"], default="rne",
                    help="profiling cases only: round to nearest even or stochastically")
    ap.add_argument("--case", choices=sorted(PROFILE_CASES), default=None,
                    help="profiling: run one matmul case three times and exit (no timing)")
    return ap.parse_args()


# Single-call cases for a profiler (each runs its call three times, so that
# `ncu -s 2 -c 1` captures a warm launch): the square 4096^3 A @ B.T matmul
# on int8 codes and on f16 containers of the same codes, and the BF16
# forward pass of a q projection at T = 16384; quantize-AxB-2048: the two
# quantizations of a 2048^3 A @ B (A by rows, B by columns in place; two
# launches per call).
PROFILE_CASES = ("square-int8-4096", "square-f16-4096", "square-f16-2048", "square-f16-1024",
                 "bf16-forward-q-T16384", "forward-q-T16384-w-codes",
                 "forward-q-T16384-w-quantized-in-prologue", "quantize-AxB-2048")


def run_profile_case(case, device):
    import torch
    import int8_mixed_precision_row_gb300 as m
    from int8_mixed_precision_row_gb300 import synth
    g = torch.Generator(device=device).manual_seed(0)
    if case.startswith("square"):
        S = int(case.rsplit("-", 1)[1])
        a = torch.randint(-127, 128, (S, S), device=device, generator=g, dtype=torch.int32)
        b = torch.randint(-127, 128, (S, S), device=device, generator=g, dtype=torch.int32)
        dt = torch.int8 if case == "square-int8-4096" else torch.float16
        a, b = a.to(dt), b.to(dt)
        sa = torch.rand(S, device=device, generator=g)
        sb = torch.rand(S, device=device, generator=g)
        out = torch.empty((S, S), dtype=torch.bfloat16, device=device)
        ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=device)
        for _ in range(3):
            m.int8mp_scaled_mm(a, sa, b, sb, out=out, workspace=ws)
    elif case.startswith("quantize-AxB"):
        S = int(case.rsplit("-", 1)[1])
        A = synth.bf16_normal((S, S), 1).to(device)
        B = synth.bf16_normal((S, S), 2).to(device)
        qa = torch.empty((S, S), dtype=torch.float16, device=device)
        qb = torch.empty((S, S), dtype=torch.float16, device=device)
        sa = torch.empty(S, dtype=torch.float32, device=device)
        sb = torch.empty(S, dtype=torch.float32, device=device)
        for _ in range(3):
            m.int8mp_quantize_rowwise(A, axis=0, codes=m.INT8MP_CODES_F16, q=qa, scale=sa)
            m.int8mp_quantize_rowwise(B, axis=m.INT8MP_GROUP_COLS, codes=m.INT8MP_CODES_F16, q=qb,
                                      scale=sb)
    elif case.startswith("forward-q-T16384"):
        # the forward matmul of a q projection on X's codes, with W's codes
        # from the row pass, or W quantized in the GEMM's prologue from its
        # row scales (the row pass's scales)
        X = synth.bf16_normal((16384, 2048), 10).to(device)
        W = synth.bf16_normal((2048, 2048), 20, std=0.02).to(device)
        (qx, sx), (qw, sw) = m.int8mp_quantize_rows_batch([X, W], codes=m.INT8MP_CODES_F16)
        Y = torch.empty((16384, 2048), dtype=torch.bfloat16, device=device)
        for _ in range(3):
            if case.endswith("in-prologue"):
                m.int8mp_debug_scaled_mm_quant_b(qx, sx, W, sw, out=Y)
            else:
                m.int8mp_scaled_mm(qx, sx, qw, sw, out=Y)
    else:
        X = synth.bf16_normal((16384, 2048), 10).to(device)
        W = synth.bf16_normal((2048, 2048), 20, std=0.02).to(device)
        cfg = m.linear_cfg(int8_fwd=0, int8_grad_in=0, int8_grad_w=0)
        Y = torch.empty((16384, 2048), dtype=torch.bfloat16, device=device)
        for _ in range(3):
            m.int8mp_linear_fwd(X, W, cfg, Y=Y)
    torch.cuda.synchronize()
    if m.int8mp_poll_device_status() != m.INT8MP_OK:
        raise RuntimeError("a bounded device wait ran out")
    print(f"profile case {case}: done")


# ------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world, device=None):
    """Largest value over all ranks (the job takes as long as its slowest
    rank).  No data-path collective: the replicas share nothing else."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "temperature.gpu,clocks.mem")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        temp = [num(r[9]) for r in rows if len(r) > 9 and num(r[9]) is not None]
        mem = [num(r[10]) for r in rows if len(r) > 10 and num(r[10]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "temp_c_max": max(temp) if temp else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- workload
class LayerStep:
    """Device-resident inputs, outputs and code/scale buffers of one decoder
    layer's linears, and the step composed of the public C-ABI calls."""

    def __init__(self, spec, mode, device, T=None, only=None, world=1, rank=0):
        import torch
        from int8_mixed_precision_row_gb300 import dp, synth
        import int8_mixed_precision_row_gb300 as m
        self.m = m
        self.dp = dp
        self.world, self.rank = world, rank
        self.spec = spec
        self.T = spec["T"] if T is None else T
        self.mode = mode
        self.device = device
        if only:
            spec = dict(spec, linears=[l for l in spec["linears"] if l[0] in only])
            self.spec = spec
        host = synth.layer_inputs(spec, T=self.T)
        self.host = host
        dev_cache = {}

        def on_dev(t):
            key = id(t)
            if key not in dev_cache:
                dev_cache[key] = t.to(device)
            return dev_cache[key]
        self.linears = []
        T = self.T
        for name, (X, W, dY) in host.items():
            N, K = W.shape
            self.linears.append({
                "name": name, "N": N, "K": K, "X": on_dev(X), "W": on_dev(W), "dY": on_dev(dY),
                "Y": torch.empty((T, N), dtype=torch.bfloat16, device=device),
                "dX": torch.empty((T, K), dtype=torch.bfloat16, device=device),
                "dW": torch.empty((N, K), dtype=torch.bfloat16, device=device)})
        nmax = max(l["N"] for l in self.linears)
        kmax = max(l["K"] for l in self.linears)
        big = max(T * kmax, T * nmax, nmax * kmax)
        f16 = torch.float16
        # code buffers (f16 containers) and scales, reused linear after linear
        self.qa = torch.empty(big, dtype=f16, device=device)
        self.qb = torch.empty(big, dtype=f16, device=device)
        self.sa = torch.empty(max(T, nmax, kmax), dtype=torch.float32, device=device)
        self.sb = torch.empty(max(T, nmax, kmax), dtype=torch.float32, device=device)
        # column absmax of X, W (recorded by their forward row passes) and dY
        # (by its grad-input row pass), per linear [K | K | N], all linears in
        # one buffer cleared once per step
        sizes = [2 * l["K"] + l["N"] for l in self.linears]
        self.colmax_all = torch.empty(sum(sizes), dtype=torch.float32, device=device)
        at = 0
        for l, n in zip(self.linears, sizes):
            l["colmax"] = self.colmax_all[at:at + n]
            at += n
        # the matmuls' scratch for splitting their last wave of tiles
        self.mm_ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=device)
        # data parallel (world > 1): each rank's fp32 part of dW per linear,
        # summed by an all-reduce and rounded once; the all-reduces run while
        # the later linears compute, and the roundings end the step
        self.dw_f32 = ([torch.empty((l["N"], l["K"]), dtype=torch.float32, device=device)
                        for l in self.linears] if world > 1 else None)
        self.flops = 6.0 * T * sum(l["N"] * l["K"] for l in self.linears)
        # GEMM operands read once (f16 codes) and bf16 outputs written, per step
        self.gemm_bytes = 6.0 * sum(T * l["K"] + T * l["N"] + l["N"] * l["K"] for l in self.linears)
        self.gemms_per_step = 3 * len(self.linears)
        # kernels of this library per step and linear: two row-quantization
        # launches (X and W together, then dY; each also recording column
        # absmax), three column quantizations (codes from that absmax), three
        # GEMMs
        self.kernels_per_step = len(self.linears) * (2 + 3 + 3 + (1 if world > 1 else 0))
        # algorithmic quantize bytes: bf16 read once, code (f16 container) and scale written
        self.quant_elems = sum(2 * (T * l["K"] + l["N"] * l["K"] + T * l["N"]) for l in self.linears)

    def _q(self, x, axis, sid, qbuf, sbuf, cfg_seed, cfg_off, colmax):
        """axis 0: row groups, recording each column's absmax into colmax;
        2: column groups, codes in x's layout, from that absmax."""
        m = self.m
        rows, cols = x.shape
        q = qbuf[:rows * cols].view(rows, cols)
        kw = dict(mode=self.mode, seed=cfg_seed, offset=cfg_off, stream_id=sid,
                  codes=m.INT8MP_CODES_F16, q=q)
        if axis == 0:
            s = sbuf[:rows]
            m.int8mp_quantize_rows_colmax(x, colmax, scale=s, **kw)
        else:
            s = sbuf[:cols]
            m.int8mp_quantize_cols_absmax(x, colmax, scale=s, **kw)
        return q, s

    def _q_rows2(self, X, W, cx, cw, seed, offset):
        """X and W by rows in one launch, each recording its column absmax."""
        m = self.m
        (T, K), N = X.shape, W.shape[0]
        return m.int8mp_quantize_rows_batch(
            [X, W], mode=self.mode, seed=seed, offsets=[offset, offset],
            stream_ids=[m.INT8MP_STREAM_FWD_X, m.INT8MP_STREAM_FWD_W], codes=m.INT8MP_CODES_F16,
            qs=[self.qa[:T * K].view(T, K), self.qb[:N * K].view(N, K)],
            scales=[self.sa[:T], self.sb[:N]], colmaxes=[cx, cw])

    def run(self, timers=None, seed=0, offset=0):
        """One step.  timers: optional dict of kernel class -> list of
        (start, end) CUDA event pairs recorded around each call."""
        m = self.m
        import torch

        def rec(kind, fn):
            if timers is None:
                return fn()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            r = fn()
            b.record()
            timers.setdefault(kind, []).append((a, b))
            return r
        # data parallel: rank r's stochastic-rounding counters start at
        # offset + r * 2^40 (disjoint streams); rank 0 (and one GPU) as given
        offset = self.dp.shard_offset(offset, self.rank)
        self.colmax_all.zero_()
        pending = []  # data parallel: (all-reduce in flight, fp32 part, dW)
        for i, l in enumerate(self.linears):
            X, W, dY = l["X"], l["W"], l["dY"]
            K = l["K"]
            cm = l["colmax"]
            cx, cw, cg = cm[:K], cm[K:2 * K], cm[2 * K:]
            # forward: X and W along K (their rows, one launch); their column
            # absmax on the way
            (qx, sx), (qw, sw) = rec("quant_rows", lambda: self._q_rows2(X, W, cx, cw, seed, offset))
            rec("gemm", lambda: m.int8mp_scaled_mm(qx, sx, qw, sw, out=l["Y"], workspace=self.mm_ws))
            # grad input: dY along N (rows), W along N (columns, codes [N, K]): A @ B
            qg, sg = rec("quant_rows", lambda: self._q(dY, 0, m.INT8MP_STREAM_GI_DY, self.qa, self.sa, seed, offset, cg))
            qwc, swc = rec("quant_cols", lambda: self._q(W, 2, m.INT8MP_STREAM_GI_W, self.qb, self.sb, seed, offset, cw))
            rec("gemm", lambda: m.int8mp_scaled_mm(qg, sg, qwc, swc, layout=m.INT8MP_AxB, out=l["dX"],
                                                   workspace=self.mm_ws))
            # grad weight: dY and X along T (columns, codes [T, N], [T, K]): A.T @ B
            qgc, sgc = rec("quant_cols", lambda: self._q(dY, 2, m.INT8MP_STREAM_GW_DY, self.qa, self.sa, seed, offset, cg))
            qxc, sxc = rec("quant_cols", lambda: self._q(X, 2, m.INT8MP_STREAM_GW_X, self.qb, self.sb, seed, offset, cx))
            if self.world == 1:
                rec("gemm", lambda: m.int8mp_scaled_mm(qgc, sgc, qxc, sxc, layout=m.INT8MP_ATxB,
                                                       out=l["dW"], workspace=self.mm_ws))
            else:
                # this rank's fp32 part of dW, its all-reduce started (it runs
                # while the next linears compute), one rounding at the end
                part = self.dw_f32[i]
                rec("gemm", lambda: m.int8mp_scaled_mm_f32(qgc, sgc, qxc, sxc, layout=m.INT8MP_ATxB,
                                                           out=part, workspace=self.mm_ws))
                work = self.dp.reduce_partials(part, async_op=True)
                pending.append((work, part, l["dW"]))
        for work, part, dW in pending:
            rec("allreduce", work.wait)
            rec("round", lambda: m.int8mp_round_bf16(part.view(-1), dW.view(-1)))


def time_steps(step, steps, warmup, world, device):
    """`steps` steps timed end to end with nothing but the workload between
    the two events; then, for the per-kernel breakdown, up to 20 more steps
    with CUDA events around every call (their per-kind sums are scaled to
    `steps` steps)."""
    import torch
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step.run()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    elapsed_ms = start.elapsed_time(end)
    timers = {}
    n_inst = max(1, min(steps, 20))
    for _ in range(n_inst):
        step.run(timers=timers)
    torch.cuda.synchronize()
    scale = steps / n_inst
    per_kind = {k: scale * sum(a.elapsed_time(b) for a, b in v) for k, v in timers.items()}
    counts = {k: round(scale * len(v)) for k, v in timers.items()}
    return elapsed_ms, per_kind, counts


def time_e2e(step, steps, warmup):
    """Same step through int8mp_linear_fwd_save / int8mp_linear_bwd_saved (the
    layer API: the forward pass keeps X's and W's column absmax for the
    backward pass), inputs copied from pinned host memory each step and dW
    copied back.  Copies run on their own streams (copy engines) and overlap
    the compute of other linears: a linear's inputs are copied in as soon as
    the previous step's last reader of that buffer is done, its compute waits
    for them, and its dW goes back while the next linear computes."""
    import torch
    m = step.m
    cfg = m.linear_cfg(mode=step.mode)
    pinned = {}
    for l, (name, (X, W, dY)) in zip(step.linears, step.host.items()):
        ins = []
        for key, t in (("X", X), ("W", W), ("dY", dY)):
            if id(t) not in pinned:
                pinned[id(t)] = (t.pin_memory(), l[key])
            ins.append(id(t))
        l["inputs"] = ins
        l["hdW"] = torch.empty(l["dW"].shape, dtype=torch.bfloat16).pin_memory()
    ws_bytes = max(m.int8mp_linear_workspace_size(step.T, l["N"], l["K"], cfg) for l in step.linears)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=step.device)
    h2d = sum(h.numel() * 2 for h, _ in pinned.values())
    d2h = sum(l["dW"].numel() * 2 for l in step.linears)
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    last_read = {}   # input buffer -> compute event of its last reader so far
    dw_back = {}     # linear -> event: its dW has reached the host

    def event(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    copies = []      # (bytes, start, end) of each timed step's input copies

    def one(timed=False):
        ready = {}
        for i, l in enumerate(step.linears):
            for hid in l["inputs"]:
                if hid not in ready:
                    host, dev = pinned[hid]
                    if hid in last_read:
                        cin.wait_event(last_read[hid])
                    with torch.cuda.stream(cin):
                        if timed:
                            c0 = torch.cuda.Event(enable_timing=True)
                            c0.record(cin)
                        dev.copy_(host, non_blocking=True)
                        if timed:
                            c1 = torch.cuda.Event(enable_timing=True)
                            c1.record(cin)
                            copies.append((host.numel() * 2, c0, c1))
                    ready[hid] = event(cin)
                comp.wait_event(ready[hid])
            if i in dw_back:
                comp.wait_event(dw_back[i])
            K = l["K"]
            am = l["colmax"][:2 * K]
            m.int8mp_linear_fwd_save(l["X"], l["W"], am, cfg, Y=l["Y"], workspace=ws)
            m.int8mp_linear_bwd_saved(l["dY"], l["X"], l["W"], am, cfg, dX=l["dX"], dW=l["dW"],
                                      workspace=ws)
            done = event(comp)
            for hid in l["inputs"]:
                last_read[hid] = done
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                l["hdW"].copy_(l["dW"], non_blocking=True)
            dw_back[i] = event(cout)
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    cin.wait_event(a)
    cout.wait_event(a)
    t0 = time.perf_counter()
    for _ in range(steps):
        one(timed=True)
    comp.wait_event(event(cin))
    comp.wait_event(event(cout))
    b.record(comp)
    host_ms = (time.perf_counter() - t0) * 1e3  # enqueueing the steps, no wait
    torch.cuda.synchronize()
    if m.int8mp_poll_device_status() != m.INT8MP_OK:
        raise RuntimeError("device status reported a timeout during the e2e run")
    # the input copies' own rate inside the run (busy time of the copy stream)
    copy_gbs = (sum(n for n, _, _ in copies) /
                (sum(c0.elapsed_time(c1) for _, c0, c1 in copies) * 1e-3) / 1e9)
    # the host link alone on this machine: the largest input copied in, nothing else running
    host, dev = max(pinned.values(), key=lambda hd: hd[0].numel())
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    dev.copy_(host, non_blocking=True)
    c0.record(comp)
    for _ in range(3):
        dev.copy_(host, non_blocking=True)
    c1.record(comp)
    torch.cuda.synchronize()
    link_gbs = 3 * host.numel() * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    return a.elapsed_time(b), h2d, d2h, link_gbs, copy_gbs, host_ms / steps


# ------------------------------------------------------------------ oracle
def oracle_layer_sample(spec, T_sample, mode=0, nthreads=None):
    """Seconds the oracle takes for the step's arithmetic on the first
    T_sample tokens of the same layer inputs (all seven linears, fwd + bwd)."""
    import numpy as np
    import torch
    import oracle
    from int8_mixed_precision_row_gb300 import synth

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    host = synth.layer_inputs(spec, T=T_sample)
    arrays = [(bits(X), bits(W), bits(dY)) for X, W, dY in host.values()]
    nthreads = nthreads or oracle.default_threads()
    oracle.lib()
    t0 = time.perf_counter()
    for X, W, dY in arrays:
        oracle.linear_fwd(X, W, mode=mode, nthreads=nthreads)
        oracle.linear_bwd(dY, X, W, mode=mode, nthreads=nthreads)
    return time.perf_counter() - t0, nthreads


def oracle_small_single_core():
    """Milliseconds the oracle takes on one core for the two small problems:
    the 256x512 single forward matmul (quantize X and W by rows, scaled mm)
    and the 1024^3 square A @ B.T (same steps)."""
    import numpy as np
    import torch
    import oracle
    from int8_mixed_precision_row_gb300 import synth

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def one(A, B):
        a, b = bits(A), bits(B)
        t0 = time.perf_counter()
        qa, sa = oracle.quantize(a, axis=0)
        qb, sb = oracle.quantize(b, axis=0)
        oracle.scaled_mm(qa, sa, qb, sb, a.shape[0], b.shape[0], a.shape[1], nthreads=1)
        return round((time.perf_counter() - t0) * 1e3, 1)
    oracle.lib()
    X, W = synth.single_matmul_inputs()
    A, B = synth.square_inputs(1024, "AxBT")
    return {"single_matmul_256x256x512_ms": one(X, W), "square_1024_AxBT_ms": one(A, B),
            "cores": 1}


def cpu_baseline(spec):
    secs, cores = oracle_layer_sample(spec, ORACLE_SAMPLE_TOKENS)
    return {"value": ORACLE_SAMPLE_TOKENS / secs, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"first {ORACLE_SAMPLE_TOKENS} tokens of the same layer inputs, all 7 linears "
                      f"fwd+grad_in+grad_w, RNE ({secs:.1f} s)",
            "small_problems_single_core": oracle_small_single_core()}


# ------------------------------------------------------------------ extras
def graph_replay_us(fn, device, reps, flush=None):
    """Median device time (us) of `fn`'s launches captured once in a CUDA
    graph and replayed `reps` times, events around each replay (one host
    call per replay, so no host gaps inside the timed interval); `flush`, if
    given, runs before each replay outside the timed interval."""
    import torch
    s = torch.cuda.Stream(device=device)
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    ev = []
    for it in range(reps + 3):
        if flush is not None:
            flush(it)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        if it >= 3:
            ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.median([x.elapsed_time(y) for x, y in ev]) * 1e3


def graph_sequence_us(fn, device, n=20, reps=5, flush=None):
    """Device time (us) per call of `fn` when n calls run back to back: n
    calls (each after `flush`, if given) captured in one CUDA graph and
    replayed, the time of a graph of the n flushes alone subtracted, divided
    by n (median of `reps` replays each).  Unlike graph_replay_us, one call's
    launch overlaps the end of the work before it, as in a stream of calls."""
    import torch
    s = torch.cuda.Stream(device=device)

    def graph_of(body):
        body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        torch.cuda.synchronize()
        return g

    def timed(g):
        ts = []
        for _ in range(reps + 1):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts[1:])

    def calls():
        for i in range(n):
            if flush is not None:
                flush(i)
            fn()

    def flushes():
        for i in range(n):
            flush(i)
    full = timed(graph_of(calls))
    base = timed(graph_of(flushes)) if flush is not None else 0.0
    return (full - base) / n


def square_sweep(device, sizes=(1024, 2048, 4096), iters=20):
    """Square quant+scaled-mm in the three layouts: quantize A and B along K
    (by columns, codes left in place, for the operands stored K-first), then
    the matmul in the stored layout.  Each of quantize, matmul and both is
    captured in a CUDA graph and replayed (device time, no host gaps), the
    L2 flushed before every replay: a 256 MB write, then a read of another
    256 MB buffer, so that the flush's dirty lines are written back before
    the timed kernels start."""
    import torch
    import int8_mixed_precision_row_gb300 as m
    from int8_mixed_precision_row_gb300 import synth
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    clean = torch.zeros(64 << 20, dtype=torch.float32, device=device)  # 256 MB, read

    def flush(it):
        flush_buf.fill_(it & 0xFF)
        clean.max()
    out = {}
    for S in sizes:
        A, B = synth.square_inputs(S, "AxBT")
        A, B = A.to(device), B.to(device)
        qa = torch.empty((S, S), dtype=torch.float16, device=device)
        qb = torch.empty((S, S), dtype=torch.float16, device=device)
        sa = torch.empty(S, dtype=torch.float32, device=device)
        sb = torch.empty(S, dtype=torch.float32, device=device)
        Y = torch.empty((S, S), dtype=torch.bfloat16, device=device)
        mm_ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=device)
        for layout, (ax_a, ax_b, lay) in (("A@B.T", (0, 0, m.INT8MP_AxBT)), ("A@B", (0, 2, m.INT8MP_AxB)),
                                          ("A.T@B", (2, 2, m.INT8MP_ATxB))):
            def quant():
                if ax_a == 0 and ax_b == 0:  # both by rows: one launch
                    m.int8mp_quantize_rows_batch([A, B], codes=m.INT8MP_CODES_F16, qs=[qa, qb],
                                                 scales=[sa, sb])
                elif ax_a == 2 and ax_b == 2:  # both by columns: one launch up to 2048 rows
                    m.int8mp_quantize_cols_batch([A, B], codes=m.INT8MP_CODES_F16, qs=[qa, qb],
                                                 scales=[sa, sb])
                else:
                    m.int8mp_quantize_rowwise(A, axis=ax_a, codes=m.INT8MP_CODES_F16, q=qa,
                                              scale=sa)
                    m.int8mp_quantize_rowwise(B, axis=ax_b, codes=m.INT8MP_CODES_F16, q=qb,
                                              scale=sb)

            def mm():
                m.int8mp_scaled_mm(qa, sa, qb, sb, layout=lay, out=Y, workspace=mm_ws)

            def both():
                quant()
                mm()
            q_us = graph_replay_us(quant, device, iters, flush)
            mm_us = graph_replay_us(mm, device, iters, flush)
            both_us = graph_replay_us(both, device, iters, flush)
            seq_us = graph_sequence_us(both, device, flush=flush)
            ops = 2.0 * S ** 3
            out[f"{S}:{layout}"] = {
                "quant_mm_tops": round(ops / (both_us * 1e-6) / 1e12, 1),
                "mm_tops": round(ops / (mm_us * 1e-6) / 1e12, 1),
                "quant_us": round(q_us, 2), "mm_us": round(mm_us, 2), "quant_mm_us": round(both_us, 2),
                "quant_gbs_f16codes": round(2 * S * S * 4 / (q_us * 1e-6) / 1e9, 1),
                "quant_mm_us_in_sequence": round(seq_us, 2),
                "quant_mm_tops_in_sequence": round(ops / (seq_us * 1e-6) / 1e12, 1)}
    out["timing"] = ("each of quantize, matmul and both replayed alone from a CUDA graph after "
                     "an L2 flush (median device time); *_in_sequence: 20 flushed calls in one "
                     "graph, the flushes' own time subtracted, per call")
    return out


def single_matmul_latency(device, reps=200):
    """The 256x512 single forward matmul (X and W quantized by rows in one
    launch, then the scaled matmul): device time per call, the two launches
    replayed from a CUDA graph (inputs resident; 0.5 MB, L2-resident)."""
    import torch
    import int8_mixed_precision_row_gb300 as m
    from int8_mixed_precision_row_gb300 import synth
    X, W = synth.single_matmul_inputs()
    X, W = X.to(device), W.to(device)
    qx = torch.empty((256, 512), dtype=torch.float16, device=device)
    qw = torch.empty((256, 512), dtype=torch.float16, device=device)
    sx = torch.empty(256, dtype=torch.float32, device=device)
    sw = torch.empty(256, dtype=torch.float32, device=device)
    Y = torch.empty((256, 256), dtype=torch.bfloat16, device=device)

    def one():
        m.int8mp_quantize_rows_batch([X, W], codes=m.INT8MP_CODES_F16, qs=[qx, qw], scales=[sx, sw])
        m.int8mp_scaled_mm(qx, sx, qw, sw, out=Y)
    us = graph_replay_us(one, device, reps)
    seq = graph_sequence_us(one, device)
    ops = 2.0 * 256 * 256 * 512
    return {"us_per_call": round(us, 2), "tops": round(ops / (us * 1e-6) / 1e12, 2),
            "us_per_call_in_sequence": round(seq, 2),
            "tops_in_sequence": round(ops / (seq * 1e-6) / 1e12, 2),
            "launches_per_call": 2,
            "timing": "CUDA-graph replays of one call, device time, median; *_in_sequence: 20 "
                      "calls in one graph, per call"}


def decoder_module_tok_s(spec, device, steps=5, warmup=2):
    """The decoder layer's seven linears as Int8MixedPrecisionDecoderLinears
    (SwiGLU between gate/up and down, glue in fp32 torch ops), forward and
    backward through torch.autograd on T tokens."""
    import torch
    import int8_mixed_precision_row_gb300 as m
    from int8_mixed_precision_row_gb300 import synth
    T = spec["T"]
    layer = m.Int8MixedPrecisionDecoderLinears(spec["hidden"], spec["inter"], device=device)
    x = synth.bf16_normal((T, spec["hidden"]), 10).to(device).requires_grad_(True)
    dy = synth.bf16_normal((T, spec["hidden"]), 30, std=1e-3).to(device)

    def one():
        layer.zero_grad(set_to_none=True)
        x.grad = None
        layer(x).backward(dy)
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    del layer, x, dy
    torch.cuda.empty_cache()
    return {"tok_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 3),
            "glue": "fp32 torch elementwise (stand-in attention a = v + q*k, SwiGLU, residuals)"}


def layer_tok_s(spec, mode, device, steps=5, warmup=2):
    import torch
    step = LayerStep(spec, mode, device)
    el, per_kind, _ = time_steps(step, steps, warmup, 1, device)
    r = {"tok_s": round(step.T * steps / (el * 1e-3), 1), "ms_per_step": round(el / steps, 3),
         "gemm_tflops": round(step.flops * steps / (per_kind.get("gemm", el) * 1e-3) / 1e12, 1)}
    del step
    torch.cuda.empty_cache()
    return r


def pass_switch_table(spec, device, steps=5, warmup=2):
    """The rows of the pages' INT8 mixed precision training table (forward /
    grad-input / grad-weight each INT8 or BF16, nearest-even) on this GPU,
    for the decoder layer's linears, through int8mp_linear_fwd_save /
    int8mp_linear_bwd_saved."""
    import torch
    import int8_mixed_precision_row_gb300 as m
    step = LayerStep(spec, m.INT8MP_RNE, device)
    ws_bytes = max(m.int8mp_linear_workspace_size(step.T, l["N"], l["K"]) for l in step.linears)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    rows = {}
    for flags in ((0, 0, 0), (1, 0, 0), (1, 1, 0), (1, 1, 1)):
        cfg = m.linear_cfg(int8_fwd=flags[0], int8_grad_in=flags[1], int8_grad_w=flags[2])

        def one():
            for l in step.linears:
                am = l["colmax"][:2 * l["K"]]
                m.int8mp_linear_fwd_save(l["X"], l["W"], am, cfg, Y=l["Y"], workspace=ws)
                m.int8mp_linear_bwd_saved(l["dY"], l["X"], l["W"], am, cfg, dX=l["dX"],
                                          dW=l["dW"], workspace=ws)
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            one()
        b.record()
        torch.cuda.synchronize()
        name = "/".join("INT8" if f else "BF16" for f in flags)
        rows[name] = round(step.T * steps / (a.elapsed_time(b) * 1e-3), 1)
    base = rows["BF16/BF16/BF16"]
    out = {k: {"tok_s": v, "speedup_vs_bf16": round(v / base, 3)} for k, v in rows.items()}
    del step, ws
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------------- main
# DRAM traffic of the dominant kernel (gemm_s8f16_pair_kernel), per launch,
# averaged over the 21 launches of one step of this workload:
# dram__bytes_read.sum + dram__bytes_write.sum from one ncu launch list of
# `python bench.py --steps 2 --warmup 3 --profile-steps` (one pass per
# launch), valid for the GEMM sources whose digest is given (reported as null
# once they change).
GEMM_TRAFFIC = {"bytes_per_launch": 406877788, "sources_sha256_16": "b888284032285bea"}
GEMM_SOURCES = ("gemm.cu", "ptx.cuh")


def gemm_sources_digest():
    """sha256 (16 hex digits) of the GEMM sources with // comments, blank
    lines and indentation removed: only a change of the code counts."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "int8_mixed_precision_row_gb300", "csrc", f)) as fh:
            for line in fh:
                code = re.sub(r"//.*$", "", line).strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def gemm_traffic():
    if gemm_sources_digest() != GEMM_TRAFFIC["sources_sha256_16"]:
        return None
    return GEMM_TRAFFIC["bytes_per_launch"]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p.get("hbm_gbs"), p.get("bf16_tflops"), p.get("bf16_tflops_sustained"), "measured"
    except (OSError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores, each step a bounded sample
    of the same workload.  Under torchrun only rank 0 works."""
    if rank != 0:
        return
    from int8_mixed_precision_row_gb300 import synth
    spec = synth.LLAMA2_1B
    T_s = 32
    for _ in range(args.warmup):
        oracle_layer_sample(spec, T_s)
    secs = 0.0
    cores = 1
    for _ in range(args.steps):
        s, cores = oracle_layer_sample(spec, T_s)
        secs += s
    value = T_s * args.steps / secs
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": T_s, "parallelism": "replicas"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {T_s} tokens of the llama2-1b layer per step"},
        "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        init_dist(world, "gloo")
        run_reference(args, world, rank)
        return
    import torch
    from int8_mixed_precision_row_gb300 import build, synth
    import int8_mixed_precision_row_gb300 as m
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    build.build()
    m.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    spec = synth.LLAMA2_1B
    only = set(args.linears.split(",")) if args.linears else None
    if (args.tokens or only or args.rounding != "rne") and not args.profile_steps:
        raise SystemExit("--tokens/--linears/--rounding select profiling cases and need "
                         "--profile-steps")
    if args.case:
        run_profile_case(args.case, device)
        return
    mode = m.INT8MP_SR if args.rounding == "sr" else m.INT8MP_RNE
    step = LayerStep(spec, mode, device, T=args.tokens, only=only, world=world, rank=rank)
    with ClockSampler(local) as clk:
        elapsed_ms, per_kind, counts = time_steps(step, args.steps, args.warmup, world, device)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    if m.int8mp_poll_device_status() != m.INT8MP_OK:
        raise RuntimeError("a bounded device wait ran out during the timed region")
    tokens = step.T * args.steps * world
    value = tokens / (elapsed_ms * 1e-3)
    hbm, bf16_burst, bf16_sust, peak_src = measured_peaks()
    gemm_ms = per_kind.get("gemm", 0.0)
    gemm_launches = counts.get("gemm", 1)
    gemm_tflops = step.flops * args.steps / (gemm_ms * 1e-3) / 1e12
    quant_ms = per_kind.get("quant_rows", 0.0) + per_kind.get("quant_cols", 0.0)
    quant_bytes = step.quant_elems * 4 * args.steps  # bf16 read + f16 code written per element
    quant_bytes_alg = step.quant_elems * 3 * args.steps  # bf16 read + one int8 code: the minimum
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": step.T, "hidden": spec["hidden"],
                   "intermediate": spec["inter"], "linears": len(step.linears),
                   "rounding": "SR" if mode == m.INT8MP_SR else "RNE",
                   "l2": "inputs larger than L2 (about 5 GB touched per step, L2 129 MB)",
                   "parallelism": (f"data parallel x{world}: {step.T} tokens per rank, dW as "
                                   f"fp32 partials all-reduced then rounded once")
                   if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor",
                     "kernel": "gemm_s8f16_pair_kernel (CTA-pair tcgen05 kind::f16, exact int32)",
                     "achieved": round(gemm_tflops, 1), "peak": bf16_burst, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / bf16_burst, 3),
                     "traffic": gemm_traffic() if step.T == spec["T"] and not only else None,
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
                     "algorithmic_bytes": round(step.gemm_bytes / step.gemms_per_step),
                     "peak_source": f"{peak_src} dense bf16 burst (f16 runs at the bf16 rate; "
                                    f"sm_103a has no faster INT8 MMA); sustained {bf16_sust} "
                                    f"TFLOP/s -> frac {round(gemm_tflops / bf16_sust, 3)}",
                     "launches_timed": gemm_launches,
                     "avg_launch_ms": round(gemm_ms / gemm_launches, 4)},
        "kernels": {
            "gemm_ms_per_step": round(gemm_ms / args.steps, 3),
            "quant_rows_ms_per_step": round(per_kind.get("quant_rows", 0.0) / args.steps, 3),
            "quant_cols_ms_per_step": round(per_kind.get("quant_cols", 0.0) / args.steps, 3),
            "quant_gbs_f16codes": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1) if quant_ms else None,
            "quant_frac_of_hbm_f16codes": round(quant_bytes / (quant_ms * 1e-3) / 1e9 / hbm, 3)
            if quant_ms else None,
            "quant_gbs_algorithmic_3B": round(quant_bytes_alg / (quant_ms * 1e-3) / 1e9, 1)
            if quant_ms else None,
            "quant_frac_of_hbm_algorithmic_3B": round(quant_bytes_alg / (quant_ms * 1e-3) / 1e9 / hbm, 3)
            if quant_ms else None,
            "quant_bytes_note": "f16codes: bytes moved (bf16 read + f16 code container written, 4 B "
                                "per element); algorithmic_3B: bf16 read + int8 code, 3 B per "
                                "element",
            "hbm_peak_gbs": hbm,
            "timing": "value: the timed steps with no per-kernel events; this breakdown: up "
                      "to 20 further steps with CUDA events around every call, scaled"},
        "gpu_launches": step.kernels_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.profile_steps:
        e2e_steps = max(3, min(args.steps, 10))
        with ClockSampler(local) as eclk:
            e2e_ms, h2d, d2h, link_gbs, copy_gbs, host_ms = time_e2e(step, e2e_steps, 1)
        e2e_ms = max_over_ranks(e2e_ms, world, device)
        line["e2e"] = {"value": round(step.T * e2e_steps * world / (e2e_ms * 1e-3), 1), "unit": "tok/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "copies": "pinned host <-> device on their own streams, overlapping the "
                                 "compute of other linears",
                       "host_link_h2d_gbs": round(link_gbs, 1),
                       "h2d_gbs_in_run": round(copy_gbs, 1),
                       "host_enqueue_ms_per_step": round(host_ms, 3),
                       "h2d_bound_tok_s": round(step.T * world / (h2d / (link_gbs * 1e9)), 1),
                       "clocks": eclk.summary()}
    del step
    torch.cuda.empty_cache()
    if rank == 0 and not args.profile_steps and not args.no_extra:
        line["extra"] = {
            "single_forward_matmul_256x256x512": single_matmul_latency(device),
            "square_quant_scaled_mm": square_sweep(device),
            "llama2-1b_decoder_module_autograd": decoder_module_tok_s(synth.LLAMA2_1B, device),
            "llama2-1b_stochastic_rounding": layer_tok_s(synth.LLAMA2_1B, m.INT8MP_SR, device),
            "llama3-8b_T16384": layer_tok_s(synth.LLAMA3_8B, m.INT8MP_RNE, device),
            "llama2-1b_pass_switches (forward/grad-input/grad-weight)":
                pass_switch_table(synth.LLAMA2_1B, device),
        }
    if rank == 0 and not args.profile_steps and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
