"""Benchmark of the CODA GEMM-plus-epilogue hot path on one GB300 (or N
replicas, one process per GPU: started by torchrun, or by this script itself
when --gpus N > 1 runs without it).

One step = one pass over every kernel of the hot path:
  * Llama-3-1B-shaped MLP block forward, M=8192, d=2048, f=8192
      (residual+RMSNorm-weight+row-stats GEMM, r, delayed-r SwiGLU GEMM,
       down projection)
  * LM head + cross-entropy, M=8192, d=2048, V=128256 (logits never written)
  * the block's reverse-fused backward (SwiGLU-bwd GEMM + s partials, s,
    RMSNorm-bwd GEMM + dgamma partials, dgamma, dW2, dW1, dW0, dx)
  * Llama-3-8B-shaped non-attention forward + backward, M=16384, d=4096,
    f=14336, QKV 6144 with RoPE (theta 5e5, positions 0..4095 per sequence)
The metric is the GEMM work of the step (2*M*N*K per GEMM) per second; the
LM head is also reported as tokens/s. Inputs are synthetic (seeded, the
workloads' distributions), resident in HBM before the timed region; L2 is
flushed (a 512 MiB write) before every timed step, outside the step's events.

--impl reference times the CPU oracle (fp64 numpy) on a bounded row sample of
the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "fused GEMM+epilogue TFLOP/s (% BF16 peak); LM-head+CE tokens/s"
UNIT = "TFLOP/s"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _smi_id(local: int) -> str:
    """nvidia-smi's name for this process's CUDA device `local` (its UUID, so
    that CUDA_VISIBLE_DEVICES renumbering does not matter)."""
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        return str(local)


class Clocks:
    """Samples nvidia-smi every 50 ms around the timed region; `stop` keeps
    the samples whose nvidia-smi timestamp falls inside the region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def parse(lines, window=None):
        """Median SM clock, max clock and the throttle reasons seen, from
        nvidia-smi CSV lines; with window = (t0, t1) (seconds since the
        epoch) only the samples stamped inside it count, if there are any."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if window and window[0] <= r[0] <= window[1]]
        use = inside or rows
        sm = sorted(r[1] for r in use)
        reasons = sorted({n for r in use for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": use[-1][2] if use else None, "reasons": reasons,
                "samples": len(use), "in_timed_region": bool(inside)}

    def summary(self, window=None):
        """The record of the samples so far (the sampler keeps running)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return self.parse(list(self.lines), window)

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return self.parse(self.lines, window)


def _kernel_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gemm_epilogue_fusion_tcgen05_gb300", "csrc")
    for base, _, files in sorted(os.walk(d)):
        for f in sorted(files):
            if f.endswith((".cu", ".cuh", ".h")):
                h.update(open(os.path.join(base, f), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ ranks

def max_over_ranks(ms: float, device) -> float:
    """Largest per-step time over all ranks (every rank holds a replica of
    the whole step; the slowest one sets the job's step time)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, ms: float) -> float:
    """Whole-job TFLOP/s: every replica does a full step in `ms` (the max
    over ranks)."""
    return flops_per_step * world / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ the step

class Step:
    """Buffers and the list of C-ABI calls of one step. Each call is wrapped
    in CUDA events on the launching (current) stream."""

    def __init__(self, dev, with_8b=True, with_1b=True, with_lm=True, tokens_8b=None):
        import gemm_epilogue_fusion_tcgen05_gb300 as C
        from gemm_epilogue_fusion_tcgen05_gb300 import blocks
        from coda_inputs import WORKLOADS, mlp_block_inputs, lmhead_inputs, block8b_inputs
        self.C = C
        self.dev = dev
        bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32
        e = lambda s, dt: torch.empty(s, dtype=dt, device=dev)
        # ---- Llama-3-1B-shaped block (forward state kept for the backward)
        s1 = WORKLOADS["llama1b_mlp_bwd"]
        self.s1 = s1
        M, d, f = s1.M, s1.d, s1.f
        self.with_1b, self.with_lm = with_1b, with_lm
        if with_1b:
            self.i1 = mlp_block_inputs(s1, device=dev)
            self.b1 = {"h": e((M, d), bf), "hg": e((M, d), bf), "part": e((C.col_tiles(d), M), f32),
                       "r": e((M,), f32), "a": e((M, f), bf), "y": e((M, 2 * f), f16),
                       "out": e((M, d), bf), "dyhat": e((M, 2 * f), bf),
                       "spart": e((C.col_tiles(f), M), f32), "s": e((M,), f32), "dh": e((M, d), bf),
                       "dgpart": e((C.row_tiles32(M), d), f32), "dgamma": e((d,), f32),
                       "dW0": e((d, d), f32), "dW1": e((d, 2 * f), f32), "dW2": e((f, d), f32),
                       "dx": e((M, d), bf)}
        # ---- LM head
        s2 = WORKLOADS["lmhead_ce"]
        self.s2 = s2
        if with_lm:
            self.i2 = lmhead_inputs(s2, device=dev)
            self.ws2 = torch.empty(C.coda_lmhead_ce_workspace_size(s2.M, s2.V), dtype=torch.uint8,
                                   device=dev)
            self.o2 = {"lse": e((s2.M,), f32), "loss": e((s2.M,), f32)}
        # ---- Llama-3-8B-shaped block
        self.with_8b = with_8b
        if with_8b:
            s4 = WORKLOADS["llama8b_block"]
            if tokens_8b:  # fewer rows (whole sequences or one partial one)
                s4 = dataclasses.replace(s4, M=tokens_8b)
            self.s4 = s4
            self.i4 = block8b_inputs(s4, device=dev)
            self.cs = blocks.rope_table(s4.seq_len, s4.head_dim, s4.theta, dev)
            M4, d4, f4, n4 = s4.M, s4.d, s4.f, s4.n_qkv
            self.b4 = {"h": e((M4, d4), bf), "hg": e((M4, d4), bf),
                       "part": e((C.col_tiles(d4), M4), f32), "r": e((M4,), f32),
                       "a": e((M4, f4), bf), "y": e((M4, 2 * f4), f16), "out": e((M4, d4), bf),
                       "outg": e((M4, d4), bf), "part1": e((C.col_tiles(d4), M4), f32),
                       "r1": e((M4,), f32), "qkv": e((M4, n4), bf), "qkv_save": e((M4, n4), f16),
                       "dqh": e((M4, n4), bf),
                       "s1": e((M4,), f32), "dout": e((M4, d4), bf),
                       "dgp1": e((C.row_tiles32(M4), d4), f32), "dgamma1": e((d4,), f32),
                       "dWqkv": e((d4, n4), f32), "dyhat": e((M4, 2 * f4), bf),
                       "spart": e((C.col_tiles(f4), M4), f32), "s": e((M4,), f32),
                       "dW2": e((f4, d4), f32), "dh": e((M4, d4), bf),
                       "dgp2": e((C.row_tiles32(M4), d4), f32), "dgamma2": e((d4,), f32),
                       "dW1": e((d4, 2 * f4), f32), "dWo": e((d4, d4), f32), "do": e((M4, d4), bf)}
        self.calls = self._build_calls()
        self.launches_per_step = sum(c[3] for c in self.calls)
        self.flops = sum(c[1] for c in self.calls)

    def _build_calls(self):
        C = self.C
        calls = []  # (name, flops, fn, launches)
        add = lambda n, fl, fn, k=1: calls.append((n, float(fl), fn, k))
        if self.with_1b:
            self._calls_1b_fwd(add)
        if self.with_lm:
            s2, i2 = self.s2, self.i2
            add("lmhead_ce", 2 * s2.M * s2.d * s2.V,
                lambda: C.coda_lmhead_ce(i2["hidden"], i2["W"], i2["targets"], self.o2["lse"],
                                         self.o2["loss"], self.ws2), 2)
        if self.with_1b:
            self._calls_1b_bwd(add)
        if self.with_8b:
            self._calls_8b(add)
        return calls

    def _calls_1b_fwd(self, add):
        C, i1, b1 = self.C, self.i1, self.b1
        M, d, f = self.s1.M, self.s1.d, self.s1.f
        add("1b.gemm_resid_norm_stats", 2 * M * d * d,
            lambda: C.coda_gemm_resid_norm_stats(i1["x"], i1["W0"], i1["z"], i1["gamma"], b1["h"],
                                                 b1["hg"], b1["part"]))
        add("1b.row_rms", 0, lambda: C.coda_row_rms(b1["part"], b1["r"], d, 1e-6))
        add("1b.gemm_rowscale_swiglu", 2 * M * d * 2 * f,
            lambda: C.coda_gemm_rowscale_swiglu(b1["hg"], i1["W1"], b1["r"], b1["a"], b1["y"]))
        add("1b.gemm_down", 2 * M * f * d, lambda: C.coda_gemm(b1["a"], i1["W2"], b1["out"]))

    def _calls_1b_bwd(self, add):
        C, i1, b1 = self.C, self.i1, self.b1
        M, d, f = self.s1.M, self.s1.d, self.s1.f
        add("1b.gemm_rowscale_swiglu_bwd", 2 * M * d * f,
            lambda: C.coda_gemm_rowscale_swiglu_bwd(i1["dout"], i1["W2"], b1["y"], b1["r"],
                                                    b1["dyhat"], b1["spart"]))
        add("1b.row_rms_bwd", 0, lambda: C.coda_row_rms_bwd(b1["spart"], b1["s"], d))
        add("1b.gemm_resid_norm_stats_bwd", 2 * M * 2 * f * d,
            lambda: C.coda_gemm_resid_norm_stats_bwd(b1["dyhat"], i1["W1"], b1["h"], i1["gamma"],
                                                     b1["r"], b1["s"], b1["dh"], b1["dgpart"]))
        add("1b.col_reduce", 0, lambda: C.coda_col_reduce(b1["dgpart"], b1["dgamma"]))
        add("1b.wgrad_W2", 2 * f * d * M, lambda: C.coda_gemm(b1["a"], i1["dout"], b1["dW2"], transA=True))
        add("1b.wgrad_W1", 2 * d * 2 * f * M, lambda: C.coda_gemm(b1["hg"], b1["dyhat"], b1["dW1"], transA=True))
        add("1b.wgrad_W0", 2 * d * d * M, lambda: C.coda_gemm(i1["x"], b1["dh"], b1["dW0"], transA=True))
        add("1b.dgrad_x", 2 * M * d * d, lambda: C.coda_gemm(b1["dh"], i1["W0"], b1["dx"], transB=True))

    def _calls_8b(self, add):
        C = self.C
        s4, i4, b4, cs = self.s4, self.i4, self.b4, self.cs
        M4, d4, f4, n4 = s4.M, s4.d, s4.f, s4.n_qkv
        sl, hd, nr = s4.seq_len, s4.head_dim, s4.n_rope_cols
        add("8b.gemm_resid_norm_stats(Wo)", 2 * M4 * d4 * d4,
            lambda: C.coda_gemm_resid_norm_stats(i4["o"], i4["Wo"], i4["z"], i4["gamma2"],
                                                 b4["h"], b4["hg"], b4["part"]))
        add("8b.row_rms", 0, lambda: C.coda_row_rms(b4["part"], b4["r"], d4, 1e-6))
        add("8b.gemm_rowscale_swiglu", 2 * M4 * d4 * 2 * f4,
            lambda: C.coda_gemm_rowscale_swiglu(b4["hg"], i4["W1"], b4["r"], b4["a"], b4["y"]))
        add("8b.gemm_resid_norm_stats(W2)", 2 * M4 * f4 * d4,
            lambda: C.coda_gemm_resid_norm_stats(b4["a"], i4["W2"], b4["h"], i4["gamma1"],
                                                 b4["out"], b4["outg"], b4["part1"]))
        add("8b.row_rms1", 0, lambda: C.coda_row_rms(b4["part1"], b4["r1"], d4, 1e-6))
        add("8b.gemm_rope", 2 * M4 * d4 * n4,
            lambda: C.coda_gemm_rope(b4["outg"], i4["Wqkv"], b4["r1"], cs, sl, hd, nr, b4["qkv"],
                                     b4["qkv_save"]))
        add("8b.rope_bwd", 0,
            lambda: C.coda_gemm_rope_bwd(i4["dqkv"], b4["qkv_save"], b4["r1"], cs, sl, hd, nr,
                                         b4["dqh"], b4["s1"], d4))
        add("8b.gemm_resid_norm_stats_bwd(Wqkv)", 2 * M4 * n4 * d4,
            lambda: C.coda_gemm_resid_norm_stats_bwd(b4["dqh"], i4["Wqkv"], b4["out"],
                                                     i4["gamma1"], b4["r1"], b4["s1"],
                                                     b4["dout"], b4["dgp1"], dresid=i4["dres"]))
        add("8b.col_reduce1", 0, lambda: C.coda_col_reduce(b4["dgp1"], b4["dgamma1"]))
        add("8b.wgrad_Wqkv", 2 * d4 * n4 * M4,
            lambda: C.coda_gemm(b4["outg"], b4["dqh"], b4["dWqkv"], transA=True))
        add("8b.gemm_rowscale_swiglu_bwd", 2 * M4 * d4 * f4,
            lambda: C.coda_gemm_rowscale_swiglu_bwd(b4["dout"], i4["W2"], b4["y"], b4["r"],
                                                    b4["dyhat"], b4["spart"]))
        add("8b.row_rms_bwd", 0, lambda: C.coda_row_rms_bwd(b4["spart"], b4["s"], d4))
        add("8b.wgrad_W2", 2 * f4 * d4 * M4,
            lambda: C.coda_gemm(b4["a"], b4["dout"], b4["dW2"], transA=True))
        add("8b.gemm_resid_norm_stats_bwd(W1)", 2 * M4 * 2 * f4 * d4,
            lambda: C.coda_gemm_resid_norm_stats_bwd(b4["dyhat"], i4["W1"], b4["h"],
                                                     i4["gamma2"], b4["r"], b4["s"], b4["dh"],
                                                     b4["dgp2"], dresid=b4["dout"]))
        add("8b.col_reduce2", 0, lambda: C.coda_col_reduce(b4["dgp2"], b4["dgamma2"]))
        add("8b.wgrad_W1", 2 * d4 * 2 * f4 * M4,
            lambda: C.coda_gemm(b4["hg"], b4["dyhat"], b4["dW1"], transA=True))
        add("8b.wgrad_Wo", 2 * d4 * d4 * M4, lambda: C.coda_gemm(i4["o"], b4["dh"], b4["dWo"], transA=True))
        add("8b.dgrad_o", 2 * M4 * d4 * d4, lambda: C.coda_gemm(b4["dh"], i4["Wo"], b4["do"], transB=True))

    def select(self, names):
        """Keep only the named calls (for single-kernel profiling); the full
        step still runs during warm-up so that every input is initialised."""
        self.all_calls = self.calls
        keep = [c for c in self.calls if c[0] in names]
        if not keep:
            raise SystemExit(f"--only matched nothing; names: {[c[0] for c in self.calls]}")
        self.calls = keep
        self.launches_per_step = sum(c[3] for c in keep)
        self.flops = sum(c[1] for c in keep)

    def run(self, events=None, calls=None):
        for k, (name, fl, fn, nl) in enumerate(calls if calls is not None else self.calls):
            if events is not None:
                events[k][0].record()
            fn()
            if events is not None:
                events[k][1].record()

    # per-step inputs and results for the end-to-end measurement
    def host_io(self):
        ins = [t for group, _ in self.input_groups() for t in group]
        outs = [self.o2["loss"], self.o2["lse"], self.b1["dgamma"]]
        return ins, outs

    def input_slots(self):
        """Every per-step input as (dict, key), grouped by the first call that
        reads the group. The calls look their tensors up in these dicts when
        they run, so replacing an entry switches a call to another buffer."""
        groups = [([(self.i1, "x"), (self.i1, "z")], "1b.gemm_resid_norm_stats"),
                  ([(self.i2, "hidden"), (self.i2, "targets")], "lmhead_ce"),
                  ([(self.i1, "dout")], "1b.gemm_rowscale_swiglu_bwd")]
        if self.with_8b:
            groups += [([(self.i4, "o"), (self.i4, "z")], "8b.gemm_resid_norm_stats(Wo)"),
                       ([(self.i4, "dqkv"), (self.i4, "dres")], "8b.rope_bwd")]
        return groups

    def input_groups(self):
        """The step's per-step input tensors in the order the step first
        reads them, each group with the first call that reads any of them."""
        return [([d[k] for d, k in slots], name) for slots, name in self.input_slots()]

    def _use_inputs(self, tensors):
        flat = [dk for slots, _ in self.input_slots() for dk in slots]
        for (d, k), t in zip(flat, tensors):
            d[k] = t

    def run_e2e(self, steps, h_ins, h_outs, copy_stream, flush, stream):
        """End-to-end steps through the public calls: every step copies its
        inputs host -> device from pinned memory (`h_ins`, in input_groups
        order) and reads its results back into `h_outs`. Two device buffer
        sets hold the inputs: while step i computes on one, step i + 1's
        inputs are copied into the other on `copy_stream` (once step i - 1 has
        finished reading it), the prefetching input pipeline of a training
        loop; step 0's copy is not overlapped. Returns one event pair per step
        on `stream` (the L2 flush before each step is outside its pair); the
        buffers the step held before are restored at the end."""
        first = [t for g, _ in self.input_groups() for t in g]
        sets = [first, [torch.empty_like(t) for t in first]]
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        outs = self.host_io()[1]

        def copy_into(dst, ev):
            with torch.cuda.stream(copy_stream):
                for hsrc, ddst in zip(h_ins, dst):
                    ddst.copy_(hsrc, non_blocking=True)
                ev.record(copy_stream)

        evs = []
        for i in range(steps):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            cur = i % 2
            if i == 0:
                copy_stream.wait_stream(stream)
                copy_into(sets[0], copied[0])
            self._use_inputs(sets[cur])
            stream.wait_event(copied[cur])
            if i + 1 < steps:
                nxt = 1 - cur
                if i >= 1:
                    copy_stream.wait_event(done[nxt])  # step i - 1 is done with that set
                copy_into(sets[nxt], copied[nxt])
            for name, fl, fn, nl in self.calls:
                fn()
            done[cur].record(stream)
            for dsrc, hdst in zip(outs, h_outs):
                hdst.copy_(dsrc, non_blocking=True)
            e1.record(stream)
            evs.append((e0, e1))
        self._use_inputs(sets[0])
        return evs


def run_coda(args):
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as C

    step = Step(dev, with_8b=not args.no_8b)
    warm_calls = step.calls
    if args.only:
        step.select(set(args.only.split(",")))
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run(calls=warm_calls)
    torch.cuda.synchronize()
    st = C.get_device_error()
    if st != 0:
        raise SystemExit(f"device error after warm-up: {st}")

    n = len(step.calls)
    step_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in range(args.steps)]
    clocks = Clocks(_smi_id(local))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    t_epoch0 = time.time()
    for i in range(args.steps):
        flush.fill_(float(i))
        step_ev[i][0].record(stream)
        step.run()  # no events between the calls: consecutive kernels overlap (PDL)
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    t_epoch1 = time.time()
    if ws > 1:
        torch.distributed.barrier()
    # one sampler runs on through the e2e leg (starting a second one right
    # before it stalled that leg's first step); each leg keeps its own window
    clk = clocks.summary(window=(t_epoch0, t_epoch1))
    st = C.get_device_error()
    if st != 0:
        raise SystemExit(f"device error in timed region: {st}")

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, dev)
    value = job_throughput(step.flops, ws, ms)

    # per-call attribution: a separate pass with an event pair around every
    # call. The events serialise the calls (no launch overlap), so this pass
    # is not the timed one; it gives each kernel's own duration.
    n_attr = max(2, min(args.steps, 5))
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in range(n)] for _ in range(n_attr)]
    attr_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in range(n_attr)]
    for i in range(n_attr):
        flush.fill_(float(i))
        attr_ev[i][0].record(stream)
        step.run(evs[i])
        attr_ev[i][1].record(stream)
    torch.cuda.synchronize()
    per_call = [sum(evs[i][k][0].elapsed_time(evs[i][k][1]) for i in range(n_attr)) / n_attr
                for k in range(n)]
    attr_ms = sum(a.elapsed_time(b) for a, b in attr_ev) / n_attr

    # end-to-end through the public API with host buffers: copy this step's
    # inputs host -> device from pinned memory, run, read the results back.
    # Run after the timed region and the per-call pass (the GPU already
    # power-capped, as in the timed region's later steps), for the same
    # number of steps and with its own clock window.
    ins, outs = step.host_io()
    h_ins = [t.cpu().pin_memory() for t in ins]
    h_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_ins)
    d2h = sum(t.numel() * t.element_size() for t in h_outs)
    e2e_steps = 0 if args.only else args.steps
    copy_stream = torch.cuda.Stream(device=dev)
    if e2e_steps:
        step.run_e2e(2, h_ins, h_outs, copy_stream, flush, stream)  # untimed first use
    torch.cuda.synchronize()
    # the steps are enqueued back to back, as in the device-timed leg, with
    # one host synchronisation at the end
    te0 = time.time()
    e2e_ev = step.run_e2e(e2e_steps, h_ins, h_outs, copy_stream, flush, stream) if e2e_steps else []
    torch.cuda.synchronize()
    te1 = time.time()
    e2e_ms_list = [a.elapsed_time(b) for a, b in e2e_ev]
    clk_e2e = clocks.stop(window=(te0, te1)) if e2e_steps else None
    if not e2e_steps:
        clocks.stop()
    e2e_ms = sum(e2e_ms_list) / len(e2e_ms_list) if e2e_ms_list else 0.0
    e2e_value = job_throughput(step.flops, ws, max_over_ranks(e2e_ms, dev)) if e2e_ms > 0 else None

    peaks, src = _peaks()
    k_dom = max(range(n), key=lambda k: per_call[k])
    name, fl, _, nl = step.calls[k_dom]
    # the burst figure is the conservative denominator: the step runs boosted
    # for its first steps and power-capped after that (the line also gives
    # the fraction of the sustained figure)
    peak = peaks.get("bf16_tflops")
    achieved = fl / (per_call[k_dom] * 1e-3) / 1e12 if per_call[k_dom] > 0 else None
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        tj = json.load(open(tp))
        ent = tj.get("kernels", {}).get(name)
        if ent and tj.get("kernel_hash") == _kernel_hash():
            traffic = ent.get("dram_bytes_per_launch")
    lm = [k for k in range(n) if step.calls[k][0] == "lmhead_ce"]
    lm_tok_s = step.s2.M / (per_call[lm[0]] * 1e-3) if lm else None

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; workloads' shapes and distributions; drawn on the GPU)",
        "config": {"workload": "llama1b_mlp_fwd+lmhead_ce+llama1b_mlp_bwd" +
                               ("+llama8b_block_fwd_bwd" if step.with_8b else ""),
                   "tokens": step.s1.M, "d": step.s1.d, "f": step.s1.f, "vocab": step.s2.V,
                   "tokens_8b": step.s4.M if step.with_8b else 0,
                   "gflop_per_step": round(step.flops / 1e9, 1),
                   "l2": "flushed before each step (512 MiB write, outside the step events)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "pct_bf16_peak": round(100 * value / ws / peak, 2),
        "pct_bf16_sustained_peak": (round(100 * value / ws / peaks["bf16_tflops_sustained"], 2)
                                    if peaks.get("bf16_tflops_sustained") else None),
        "lmhead_ce_tokens_per_s": round(lm_tok_s, 1) if lm_tok_s else None,
        "gpu_launches": step.launches_per_step * args.steps,
        "wall_s_timed_region": round(wall, 4),
        "roofline": {"kernel": name, "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{src} bf16_tflops (burst, the conservative denominator; "
                                    "frac_of_sustained_peak uses bf16_tflops_sustained)",
                     "frac_of_sustained_peak": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                                if peaks.get("bf16_tflops_sustained") else None),
                     "flops_per_launch": fl, "ms_per_launch": round(per_call[k_dom], 4),
                     "traffic": traffic},
        "e2e": {"value": round(e2e_value, 2) if e2e_value else None, "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "step_ms": [round(t, 3) for t in e2e_ms_list],
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "each step's activations, upstream gradients and targets copied "
                          "host -> device from pinned memory on a copy stream into one of two "
                          "device buffer sets, a step ahead (step 0's copy not overlapped); the "
                          "weights stay resident on the device and are not copied; each step's "
                          "losses and dgamma are read back",
                "timing": "the same number of steps as the timed region, run after it and "
                          "the per-call pass, enqueued back to back with one host "
                          "synchronisation at the end",
                "clocks": clk_e2e},
        "clocks": clk,
        "step_ms_spread": {"min": round(min(step_ms), 4), "median": round(sorted(step_ms)[len(step_ms) // 2], 4),
                           "max": round(max(step_ms), 4), "all": [round(t, 3) for t in step_ms]},
        "parts_ms": {step.calls[k][0]: round(per_call[k], 4) for k in range(n)},
        "parts_note": ("per-call CUDA-event times from a separate pass with events between "
                       f"the calls (that pass: {attr_ms:.4f} ms/step; the timed steps have no "
                       "events between calls, so consecutive kernels overlap their launch)"),
    }
    if args.only:
        line["config"]["only"] = args.only
    else:
        line["per_config"] = per_config(step, per_call, peak)
        line["aux_hbm"] = aux_hbm(step, per_call, peaks.get("hbm_gbs"))
        line["l2_warm"] = l2_warm(step, args.steps, stream)
        line["graph"] = graph_step(step, flush, args.steps, stream)
    if not args.only and not args.no_next_rows:
        line["next_rows"] = next_rows(step, flush)
    if not args.only and not args.no_primitives:
        clk_p = Clocks(_smi_id(local))
        clk_p.start()
        time.sleep(0.2)
        tp0 = time.time()
        prim = primitives_table(C, dev, reps=5)
        tp1 = time.time()
        prim["clocks"] = clk_p.stop(window=(tp0, tp1))
        line["primitives"] = prim
    if not args.only and not args.no_unfused:
        ref_ms = unfused_reference(step, flush)
        line["unfused_reference"] = {
            "what": "PyTorch eager bf16 on the same inputs: cuBLAS matmuls, separate residual, "
                    "rms_norm, SiLU*mul, RoPE and cross_entropy kernels (logits materialised), "
                    "autograd backward",
            "ms_per_step": round(ref_ms, 4), "value": round(step.flops / (ref_ms * 1e-3) / 1e12, 2),
            "unit": UNIT, "fused_speedup": round(ref_ms / ms, 3)}
    if rank == 0 and not args.no_cpu_baseline and not args.only:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ rows beyond the step

def per_config(step, per_call, peak):
    """The step's workloads one by one (sums of their calls' event times):
    the 1B-shaped block forward and backward, the LM head + CE, the 8B-shaped
    block forward + backward; GEMM FLOPs only."""
    groups = {"llama1b_mlp_fwd": lambda n: n in ("1b.gemm_resid_norm_stats", "1b.row_rms",
                                                    "1b.gemm_rowscale_swiglu", "1b.gemm_down"),
              "lmhead_ce": lambda n: n == "lmhead_ce",
              "llama1b_mlp_bwd": lambda n: n.startswith("1b.") and n not in (
                  "1b.gemm_resid_norm_stats", "1b.row_rms", "1b.gemm_rowscale_swiglu",
                  "1b.gemm_down"),
              "llama8b_block_fwd_bwd": lambda n: n.startswith("8b.")}
    out = {}
    for gname, pred in groups.items():
        ks = [k for k, c in enumerate(step.calls) if pred(c[0])]
        if not ks:
            continue
        ms = sum(per_call[k] for k in ks)
        fl = sum(step.calls[k][1] for k in ks)
        ent = {"ms": round(ms, 4), "gflop": round(fl / 1e9, 1),
               "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
               "frac_of_burst_peak": round(fl / (ms * 1e-3) / 1e12 / peak, 3)}
        if gname == "lmhead_ce":
            ent["tokens_per_s"] = round(step.s2.M / (ms * 1e-3), 1)
        out[gname] = ent
    return out


def aux_hbm(step, per_call, hbm_gbs):
    """The bandwidth-bound auxiliary kernels: algorithmic bytes / event time
    against the measured copy bandwidth."""
    out = {}
    names = [c[0] for c in step.calls]
    if "8b.rope_bwd" in names:
        s4 = step.s4
        M, N = s4.M, s4.n_qkv
        # dqkv_rot bf16 and the fp16 saved copy in, dqkv_hat bf16 out, r in, s out,
        # the cos/sin table once
        byts = 3 * 2 * M * N + 8 * M + 4 * 2 * s4.seq_len * (s4.head_dim // 2)
        ms = per_call[names.index("8b.rope_bwd")]
        gbs = byts / (ms * 1e-3) / 1e9
        out["rope_bwd"] = {"bytes": byts, "ms": round(ms, 4), "gb_s": round(gbs, 1),
                           "frac_of_hbm_peak": round(gbs / hbm_gbs, 3) if hbm_gbs else None}
    for n in ("1b.row_rms", "1b.row_rms_bwd", "1b.col_reduce"):
        if n in names:
            out[n.split(".", 1)[1] + "_us"] = round(1e3 * per_call[names.index(n)], 1)
    return out


def l2_warm(step, steps, stream):
    """The same step back to back without the L2 flush in between (inputs and
    weights partly L2-resident from the previous step)."""
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step.run()
    b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"ms_per_step": round(ms, 4), "tflops": round(step.flops / (ms * 1e-3) / 1e12, 2)}


def graph_step(step, flush, steps, stream):
    """The same step captured once into a CUDA graph (blocks.CapturedStep)
    and replayed, L2 flushed before each replay: one host launch per step."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    cap = blocks.CapturedStep(step.run, warmup=1)
    ts = []
    for i in range(steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cap.replay()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = sum(ts) / len(ts)
    return {"ms_per_step": round(ms, 4), "tflops": round(step.flops / (ms * 1e-3) / 1e12, 2),
            "what": "the timed step captured once in a CUDA graph and replayed"}


def next_rows(step, flush, reps=5):
    """Kernels built beyond the step's rows, timed on the step's LM-head
    inputs: the cross-entropy backward (logits recomputed per vocabulary
    chunk; three GEMMs of 2*M*d*V each)."""
    C = step.C
    s2, i2 = step.s2, step.i2
    dev = step.dev
    dl = torch.full((s2.M,), 1.0 / s2.M, dtype=torch.float32, device=dev)
    dh = torch.empty((s2.M, s2.d), dtype=torch.float32, device=dev)
    dW = torch.empty((s2.d, s2.V), dtype=torch.float32, device=dev)
    ws = torch.empty(C.coda_lmhead_ce_bwd_workspace_size(s2.M, s2.V), dtype=torch.uint8, device=dev)
    fn = lambda: C.coda_lmhead_ce_bwd(i2["hidden"], i2["W"], i2["targets"], step.o2["lse"], dl,
                                      dh, dW, ws)
    fn()
    torch.cuda.synchronize()
    ts = []
    for i in range(reps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = sorted(ts)[len(ts) // 2]
    fl = 3 * 2.0 * s2.M * s2.d * s2.V
    chunk = min(16384, (s2.V + 255) // 256 * 256)  # the recommended workspace's chunk
    rows = {"lmhead_ce_bwd": {"ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
                              "tokens_per_s": round(s2.M / (ms * 1e-3), 1),
                              "launches": 3 * ((s2.V + chunk - 1) // chunk)}}
    rows.update(layernorm_row(step, flush, reps))
    return rows


def _median_ms(fn, flush, reps):
    fn()
    torch.cuda.synchronize()
    ts = []
    for i in range(reps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return sorted(ts)[len(ts) // 2]


def layernorm_row(step, flush, reps=5):
    """The LayerNorm variant of the MLP block, forward + backward, on the
    Llama-1B MLP shape (M=8192, d=2048, f=8192), timed beside the RMSNorm
    block run the same way (block-level calls, buffers from torch's caching
    allocator). GEMM FLOPs: forward 2M(d^2 + 3df), backward twice that."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    from coda_inputs import BlockShape, ln_block_inputs
    s1 = step.s1
    sh = BlockShape("llama1b_ln_mlp", M=s1.M, d=s1.d, f=s1.f, seed=7)
    g = ln_block_inputs(sh, device=step.dev)

    def ln():
        fw = blocks.ln_mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"],
                                     g["beta"])
        blocks.ln_mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"],
                                g["dout"])

    def rms():
        fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
        blocks.mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["dout"])

    ms_ln = _median_ms(ln, flush, reps)
    ms_rms = _median_ms(rms, flush, reps)
    fl = 3 * 2.0 * sh.M * (sh.d * sh.d + 3 * sh.d * sh.f)
    return {"layernorm_mlp_fwd_bwd": {
        "ms": round(ms_ln, 4), "tflops": round(fl / (ms_ln * 1e-3) / 1e12, 2),
        "rmsnorm_same_calls_ms": round(ms_rms, 4),
        "ratio_to_rmsnorm": round(ms_ln / ms_rms, 3), "launches": 15}}


# ------------------------------------------------------------------ unfused GPU reference

def unfused_reference(step, flush, steps=3, warmup=2):
    """The same step written the way a framework runs it unfused (PyTorch
    eager, bf16): cuBLAS GEMMs plus separate elementwise / normalisation /
    loss kernels, autograd for the backward. Reported as a reference point;
    it runs none of this library's kernels."""
    import warnings
    import torch.nn.functional as F
    warnings.filterwarnings("ignore", message="Attempting to run cuBLAS")
    s1, i1 = step.s1, step.i1
    i2 = step.i2
    d = s1.d

    def leaf(t):
        return t.detach().clone().requires_grad_(True)

    def one():
        x, z, W0, W1, W2, gm = (leaf(i1[k]) for k in ("x", "z", "W0", "W1", "W2", "gamma"))
        h = x @ W0 + z
        y = F.rms_norm(h, (d,), gm, 1e-6) @ W1
        out = (F.silu(y[:, 0::2]) * y[:, 1::2]) @ W2
        out.backward(i1["dout"])
        logits = i2["hidden"] @ i2["W"]
        F.cross_entropy(logits.float(), i2["targets"].long(), reduction="none")
        if step.with_8b:
            s4, i4 = step.s4, step.i4
            o, z4, Wo, W14, W24, g2, g1, Wq = (leaf(i4[k]) for k in
                                               ("o", "z", "Wo", "W1", "W2", "gamma2", "gamma1", "Wqkv"))
            h4 = o @ Wo + z4
            y4 = F.rms_norm(h4, (s4.d,), g2, 1e-6) @ W14
            out4 = (F.silu(y4[:, 0::2]) * y4[:, 1::2]) @ W24 + h4
            pre = F.rms_norm(out4, (s4.d,), g1, 1e-6) @ Wq
            nr, hd = s4.n_rope_cols, s4.head_dim
            pos = torch.arange(s4.M, device=o.device) % s4.seq_len
            inv = torch.pow(torch.tensor(s4.theta, dtype=torch.float64, device=o.device),
                            -2.0 * torch.arange(hd // 2, device=o.device, dtype=torch.float64) / hd)
            ang = (pos[:, None].double() * inv[None, :]).float().repeat(1, nr // hd)
            c, sn = torch.cos(ang), torch.sin(ang)
            e, od = pre[:, :nr:2].float(), pre[:, 1:nr:2].float()
            rot = torch.stack([e * c - od * sn, e * sn + od * c], dim=-1).reshape(s4.M, nr)
            qkv = torch.cat([rot.to(pre.dtype), pre[:, nr:]], dim=1)
            torch.autograd.backward([qkv, out4], [i4["dqkv"], i4["dres"]])

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    tot = 0.0
    for i in range(steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        b.synchronize()
        tot += a.elapsed_time(b)
    torch.cuda.empty_cache()
    return tot / steps


# ------------------------------------------------------------------ profiling cases

# Reduced shapes of the step's kernels (a few GB on the device at most) for
# multi-pass ncu captures; each runs 2 warm-up launches and 1 more launch.
KERNEL_CASES = {
    # weight gradient dW = X^T dY (both operands MN-major, fp32 out), K = tokens
    "wgrad_4096x7168x16384": dict(M=4096, N=7168, K=16384, transA=True, f32=True),
    # the forward-like GEMM with the same FLOPs (A K-major, B MN-major, bf16 out)
    "fwd_16384x7168x4096": dict(M=16384, N=7168, K=4096, transA=False, f32=False),
    # the row-scale + RoPE GEMM of the 8B block at half its rows (bf16 out + fp16 copy)
    "rope_8192x6144x4096": dict(M=8192, N=6144, K=4096, kind="rope"),
    # the plain GEMM of the same shape, for comparison
    "fwd_8192x6144x4096": dict(M=8192, N=6144, K=4096, transA=False, f32=False),
    # the 1B block's SwiGLU GEMM at half its rows (a bf16 + the fp16 saved y)
    "swiglu_4096x16384x2048": dict(M=4096, N=16384, K=2048, kind="swiglu"),
    "fwd_4096x16384x2048": dict(M=4096, N=16384, K=2048, transA=False, f32=False),
    # the LM head + CE at a quarter of its tokens (W, 525 MB, still far larger than L2)
    "lmhead_2048x128256x2048": dict(M=2048, N=128256, K=2048, kind="lmhead"),
}


def run_kernel_case(args):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as C
    cs = KERNEL_CASES[args.kernel_case]
    gen = torch.Generator(device=dev).manual_seed(0)
    M, N, K = cs["M"], cs["N"], cs["K"]
    if cs.get("kind") == "swiglu":
        A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
        B = (torch.randn((K, N), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        r = torch.rand(M, generator=gen, device=dev) + 0.5
        a_out = torch.empty((M, N // 2), dtype=torch.bfloat16, device=dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        fn = lambda: C.coda_gemm_rowscale_swiglu(A, B, r, a_out, y)
    elif cs.get("kind") == "rope":
        from gemm_epilogue_fusion_tcgen05_gb300 import blocks
        A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
        B = (torch.randn((K, N), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        r = torch.rand(M, generator=gen, device=dev) + 0.5
        table = blocks.rope_table(4096, 128, 500000.0, dev)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        save = torch.empty((M, N), dtype=torch.float16, device=dev)
        fn = lambda: C.coda_gemm_rope(A, B, r, table, 4096, 128, N - 1024, out, save)
    elif cs.get("kind") == "lmhead":
        A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
        B = (torch.randn((K, N), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        t = torch.randint(0, N, (M,), generator=gen, device=dev, dtype=torch.int32)
        lse = torch.empty(M, dtype=torch.float32, device=dev)
        loss = torch.empty(M, dtype=torch.float32, device=dev)
        ws = torch.empty(C.coda_lmhead_ce_workspace_size(M, N), dtype=torch.uint8, device=dev)
        fn = lambda: C.coda_lmhead_ce(A, B, t, lse, loss, ws)
    else:
        A = torch.randn((K, M) if cs["transA"] else (M, K), generator=gen, device=dev).to(torch.bfloat16)
        B = torch.randn((K, N), generator=gen, device=dev).to(torch.bfloat16)
        Cm = torch.empty((M, N), dtype=torch.float32 if cs["f32"] else torch.bfloat16, device=dev)
        fn = lambda: C.coda_gemm(A, B, Cm, transA=cs["transA"])
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    b.synchronize()
    st = C.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {st}")
    ms = a.elapsed_time(b)
    print(json.dumps({"kernel_case": args.kernel_case, "ms": round(ms, 4),
                      "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)}))


PROFILE_PASSES = ("1b", "lmhead", "8b", "ln")


def run_profile_pass(args):
    """One pass over one workload's library calls, without warm-up, so that
    an ncu capture of any kernel sees few launches before it and a few GB on
    the device:
      1b      the Llama-3-1B-shaped MLP block forward + backward (M = 8192)
      lmhead  LM head + CE forward and the chunked CE backward
              (M = 8192, V = 128256)
      8b      the Llama-3-8B-shaped non-attention block forward + backward
              at 4096 tokens (one sequence; the bench step has four)
      ln      the LayerNorm form of the 1B-shaped MLP block, forward +
              backward (M = 8192)"""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as C
    ph = args.profile_pass
    names = []
    if ph in ("1b", "lmhead", "8b"):
        step = Step(dev, with_1b=ph == "1b", with_lm=ph == "lmhead", with_8b=ph == "8b",
                    tokens_8b=4096)
        for name, fl, fn, nl in step.calls:
            fn()
            names.append(name)
        if ph == "lmhead":
            s2, i2 = step.s2, step.i2
            dl = torch.full((s2.M,), 1.0 / s2.M, dtype=torch.float32, device=dev)
            dh = torch.empty((s2.M, s2.d), dtype=torch.float32, device=dev)
            dW = torch.empty((s2.d, s2.V), dtype=torch.float32, device=dev)
            ws = torch.empty(C.coda_lmhead_ce_bwd_workspace_size(s2.M, s2.V), dtype=torch.uint8,
                             device=dev)
            C.coda_lmhead_ce_bwd(i2["hidden"], i2["W"], i2["targets"], step.o2["lse"], dl, dh, dW, ws)
            names.append("lmhead_ce_bwd")
    else:
        from gemm_epilogue_fusion_tcgen05_gb300 import blocks
        from coda_inputs import BlockShape, WORKLOADS, ln_block_inputs
        s1 = WORKLOADS["llama1b_mlp_bwd"]
        sh = BlockShape("llama1b_ln_mlp", M=s1.M, d=s1.d, f=s1.f, seed=7)
        gi = ln_block_inputs(sh, device=dev)
        fw = blocks.ln_mlp_block_fwd(gi["x"], gi["z"], gi["W0"], gi["W1"], gi["W2"], gi["gamma"],
                                     gi["beta"])
        blocks.ln_mlp_block_bwd(fw, gi["x"], gi["W0"], gi["W1"], gi["W2"], gi["gamma"], gi["beta"],
                                gi["dout"])
        names += ["ln_mlp_block_fwd", "ln_mlp_block_bwd"]
    torch.cuda.synchronize()
    st = C.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {st}")
    print(json.dumps({"profile_pass": ph, "calls": names,
                      "device_gb": round(torch.cuda.max_memory_allocated(dev) / 1e9, 2)}))


# ------------------------------------------------------------------ primitive microbenchmarks

def primitives_table(C, dev, reps=7):
    """One GEMM shape (8192 x 8192 x 4096, bf16) with one epilogue primitive
    of each class ("Reading notes on CODA", s1; the pages' Fig. 8 measures
    the same kind of table on H100), fused here vs cuBLAS followed by a
    separate PyTorch kernel:
      elementwise/pairwise map   SwiGLU on adjacent columns
      row/column vector load     row scale r[m] (delayed RMSNorm factor)
      tile load/store            residual add
      tile reduction             per-row sum of squares
      stateful transform         running max / sum-exp (LSE + CE, V = N)
    Medians of `reps` runs, L2 flushed before each."""
    import torch.nn.functional as F
    gen = torch.Generator(device=dev).manual_seed(7)
    M, N, K = 8192, 8192, 4096
    bf, f32 = torch.bfloat16, torch.float32
    A = torch.randn(M, K, device=dev, generator=gen).to(bf)
    B = (torch.randn(K, N, device=dev, generator=gen) * 0.02).to(bf)
    R = torch.randn(M, N, device=dev, generator=gen).to(bf)
    r = torch.rand(M, device=dev, generator=gen) + 0.5
    t = torch.randint(0, N, (M,), device=dev, generator=gen, dtype=torch.int32)
    out = torch.empty(M, N, dtype=bf, device=dev)
    half = torch.empty(M, N // 2, dtype=bf, device=dev)
    part = torch.empty(C.col_tiles(N), M, dtype=f32, device=dev)
    cs = torch.zeros(16, 64, 2, dtype=f32, device=dev)
    lse = torch.empty(M, dtype=f32, device=dev)
    loss = torch.empty(M, dtype=f32, device=dev)
    ws = torch.empty(C.coda_lmhead_ce_workspace_size(M, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(128 * 1024 * 1024, dtype=f32, device=dev)

    def timeit(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for i in range(reps):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return sorted(ts)[len(ts) // 2]

    cases = {
        "pairwise map (SwiGLU)": (
            lambda: C.coda_gemm_rowscale_swiglu(A, B, torch.ones_like(r), half, None),
            lambda: (lambda y: F.silu(y[:, 0::2]) * y[:, 1::2])(A @ B)),
        "row vector (scale r[m])": (
            lambda: C.coda_gemm_rope(A, B, r, cs, 16, 128, 0, out),
            lambda: (A @ B) * r[:, None].to(bf)),
        "tile load (residual)": (
            lambda: C.coda_gemm(A, B, out, resid=R),
            lambda: A @ B + R),
        "tile reduction (row sum of squares)": (
            lambda: C.coda_gemm(A, B, out, rowsq_part=part),
            lambda: (lambda y: (y, y.float().square().sum(1)))(A @ B)),
        "stateful max/sum-exp (LSE + CE)": (
            lambda: C.coda_lmhead_ce(A, B, t, lse, loss, ws),
            lambda: F.cross_entropy((A @ B).float(), t.long(), reduction="none")),
    }
    # what each fused call produced, to set against the unfused result
    fused_out = {
        "pairwise map (SwiGLU)": lambda: half,
        "row vector (scale r[m])": lambda: out,
        "tile load (residual)": lambda: out,
        "tile reduction (row sum of squares)": lambda: part.sum(0),
        "stateful max/sum-exp (LSE + CE)": lambda: loss,
    }
    unfused_out = {"tile reduction (row sum of squares)": lambda u: u[1]}

    def maxrel(a, b):
        a, b = a.float(), b.float()
        return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))

    gemm_ms = timeit(lambda: torch.matmul(A, B, out=out))
    res = {}
    for name, (fused, unfused) in cases.items():
        fm, um = timeit(fused), timeit(unfused)
        fused()
        got = fused_out[name]().clone()
        want = unfused_out.get(name, lambda u: u)(unfused())
        res[name] = {"fused_ms": round(fm, 4), "cublas_plus_kernel_ms": round(um, 4),
                     "speedup": round(um / fm, 3),
                     # the unfused path rounds its GEMM output to bf16 first
                     "max_rel_diff_vs_unfused": round(maxrel(got, want), 6)}
    st = C.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {st}")
    return {"shape": [M, N, K], "cublas_gemm_alone_ms": round(gemm_ms, 4), "reps": reps,
            "primitives": res}


def run_primitives(args):
    """The primitive table alone, as its own JSON line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as C
    clk = Clocks(_smi_id(0))
    clk.start()
    time.sleep(0.2)
    t0 = time.time()
    tab = primitives_table(C, dev)
    t1 = time.time()
    line = {"metric": "epilogue primitives: fused GEMM+epilogue vs cuBLAS + separate kernel",
            **tab, "clocks": clk.stop(window=(t0, t1))}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ CPU oracle

def _oracle_sample(rows1, rows_ce, rows8):
    """The CPU oracle, as it stands, on the first rows of each part of the
    step. Returns (flops, seconds); flops counted like the GPU metric."""
    import numpy as np
    from coda_inputs import WORKLOADS, BlockShape, LMHeadShape, Block8BShape, \
        mlp_block_inputs, lmhead_inputs, block8b_inputs, positions
    from oracle import coda_oracle as O
    s1 = WORKLOADS["llama1b_mlp_bwd"]
    s2 = WORKLOADS["lmhead_ce"]
    s4 = WORKLOADS["llama8b_block"]
    # draw the sample directly at its row count (same recipe, fewer rows)
    i1 = mlp_block_inputs(BlockShape("s", rows1, s1.d, s1.f, s1.seed))
    i2 = lmhead_inputs(LMHeadShape("s", rows_ce, s2.d, s2.V, s2.seed))
    i4 = block8b_inputs(Block8BShape("s", rows8, s4.d, s4.f, s4.seq_len, s4.head_dim,
                                     s4.n_q_heads, s4.n_kv_heads, s4.theta, s4.seed))
    n1 = {k: O.to64(v) for k, v in i1.items()}
    n2 = {k: O.to64(v) for k, v in i2.items()}
    n4 = {k: O.to64(v) for k, v in i4.items()}
    pos = positions(rows8, s4.seq_len).numpy()
    t0 = time.perf_counter()
    fw = O.mlp_fwd(n1["x"], n1["z"], n1["W0"], n1["W1"], n1["W2"], n1["gamma"])
    O.mlp_bwd(fw, n1["x"], n1["W0"], n1["W1"], n1["W2"], n1["gamma"], n1["dout"])
    O.lmhead_ce(n2["hidden"], n2["W"], i2["targets"].numpy())
    f4 = O.block8b_fwd(n4["o"], n4["z"], n4["Wo"], n4["W1"], n4["W2"], n4["gamma2"], n4["gamma1"],
                       n4["Wqkv"], pos, s4.n_rope_cols, s4.head_dim, s4.theta)
    O.block8b_bwd(f4, n4["o"], n4["Wo"], n4["W1"], n4["W2"], n4["gamma2"], n4["gamma1"],
                  n4["Wqkv"], n4["dqkv"], n4["dres"], pos, s4.n_rope_cols, s4.head_dim, s4.theta)
    dt = time.perf_counter() - t0
    d, f = s1.d, s1.f
    fl1 = rows1 * 3 * 2 * (d * d + d * 2 * f + f * d)
    fl2 = rows_ce * 2 * s2.d * s2.V
    d4, f4_, n4q = s4.d, s4.f, s4.n_qkv
    fl4 = rows8 * 3 * 2 * (d4 * d4 + d4 * 2 * f4_ + f4_ * d4 + d4 * n4q)
    return float(fl1 + fl2 + fl4), dt


def cpu_baseline(seconds_target=15.0):
    """The oracle on a row sample of the step's workloads, scaled from a
    short probe so that the measured sample takes about `seconds_target`
    (each part at most its workload's rows)."""
    from coda_inputs import WORKLOADS
    full = (WORKLOADS["llama1b_mlp_bwd"].M, WORKLOADS["lmhead_ce"].M, WORKLOADS["llama8b_block"].M)
    rows = (512, 64, 64)
    fl, dt = _oracle_sample(*rows)
    scale = max(1.0, min(32.0, seconds_target / max(dt, 1e-3)))
    if scale > 1.5:
        rows = tuple(min(f, max(8, int(r * scale) // 8 * 8)) for r, f in zip(rows, full))
        fl, dt = _oracle_sample(*rows)
    return {"value": round(fl / dt / 1e12, 5), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle on {rows[0]} rows of the 1B block fwd+bwd, {rows[1]} rows "
                      f"of the LM head, {rows[2]} rows of the 8B block fwd+bwd ({dt:.1f} s, "
                      f"{fl / 1e12:.2f} TFLOP)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    rows = (256, 32, 32)
    for _ in range(args.warmup):
        _oracle_sample(*rows)
    fl_tot, dt_tot = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = _oracle_sample(*rows)
        fl_tot += fl
        dt_tot += dt
    v = fl_tot / dt_tot / 1e12
    line = {"metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt_tot / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic (seeded; CPU draws)",
            "config": {"workload": "llama1b_mlp_fwd+lmhead_ce+llama1b_mlp_bwd+llama8b_block_fwd_bwd",
                       "sample_rows": {"1b": rows[0], "lmhead": rows[1], "8b": rows[2]}},
            "cpu_baseline": {"value": round(v, 5), "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"fp64 numpy oracle, {rows[0]}/{rows[1]}/{rows[2]} rows "
                                       "of the 1B block / LM head / 8B block per step"},
            "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def launch_ranks(n, argv, timeout_s=3600):
    """Start n ranks of this script on this node, one process per GPU, the way
    torchrun does: RANK = LOCAL_RANK = i, WORLD_SIZE = n, rendezvous on
    127.0.0.1. Each rank is a replica (the path needs no exchange); rank 0
    prints the line. Returns the worst exit code; if any rank fails, the
    others are stopped."""
    port = _free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env))
    rc = 0
    t0 = time.time()
    pending = list(procs)
    while pending:
        for p in list(pending):
            c = p.poll()
            if c is None:
                continue
            pending.remove(p)
            rc = max(rc, abs(c))
            if c != 0:
                for q in pending:
                    q.terminate()
        if time.time() - t0 > timeout_s:
            for q in pending:
                q.kill()
            rc = max(rc, 124)
            break
        time.sleep(0.1)
    for p in procs:
        p.wait()
    return rc


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def run_probe_ranks(args):
    """The rank plumbing alone (no GPU work): every rank joins the process
    group, reports its rank and the device it would use (LOCAL_RANK), and
    rank 0 prints them. With --backend gloo it runs on CPU."""
    import torch.distributed as dist
    ws, rank, local = _dist()
    backend = args.backend or ("nccl" if torch.cuda.is_available() else "gloo")
    if ws > 1:
        dist.init_process_group(backend)
    me = {"rank": rank, "local_rank": local, "device_index": local, "pid": os.getpid()}
    allr = [None] * ws
    if ws > 1:
        dist.all_gather_object(allr, me)
        dist.barrier()
    else:
        allr = [me]
    if rank == 0:
        print(json.dumps({"probe": "ranks", "n_gpus": ws, "backend": backend if ws > 1 else None,
                          "ranks": allr}), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (ranks) on this node; under torchrun it must equal WORLD_SIZE, "
                         "without it N > 1 starts the N ranks itself")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["coda", "reference"], default="coda")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-8b", action="store_true", help="leave the 8B-shaped block out of the step")
    ap.add_argument("--primitives", action="store_true",
                    help="epilogue-primitive microbenchmarks instead of the step")
    ap.add_argument("--kernel-case", default="", choices=[""] + sorted(KERNEL_CASES),
                    help="run one reduced-shape GEMM three times (for ncu captures)")
    ap.add_argument("--profile-pass", default="", choices=[""] + list(PROFILE_PASSES),
                    help="run one workload's calls once, without warm-up (for per-kernel ncu "
                         "captures)")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the rows timed beyond the step (CE backward, LayerNorm block)")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip the unfused PyTorch reference sequence")
    ap.add_argument("--only", default="", help="time only these calls (comma-separated names; "
                    "profiling aid, not a bench line)")
    ap.add_argument("--no-primitives", action="store_true",
                    help="leave the epilogue-primitive table out of the default line")
    ap.add_argument("--probe-ranks", action="store_true",
                    help="start the ranks and report them, with no GPU work")
    ap.add_argument("--backend", default="", help="process-group backend for --probe-ranks")
    args = ap.parse_args(argv)
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" in os.environ:
        if int(os.environ["WORLD_SIZE"]) != args.gpus:
            raise SystemExit(f"--gpus {args.gpus} does not match WORLD_SIZE "
                             f"{os.environ['WORLD_SIZE']} (one rank per GPU)")
    elif args.gpus > 1:
        sys.exit(launch_ranks(args.gpus, argv))
    if args.warmup < 3:
        print("note: at least 3 warm-up steps are required; using 3", file=sys.stderr)
        args.warmup = 3
    if args.probe_ranks:
        run_probe_ranks(args)
    elif args.kernel_case:
        run_kernel_case(args)
    elif args.profile_pass:
        run_profile_pass(args)
    elif args.primitives:
        run_primitives(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_coda(args)


if __name__ == "__main__":
    main()
