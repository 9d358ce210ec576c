"""Benchmark: one Ulysses attention layer step (fwd + bwd) on the GPU.

A step is one pass of the whole hot path over one batch of synthetic input,
in a layer's order: for every virtual rank and UPipe chunk, seq2head of
Q/K/V, attention forward, head2seq of O; then for every stage again seq2head
of Q/K/V/O/dO, attention backward, head2seq of dQ/dK/dV.  Default workload: the Qwen3-4B-shaped layer at S=65536
(H_q=32, H_kv=8, D=128, P=4 virtual ranks, head_chunk=8, bf16 N(0,1) inputs).

Prints one JSON line.  `value` is tokens/s of the whole step with inputs
resident in HBM; `e2e` is the same through the public layer API with the
inputs copied from pinned host memory and the outputs copied back inside the
timed region.  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from long_context_sequence_seq_gb300 import inputs  # noqa: E402

METRIC = "causal attn fwd+bwd tokens/s & TFLOPS at S=64K (% BF16 peak); re-layout GB/s"
UNIT = "tokens/s"

# Nominal dense GB300 figures (bf16 tensor, HBM3e), reported beside the
# measured peaks for context.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0

# DRAM bytes per launch of the dominant kernel from an ncu capture of this
# workload, valid only for the kernel source it was taken on (sha256 prefix);
# any other source reports null.
TRAFFIC = {"qwen3_4b_64k": ("attn_tc_bwd.cu", "b5a16aedd5cff6b1", 3267981760)}


def measured_traffic(workload):
    import hashlib
    if workload not in TRAFFIC:
        return None
    fname, sha, nbytes = TRAFFIC[workload]
    path = os.path.join(ROOT, "long_context_sequence_seq_gb300", "csrc", fname)
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return nbytes if digest.startswith(sha) else None


def reduce_max(value, device=None):
    """Max of a per-rank float over the default process group (identity when
    no group is initialised)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, B, S, t_step):
    """Whole-job throughput: every replica processes B*S tokens per step."""
    return world * B * S / t_step


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def pairs_total(w, cu):
    """Unmasked (i, j) pairs per head (host arithmetic on the mask only)."""
    if cu is None:
        return w.S * (w.S + 1) // 2 if w.causal else w.S * w.S
    L = np.diff(np.asarray(cu, dtype=np.int64))
    return int(np.sum(L * (L + 1) // 2)) if w.causal else int(np.sum(L * L))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class LayerStep:
    """Device-resident buffers and the per-stage C-ABI call sequence of one step.

    The step does what a layer does: the forward over every UPipe stage, then
    the backward over every stage, which gathers the stage's Q, K, V, O and
    dO again (dO only exists after the whole forward).  Per stage each
    direction is one batched gather, the attention call and one batched
    scatter, the same launches as the native layer drivers.  CUDA events on
    the launching stream bracket every launch group, so the attention and
    re-layout durations come from the timed region itself.
    """

    def __init__(self, w, dev, cu_np):
        from long_context_sequence_seq_gb300 import ulysses as U
        self.U = U
        self.w = w
        q, k, v, do = inputs.make_seq_inputs(w, device=dev, small_on_host=False)
        self.q, self.k, self.v, self.do = q, k, v, do
        self.cu = None if cu_np is None else torch.from_numpy(cu_np).to(dev)
        self.o = torch.empty_like(q)
        self.lse = torch.empty((w.B, w.H_q, w.S), dtype=torch.float32, device=dev)
        self.dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        self.dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        self.dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        C, G = w.head_chunk, w.G
        S, B, D = w.S, w.B, w.D
        mk = lambda n, dt: torch.empty((B, n, S, D), dtype=dt, device=dev)  # noqa: E731
        dt = q.dtype
        self.qh, self.oh, self.doh = mk(C, dt), mk(C, dt), mk(C, dt)
        self.kh, self.vh = mk(C // G, dt), mk(C // G, dt)
        self.dqh = mk(C, torch.float32)
        self.dkh, self.dvh = mk(C // G, torch.float32), mk(C // G, torch.float32)
        # B > 1: a stage's LSE rows are not contiguous in [B, H_q, S]; keep one
        # [B, C, S] buffer per stage (the backward reads it after every forward)
        self.stages = w.P * (w.H_q // w.P // C)
        self.lse_st = [] if B == 1 else [torch.empty((B, C, S), dtype=torch.float32, device=dev)
                                         for _ in range(self.stages)]
        wsb = U.attn_bwd_workspace_bytes(S, B, w.H_q, w.H_kv, D, w.P, C, 0,
                                         U.BF16 if w.dtype == "bf16" else U.FP32)
        self.ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        self.events = []      # per timed step: lists of (r0, r1, r2, r3) for fwd and bwd stages

    def _lse_stage(self, st):
        w = self.w
        hq = w.H_q // w.P
        r, c = divmod(st, hq // w.head_chunk)
        h0 = r * hq + c * w.head_chunk
        # B == 1: the stage's rows of the global [B, H_q, S] LSE are contiguous
        return self.lse[:, h0:h0 + w.head_chunk] if w.B == 1 else self.lse_st[st]

    def run(self, timed=False):
        U, w = self.U, self.w
        C, G, P = w.head_chunk, w.G, w.P
        ev_f, ev_b = [], []

        def marks():
            if not timed:
                return None
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            return e

        for st in range(self.stages):
            e = marks()
            if e:
                e[0].record()
            U.seq2head_n([(self.q, self.qh, C, st), (self.k, self.kh, C // G, st),
                          (self.v, self.vh, C // G, st)], P)
            if e:
                e[1].record()
            U.attn_fwd(self.qh, self.kh, self.vh, w.H_q, w.H_kv, P, C, st, self.cu, w.causal,
                       out=self.oh, lse=self._lse_stage(st))
            if e:
                e[2].record()
            U.head2seq(self.oh, self.o, P, C, st)
            if e:
                e[3].record()
                ev_f.append(e)
        for st in range(self.stages):
            e = marks()
            if e:
                e[0].record()
            U.seq2head_n([(self.q, self.qh, C, st), (self.k, self.kh, C // G, st),
                          (self.v, self.vh, C // G, st), (self.o, self.oh, C, st),
                          (self.do, self.doh, C, st)], P)
            if e:
                e[1].record()
            U.attn_bwd(self.qh, self.kh, self.vh, self.oh, self.doh, self._lse_stage(st), w.H_q, w.H_kv,
                       P, C, st, self.cu, w.causal, workspace=self.ws, dq=self.dqh,
                       dk=self.dkh, dv=self.dvh)
            if e:
                e[2].record()
            U.head2seq_n([(self.dqh, self.dq, C, st), (self.dkh, self.dk, C // G, st),
                          (self.dvh, self.dv, C // G, st)], P)
            if e:
                e[3].record()
                ev_b.append(e)
        if timed:
            self.events.append((ev_f, ev_b))

    def durations(self):
        """Mean per step of (forward attention, backward attention, all
        re-layouts) in seconds, from the events of the timed steps."""
        fw, bw, rl = [], [], []
        for ev_f, ev_b in self.events:
            f = sum(e[1].elapsed_time(e[2]) for e in ev_f) / 1e3
            b = sum(e[1].elapsed_time(e[2]) for e in ev_b) / 1e3
            r = sum(e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in ev_f + ev_b) / 1e3
            fw.append(f)
            bw.append(b)
            rl.append(r)
        return statistics.mean(fw), statistics.mean(bw), statistics.mean(rl)


def relayout_bytes_per_step(w):
    """Bytes the step's re-layouts read plus write (STREAM-copy convention):
    forward Q, K, V gathered and O scattered; backward Q, K, V, O, dO gathered
    and the fp32 dQ, dK, dV scattered."""
    elt = 2 if w.dtype == "bf16" else 4
    n_q = w.B * w.S * w.H_q * w.D
    n_kv = w.B * w.S * w.H_kv * w.D
    fwd = 2 * (n_q + 2 * n_kv) * elt + 2 * n_q * elt
    bwd = 2 * (3 * n_q + 2 * n_kv) * elt + 2 * (n_q + 2 * n_kv) * 4
    return fwd + bwd


def measure_relayout(w, dev, reps=10):
    """Isolated K1 timing on the Q tensor (inputs larger than L2)."""
    from long_context_sequence_seq_gb300 import ulysses as U
    x = torch.empty((w.B, w.S, w.H_q, w.D), dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32,
                    device=dev)
    x.view(torch.int16 if x.element_size() == 2 else torch.int32).random_(0, 1000)
    out = torch.empty((w.B, w.H_q, w.S, w.D), dtype=x.dtype, device=dev)
    for _ in range(3):
        U.seq2head(x, w.P, None, None, out=out)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        U.seq2head(x, w.P, None, None, out=out)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / 1e3)
    byts = 2 * x.numel() * x.element_size()
    del x, out
    return byts / statistics.median(ts) / 1e9, byts


def e2e_measure(w, dev, cu_np, steps, warmup):
    """The public layer API with host buffers: H2D inputs, fwd+bwd, D2H outputs."""
    from long_context_sequence_seq_gb300 import ulysses as U
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in inputs.make_seq_inputs(w, device=dev, small_on_host=False))
    # two device copies of the inputs: step i+1's upload runs under step i
    bufs = [[torch.empty(t.shape, dtype=dt, device=dev) for t in (hq, hk, hv, hdo)] for _ in range(2)]
    ws = U.layer_workspace(w.S, w.B, w.H_q, w.H_kv, w.D, w.P, w.head_chunk,
                           U.BF16 if w.dtype == "bf16" else U.FP32, dev)
    cu = None if cu_np is None else torch.from_numpy(cu_np).to(dev)
    o = torch.empty(hq.shape, dtype=dt, device=dev)
    lse = torch.empty((w.B, w.H_q, w.S), dtype=torch.float32, device=dev)
    # two sets of device gradients: step i's download runs under step i+1
    grads = [[torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (hq, hk, hv)] for _ in range(2)]
    ho = torch.empty(o.shape, dtype=dt).pin_memory()
    hdq = torch.empty(hq.shape, dtype=torch.float32).pin_memory()
    hdk = torch.empty(hk.shape, dtype=torch.float32).pin_memory()
    hdv = torch.empty(hv.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hdq, hdk, hdv))

    # Copies run on two side streams, one per direction (separate copy
    # engines): step i's inputs are uploaded into buffer set i % 2 while step
    # i-1 computes from the other set; O is downloaded under the backward, and
    # dQ/dK/dV (gradient set i % 2) under the whole next step.  Events order
    # every reuse of a buffer, so every step still moves all of its inputs and
    # results.
    main = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]        # set j uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]      # set j no longer read
    ev = {name: torch.cuda.Event() for name in ("fwd", "o_out", "bwd")}
    ev_g_out = [torch.cuda.Event() for _ in range(2)]     # gradient set j is on the host
    state = {"i": 0}

    def upload(i):
        j = i % 2
        if i >= 2:
            up.wait_event(ev_used[j])
        with torch.cuda.stream(up):
            for d_, h_ in zip(bufs[j], (hq, hk, hv, hdo)):
                d_.copy_(h_, non_blocking=True)
            ev_in[j].record(up)

    def step(last):
        i = state["i"]
        j = i % 2
        q, k, v, do = bufs[j]
        main.wait_event(ev_in[j])
        if i > 0:
            main.wait_event(ev["o_out"])          # O of the previous step is on the host
        U.layer_fwd(q, k, v, w.P, w.head_chunk, cu, w.causal, workspace=ws, out=o, lse=lse)
        ev["fwd"].record(main)
        with torch.cuda.stream(down):
            down.wait_event(ev["fwd"])
            ho.copy_(o, non_blocking=True)
            ev["o_out"].record(down)
        if not last:
            upload(i + 1)                         # the next step's inputs, under this step
        dq, dk, dv = grads[j]
        if i >= 2:
            main.wait_event(ev_g_out[j])          # this set's gradients (step i-2) are on the host
        U.layer_bwd(q, k, v, o, do, lse, w.P, w.head_chunk, cu, w.causal, workspace=ws,
                    dq=dq, dk=dk, dv=dv)
        ev_used[j].record(main)
        ev["bwd"].record(main)
        with torch.cuda.stream(down):
            down.wait_event(ev["bwd"])
            for h_, d_ in ((hdq, dq), (hdk, dk), (hdv, dv)):
                h_.copy_(d_, non_blocking=True)
            ev_g_out[j].record(down)
        state["i"] = i + 1

    def run(n):
        state["i"] = 0
        upload(0)
        for s_ in range(n):
            step(s_ == n - 1)
        for e_ in ev_g_out:                       # every step's results are on the host
            main.wait_event(e_)

    run(warmup)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    up.wait_stream(main)
    run(steps)                                    # the first upload is inside the timed region
    b.record(main)
    torch.cuda.synchronize()
    U.check()
    t = a.elapsed_time(b) / 1e3 / steps

    # the host link on its own (one large pinned copy each way), which tells
    # how much of the per-step traffic the compute can hide on this machine
    def copy_gbs(dst, src):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        dst.copy_(src, non_blocking=True)
        e1.record(main)
        torch.cuda.synchronize()
        return src.numel() * src.element_size() / (e0.elapsed_time(e1) / 1e3) / 1e9
    link = {"h2d_gbs": copy_gbs(bufs[0][0], hq), "d2h_gbs": copy_gbs(hdq, grads[0][0])}
    return {"value": w.B * w.S / t, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": t * 1e3, "host_link": link}


def ring_measure(w, dev, steps, warmup):
    """The ring-attention variant of the same layer (P virtual ranks, KV
    chunks met one ring step at a time, partial results merged by LSE), timed
    forward + backward with CUDA events on inputs resident on the device."""
    from long_context_sequence_seq_gb300 import ulysses as U
    if w.B != 1 or w.packed:
        return None
    q, k, v, do = inputs.make_seq_inputs(w, device=dev)

    def step():
        o, lse = U.ring_attention_fwd(q, k, v, w.P, causal=w.causal)
        U.ring_attention_bwd(q, k, v, o, do, lse, w.P, causal=w.causal)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    U.check()
    t = a.elapsed_time(b) / 1e3 / steps
    fl = 14.0 * w.D * pairs_total(w, None) * w.H_q
    return {"ms_per_step": t * 1e3, "tflops_fwd_bwd": fl / t / 1e12,
            "note": "same layer as the ring variant: attention blocks of S/P tokens, LSE merges"}


def proj_measure(w, dev, reps=10):
    """The QKV projection with its head-layout epilogue and the output
    projection reading O from head layout, at the workload's model width,
    on synthetic weights (N(0, 1/fan_in)); CUDA events, median of reps."""
    from long_context_sequence_seq_gb300 import ulysses as U
    if not w.hidden or w.dtype != "bf16" or w.B != 1:
        return None
    g = torch.Generator(device=dev).manual_seed(inputs.SEED_Q + 100)
    nf = (w.H_q + 2 * w.H_kv) * w.D
    x = torch.randn(w.S, w.hidden, device=dev, generator=g).to(torch.bfloat16)
    wq = (torch.randn(nf, w.hidden, device=dev, generator=g) / w.hidden ** 0.5).to(torch.bfloat16)
    o = torch.randn(w.H_q, w.S, w.D, device=dev, generator=g).to(torch.bfloat16)
    wo = (torch.randn(w.hidden, w.H_q * w.D, device=dev, generator=g) / (w.H_q * w.D) ** 0.5).to(torch.bfloat16)
    qkv = torch.empty((w.H_q + 2 * w.H_kv, w.S, w.D), dtype=torch.bfloat16, device=dev)
    y = torch.empty((w.S, w.hidden), dtype=torch.bfloat16, device=dev)
    res = {}
    for name, fn, fl in (("qkv_proj", lambda: U.qkv_proj(x, wq, w.H_q, w.H_kv, out=qkv), 2.0 * w.S * nf * w.hidden),
                         ("out_proj", lambda: U.out_proj(o, wo, out=y), 2.0 * w.S * w.hidden * w.H_q * w.D)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        t = statistics.median(ts)
        res[name] = {"ms": t * 1e3, "tflops": fl / t / 1e12}
    U.check()
    res["hidden"] = w.hidden
    res["weights"] = "synthetic N(0, 1/fan_in)"
    return res


def fused_measure(w, dev, cu_np, steps, warmup):
    """The same layer step with the all-to-alls folded into the attention
    kernels (no re-layout launches, no head-layout copies), inputs resident on
    the device, CUDA events around the whole step."""
    from long_context_sequence_seq_gb300 import ulysses as U
    if w.B != 1 or w.dtype != "bf16" or w.D != 128:
        return None
    q, k, v, do = inputs.make_seq_inputs(w, device=dev)
    cu = None if cu_np is None else torch.from_numpy(cu_np).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H_q, w.S), dtype=torch.float32, device=dev)
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
    nb = U.lib().ulysses_layer_fused_workspace(w.S, w.B, w.H_q, w.H_kv, w.D, w.P, w.head_chunk, U.BF16)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)

    def step():
        U.layer_fwd_fused(q, k, v, w.P, w.head_chunk, cu, w.causal, out=o, lse=lse)
        U.layer_bwd_fused(q, k, v, o, do, lse, w.P, w.head_chunk, cu, w.causal, workspace=ws, dq=dq, dk=dk, dv=dv)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    U.check()
    t = a.elapsed_time(b) / 1e3 / steps
    return {"ms_per_step": t * 1e3, "tokens_per_s": w.B * w.S / t,
            "note": "all-to-alls folded into the attention kernels' addressing"}


def cpu_baseline(w, cu_np, min_sample_s=7.5):
    """The fp64 oracle as it stands on the host cores, on a bounded sample:
    forward + backward of one (q head, kv head) pair over a causal prefix of
    the sequence, the prefix doubled until one pass takes more than
    min_sample_s (so the timed pass takes ~8-30 s).  Reported as the
    full-workload tokens/s it implies (pairs per second of the oracle, scaled
    to all heads and pairs)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    L = 2048
    rng = np.random.Generator(np.random.PCG64(0))
    while True:
        q = rng.standard_normal((1, L, w.D))
        k = rng.standard_normal((1, L, w.D))
        v = rng.standard_normal((1, L, w.D))
        do = rng.standard_normal((1, L, w.D))
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v)
        oracle.attn_bwd(q, k, v, do)
        dt = time.perf_counter() - t0
        if dt > min_sample_s or L >= w.S:
            break
        L = min(w.S, L * 2)
    pairs_s = (L * (L + 1) / 2) / dt
    cu = cu_np
    total = pairs_total(w, cu) * w.H_q * w.B
    step_s = total / pairs_s
    return {"value": w.B * w.S / step_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of one q head over a {L}-token causal prefix "
                      f"({dt:.2f} s), scaled by unmasked pairs to all {w.H_q} heads",
            "sample_seconds": dt}


def gpu_arm(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from long_context_sequence_seq_gb300 import ulysses as U
    U.lib()
    w = workload_from_args(args)
    cu_np = inputs.workload_cu_seqlens(w)
    step = LayerStep(w, dev, cu_np)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    U.check()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    n0 = U.launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        step.run(timed=True)
    end.record()
    torch.cuda.synchronize()
    launches = U.launch_count() - n0
    clk = clocks.stop()
    U.check()
    elapsed = reduce_max(start.elapsed_time(end) / 1e3, dev)
    if world > 1:
        dist.barrier()
    t_step = elapsed / args.steps
    t_fwd, t_bwd, t_relayout = step.durations()
    n_launch_attn = step.stages
    pairs = pairs_total(w, cu_np) * w.H_q * w.B
    fl_fwd, fl_bwd = 4.0 * w.D * pairs, 10.0 * w.D * pairs
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    relay_bytes = relayout_bytes_per_step(w)
    relay_step_gbs = relay_bytes / t_relayout / 1e9
    relay_gbs = None
    e2e = None
    ring = None
    proj = None
    fused = None
    del step
    torch.cuda.empty_cache()
    if not args.kernels_only:
        relay_gbs, _ = measure_relayout(w, dev)
        e2e = e2e_measure(w, dev, cu_np, max(1, args.steps), max(1, args.warmup // 2))
        # whole job, like `value`: every replica's tokens over the slowest replica's time
        e2e_t = reduce_max(e2e["ms_per_step"] / 1e3, dev)
        e2e["ms_per_step"] = e2e_t * 1e3
        e2e["value"] = job_tokens_per_s(world, w.B, w.S, e2e_t)
        ring = ring_measure(w, dev, max(1, args.steps // 2), 1) if args.ring else None
        proj = proj_measure(w, dev) if args.proj else None
        fused = fused_measure(w, dev, cu_np, max(1, args.steps // 2), 1) if args.fused else None
    # dominant kernel = attention backward (2.5x the forward's FLOPs)
    bwd_per_launch_s = t_bwd / n_launch_attn
    achieved = fl_bwd / n_launch_attn / bwd_per_launch_s / 1e12
    res = {
        "metric": METRIC, "value": job_tokens_per_s(world, w.B, w.S, t_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic N(0,1), seeded",
        "config": workload_config(w, world),
        "tflops_fwd_bwd": (fl_fwd + fl_bwd) / (t_fwd + t_bwd) / 1e12,
        "attn_fwd_ms": t_fwd * 1e3, "attn_bwd_ms": t_bwd * 1e3,
        "attn_fwd_tflops": fl_fwd / t_fwd / 1e12, "attn_bwd_tflops": fl_bwd / t_bwd / 1e12,
        "frac_fwd_bwd_of_bf16_peak": (fl_fwd + fl_bwd) / (t_fwd + t_bwd) / 1e12 / bf16,
        "frac_fwd_bwd_of_nominal_bf16": (fl_fwd + fl_bwd) / (t_fwd + t_bwd) / 1e12 / NOMINAL_BF16_TFLOPS,
        "peaks": {"bf16_tflops": bf16, "hbm_gbs": hbm, "source": peak_src,
                  "nominal_bf16_tflops": NOMINAL_BF16_TFLOPS, "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                  "targets_measured_against": "the measured peaks (frac_* keys without 'nominal')"},
        "relayout_gbs": relay_step_gbs, "relayout_frac_hbm": relay_step_gbs / hbm,
        "relayout_ms_per_step": t_relayout * 1e3,
        "relayout_bytes_per_step": relay_bytes,
        "relayout_frac_nominal_hbm": relay_step_gbs / NOMINAL_HBM_GBS,
        "relayout_isolated_q_gather_gbs": relay_gbs,
        "relayout_isolated_q_gather_frac_hbm": None if relay_gbs is None else relay_gbs / hbm,
        "roofline": {"kernel": "attn_bwd", "bound": "tensor", "achieved": achieved,
                     "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16,
                     "traffic": measured_traffic(w.name),
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "frac_of_sustained_peak": achieved / bf16_sus if bf16_sus else None},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    if ring is not None:
        res["ring_variant"] = ring
    if proj is not None:
        res["projections_fused_relayout"] = proj
    if fused is not None:
        res["fused_relayout_step"] = fused
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, cu_np)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args):
    """The fp64 CPU oracle on the host cores (rank 0 only), one bounded sample
    per step, reported as the full-workload tokens/s the sample implies."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    w = workload_from_args(args)
    cu_np = inputs.workload_cu_seqlens(w)
    for _ in range(args.warmup):
        cpu_baseline(w, cu_np, min_sample_s=0.5)
    vals, secs = [], []
    for _ in range(args.steps):
        r = cpu_baseline(w, cu_np, min_sample_s=0.5)
        vals.append(r["value"])
        secs.append(r["sample_seconds"])
    v = statistics.median(vals)
    res = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic N(0,1), seeded", "impl": "reference",
           "config": workload_config(w, world),
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                            "sample": r["sample"]},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def workload_config(w, world):
    """The `config` object of both arms' JSON lines (same keys, same values)."""
    return {"workload": w.name, "S": w.S, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv,
            "D": w.D, "P": w.P, "head_chunk": w.head_chunk, "causal": w.causal,
            "packed": w.packed, "l2": "inputs larger than L2 (no flush needed)",
            "parallelism": f"{w.P} virtual ranks on one GPU" + (f", {world} replicas" if world > 1 else "")}


def workload_from_args(args):
    w = inputs.WORKLOADS[args.workload]
    if args.seq_len:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}@S={args.seq_len}", S=args.seq_len)
    return w


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qwen3_4b_64k", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ring", action="store_true",
                    help="also time the ring-attention variant of the same layer")
    ap.add_argument("--proj", action="store_true",
                    help="also time the projections with the re-layout fused in")
    ap.add_argument("--fused", action="store_true",
                    help="also time the layer step with the all-to-alls folded into the attention kernels")
    ap.add_argument("--kernels-only", action="store_true",
                    help="skip the isolated re-layout and end-to-end measurements (profiling runs)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override S of the workload (smaller profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
