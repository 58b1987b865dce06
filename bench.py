#!/usr/bin/env python
"""Benchmark of the slot-indexed recurrent-state layer step on one GB300 (or N replicas).

Headline (one JSON line on stdout): KDA decode over a Kimi-K3 TP8-shard pool -- 69
layers, H=12 heads, K=V=128, bf16 state and io, 320 usable slots, 64 requests with
distinct random slots, one token per request per step.  A step runs all 69 layer
launches (replayed from a CUDA graph) through kda_decode_step_overlap, each layer's decode
a programmatic dependent of the previous layer's (its state reads overlap that layer's
tail; the plain kda_decode_step is timed beside it as the decode_plain leg); value =
decode tokens/s per layer = batch * layers / step time.  The per-step state working set (64 x 69 x 786 KB moved)
is ~14x the 129 MB L2, so no flush is needed between steps.

Legs reported in the same line (each timed separately with CUDA events):
  gdn_decode   GDN decode, H=32, K=V=128, fp32 state, 48 layers, 1024-slot pool,
               batch 1/16/64/256
  prefill      one KDA layer, 13600 tokens in chunked-prefill calls of 6144/6144/1312,
               a slot snapshot (ssm_slot_copy) after each call; bf16 state (tensor cores),
               then fp32 state (blocked closed form) on the same prompt and on 64 packed
               212-token sequences; the two forms' outputs and final states on the prompt
               are compared (cross_check)
  slot_copy    64 (src, dst) pairs of the 69-layer decode pool, all layers, one launch
  spec         verify of 8 tokens (anchor + 7 drafts) for 64 requests into a 16-deep
               cache, then commit of a seeded accept count per request
The oracle (plain fp64 C) is timed on a bounded sample, on one and on all host cores, as
cpu_baseline.

--impl reference times the oracle itself on the same workload (rank 0 only).
Multi-GPU: replicas only (the layer step has no exchange between requests or heads);
under torchrun every rank runs the full workload on its own GPU.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE_METRIC = "decode tokens/s per layer and achieved HBM GB/s (% of peak); prefill tok/s"

# DRAM bytes (read + write) per launch of the headline decode kernel in a one-pass ncu capture
# of the same launch shape (64 requests, 12 heads, second of two captured launches' first),
# keyed by a hash of the kernel's source files: reported only while the kernel is the one
# that was captured.
DECODE_SOURCES = ("decode.cu", "rsc_step.cuh", "rsc_common.cuh")
# Layers per host<->device copy in the end-to-end step (fewer, larger copies against a finer
# overlap of copies and compute).
E2E_GROUP = 16


def e2e_bounds(layers: int, mid: int = E2E_GROUP) -> list:
    """Group boundaries of the end-to-end step: small groups first (nothing hides the first
    input copy), then `mid`-layer groups, then a short and a 2-layer group (nothing hides the
    last output copy).  69 layers: [0, 2, 6, 14, 30, 46, 62, 67, 69]."""
    b = [0]
    for s in (2, 4, 8):
        if b[-1] + s < layers - 7:
            b.append(b[-1] + s)
    while b[-1] + mid <= layers - 7:
        b.append(b[-1] + mid)
    if b[-1] < layers - 2:
        b.append(layers - 2)
    b.append(layers)
    return b
CAPTURED_DECODE_TRAFFIC = {"3f787822c76e207d": 28_088_320}


# --------------------------------------------------------------------------- plumbing

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--legs", default="all", help="comma list of gdn,prefill,copy,spec,replay,gated,track or all/none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=2.0,
                    help="wall seconds of each oracle baseline run (six runs)")
    ap.add_argument("--layers", type=int, default=69,
                    help="layers of the headline decode pool (69 = the Kimi-K3 shard; fewer "
                         "only for small profiling captures)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device=None) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while a region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); smax.append(float(f[2])); power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def timed(fn, steps, warmup, stream, dist=None):
    """Run fn warmup times, then time exactly `steps` calls with CUDA events on `stream`,
    bracketed by barrier + synchronize.  Returns milliseconds per step."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / steps


def graph_of(fn, stream):
    """Capture fn (a sequence of library launches on `stream`) into a CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm: loads every kernel module before capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def decode_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "recurrent_state_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- roofline arithmetic

def decode_bytes_per_launch(B, H, K, V, state_bytes, io_bytes, per_channel_gate=True):
    """Algorithmic bytes of one decode launch: per request the state read + written, the
    window read + written, qkv, g, beta, out and its slot id; plus the layer's conv taps."""
    D = H * (2 * K + V)
    gw = K if per_channel_gate else 1
    per_req = (2 * H * V * K * state_bytes + 2 * 3 * D * io_bytes + D * io_bytes + H * gw * 4
               + H * 4 + H * V * io_bytes + 4)
    return B * per_req + D * 4 * 4


def prefill_flops(T, H, K, V, C=64):
    """Algorithmic tensor flops of a chunked prefill of T tokens: per token and head
    6CK + 4CV + 6KV (A, P, W; U', P U'; W S^T, Q S^T, U^T K)."""
    return T * H * (6 * C * K + 4 * C * V + 6 * K * V)


def spec_verify_bytes(B, T, H, K, V, state_bytes=2, io_bytes=2):
    """Algorithmic bytes of a snapshot verify: per request the slot state read and T states
    written, the window read and T window entries written, and per token qkv, g, beta, out;
    plus the slot id."""
    D = H * (2 * K + V)
    S, Wb = H * V * K * state_bytes, 3 * D * io_bytes
    return B * (S + T * S + Wb + T * Wb + T * D * io_bytes + T * H * K * 4 + T * H * 4
                + T * H * V * io_bytes + 4)


# --------------------------------------------------------------------------- workloads

def _softplus_neg(t):
    import torch
    return -torch.nn.functional.softplus(t)


class DecodeWorkload:
    """Per-layer inputs of one decode step, resident on the device; seeded."""

    def __init__(self, dev, layers, P, B, H, K, V, st, io, gate, seed=0):
        import torch
        import recurrent_state_cache_gb300 as rsc
        from recurrent_state_cache_gb300 import inputs
        self.rsc = rsc
        self.layers, self.P, self.B, self.H, self.K, self.V = layers, P, B, H, K, V
        self.st, self.io, self.gate = st, io, gate
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        sdt, idt = rsc.binding.TORCH_DTYPE[st], rsc.binding.TORCH_DTYPE[io]
        D = H * (2 * K + V)
        self.D = D
        ssm = torch.empty((layers, P + 1, H, V, K), dtype=sdt, device=dev).normal_(0, 0.1, generator=gen)
        conv = torch.empty((layers, P + 1, 3, D), dtype=idt, device=dev).normal_(0, 0.1, generator=gen)
        self.pool = rsc.SlotPool(layers, P, H, K, V, st, io, gate, dev, ssm=ssm, conv=conv)
        r = inputs.rng(seed)
        self.slots = torch.from_numpy(inputs.distinct_slots(r, B, P)).to(dev)
        gshape = (layers, B, H, K) if gate == rsc.KDA else (layers, B, H)
        self.qkv = torch.empty((layers, B, D), dtype=idt, device=dev).normal_(0, 1, generator=gen)
        self.g = _softplus_neg(torch.empty(gshape, device=dev).normal_(0, 1, generator=gen))
        self.beta = torch.sigmoid(torch.empty((layers, B, H), device=dev).normal_(0, 1, generator=gen))
        self.w = torch.empty((layers, D, 4), device=dev).normal_(0, 0.5, generator=gen)
        self.out = torch.empty((layers, B, H, V), dtype=idt, device=dev)
        # consecutive calls are different layers, so the overlapped launch's precondition holds
        self.overlap = True

    def step(self):
        rsc = self.rsc
        for l in range(self.layers):
            rsc.kda_decode_step(self.pool, l, self.slots, self.qkv[l], self.w[l], self.g[l],
                                self.beta[l], self.out[l], overlap=self.overlap)

    def bytes_per_launch(self):
        """Algorithmic bytes of one layer launch (decode_bytes_per_launch)."""
        return decode_bytes_per_launch(self.B, self.H, self.K, self.V,
                                       4 if self.st == 0 else 2, 4 if self.io == 0 else 2,
                                       self.gate == 0)


# --------------------------------------------------------------------------- legs

def leg_gdn(dev, peaks, stream, batches=(1, 16, 64, 256)):
    import torch
    from recurrent_state_cache_gb300 import binding as b
    res = {"config": "GDN decode, H=32, K=V=128, fp32 state, bf16 io, 48 layers, 1024 slots"}
    wl = DecodeWorkload(dev, 48, 1024, max(batches), 32, 128, 128, b.F32, b.BF16, b.GDN, seed=1)
    full_slots = wl.slots
    rows = []
    for B in batches:
        wl.B = B
        wl.slots = full_slots[:B].contiguous()
        sub = (wl.qkv, wl.g, wl.beta, wl.out)
        wl.qkv, wl.g, wl.beta, wl.out = (x[:, :B].contiguous() for x in sub)
        graph = graph_of(wl.step, stream)
        ms = timed(graph.replay, 20, 3, stream)
        wl.qkv, wl.g, wl.beta, wl.out = sub
        per_launch = ms / wl.layers
        gbs = wl.bytes_per_launch() / (per_launch * 1e-3) / 1e9
        rows.append({"batch": B, "us_per_layer": round(per_launch * 1e3, 3),
                     "tokens_per_s_per_layer": round(B / (per_launch * 1e-3), 1),
                     "hbm_gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)})
    res["sweep"] = rows
    del wl
    torch.cuda.empty_cache()
    return res


PROMPT_CHUNKS = (6144, 6144, 1312)


def _prompt_run(dev, stream, st, seed):
    """ms per 13600-token prompt: three kda_prefill_chunk calls of 6144/6144/1312 tokens chained
    through one slot of a 1-layer pool (H=12, K=V=128, bf16 inputs, state dtype st), a slot
    snapshot after each; captured once in a CUDA graph and replayed.  Also returns the outputs
    and the slot's final state (every replay starts the prompt from a fresh state, so they are
    the prompt's)."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    from recurrent_state_cache_gb300 import binding as b
    H, K, V = 12, 128, 128
    chunks = PROMPT_CHUNKS
    T = sum(chunks)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    D = H * (2 * K + V)
    pool = rsc.SlotPool(1, 8, H, K, V, st, b.BF16, b.KDA, dev)
    qkv = torch.empty((T, D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=gen)
    g = -torch.nn.functional.softplus(torch.empty((T, H, K), device=dev).normal_(0, 1, generator=gen))
    beta = torch.sigmoid(torch.empty((T, H), device=dev).normal_(0, 1, generator=gen))
    w = torch.empty((D, 4), device=dev).normal_(0, 0.5, generator=gen)
    out = torch.empty((T, H, V), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(rsc.kda_prefill_workspace_size(pool, 1, max(chunks)), dtype=torch.uint8, device=dev)
    slot = torch.tensor([1], dtype=torch.int32, device=dev)
    snaps = [torch.tensor([s], dtype=torch.int32, device=dev) for s in (2, 3, 4)]
    fresh = torch.tensor([0], dtype=torch.uint8, device=dev)
    cus = [torch.tensor([0, c], dtype=torch.int32, device=dev) for c in chunks]
    offs = np.cumsum((0,) + chunks)

    def run():
        for i, c in enumerate(chunks):
            a, e = int(offs[i]), int(offs[i + 1])
            rsc.kda_prefill_chunk(pool, 0, slot, cus[i], qkv[a:e], w, g[a:e], beta[a:e],
                                  has_initial_state=fresh if i == 0 else None, out=out[a:e],
                                  workspace=ws)
            rsc.ssm_slot_copy(pool, 0, slot, snaps[i])

    ms = timed(graph_of(run, stream).replay, 5, 2, stream)
    assert rsc.rsc_get_device_error(pool) == 0
    return ms, out, pool.ssm[0, 1]


def _max_rel_err(got, ref) -> float:
    got, ref = got.float(), ref.float()
    return float((got - ref).abs().max() / ref.abs().max().clamp_min(1e-30))


def leg_prefill(dev, peaks, stream):
    from recurrent_state_cache_gb300 import binding as b
    H, K, V = 12, 128, 128
    T = sum(PROMPT_CHUNKS)
    D = H * (2 * K + V)
    ms, out_tc, state_tc = _prompt_run(dev, stream, b.BF16, 2)
    flops = prefill_flops(T, H, K, V)
    io_bytes = T * D * 2 + T * H * K * 4 + T * H * 4 + T * H * V * 2
    res = {"config": "1 KDA layer, H=12, K=V=128, bf16, 13600 tokens as 6144/6144/1312, snapshot copy after each",
           "ms_per_prefill": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1),
           "algorithmic_tflops": round(flops / (ms * 1e-3) / 1e12, 3),
           "tensor_frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 5),
           "io_gbs": round(io_bytes / (ms * 1e-3) / 1e9, 1),
           "hbm_frac": round(io_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "path": "chunkwise, tcgen05 tensor cores"}
    res["f32_state"], out_f32, state_f32 = leg_prefill_f32(dev, stream)
    # The two forms on the same prompt (same seed): the tensor-core form's bf16 operands
    # against the fp32 closed form, at the bf16 bar (max |difference| / max |fp32 value|).
    res["cross_check"] = {
        "what": "bf16-state tensor-core prefill against the fp32-state blocked prefill on the same "
                "13600-token prompt: every output, and the final state",
        "out_max_rel_err": round(_max_rel_err(out_tc, out_f32), 5),
        "state_max_rel_err": round(_max_rel_err(state_tc, state_f32), 5),
        "bar": 0.02}
    return res


def leg_prefill_f32(dev, stream, nseq=64, seqlen=212):
    """The fp32-state prefill (the recurrence eight tokens at a time in closed form, fp32 on the
    CUDA cores) at the same head shape (H=12, K=V=128, bf16 inputs): the bf16 leg's 13600-token
    prompt (same inputs), and a batch of 64 packed 212-token sequences from fresh slots.
    Returns the leg's figures, and the prompt's outputs and final state."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    from recurrent_state_cache_gb300 import binding as b
    T = sum(PROMPT_CHUNKS)
    ms_prompt, out_prompt, state_prompt = _prompt_run(dev, stream, b.F32, 2)
    H, K, V = 12, 128, 128
    Tb = nseq * seqlen
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    D = H * (2 * K + V)
    pool = rsc.SlotPool(1, nseq + 1, H, K, V, b.F32, b.BF16, b.KDA, dev)
    qkv = torch.empty((Tb, D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=gen)
    g = -torch.nn.functional.softplus(torch.empty((Tb, H, K), device=dev).normal_(0, 1, generator=gen))
    beta = torch.sigmoid(torch.empty((Tb, H), device=dev).normal_(0, 1, generator=gen))
    w = torch.empty((D, 4), device=dev).normal_(0, 0.5, generator=gen)
    out = torch.empty((Tb, H, V), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(rsc.kda_prefill_workspace_size(pool, nseq, Tb), dtype=torch.uint8, device=dev)
    slots = torch.arange(1, nseq + 1, dtype=torch.int32, device=dev)
    fresh = torch.zeros(nseq, dtype=torch.uint8, device=dev)
    cu = torch.arange(0, Tb + 1, seqlen, dtype=torch.int32, device=dev)
    run = lambda: rsc.kda_prefill_chunk(pool, 0, slots, cu, qkv, w, g, beta,
                                        has_initial_state=fresh, out=out, workspace=ws)
    ms_batch = timed(graph_of(run, stream).replay, 5, 2, stream)
    assert rsc.rsc_get_device_error(pool) == 0
    leg = {"config": f"1 KDA layer, H=12, K=V=128, fp32 state, bf16 io: the {T}-token prompt as "
                      f"6144/6144/1312 with snapshots; {nseq} packed {seqlen}-token sequences",
            "ms_per_prefill": round(ms_prompt, 4), "tokens_per_s": round(T / (ms_prompt * 1e-3), 1),
            "us_per_token": round(ms_prompt * 1e3 / T, 4),
            "batch_ms": round(ms_batch, 4), "batch_tokens_per_s": round(Tb / (ms_batch * 1e-3), 1),
            "path": "8-token blocks in closed form (per-block conv/norm/operand kernel, blocked "
                    "recurrence, window kernel)"}
    return leg, out_prompt, state_prompt


def leg_copy(dev, peaks, stream, wl):
    import torch
    import recurrent_state_cache_gb300 as rsc
    from recurrent_state_cache_gb300 import inputs
    r = inputs.rng(3)
    perm = r.permutation(wl.P) + 1
    src = torch.from_numpy(perm[:64].astype(np.int32)).to(dev)
    dst = torch.from_numpy(perm[64:128].astype(np.int32)).to(dev)
    fn = lambda: rsc.ssm_slot_copy(wl.pool, -1, src, dst)
    ms = timed(fn, 10, 3, stream)
    ss, io = 2, 2
    row = wl.H * wl.V * wl.K * ss + 3 * wl.D * io
    nbytes = 2 * row * wl.layers * 64
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"config": "64 pairs x 69 layers of the decode pool, one launch",
            "ms": round(ms, 4), "bytes": nbytes, "hbm_gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4)}


SPEC_ROTATIONS = 8  # distinct (layer, cache, accept) sets cycled through by the spec legs


def _spec_inputs(dev, seed, R, B, T, H, K, V):
    """Inputs of R verify calls of the speculative workload (one set per rotation)."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    D = H * (2 * K + V)
    qkv = torch.empty((R, B, T, D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=gen)
    g = -torch.nn.functional.softplus(torch.empty((R, B, T, H, K), device=dev).normal_(0, 1, generator=gen))
    beta = torch.sigmoid(torch.empty((R, B, T, H), device=dev).normal_(0, 1, generator=gen))
    w = torch.empty((D, 4), device=dev).normal_(0, 0.5, generator=gen)
    return gen, qkv, g, beta, w


def leg_spec(dev, peaks, stream):
    """Snapshot-form verify and commit on the speculative workload (B=64, T=8, cache depth
    16).  Each timed graph cycles through SPEC_ROTATIONS calls on distinct pool layers, spec
    caches and accept vectors, so a call's rows were last touched seven calls (>= 370 MB of
    other traffic) earlier and are read from HBM, not from L2."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    from recurrent_state_cache_gb300 import binding as b, inputs
    H, K, V, B, T, L, P, R = 12, 128, 128, 64, 8, 16, 320, SPEC_ROTATIONS
    D = H * (2 * K + V)
    gen, qkv, g, beta, w = _spec_inputs(dev, 4, R, B, T, H, K, V)
    ssm = torch.empty((R, P + 1, H, V, K), dtype=torch.bfloat16, device=dev).normal_(0, 0.1, generator=gen)
    conv = torch.empty((R, P + 1, 3, D), dtype=torch.bfloat16, device=dev).normal_(0, 0.1, generator=gen)
    pool = rsc.SlotPool(R, P, H, K, V, b.BF16, b.BF16, b.KDA, dev, ssm=ssm, conv=conv)
    r = inputs.rng(4)
    slots = [torch.from_numpy(inputs.distinct_slots(r, B, P)).to(dev) for _ in range(R)]
    accept_np = [inputs.accept_counts(r, B, T) for _ in range(R)]
    accept = [torch.from_numpy(a).to(dev) for a in accept_np]
    out = torch.empty((R, B, T, H, V), dtype=torch.bfloat16, device=dev)
    spec_ssm = [torch.empty((B, L, H, V, K), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    spec_conv = [torch.empty((B, L, 3, D), dtype=torch.bfloat16, device=dev) for _ in range(R)]

    def verify():
        for i in range(R):
            rsc.kda_spec_verify_commit(pool, i, rsc.VERIFY, slots[i], T, L, spec_ssm[i],
                                       spec_conv[i], qkv[i], w, g[i], beta[i], out[i])

    def commit():
        for i in range(R):
            rsc.kda_spec_verify_commit(pool, i, rsc.COMMIT, slots[i], T, L, spec_ssm[i],
                                       spec_conv[i], accept=accept[i])
    ms_v = timed(graph_of(verify, stream).replay, 20, 3, stream) / R
    ms_c = timed(graph_of(commit, stream).replay, 20, 3, stream) / R
    S, Wb = H * V * K * 2, 3 * D * 2
    vb = spec_verify_bytes(B, T, H, K, V)
    cb = B * 2 * (S + Wb)
    vw = B * (T * S + T * Wb + T * H * V * 2)  # bytes written by verify
    return {"config": "KDA H=12 K=V=128 bf16, batch 64, T=8 (anchor+7 drafts), cache depth 16; "
                      f"graphs of {R} calls on distinct layers, caches and accept vectors",
            "verify_ms": round(ms_v, 4), "verify_gbs": round(vb / (ms_v * 1e-3) / 1e9, 1),
            "verify_frac": round(vb / (ms_v * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "verify_write_gbs": round(vw / (ms_v * 1e-3) / 1e9, 1),
            "commit_ms": round(ms_c, 4), "commit_gbs": round(cb / (ms_c * 1e-3) / 1e9, 1),
            "commit_frac": round(cb / (ms_c * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}


def leg_gated(dev, peaks, stream, wl):
    """The headline decode step with the gates formed in the kernel from raw projections
    (a [B][H][K], b [B][H], per-head A_log and per-channel dt_bias) instead of given g, beta:
    the same 69-layer graph, the raw projections in place of g and beta."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    gen = torch.Generator(device=dev)
    gen.manual_seed(6)
    H, K = wl.H, wl.K
    A_log = torch.empty((wl.layers, H), device=dev).normal_(0, 0.5, generator=gen)
    dt = torch.empty((wl.layers, H, K), device=dev).normal_(0, 1, generator=gen)

    def step(overlap):
        for l in range(wl.layers):
            rsc.kda_decode_step_ex(wl.pool, l, wl.slots, wl.qkv[l], wl.w[l], wl.g[l], wl.beta[l],
                                   out=wl.out[l], A_log=A_log[l], dt_bias=dt[l], overlap=overlap)
    ms = timed(graph_of(lambda: step(True), stream).replay, 50, 5, stream)
    ms_plain = timed(graph_of(lambda: step(False), stream).replay, 50, 5, stream)
    tok = wl.B / (ms * 1e-3 / wl.layers)
    bytes_layer = wl.bytes_per_launch() + H * 4 + H * K * 4
    gbs = bytes_layer * wl.layers / (ms * 1e-3) / 1e9
    return {"config": "headline decode workload, gates from raw projections in the kernel "
                      "(kda_decode_step_ex, overlapped launch)",
            "ms_per_step": round(ms, 4), "tokens_per_s_per_layer": round(tok, 1),
            "hbm_gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
            "plain_launch_ms_per_step": round(ms_plain, 4)}


def leg_track(dev, peaks, stream, wl):
    """The headline decode step with every request tracked (the worst case of the pages'
    mamba_track_interval copy): the track copy fused into decode against decode followed by
    the masked slot copy of each layer."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    used = set(wl.slots.cpu().tolist())
    free = [s for s in range(1, wl.P + 1) if s not in used][:wl.B]
    track = torch.tensor(free, dtype=torch.int32, device=dev)
    mask = torch.ones(wl.B, dtype=torch.uint8, device=dev)

    def fused(overlap=True):
        for l in range(wl.layers):
            rsc.kda_decode_step_ex(wl.pool, l, wl.slots, wl.qkv[l], wl.w[l], wl.g[l], wl.beta[l],
                                   out=wl.out[l], track_mask=mask, track_slots=track,
                                   overlap=overlap)

    def separate():
        for l in range(wl.layers):
            rsc.kda_decode_step(wl.pool, l, wl.slots, wl.qkv[l], wl.w[l], wl.g[l], wl.beta[l],
                                wl.out[l], overlap=True)
            rsc.ssm_slot_copy(wl.pool, l, wl.slots, track, mask)
    ms_f = timed(graph_of(fused, stream).replay, 30, 5, stream)
    ms_fp = timed(graph_of(lambda: fused(False), stream).replay, 30, 5, stream)
    ms_s = timed(graph_of(separate, stream).replay, 30, 5, stream)
    row = wl.H * wl.V * wl.K * 2 + 3 * wl.D * 2          # one slot row of a layer (bf16)
    bytes_f = (wl.bytes_per_launch() + wl.B * row) * wl.layers  # the track rows written once more
    return {"config": "headline decode workload, all 64 requests tracked every step "
                      "(kda_decode_step_ex, overlapped launch; separate = overlapped decode then "
                      "ssm_slot_copy per layer)",
            "fused_ms_per_step": round(ms_f, 4), "separate_ms_per_step": round(ms_s, 4),
            "fused_plain_launch_ms_per_step": round(ms_fp, 4),
            "fused_tokens_per_s_per_layer": round(wl.B / (ms_f * 1e-3 / wl.layers), 1),
            "fused_hbm_gbs": round(bytes_f / (ms_f * 1e-3) / 1e9, 1),
            "fused_frac": round(bytes_f / (ms_f * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}


def leg_replay(dev, peaks, stream):
    """ReplaySSM verify / commit on the speculative workload of leg_spec: verify writes ring
    records (d, k, rawv, rawk, g, beta) instead of 8 states per request; commit replays the
    accepted tokens from the slot state.  Timed like leg_spec: graphs cycling through
    SPEC_ROTATIONS distinct layers (each with its own rings), slot sets and accept vectors."""
    import torch
    import recurrent_state_cache_gb300 as rsc
    from recurrent_state_cache_gb300 import binding as b, inputs
    H, K, V, B, T, L, P, R = 12, 128, 128, 64, 8, 16, 320, SPEC_ROTATIONS
    D = H * (2 * K + V)
    gen, qkv, g, beta, w = _spec_inputs(dev, 5, R, B, T, H, K, V)
    ssm = torch.empty((R, P + 1, H, V, K), dtype=torch.bfloat16, device=dev).normal_(0, 0.1, generator=gen)
    conv = torch.empty((R, P + 1, 3, D), dtype=torch.bfloat16, device=dev).normal_(0, 0.1, generator=gen)
    pool = rsc.SlotPool(R, P, H, K, V, b.BF16, b.BF16, b.KDA, dev, ssm=ssm, conv=conv)
    rings = rsc.ReplayRings(pool, L)
    r = inputs.rng(4)
    slots = [torch.from_numpy(inputs.distinct_slots(r, B, P)).to(dev) for _ in range(R)]
    accept_np = [inputs.accept_counts(r, B, T) for _ in range(R)]
    accept = [torch.from_numpy(a).to(dev) for a in accept_np]
    r5 = inputs.rng(5)
    pos = [torch.from_numpy(r5.integers(0, L, B).astype("int32")).to(dev) for _ in range(R)]
    out = torch.empty((R, B, T, H, V), dtype=torch.bfloat16, device=dev)
    spec_conv = [torch.empty((B, L, 3, D), dtype=torch.bfloat16, device=dev) for _ in range(R)]

    def verify():
        for i in range(R):
            rsc.kda_replay_verify_commit(pool, rings, i, rsc.VERIFY, slots[i], pos[i], T,
                                         spec_conv[i], qkv[i], w, g[i], beta[i], out[i])

    def commit():
        for i in range(R):
            rsc.kda_replay_verify_commit(pool, rings, i, rsc.COMMIT, slots[i], pos[i], T,
                                         spec_conv[i], accept=accept[i])
    ms_v = timed(graph_of(verify, stream).replay, 20, 3, stream) / R
    ms_c = timed(graph_of(commit, stream).replay, 20, 3, stream) / R
    S, Wb = H * V * K * 2, 3 * D * 2
    rec = H * (2 * V * 2 + 2 * K * 2 + K * 4 + 4)   # one token's records over the heads
    rep_ = H * (V * 2 + K * 2 + K * 4 + 4)          # what commit reads of one token's records
    vb = B * (S + T * rec + Wb + T * Wb + T * D * 2 + T * H * K * 4 + T * H * 4 + T * H * V * 2 + 8)
    acc_tokens = sum(int(a.astype("int64").sum()) + B for a in accept_np) / R
    cb = int(2 * B * S + 2 * B * Wb + acc_tokens * rep_ + 12 * B)
    return {"config": "KDA H=12 K=V=128 bf16, batch 64, T=8 (anchor+7 drafts), ring depth 16; "
                      f"graphs of {R} calls on distinct layers, slot sets and accept vectors",
            "verify_ms": round(ms_v, 4), "verify_bytes": vb,
            "verify_gbs": round(vb / (ms_v * 1e-3) / 1e9, 1),
            "verify_frac": round(vb / (ms_v * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "commit_ms": round(ms_c, 4), "commit_bytes": cb,
            "commit_gbs": round(cb / (ms_c * 1e-3) / 1e9, 1),
            "commit_frac": round(cb / (ms_c * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}


# --------------------------------------------------------------------------- oracle timing

class OracleWork:
    """One unit of oracle work on synthetic inputs built once, outside any timing.
    kind "kda_decode": a layer-step of `part` requests of the headline workload (H=12,
      K=V=128, bf16 state and io, per-channel gate);
    kind "gdn_decode": a layer-step of `part` requests of the GDN workload (H=32, K=V=128, fp32
      state, bf16 io, per-head gate);
    kind "prefill": a recurrent prefill call of `tokens` tokens over `part` heads of the
      chunked-prefill workload (K=V=128, bf16), continuing from the slot.
    units() = tokens processed per step (requests for decode, tokens for prefill; a prefill
    over a share of the heads counts its tokens divided by the share)."""

    SHAPES = {"kda_decode": (12, 0, 0, 1, 1), "gdn_decode": (32, 1, 1, 0, 1),
              "prefill": (12, 0, 0, 1, 1)}

    def __init__(self, kind, part, seed=0, tokens=2048):
        import oracle
        from recurrent_state_cache_gb300 import inputs
        self.oracle, self.kind, self.part = oracle, kind, part
        H_full, gate, _, st, io = self.SHAPES[kind]
        st = oracle.BF16 if st else oracle.F32
        io = oracle.BF16 if io else oracle.F32
        gate = oracle.GDN if gate else oracle.KDA
        K = V = 128
        r = inputs.rng(seed)
        if kind == "prefill":
            H, B, self.T = part, 1, tokens
            self.share = part / H_full
        else:
            H, B = H_full, part
            self.share = 1.0
        ssm, conv = inputs.pool_arrays(r, 1, B, H, K, V, st, io)
        self.pool = oracle.Pool(1, B, H, K, V, st, io, gate, ssm, conv)
        self.w = inputs.conv_weights(r, H, K, V)
        self.slots = inputs.distinct_slots(r, B, B)
        lead = (self.T,) if kind == "prefill" else (B,)
        self.x = inputs.projections(r, lead, H, K, V, io)
        self.g, self.beta = inputs.gates(r, lead, H, K, gate)
        self.cu = np.int32([0, self.T]) if kind == "prefill" else None

    def step(self):
        if self.kind == "prefill":
            self.oracle.prefill(self.pool, 0, self.slots, self.cu, self.x, self.w, self.g, self.beta)
        else:
            self.oracle.decode_step(self.pool, 0, self.slots, self.x, self.w, self.g, self.beta)

    def units(self):
        return self.T * self.share if self.kind == "prefill" else self.part


def _oracle_worker(kind, part, seed, tokens, steps, barrier, q):
    w = OracleWork(kind, part, seed, tokens)
    w.step()  # warm
    barrier.wait()
    t0 = time.time()
    for _ in range(steps):
        w.step()
    q.put((t0, time.time(), w.units() * steps))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _split(n, parts):
    """n work items over at most `parts` workers, as even as possible (no empty share)."""
    parts = max(1, min(parts, n))
    return [n // parts + (1 if i < n % parts else 0) for i in range(parts)]


def oracle_rate(kind, total, seconds, cores=1, seed=0, tokens=2048, steps=None):
    """Oracle throughput (tokens/s) on `kind` over `total` requests (decode) or heads
    (prefill), single-threaded (cores = 1) or split over `cores` worker processes (spawned,
    each with its own share and inputs) that start together; the steps are sized to about
    `seconds` of wall time unless given.  Returns (tokens/s, workers used, steps, wall s)."""
    one = OracleWork(kind, total if cores == 1 else _split(total, cores)[0], seed, tokens)
    t0 = time.perf_counter()
    one.step()
    t_step = time.perf_counter() - t0
    if steps is None:
        steps = max(1, int(seconds / max(t_step, 1e-6)))
    if cores == 1:
        t0 = time.perf_counter()
        for _ in range(steps):
            one.step()
        el = time.perf_counter() - t0
        return one.units() * steps / el, 1, steps, el
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    shares = _split(total, cores)
    barrier = ctx.Barrier(len(shares))
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(kind, n, seed + i, tokens, steps, barrier, q))
             for i, n in enumerate(shares)]
    for p in procs:
        p.start()
    import queue
    res = []
    limit = time.time() + 120 + 20 * max(seconds, t_step * steps)
    try:
        while len(res) < len(procs):
            try:
                res.append(q.get(timeout=1.0))
            except queue.Empty:
                if any(p.exitcode not in (None, 0) for p in procs) or time.time() > limit:
                    raise RuntimeError("an oracle worker process failed or did not finish")
    finally:
        for p in procs:
            p.join(timeout=5)
            if p.is_alive():
                p.kill()
    start = min(r[0] for r in res)
    end = max(r[1] for r in res)
    units = sum(r[2] for r in res)
    return units / (end - start), len(shares), steps, end - start


def oracle_baselines(seconds: float):
    """The oracle on the machine's host cores, single-threaded and on all cores, for the three
    workloads: KDA decode (64 requests), GDN decode (16 requests, one layer), chunked-prefill
    workload in recurrent form (a 2048-token sample of the 13600-token prompt, 12 heads)."""
    cores = host_cores()
    out = {}
    for name, kind, total in (("kda_decode_b64", "kda_decode", 64),
                              ("gdn_decode_b16", "gdn_decode", 16),
                              ("prefill_13600_sample2048", "prefill", 12)):
        r1, _, n1, e1 = oracle_rate(kind, total, seconds, 1)
        rn, used, nn, en = oracle_rate(kind, total, seconds, cores)
        out[name] = {"single_core": round(r1, 3), "all_cores": round(rn, 3), "cores": used,
                     "unit": "tokens/s per layer",
                     "steps": [n1, nn], "seconds": [round(e1, 2), round(en, 2)]}
    return cores, out


# --------------------------------------------------------------------------- main

def run_reference(args):
    """The reference arm: the oracle itself on the host cores, on the headline workload.  A
    step is one layer-step of the 64 requests, split by request over worker processes on all
    host cores (the oracle's code as it stands, each worker with its share of the requests)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    total_t0 = time.perf_counter()
    cores = host_cores()
    rate, used, steps, wall = oracle_rate("kda_decode", 64, 0.0, cores, steps=args.steps)
    ms = 1e3 * wall / steps
    value = rate
    line = {"metric": HEADLINE_METRIC, "value": round(value, 3), "unit": "tokens/s per layer",
            "impl": "reference", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "kda_decode_kimi_k3_tp8_shard", "layers_per_step": 1,
                       "batch": 64, "H": 12, "K": 128, "V": 128, "state_dtype": "bf16"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s per layer", "cores": used,
                             "kind": "oracle",
                             "sample": f"each step: one layer-step of the 64 requests of the headline "
                                       f"workload, split by request over {used} worker processes "
                                       f"({cores} host cores); each worker warmed by one step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s per layer",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - total_t0, 1)}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    from recurrent_state_cache_gb300 import _build, binding as b
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    # ---- headline: Kimi-K3 shard KDA decode, 69 layers, batch 64
    wl = DecodeWorkload(dev, args.layers, 320, 64, 12, 128, 128, b.BF16, b.BF16, b.KDA, seed=0)
    graph = graph_of(wl.step, stream)
    with ClockSampler(local) as clk:
        ms = timed(graph.replay, args.steps, args.warmup, stream, dist)
    ms_max = max_over_ranks(ms, dist, dev)
    units = wl.B * wl.layers
    value = sum_over_ranks(units, dist, dev) / (ms_max * 1e-3)
    per_launch_s = ms * 1e-3 / wl.layers
    bpl = wl.bytes_per_launch()
    achieved = bpl / per_launch_s / 1e9

    # ---- e2e through the public API with pinned host buffers
    # a layer's inputs packed as [qkv | g | beta] in one row, on the host and on the device,
    # so that a group of layers moves in one copy
    QB = wl.B * wl.D * wl.qkv.element_size()
    GB = wl.g[0].numel() * 4
    BB = wl.beta[0].numel() * 4
    dpack = torch.empty((wl.layers, QB + GB + BB), dtype=torch.uint8, device=dev)
    p_qkv = [dpack[l, :QB].view(wl.qkv.dtype).view(wl.qkv[l].shape) for l in range(wl.layers)]
    p_g = [dpack[l, QB:QB + GB].view(torch.float32).view(wl.g[l].shape) for l in range(wl.layers)]
    p_beta = [dpack[l, QB + GB:].view(torch.float32).view(wl.beta[l].shape) for l in range(wl.layers)]
    for l in range(wl.layers):
        p_qkv[l].copy_(wl.qkv[l]); p_g[l].copy_(wl.g[l]); p_beta[l].copy_(wl.beta[l])
    h_pack = dpack.cpu().pin_memory()
    h_out = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()

    cin = torch.cuda.Stream(device=dev)   # host -> device input copies
    cout = torch.cuda.Stream(device=dev)  # device -> host output copies
    ev_in = [torch.cuda.Event() for _ in range(wl.layers)]
    ev_out = [torch.cuda.Event() for _ in range(wl.layers)]

    def e2e_step():
        # pipelined by groups of layers (e2e_bounds): a group's inputs arrive while the previous
        # group computes, and its outputs leave while the next one computes; every stream joins
        # back before the step ends
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        cin.wait_event(fork)
        cout.wait_event(fork)
        bounds = e2e_bounds(wl.layers)
        with torch.cuda.stream(cin):
            for i in range(len(bounds) - 1):
                a, z = bounds[i], bounds[i + 1]
                dpack[a:z].copy_(h_pack[a:z], non_blocking=True)
                ev_in[i].record(cin)
        for i in range(len(bounds) - 1):
            a, z = bounds[i], bounds[i + 1]
            cur.wait_event(ev_in[i])
            for l in range(a, z):
                wl.rsc.kda_decode_step(wl.pool, l, wl.slots, p_qkv[l], wl.w[l], p_g[l],
                                       p_beta[l], wl.out[l], overlap=True)
            ev_out[i].record(cur)
            cout.wait_event(ev_out[i])
            with torch.cuda.stream(cout):
                h_out[a:z].copy_(wl.out[a:z], non_blocking=True)
        join_in, join_out = torch.cuda.Event(), torch.cuda.Event()
        join_in.record(cin)
        join_out.record(cout)
        cur.wait_event(join_in)
        cur.wait_event(join_out)

    # The step as a serving engine runs it: captured once into a CUDA graph (the pinned
    # host->device input copies, the 69 public-API decode calls, the device->host copies of
    # the outputs, overlapped layer by layer on three streams) and replayed every step.
    e2e_graph = graph_of(e2e_step, stream)
    e2e_steps = max(10, min(args.steps, 200))
    ms_e2e = timed(e2e_graph.replay, e2e_steps, args.warmup, stream, dist)
    ms_e2e = max_over_ranks(ms_e2e, dist, dev)
    # The same step issued eagerly every time (69 binding calls through ctypes, their argument
    # checks and launches, plus the stream forks and copies), without a graph.
    ms_eager = timed(e2e_step, max(10, min(args.steps, 100)), args.warmup, stream, dist)
    ms_eager = max_over_ranks(ms_eager, dist, dev)
    h2d = h_pack.numel()
    d2h = h_out.numel() * h_out.element_size()

    legs = {}
    # the plain launch (kda_decode_step) of the same workload
    wl.overlap = False
    ms_plain = timed(graph_of(wl.step, stream).replay, max(10, min(args.steps, 300)),
                     args.warmup, stream)
    wl.overlap = True
    gbs_plain = bpl / (ms_plain * 1e-3 / wl.layers) / 1e9
    legs["decode_plain"] = {"config": "the headline workload through kda_decode_step (no overlap)",
                            "us_per_layer": round(ms_plain * 1e3 / wl.layers, 3),
                            "tokens_per_s_per_layer": round(wl.B * wl.layers / (ms_plain * 1e-3), 1),
                            "hbm_gbs": round(gbs_plain, 1),
                            "frac": round(gbs_plain / peaks["hbm_gbs"], 4)}
    want = set(["gdn", "prefill", "copy", "spec", "replay", "gated", "track"] if args.legs == "all" else
               ([] if args.legs == "none" else args.legs.split(",")))
    if "copy" in want:
        legs["slot_copy"] = leg_copy(dev, peaks, stream, wl)
    del graph
    if "spec" in want:
        legs["spec"] = leg_spec(dev, peaks, stream)
    if "replay" in want:
        legs["replay_spec"] = leg_replay(dev, peaks, stream)
    if "gated" in want:
        legs["decode_gated"] = leg_gated(dev, peaks, stream, wl)
    if "track" in want:
        legs["decode_track"] = leg_track(dev, peaks, stream, wl)
    if "prefill" in want:
        legs["prefill"] = leg_prefill(dev, peaks, stream)
    del wl
    torch.cuda.empty_cache()
    if "gdn" in want:
        legs["gdn_decode"] = leg_gdn(dev, peaks, stream)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cores, wls = oracle_baselines(args.cpu_seconds)
        head = wls["kda_decode_b64"]
        cpu = {"value": head["all_cores"], "unit": "tokens/s per layer", "cores": head["cores"],
               "kind": "oracle",
               "sample": f"layer-steps of the headline workload (64 requests, H=12, K=V=128, bf16) "
                         f"split by request over {head['cores']} worker processes of the {cores} "
                         f"host cores; about {args.cpu_seconds:g} s per run; single-threaded "
                         f"{head['single_core']} tokens/s",
               "single_core": head["single_core"], "host_cores": cores, "workloads": wls}

    clocks = clk.summary()
    line = {
        "metric": HEADLINE_METRIC, "value": round(value, 1), "unit": "tokens/s per layer",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "kda_decode_kimi_k3_tp8_shard" + ("" if args.layers == 69 else
                                                                  f"_layers{args.layers}"),
                   "layers": args.layers, "batch": 64,
                   "pool_slots": 320, "H": 12, "K": 128, "V": 128, "state_dtype": "bf16",
                   "io_dtype": "bf16", "tokens_per_request_per_step": 1,
                   "l2": "inputs larger than L2: 1.74 GB of state moved per step, no flush",
                   "launch": f"{args.layers} kda_decode_step_overlap launches per step replayed from a CUDA graph",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": CAPTURED_DECODE_TRAFFIC.get(decode_source_hash()),
                     "traffic_note": "ncu dram read+write of one launch; the in-place state "
                                     "writes stay in L2 until later layers evict them",
                     "kernel": "kda_decode_kernel",
                     "bytes_per_launch": bpl, "peak_source": peaks["source"]},
        "e2e": {"value": round(sum_over_ranks(units, dist, dev) / (ms_e2e * 1e-3), 1),
                "unit": "tokens/s per layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "per step: pinned host->device copies of every layer's qkv, g, beta (packed per layer, one copy per group of layers: 2, 4, 8, then 16-layer groups, then 5 and 2), "
                       "the kda_decode_step_overlap calls, device->host copies of every layer's output, "
                       "overlapped layer by layer on a copy-in, a compute and a copy-out stream; "
                       "captured once in a CUDA graph and replayed",
                "eager_value": round(sum_over_ranks(units, dist, dev) / (ms_eager * 1e-3), 1),
                "eager_ms_per_step": round(ms_eager, 4),
                "eager_how": "the same step issued from Python every time, without a graph"},
        "gpu_launches": args.layers * args.steps,
        "clocks": clocks,
        "legs": legs,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
