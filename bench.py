#!/usr/bin/env python
"""Bench: one DeepSeek-V4-Flash CSA layer on GB300.

Headline workload: batched decode, 32 sequences with 32768-token caches
(8192 ratio-4 rows + 128-token window each), Flash shapes, bf16.  One step =
the whole hot path for every sequence: compress (attention pool), compress
(index pool), indexer top-k, attention + merge.  Metric: layer-steps/s (one
step advances all 32 sequences by a token) and the achieved HBM GB/s of the
step's algorithmic bytes.  Also measured: prefill tok/s of a 4096-token chunk
on a 65536-token cache.

Timing: CUDA events around each step on the launching stream; the 129 MB L2 is
flushed (a 512 MB write) before every timed step, outside the events, because
in a full model 42 other layers run between two steps of this one.  A timed
step is a model step of --layers layers (default 8), each with its own data.
The end-to-end figure runs the same model steps through the public calls with
every layer's inputs copied from pinned host memory and the output read back,
pipelined as a serving loop (the next step's copies under the current step).

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA decode layer-steps/s + achieved HBM GB/s (B=32, 32K ctx); prefill tok/s"
UNIT = "layer-steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# DRAM traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum, every kernel captured cold) of one decode
# layer-step of the headline workload and of one prefill chunk, with the hash of the kernel sources the counters
# were taken on (csrc_digest()); the bench reports them only while the sources still hash the same.
TRAFFIC = {"csrc_sha256": "36a6e608430072f3", "decode_layer_step_bytes": 117_480_000,
           "decode_fp8_layer_step_bytes": 87_534_000, "prefill_chunk_bytes": 1_234_002_000,
           "profile": "profiles/traffic_decode_b32_ctx32k_and_prefill_t4096.md"}


def csrc_digest() -> str:
    """sha256 (first 16 hex digits) of the library's kernel sources."""
    import hashlib
    d = os.path.join(ROOT, "deepseek_v4_compressed_csa_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def _traffic(key: str, units: int):
    if TRAFFIC.get(key) is None or TRAFFIC.get("csrc_sha256") != csrc_digest():
        return None
    return int(TRAFFIC[key] * units)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            self.path = tempfile.mktemp(suffix=".csv")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_sample(cid: int, seqs: list[int], warmup: int, steps: int, budget_s: float) -> dict:
    """Time the CPU oracle stepping sequences ``seqs`` of workload ``cid`` through ``warmup`` untimed and up to
    ``steps`` timed decode steps (stopping early once ``budget_s`` of timed work is spent).  Runs in its own
    process with single-threaded BLAS; returns the per-step times (the sum over its sequences)."""
    import numpy as np

    import csa_synth
    from oracle import csa_oracle as O
    cfg = csa_synth.CONFIGS[cid]
    cap = cfg.ctx // cfg.ratio + (warmup + steps) // cfg.ratio + 8
    host = csa_synth.synth_cache(cfg, cap, B=max(seqs) + 1)
    f = lambda t: None if t is None else t.float().numpy().astype(np.float64)  # noqa: E731
    layer = O.Layer(dtype=cfg.dtype, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                    topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps)
    comp = lambda c: O.Compressor(wkv=f(c.wkv), wgate=f(c.wgate), ape=f(c.ape), norm_w=f(c.norm_w), d=c.d)  # noqa
    ca = comp(csa_synth.compressor(cfg, "attn"))
    ci = comp(csa_synth.compressor(cfg, "index")) if cfg.has_indexer else None
    sl = lambda t, b: None if t is None else f(t[b:b + 1])  # noqa: E731
    states = {b: dict(pool=sl(host.pool, b), ikeys=sl(host.ikeys, b), window=sl(host.window, b),
                      front_a=sl(host.front_attn, b), front_i=sl(host.front_index, b),
                      n_rows=host.n_rows[b:b + 1].numpy().astype(np.int64),
                      pos=host.pos[b:b + 1].numpy().astype(np.int64)) for b in seqs}
    del host
    sink, invf = f(csa_synth.sinks(cfg)), csa_synth.inv_freq(cfg).numpy()
    times = []
    spent = 0.0
    for step in range(warmup + steps):
        si = csa_synth.step_inputs(cfg, step, B=max(seqs) + 1)
        t0 = time.perf_counter()
        for b in seqs:
            O.decode_step(layer, ca, ci, states[b], (sl(si.x, b), sl(si.q, b), sl(si.kv, b), sl(si.iq, b),
                                                     sl(si.iw, b)), sink, invf)
        dt = time.perf_counter() - t0
        if step >= warmup:
            times.append(dt)
            spent += dt
            if spent > budget_s:
                break
    return {"times": times, "seqs": list(seqs)}


def cpu_info() -> dict:
    """Host core count and CPU model (for the CPU-baseline figures)."""
    import platform
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            k = line.split(":")[0].strip().lower()
            if k in ("model name", "cpu model", "hardware") and ":" in line:
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith(("model name", "vendor id")):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine(),
            "arch": platform.machine()}


def run_oracle_processes(cid: int, groups: list[list[int]], warmup: int, steps: int, budget_s: float) -> dict:
    """The oracle on len(groups) host cores at once: one process per group of sequences (spawned as fresh
    interpreters, single-threaded BLAS each), all stepping the same decode steps.  A layer-step's time is the
    slowest process's time for that step (as if the processes met at a barrier after each step)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    procs = []
    for g in groups:
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", str(cid), ",".join(map(str, g)),
               str(warmup), str(steps), str(budget_s)]
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    results = []
    for pr in procs:
        out, err = pr.communicate(timeout=max(900, 6 * budget_s))
        if pr.returncode != 0:
            raise RuntimeError(f"oracle sample failed:\n{err[-2000:]}")
        results.append(json.loads(out.strip().splitlines()[-1]))
    n = min(len(r["times"]) for r in results)
    per_step = [max(r["times"][i] for r in results) for i in range(n)]
    return {"step_s": per_step, "steps": n, "processes": len(groups),
            "sequences": sum(len(r["seqs"]) for r in results)}


# ----------------------------------------------------------------------------- distributed plumbing

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("CSA_BENCH_GLOO") is None else "gloo")
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def whole_job_rate(world: int, units_per_rank: float, slowest_ms: float) -> float:
    """Units per second of the whole job: each of the world's replicas processes units_per_rank units in the timed
    region, whose length is the slowest rank's (the max over ranks)."""
    return world * units_per_rank / (slowest_ms / 1e3)


def _max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- our arm

class DecodeWorkload:
    """Config 3 state, weights and per-step inputs resident on one GPU."""

    def __init__(self, cfg, cap: int, n_inputs: int, device, serial_indexer: bool = False, host=None,
                 host_comp=None, pos=None, input_tag: int = 0, index_fp8: bool = False):
        """host / host_comp: a synthetic cache and compressor weights generated once and copied here (several
        layers hold copies in distinct device memory); pos: a position tensor shared with other layers;
        input_tag: offset of this layer's per-step input sets; index_fp8: the index pool as fp8 rows (the
        cache's model-dtype index rows converted by csa_index_rows_fp8)."""
        import torch

        import csa_synth
        import deepseek_v4_compressed_csa_gb300 as csa
        self.cfg, self.cap, self.dev = cfg, cap, device
        self.serial_indexer = serial_indexer
        self.one_stream_overlap = False
        # where the main stream joins the attention pool's compress call (one-stream indexer order): before the
        # indexer, or after it (then attention has two predecessors)
        self.join_before_index = False
        self.L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi,
                           Di=cfg.Di, topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps,
                           index_fp8=index_fp8)
        d = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731

        def comp(c):
            return csa.Compressor(wkv=d(c.wkv), wgate=d(c.wgate), ape=d(c.ape), norm_w=d(c.norm_w), d=c.d)
        if host_comp is None:
            host_comp = (csa_synth.compressor(cfg, "attn"), csa_synth.compressor(cfg, "index") if cfg.has_indexer
                         else None)
        self.ca = comp(host_comp[0])
        self.ci = comp(host_comp[1]) if cfg.has_indexer else None
        if host is None:
            host = csa_synth.synth_cache(cfg, cap)
        self.pool, self.ikeys, self.window = d(host.pool), d(host.ikeys), d(host.window)
        if index_fp8:
            keys = self.ikeys
            self.ikeys = torch.empty(cfg.B, cap, csa.FP8_ROW_BYTES, dtype=torch.uint8, device=device)
            csa.index_rows_fp8(self.L, keys, self.ikeys)
            del keys
        self.front_a, self.front_i = d(host.front_attn), d(host.front_index)
        self.n_a, self.n_i = d(host.n_rows), d(host.n_rows)
        self.pos = d(host.pos) if pos is None else pos
        self.sink, self.invf = d(csa_synth.sinks(cfg)), d(csa_synth.inv_freq(cfg))
        B = cfg.B
        self.host_inputs = [csa_synth.step_inputs(cfg, input_tag + i) for i in range(n_inputs)]
        # each input set lives in one packed device buffer (256-byte aligned fields), so that a step's inputs
        # can arrive from pinned host memory in a single copy
        names = ("x", "q", "kv", "iq", "iw")
        t0 = self.host_inputs[0]
        self.fields, off = [], 0
        for k in names:
            t = getattr(t0, k)
            nb = t.numel() * t.element_size()
            self.fields.append((k, off, nb, t.dtype, tuple(t.shape)))
            off = (off + nb + 255) // 256 * 256
        self.packed_bytes = off
        self.packed = [torch.empty(off, dtype=torch.uint8, device=device) for _ in self.host_inputs]
        self.inputs = []
        for buf, si in zip(self.packed, self.host_inputs):
            views = {}
            for k, o, nb, dt, shape in self.fields:
                views[k] = buf[o:o + nb].view(dt).view(shape)
                views[k].copy_(getattr(si, k))
            self.inputs.append(views)
        self.sel = torch.empty(B, cfg.topk, dtype=torch.int32, device=device)
        self.n_sel = torch.empty(B, dtype=torch.int32, device=device)
        self.out = torch.empty(B, cfg.H, cfg.D, dtype=cfg.storage, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        u8 = lambda n: torch.empty(max(n, 256), dtype=torch.uint8, device=device)  # noqa: E731
        self.ws_c = u8(csa.workspace_size(self.L, csa.OP_COMPRESS, B, 1, cap))
        self.ws_c2 = u8(csa.workspace_size(self.L, csa.OP_COMPRESS, B, 1, cap))  # the concurrent second call
        self.pair = cfg.has_indexer  # both pools through csa_compress_append_pair
        self.ws_pair = u8(csa.workspace_size(self.L, csa.OP_COMPRESS_PAIR, B, 1, cap)) if self.pair else None
        self.side = torch.cuda.Stream(device)
        self.side2 = torch.cuda.Stream(device)
        self.pool_ready = torch.cuda.Event()
        self.ws_i = u8(csa.workspace_size(self.L, csa.OP_INDEX_TOPK, B, 1, cap))
        self.ws_a = u8(csa.workspace_size(self.L, csa.OP_ATTEND_DECODE, B, 1, cap))
        self.csa = csa

    def packed_host(self, i):
        """Input set i packed as in its device buffer, in pinned host memory."""
        import torch
        h = torch.zeros(self.packed_bytes, dtype=torch.uint8).pin_memory()
        for k, o, nb, dt, shape in self.fields:
            h[o:o + nb].view(dt).view(shape).copy_(getattr(self.host_inputs[i], k))
        return h

    def front(self, inp):
        """Phase 1: both pools' compress call (csa_compress_append_pair) and the indexer on one stream; with
        pair off, the attention pool's compress call on a side stream and, on the main stream, the index pool's
        call and the indexer (or, with serial_indexer off, the index pool's call on a second side stream and
        csa_index_topk_overlapped beside it, its selection waiting for that call's event).  Each concurrent
        call has its own workspace."""
        import torch
        csa = self.csa
        main = torch.cuda.current_stream()
        if not self.cfg.has_indexer:
            # a layer without an indexer (ratio 128): its one compress call, then attention, on one stream
            csa.compress_append(self.L, self.ca, inp["x"], self.pos, self.front_a, self.pool, self.n_a, self.invf,
                                ws=self.ws_c, err=self.err)
            return
        if self.cfg.has_indexer and self.serial_indexer and self.pair:
            # both pools in one call (one projection grid, one pooling launch), then the indexer: one stream, so
            # every kernel of the step follows its predecessor by programmatic launch.  With one_stream_overlap the
            # indexer is csa_index_topk_overlapped without an event: its scan of the rows complete before the token
            # runs beside the projection and pooling kernels
            csa.compress_append_pair(self.L, self.ca, self.ci, inp["x"], self.pos, self.front_a, self.pool, self.n_a,
                                     self.front_i, self.ikeys, self.n_i, self.invf, ws=self.ws_pair, err=self.err)
            if self.one_stream_overlap:
                csa.index_topk_overlapped(self.L, inp["iq"], inp["iw"], self.ikeys, self.n_i, self.pos, self.invf,
                                          self.sel, self.n_sel, ws=self.ws_i, err=self.err)
            else:
                csa.index_topk(self.L, inp["iq"], inp["iw"], self.ikeys, self.n_i, self.pos, self.invf, self.sel,
                               self.n_sel, ws=self.ws_i, err=self.err)
            return
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            csa.compress_append(self.L, self.ca, inp["x"], self.pos, self.front_a, self.pool, self.n_a, self.invf,
                                ws=self.ws_c2, err=self.err)
        if self.cfg.has_indexer and self.serial_indexer:
            csa.compress_append(self.L, self.ci, inp["x"], self.pos, self.front_i, self.ikeys, self.n_i, self.invf,
                                ws=self.ws_c, err=self.err)
            if self.join_before_index:
                main.wait_stream(self.side)
            csa.index_topk(self.L, inp["iq"], inp["iw"], self.ikeys, self.n_i, self.pos, self.invf, self.sel,
                           self.n_sel, ws=self.ws_i, err=self.err)
        elif self.cfg.has_indexer:
            self.side2.wait_stream(main)
            with torch.cuda.stream(self.side2):
                csa.compress_append(self.L, self.ci, inp["x"], self.pos, self.front_i, self.ikeys, self.n_i,
                                    self.invf, ws=self.ws_c, err=self.err)
                self.pool_ready.record(self.side2)
            csa.index_topk_overlapped(self.L, inp["iq"], inp["iw"], self.ikeys, self.n_i, self.pos, self.invf,
                                      self.sel, self.n_sel, pool_ready=self.pool_ready, ws=self.ws_i, err=self.err)
            main.wait_stream(self.side2)
        if not (self.cfg.has_indexer and self.serial_indexer and self.join_before_index):
            main.wait_stream(self.side)

    def attend(self, inp, advance: bool = True):
        """Phase 2: attention over the selected rows and the window, merge; then (advance) the positions move on
        (in a model step that is done once, after the last layer)."""
        sel, n_sel = (self.sel, self.n_sel) if self.cfg.has_indexer else (None, None)
        self.csa.attend_decode(self.L, inp["q"], inp["kv"], self.sink, self.window, self.pool, self.n_a, sel, n_sel,
                               self.pos, self.invf, self.out, ws=self.ws_a, err=self.err)
        if advance:
            self.csa.advance_positions(self.pos, 1)

    def step(self, inp):
        self.front(inp)
        self.attend(inp)

    def capture(self, per_phase: bool = False):
        """Per input set, one CUDA graph holding the whole step (both phases), or with per_phase one graph per
        phase (compress + indexer | attention) so that events can separate them."""
        import torch
        self.graphs = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for inp in self.inputs:
                gs = []
                parts = ((self.front, self.attend),) if not per_phase else ((self.front,), (self.attend,))
                for part in parts:
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                        for fn in part:
                            fn(inp)
                    gs.append(g)
                self.graphs.append(gs)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def replay(self, i, ev=None):
        """Step i: its graph(s) (or, eagerly, the same calls); an event before each graph and one after."""
        if self.graphs is None:
            inp = self.inputs[i % len(self.inputs)]
            parts = [lambda: self.step(inp)]
        else:
            parts = [g.replay for g in self.graphs[i % len(self.graphs)]]
        for k, run in enumerate(parts):
            if ev is not None:
                ev[k].record()
            run()
        if ev is not None:
            ev[len(parts)].record()


class ModelStep:
    """One decode step of `n_layers` layers, as a model step runs them: each layer its own weights, caches, step
    inputs and workspaces in distinct device memory (so every layer reads its data cold from HBM, as after the
    other layers of a model), one shared position tensor advanced once after the last layer.  Each step is one
    CUDA graph replay holding every layer."""

    def __init__(self, cfg, cap: int, n_inputs: int, device, n_layers: int, pair: bool = True, host=None,
                 one_stream_overlap: bool = False, index_fp8: bool = False):
        import torch

        import csa_synth
        host = csa_synth.synth_cache(cfg, cap) if host is None else host
        host_comp = (csa_synth.compressor(cfg, "attn"),
                     csa_synth.compressor(cfg, "index") if cfg.has_indexer else None)
        self.layers = []
        pos = None
        for i in range(n_layers):
            wl = DecodeWorkload(cfg, cap, n_inputs, device, serial_indexer=True, host=host, host_comp=host_comp,
                                pos=pos, input_tag=1000 * i, index_fp8=index_fp8)
            wl.pair = wl.pair and pair
            wl.one_stream_overlap = one_stream_overlap
            pos = wl.pos
            self.layers.append(wl)
        self.pos, self.csa, self.n_inputs = pos, self.layers[0].csa, n_inputs
        self.graphs = None
        self.torch = torch

    def step(self, i):
        for wl in self.layers:
            inp = wl.inputs[i % self.n_inputs]
            wl.front(inp)
            wl.attend(inp, advance=False)
        self.csa.advance_positions(self.pos, 1)

    def capture(self):
        torch = self.torch
        self.graphs = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(self.n_inputs):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                    self.step(i)
                self.graphs.append(g)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def replay(self, i, ev=None):
        if ev is not None:
            ev[0].record()
        if self.graphs is None:
            self.step(i)
        else:
            self.graphs[i % self.n_inputs].replay()
        if ev is not None:
            ev[1].record()


class ConsumerLayer:
    """A layer that owns no compressor (DeepSeek-V4.1 cross-layer sharing): its own queries, new token, sinks,
    window ring and workspaces; the owner's compressed rows, index keys, row counts and positions.  kind "index":
    its own top-k over the owner's index keys (an index-source layer); "plain": the owner's selection."""

    def __init__(self, owner, kind: str, n_inputs: int, device, tag: int):
        import torch

        import csa_synth
        csa, cfg = owner.csa, owner.cfg
        self.owner, self.kind, self.csa, self.cfg = owner, kind, csa, cfg
        c = cfg.replace(cid=cfg.cid + 700 + tag)
        d = lambda t: t.to(device).contiguous()  # noqa: E731
        self.inputs = []
        for i in range(n_inputs):
            si = csa_synth.step_inputs(c, i)
            self.inputs.append({k: d(getattr(si, k)) for k in ("q", "kv", "iq", "iw")})
        self.window = owner.window.clone()
        self.sink = d(csa_synth.sinks(c))
        B, cap = cfg.B, owner.cap
        self.sel = torch.empty(B, cfg.topk, dtype=torch.int32, device=device)
        self.n_sel = torch.empty(B, dtype=torch.int32, device=device)
        self.out = torch.empty(B, cfg.H, cfg.D, dtype=cfg.storage, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        u8 = lambda n: torch.empty(max(n, 256), dtype=torch.uint8, device=device)  # noqa: E731
        self.ws_i = u8(csa.workspace_size(owner.L, csa.OP_INDEX_TOPK, B, 1, cap))
        self.ws_a = u8(csa.workspace_size(owner.L, csa.OP_ATTEND_DECODE, B, 1, cap))

    def step(self, i):
        o, csa = self.owner, self.csa
        inp = self.inputs[i % len(self.inputs)]
        if self.kind == "index":
            csa.index_topk(o.L, inp["iq"], inp["iw"], o.ikeys, o.n_i, o.pos, o.invf, self.sel, self.n_sel,
                           ws=self.ws_i, err=self.err)
            sel, n_sel = self.sel, self.n_sel
        else:
            sel, n_sel = o.sel, o.n_sel
        csa.attend_decode(o.L, inp["q"], inp["kv"], self.sink, self.window, o.pool, o.n_a, sel, n_sel, o.pos, o.invf,
                          self.out, ws=self.ws_a, err=self.err)


SHARED_PATTERN = ("owner", "plain", "plain", "index", "index", "index", "plain", "plain")


def shared_line(csa, csa_synth, dev, flush, steps: int, warmup: int) -> dict:
    """A DeepSeek-V4.1-style model step of 8 layers sharing one owner's caches (the README's pattern: one
    compressor-owning layer, then layers consuming its caches, a run of them index-source layers), B = 32 on 32K
    caches, one CUDA graph per model step, the L2 flushed before each, timed like the headline."""
    import torch
    cfg = csa_synth.CONFIGS[3]
    cap = cfg.ctx // cfg.ratio + (warmup + steps + 8) // cfg.ratio + 8
    owner = DecodeWorkload(cfg, cap, 4, dev, serial_indexer=True)
    layers = [ConsumerLayer(owner, k, 4, dev, i) for i, k in enumerate(SHARED_PATTERN) if k != "owner"]

    class _Step:
        def __init__(self):
            self.graphs = None

        def step(self, i):
            inp = owner.inputs[i % 4]
            owner.front(inp)
            owner.attend(inp, advance=False)
            for c in layers:
                c.step(i)
            csa.advance_positions(owner.pos, 1)

        def replay(self, i, ev=None):
            if ev is not None:
                ev[0].record()
            self.graphs[i % 4].replay()
            if ev is not None:
                ev[1].record()

    ms = _Step()
    ms.step(0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    ms.graphs = []
    with torch.cuda.stream(s):
        for i in range(4):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                ms.step(i)
            ms.graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in range(warmup):
        ms.replay(1 + i)
    n0 = owner.n_a.float().mean().item()
    t = time_model_steps(ms, 1 + warmup, steps, flush)
    n1 = owner.n_a.float().mean().item()
    assert owner.err.item() == 0 and all(c.err.item() == 0 for c in layers)
    nl = len(SHARED_PATTERN)
    per_step_ms = statistics.mean(t)
    n = 0.5 * (n0 + n1)
    full = step_bytes(cfg, n)
    e = 2
    rows = full["attended_rows"] + full["q_out"]
    idx = full["index_keys"] + cfg.B * (cfg.Hi * cfg.Di * e + cfg.Hi * e + cfg.topk * 4)
    by_kind = {"owner": full["total"], "index": rows + idx, "plain": rows}
    total = sum(by_kind[k] for k in SHARED_PATTERN)
    hbm, _, _ = _peaks()
    gbs = total / (per_step_ms / 1e3) / 1e9
    del layers, owner
    return {"pattern": list(SHARED_PATTERN), "layer_steps_per_s": round(nl * 1e3 / per_step_ms, 1),
            "tokens_per_s": round(cfg.B * nl * 1e3 / per_step_ms, 1), "us_per_layer_step": round(
                1e3 * per_step_ms / nl, 2), "ms_per_model_step_p10_p50_p90": [round(x, 4) for x in _percentiles(t)],
            "algorithmic_bytes_per_model_step": int(total),
            "bytes_by_layer_kind": {k: int(v) for k, v in by_kind.items()},
            "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4), "steps": steps,
            "note": ("layer 0 owns the compressors and index keys; the others attend to its rows with their own "
                     "queries, sinks and windows, index-source layers through their own top-k over its keys")}


class VerifyLayer:
    """One layer's state for verify blocks of T tokens per sequence (config 3 shapes, rollback T - 1 + 8)."""

    def __init__(self, cfg, T: int, cap: int, n_inputs: int, device, host, host_comp, pos, tag: int):
        import torch

        import csa_synth
        import deepseek_v4_compressed_csa_gb300 as csa
        self.csa, self.cfg, self.T = csa, cfg, T
        self.L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi,
                           Di=cfg.Di, topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps,
                           rollback=cfg.rollback)
        d = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731

        def comp(c):
            return csa.Compressor(wkv=d(c.wkv), wgate=d(c.wgate), ape=d(c.ape), norm_w=d(c.norm_w), d=c.d)
        self.ca, self.ci = comp(host_comp[0]), comp(host_comp[1])
        self.pool, self.ikeys, self.window = d(host.pool), d(host.ikeys), d(host.window)
        self.front_a, self.front_i = d(host.front_attn), d(host.front_index)
        self.n_a, self.n_i, self.pos = d(host.n_rows), d(host.n_rows), pos
        self.sink, self.invf = d(csa_synth.sinks(cfg)), d(csa_synth.inv_freq(cfg))
        B = cfg.B
        self.inputs = []
        for i in range(n_inputs):
            si = [csa_synth.step_inputs(cfg, tag + T * i + j) for j in range(T)]
            st = lambda f: d(torch.stack([getattr(x, f) for x in si], dim=1))  # noqa: E731
            self.inputs.append(dict(x=d(torch.cat([x.x for x in si], dim=1)), q=st("q"), kv=st("kv"), iq=st("iq"),
                                    iw=st("iw")))
        self.sel = torch.empty(B, T, cfg.topk, dtype=torch.int32, device=device)
        self.n_sel = torch.empty(B, T, dtype=torch.int32, device=device)
        self.out = torch.empty(B, T, cfg.H, cfg.D, dtype=cfg.storage, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        u8 = lambda n: torch.empty(max(n, 256), dtype=torch.uint8, device=device)  # noqa: E731
        self.ws_pair = u8(csa.workspace_size(self.L, csa.OP_COMPRESS_PAIR, B, T, cap))
        self.ws_i = u8(csa.workspace_size(self.L, csa.OP_INDEX_TOPK, B * T, 1, cap))
        self.ws_a = u8(csa.workspace_size(self.L, csa.OP_ATTEND_DECODE, B * T, 1, cap))

    def step(self, i):
        csa, inp = self.csa, self.inputs[i % len(self.inputs)]
        csa.compress_append_pair(self.L, self.ca, self.ci, inp["x"], self.pos, self.front_a, self.pool, self.n_a,
                                 self.front_i, self.ikeys, self.n_i, self.invf, ws=self.ws_pair, err=self.err)
        csa.index_topk_verify(self.L, inp["iq"], inp["iw"], self.ikeys, self.n_i, self.pos, self.invf, self.sel,
                              self.n_sel, ws=self.ws_i, err=self.err)
        csa.attend_verify(self.L, inp["q"], inp["kv"], self.sink, self.window, self.pool, self.n_a, self.sel,
                          self.n_sel, self.pos, self.invf, self.out, ws=self.ws_a, err=self.err)


def verify_line(csa, csa_synth, dev, flush, steps: int, warmup: int, nl: int, T: int = 4) -> dict:
    """Verify blocks of T tokens per sequence (a speculative step with T - 1 drafts), B = 32 on 32K caches, as a
    model step of nl layers in one CUDA graph, the positions advancing by T after the last layer."""
    import torch
    cfg = csa_synth.CONFIGS[3].replace(rollback=T - 1 + 8)
    cap = cfg.ctx // cfg.ratio + T * (warmup + steps + 8) // cfg.ratio + 8
    host = csa_synth.synth_cache(cfg, cap)
    host_comp = (csa_synth.compressor(cfg, "attn"), csa_synth.compressor(cfg, "index"))
    pos = host.pos.to(dev)
    layers = [VerifyLayer(cfg, T, cap, 4, dev, host, host_comp, pos, 5000 + 100 * i) for i in range(nl)]

    class _Step:
        graphs = None

        def step(self, i):
            for layer in layers:
                layer.step(i)
            csa.advance_positions(pos, T)

        def replay(self, i, ev=None):
            if ev is not None:
                ev[0].record()
            self.graphs[i % 4].replay()
            if ev is not None:
                ev[1].record()

    ms = _Step()
    ms.step(0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    ms.graphs = []
    with torch.cuda.stream(s):
        for i in range(4):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                ms.step(i)
            ms.graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in range(warmup):
        ms.replay(1 + i)
    n0 = layers[0].n_a.float().mean().item()
    t = time_model_steps(ms, 1 + warmup, steps, flush)
    n1 = layers[0].n_a.float().mean().item()
    assert all(layer.err.item() == 0 for layer in layers)
    per = statistics.mean(t) / nl
    b = step_bytes(cfg, 0.5 * (n0 + n1))
    # per layer-step: the weights and the index keys once (four queries share each key tile), every query's rows
    total = b["weights"] + b["index_keys"] + T * (b["attended_rows"] + b["q_out"]) + T * b["small"]
    hbm, _, _ = _peaks()
    gbs = total / (per / 1e3) / 1e9
    del layers
    return {"T": T, "B": cfg.B, "layer_steps_per_s": round(1e3 / per, 1),
            "verified_tokens_per_s": round(cfg.B * T * 1e3 / per, 1), "us_per_layer_step": round(1e3 * per, 2),
            "us_per_layer_step_p10_p50_p90": [round(1e3 * x / nl, 2) for x in _percentiles(t)],
            "algorithmic_bytes_per_layer_step": int(total), "achieved_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm, 4), "layers_per_step": nl, "steps": steps,
            "calls": "per layer: csa_compress_append_pair (T tokens), csa_index_topk_verify, csa_attend_verify"}


def step_bytes(cfg, n_rows_mean: float, index_fp8: bool = False) -> dict:
    """Algorithmic HBM bytes of one decode step (each byte the step must move once); index_fp8: index-key rows of
    144 bytes (128 codes and the row's scale) instead of Di model-dtype values."""
    B, e = cfg.B, 2
    L = cfg.lanes
    w = (2 * L * cfg.D * cfg.X + (2 * L * cfg.Di * cfg.X if cfg.has_indexer else 0)) * e
    key_row = 144 if index_fp8 else cfg.Di * e
    keys = B * n_rows_mean * key_row if cfg.has_indexer else 0
    rows = B * ((cfg.topk if cfg.has_indexer else n_rows_mean) + cfg.W) * cfg.D * e
    qo = 2 * B * cfg.H * cfg.D * e
    small = B * (cfg.X * e + cfg.D * e + cfg.Hi * cfg.Di * e + cfg.Hi * e + cfg.topk * 4)
    fr = B * 2 * (2 * L * (cfg.D + (cfg.Di if cfg.has_indexer else 0))) * e  # frontier slot write + window row
    return {"weights": w, "index_keys": keys, "attended_rows": rows, "q_out": qo, "small": small + fr,
            "total": w + keys + rows + qo + small + fr}


def time_model_steps(ms, first: int, steps: int, flush) -> list[float]:
    """CUDA-event times (ms) of `steps` model steps (graph replays), the L2 flushed before each, outside the events."""
    import torch
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        ms.replay(first + i, ev=ev[i])
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def built_cache_b1(csa, csa_synth, cfg, cap, dev):
    """Config 2's cache: 8192 seeded hidden tokens compressed into both pools by the library (one chunk call per
    pool) from an empty cache, copied back as a host cache; the window ring stays as decode will fill it."""
    import torch
    host = csa_synth.empty_cache(cfg, cap)
    d = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                  topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps)
    x = d(csa_synth.hidden(cfg, cfg.prefill_tokens))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = {k: d(getattr(host, k)) for k in ("pool", "ikeys", "front_attn", "front_index", "n_rows", "pos")}
    n_i = st["n_rows"].clone()
    for which, front, pool, n in (("attn", "front_attn", "pool", st["n_rows"]), ("index", "front_index", "ikeys", n_i)):
        c = csa_synth.compressor(cfg, which)
        comp = csa.Compressor(wkv=d(c.wkv), wgate=d(c.wgate), ape=d(c.ape), norm_w=d(c.norm_w), d=c.d)
        csa.compress_append(L, comp, x, st["pos"], st[front], st[pool], n, d(csa_synth.inv_freq(cfg)), err=err)
    torch.cuda.synchronize()
    assert err.item() == 0 and int(st["n_rows"][0]) == cfg.prefill_tokens // cfg.ratio
    for k in ("pool", "ikeys", "front_attn", "front_index", "n_rows"):
        getattr(host, k).copy_(st[k].cpu())
    host.pos[:] = cfg.prefill_tokens
    return host


def decode_config_line(csa, csa_synth, cid: int, dev, flush, steps: int, warmup: int, nl: int,
                       overlap: bool = False, index_fp8: bool = False) -> dict:
    """Throughput and HBM fraction of another decode workload as a model step of `nl` layers (config 2: B = 1
    on an 8K cache the library compressed from seeded hidden states; config 4: ratio 128, B = 16, 256K context,
    every row attended; config 3 with index_fp8: the headline workload with the index pool as fp8 rows), timed
    like the headline."""
    cfg = csa_synth.CONFIGS[cid]
    n_ctx = cfg.prefill_tokens if cid == 2 else cfg.ctx
    cap = n_ctx // cfg.ratio + (warmup + steps + 8) // cfg.ratio + 8
    host = built_cache_b1(csa, csa_synth, cfg, cap, dev) if cid == 2 else None
    ms = ModelStep(cfg, cap, n_inputs=4, device=dev, n_layers=nl, host=host, one_stream_overlap=overlap,
                   index_fp8=index_fp8)
    wl = ms.layers[0]
    ms.step(0)
    ms.capture()
    for i in range(warmup):
        ms.replay(1 + i)
    n0 = wl.n_a.float().mean().item()
    t = time_model_steps(ms, 1 + warmup, steps, flush)
    n1 = wl.n_a.float().mean().item()
    for layer in ms.layers:
        assert layer.err.item() == 0, f"device error word {layer.err.item()}"
    per = [x / nl for x in t]
    mean_ms = statistics.mean(per)
    nb = step_bytes(cfg, 0.5 * (n0 + n1), index_fp8)
    hbm, _, _ = _peaks()
    gbs = nb["total"] / (mean_ms / 1e3) / 1e9
    del ms
    return {"workload": cfg.name + (" fp8-index-keys" if index_fp8 else ""), "B": cfg.B, "context": n_ctx, "ratio": cfg.ratio, "compressed_rows": [n0, n1],
            "layer_steps_per_s": round(1e3 / mean_ms, 1), "tokens_per_s": round(cfg.B * 1e3 / mean_ms, 1),
            "us_per_layer_step": round(1e3 * mean_ms, 2),
            "us_per_layer_step_p10_p50_p90": [round(1e3 * x, 2) for x in _percentiles(per)],
            "step_algorithmic_bytes": int(nb["total"]), "achieved_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm, 4), "layers_per_step": nl, "steps": steps,
            "dram_traffic_bytes_per_layer_step": _traffic("decode_fp8_layer_step_bytes", 1) if index_fp8 else None,
            "cache": ("compressed from 8192 seeded hidden tokens by the library" if cid == 2 else
                      "synthetic rows drawn directly (seeded N(0,1))" + (
                          "; index rows converted to fp8 rows by csa_index_rows_fp8" if index_fp8 else ""))}


def trim_line(csa, csa_synth, dev) -> dict:
    """Latency of csa_trim for the headline batch (B = 32, rollback 64): one graph of 64 trims (a trim moves no
    data, so its cost is one small kernel whatever it rewinds), timed with CUDA events."""
    import torch
    cfg = csa_synth.CONFIGS[3].replace(rollback=64)
    L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                  topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps, rollback=cfg.rollback)
    i32 = lambda v: torch.full((cfg.B,), v, dtype=torch.int32, device=dev)  # noqa: E731
    pos, n_a, n_i, hw = i32(cfg.ctx), i32(cfg.ctx // 4), i32(cfg.ctx // 4), i32(cfg.ctx)
    n_back, err = i32(0), torch.zeros(1, dtype=torch.int32, device=dev)
    reps = 64
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        csa.trim(L, n_back, pos, n_a, n_i, hw, err=err)
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                csa.trim(L, n_back, pos, n_a, n_i, hw, err=err)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    assert err.item() == 0
    return {"batch": cfg.B, "rollback": cfg.rollback, "us_per_trim": round(1e3 * e0.elapsed_time(e1) / reps, 3),
            "how": f"one CUDA graph of {reps} back-to-back csa_trim calls (B = {cfg.B}), CUDA events"}


def run_ours(args):
    import torch
    dist, rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import csa_synth
    import deepseek_v4_compressed_csa_gb300 as csa
    csa.load_library()
    cfg = csa_synth.CONFIGS[3]
    nl = args.layers
    n_single = args.steps  # the one-layer comparison run (layer 0 alone, one graph per layer-step)
    total_steps = args.warmup + args.steps + args.e2e_steps + 2 * (args.warmup + n_single) + 24
    cap = cfg.ctx // cfg.ratio + total_steps // cfg.ratio + 8
    ms = ModelStep(cfg, cap, n_inputs=4, device=dev, n_layers=nl, pair=not args.two_streams,
                   one_stream_overlap=args.indexer == "overlap", index_fp8=args.index_fp8)
    wl = ms.layers[0]
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    ms.step(0)  # first calls outside capture (one-time host set-up inside the library)
    torch.cuda.synchronize()
    if args.eager:
        ms.graphs = None  # same kernels launched one by one (for profilers that do not follow graphs)
    else:
        ms.capture()  # capturing does not run anything: the graphs replay the steps below
    for i in range(args.warmup):
        ms.replay(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    n_start = wl.n_a.float().mean().item()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(args.steps):
        flush.zero_()
        ms.replay(args.warmup + i, ev=ev[i])
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = _max_over_ranks(dist, sum(step_ms), dev)
    for layer in ms.layers:
        assert layer.err.item() == 0, f"device error word {layer.err.item()}"
    n_end = wl.n_a.float().mean().item()
    # kernels per model step: counted on one eager step (graph replays enqueue the same kernels)
    k0 = csa.kernel_launches()
    ms.step(0)
    torch.cuda.synchronize()
    launches = (csa.kernel_launches() - k0) * args.steps

    # ---- end to end: per model step, each layer's inputs from pinned host memory (one copy per layer, its five
    # inputs packed as in its graph's input buffer), the step, the last layer's output back to pinned memory.  The
    # loop is pipelined as a serving loop would be: step i+1's inputs are copied on a second stream (into another
    # of the n_inputs buffer sets, once the step that last used it is done) while step i computes; one timed region
    # spans every copy, step and read-back (no L2 flush inside it: a model step's data is far larger than L2).
    pinned = [[layer.packed_host(i) for i in range(ms.n_inputs)] for layer in ms.layers]
    out_host = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
    h2d = wl.packed_bytes  # per layer-step: the bytes its one copy moves (fields plus alignment padding)
    d2h = out_host.numel() * out_host.element_size()  # per model step (the last layer's output)
    n2 = max(1, args.e2e_steps)
    copy_stream = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(n2)]
    step_done = [torch.cuda.Event() for _ in range(n2)]

    def copy_inputs(i):
        k = i % ms.n_inputs
        with torch.cuda.stream(copy_stream):
            if i >= ms.n_inputs:
                copy_stream.wait_event(step_done[i - ms.n_inputs])  # buffer set k is free again
            for layer, pin in zip(ms.layers, pinned):
                layer.packed[k].copy_(pin[k], non_blocking=True)
            in_ready[i].record(copy_stream)

    e2e_t = (mk(), mk())
    torch.cuda.synchronize()
    e2e_t[0].record(stream)
    copy_stream.wait_stream(stream)
    copy_inputs(0)
    for i in range(n2):
        stream.wait_event(in_ready[i])
        if i + 1 < n2:
            copy_inputs(i + 1)
        ms.replay(i % ms.n_inputs)
        step_done[i].record(stream)
        out_host.copy_(ms.layers[-1].out, non_blocking=True)
    e2e_t[1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(dist, e2e_t[0].elapsed_time(e2e_t[1]), dev) / n2

    # ---- comparison (not the headline): layer 0 alone, one CUDA graph per layer-step (each step's graph
    # launch latency falls on that one layer); then the per-phase diagnostic on the same layer.  These advance
    # the shared positions for layer 0 only, so they run after every model step.
    single = None
    phase_us = None
    if not args.eager:
        wl.capture()
        for i in range(args.warmup):
            wl.replay(i)
        ev1 = [(mk(), mk()) for _ in range(n_single)]
        torch.cuda.synchronize()
        for i in range(n_single):
            flush.zero_()
            wl.replay(i, ev=ev1[i])
        torch.cuda.synchronize()
        single_ms = sum(a.elapsed_time(b) for a, b in ev1) / n_single
        single = {"layer_steps_per_s": round(1e3 / single_ms, 3), "ms_per_layer_step": round(single_ms, 5)}
        wl.capture(per_phase=True)
        n_diag = min(args.steps, 16)
        evd = [(mk(), mk(), mk()) for _ in range(n_diag)]
        for i in range(3):
            wl.replay(i)
        torch.cuda.synchronize()
        for i in range(n_diag):
            flush.zero_()
            wl.replay(i, ev=evd[i])
        torch.cuda.synchronize()
        phase_us = {name: round(1e3 * statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evd), 2)
                    for k, name in enumerate(("compress_x2_and_index", "attend"))}
        assert wl.err.item() == 0, f"device error word {wl.err.item()}"

    # ---- prefill chunk (config 5), timed once per repeat from a restored snapshot
    prefill = prefill_varlen = prefill_fp8 = None
    if not args.no_prefill:
        prefill = run_prefill(csa, csa_synth, dev, flush, repeats=args.prefill_repeats)
        if not args.no_other_configs:
            prefill_varlen = run_prefill_varlen(csa, csa_synth, dev, flush, repeats=args.prefill_repeats)
            prefill_fp8 = run_prefill(csa, csa_synth, dev, flush, repeats=args.prefill_repeats, index_fp8=True)

    trim = trim_line(csa, csa_synth, dev)
    shared = None if args.no_other_configs else shared_line(csa, csa_synth, dev, flush, args.steps, args.warmup)
    verify = None if args.no_other_configs else verify_line(csa, csa_synth, dev, flush, args.steps, args.warmup, nl)

    # ---- the other decode workloads (configs 2 and 4), each as its own model step of nl layers
    others = None
    if not args.no_other_configs:
        del ms, wl
        torch.cuda.empty_cache()
        others = {}
        for cid, fp8 in ((2, False), (4, False), (3, True)):
            line = decode_config_line(csa, csa_synth, cid, dev, flush, args.steps, args.warmup, nl,
                                      overlap=args.indexer == "overlap" and not fp8, index_fp8=fp8)
            others[line["workload"]] = line

    hbm, tflops, peak_src = _peaks()
    ms_per_step = total_ms / (args.steps * nl)  # per layer-step
    value = whole_job_rate(world, args.steps * nl, total_ms)
    nb = step_bytes(cfg, 0.5 * (n_start + n_end), args.index_fp8)
    tkey = "decode_fp8_layer_step_bytes" if args.index_fp8 else "decode_layer_step_bytes"
    step_avg_s = ms_per_step / 1e3
    result = None
    if rank == 0:
        cpu = cpu_baseline(cfg, args.cpu_budget)
        result = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": cfg.name, "global_batch": cfg.B * world, "seq_len": cfg.ctx, "B_per_gpu": cfg.B,
                "heads": cfg.H, "latent": cfg.D, "window": cfg.W, "ratio": cfg.ratio, "index_heads": cfg.Hi,
                "index_dim": cfg.Di, "topk": cfg.topk, "hidden": cfg.X, "compressed_rows": [n_start, n_end],
                "tokens_per_s": round(value * cfg.B, 1),
                "step_algorithmic_bytes": int(nb["total"]),
                "step_hbm_gbs": round(nb["total"] / (ms_per_step / 1e3) / 1e9, 1),
                "step_hbm_frac": round(nb["total"] / (ms_per_step / 1e3) / 1e9 / hbm, 4),
                "layers_per_step": nl,
                "layer_steps_timed": args.steps * nl,
                "ms_per_layer_step_p10_p50_p90": [round(x / nl, 5) for x in _percentiles(step_ms)],
                "model_step": (f"each timed step is one decode step of {nl} layers (distinct weights, caches, inputs "
                               f"and workspaces: {nl} x ~0.4 GB, every layer's data cold in HBM as after the other "
                               "layers of a model), one CUDA graph replay; value = layer-steps / time; positions "
                               "advance once per model step"),
                "single_layer_graph": single,
                "l2": ("flushed (512 MB write) before every timed model step, outside the events; within a model "
                       "step each layer's data is distinct and the step's working set is far above L2"),
                "phase_us": phase_us,
                "phase_us_note": ("diagnostic: layer 0 alone, its step as two graphs (compress x2 + indexer | "
                                  "attention), events between them; each includes its graph's launch latency"),
                "launch": ("kernels launched one by one" if args.eager else
                           "each model step = 1 CUDA graph replay; per layer one stream: csa_compress_append_pair, "
                           + ("csa_index_topk_overlapped (no event: its scan of the rows complete before the token "
                              "runs beside the projection and pooling kernels), " if args.indexer == "overlap" else
                              "csa_index_topk, ") +
                           "csa_attend_decode, every kernel after its predecessor by programmatic launch; "
                           "csa_advance_positions after the last layer"),
                "indexer": args.indexer,
                "index_fp8": bool(args.index_fp8),
                "prefill": prefill,
                "prefill_varlen": prefill_varlen,
                "prefill_fp8_index_keys": prefill_fp8,
                "other_decode_workloads": others,
                "trim": trim,
                "v41_shared_caches": shared,
                "verify_blocks": verify,
            },
            "roofline": {
                "kernel": (f"model step graph: every kernel of one decode step of {nl} layers (per layer: both "
                           "projections, both pooling steps, index scan + top-k, attention + merge); algorithmic "
                           "bytes per layer = weights + index keys + attended rows + q/out + small terms"),
                "bound": "hbm",
                "achieved": round(nb["total"] / step_avg_s / 1e9, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(nb["total"] / step_avg_s / 1e9 / hbm, 4),
                "traffic": _traffic(tkey, nl),
                "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum summed over one layer-step's "
                                   f"kernels x {nl} layers ({TRAFFIC['profile']})" if _traffic(tkey, nl) else
                                   "null: no counters taken on the current kernel sources"),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6800 GB/s", "avg_launch_ms": round(total_ms / args.steps, 5),
                "algorithmic_bytes_per_launch": int(nb["total"] * nl),
            },
            "cpu_baseline": cpu,
            "e2e": {"value": round(whole_job_rate(world, nl, e2e_ms), 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": round(d2h / nl),
                    "per_model_step": {"layers": nl, "h2d_copies": nl, "h2d_bytes": h2d * nl, "d2h_bytes": d2h},
                    "pipeline": "step i+1's input copies run on a second stream during step i; one timed region over "
                                "all copies, steps and read-backs"},
            "gpu_launches": int(launches),
            "clocks": clk,
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_prefill(csa, csa_synth, dev, flush, repeats: int, index_fp8: bool = False):
    """One 4096-token chunk on a 64K cache (both compress calls + csa_attend_prefill_chunk), timed from a restored
    snapshot; index_fp8: the index pool as fp8 rows (the cache's bf16 rows converted by csa_index_rows_fp8)."""
    import torch
    cfg = csa_synth.CONFIGS[5]
    cap = (cfg.ctx + cfg.T) // cfg.ratio + 8
    host = csa_synth.synth_cache(cfg, cap)
    d = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                  topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps, index_fp8=index_fp8)

    def comp(c):
        return csa.Compressor(wkv=d(c.wkv), wgate=d(c.wgate), ape=d(c.ape), norm_w=d(c.norm_w), d=c.d)
    ca, ci = comp(csa_synth.compressor(cfg, "attn")), comp(csa_synth.compressor(cfg, "index"))
    snap = {k: d(getattr(host, k)) for k in ("pool", "ikeys", "window", "front_attn", "front_index", "n_rows", "pos")}
    if index_fp8:
        rows = torch.empty(snap["ikeys"].shape[:-1] + (csa.FP8_ROW_BYTES,), dtype=torch.uint8, device=dev)
        csa.index_rows_fp8(L, snap["ikeys"], rows)
        snap["ikeys"] = rows
    st = {k: v.clone() for k, v in snap.items()}
    n_i = st["n_rows"].clone()
    ch = csa_synth.chunk_inputs(cfg)
    x, q, kv, iq, iw = d(ch.x), d(ch.q), d(ch.kv), d(ch.iq), d(ch.iw)
    sink, invf = d(csa_synth.sinks(cfg)), d(csa_synth.inv_freq(cfg))
    out = torch.empty(cfg.T, cfg.H, cfg.D, dtype=cfg.storage, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    u8 = lambda n: torch.empty(max(n, 256), dtype=torch.uint8, device=dev)  # noqa: E731
    ws_c = u8(csa.workspace_size(L, csa.OP_COMPRESS, 1, cfg.T, cap))
    ws_p = u8(csa.workspace_size(L, csa.OP_ATTEND_PREFILL, 1, cfg.T, cap))
    times = []
    for r in range(repeats + 1):
        for k in st:
            st[k].copy_(snap[k])
        n_i.copy_(snap["n_rows"])
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        csa.compress_append(L, ca, x, st["pos"], st["front_attn"], st["pool"], st["n_rows"], invf, ws=ws_c, err=err)
        csa.compress_append(L, ci, x, st["pos"], st["front_index"], st["ikeys"], n_i, invf, ws=ws_c, err=err)
        csa.attend_prefill_chunk(L, q, kv, iq, iw, sink, cfg.ctx, st["window"][0], st["pool"][0], st["ikeys"][0],
                                 st["n_rows"], invf, out, ws=ws_p, err=err)
        e1.record()
        torch.cuda.synchronize()
        if r > 0:
            times.append(e0.elapsed_time(e1))
    assert err.item() == 0
    ms = statistics.median(times)
    nvis_sum = sum(min((cfg.ctx + cfg.T) // 4, (cfg.ctx + i + 1) // 4) for i in range(cfg.T))
    flops = (nvis_sum * cfg.Hi * cfg.Di * 2 + cfg.T * (cfg.topk + cfg.W) * cfg.H * cfg.D * 4 +
             cfg.T * cfg.X * (2 * 2 * (cfg.D + cfg.Di)) * 2)
    _, tflops, _ = _peaks()
    return {"workload": cfg.name + (" fp8-index-keys" if index_fp8 else ""), "tok_per_s": round(cfg.T / (ms / 1e3), 1),
            "ms_per_chunk": round(ms, 4), "ms_per_chunk_p10_p50_p90": [round(x, 4) for x in _percentiles(times)],
            "algorithmic_tflop": round(flops / 1e12, 4),
            "tensor_frac": round(flops / (ms / 1e3) / 1e12 / tflops, 4), "repeats": repeats,
            "tensor_frac_note": ("the same bf16-equivalent flop count and bf16 peak; the index products here are "
                                 "e4m3 (twice the bf16 rate)") if index_fp8 else None,
            "dram_traffic_bytes": None if index_fp8 else _traffic("prefill_chunk_bytes", 1)}


# A ragged prefill batch: eight requests' chunks (4096 tokens in all) at contexts from 2K to 64K, packed.
VARLEN_SPECS = [(65536, 256), (32768, 512), (16384, 384), (8192, 640), (4096, 128), (49152, 1024), (24576, 768),
                (2048, 384)]


def run_prefill_varlen(csa, csa_synth, dev, flush, repeats: int) -> dict:
    """csa_compress_append_varlen (both pools) + csa_attend_prefill_varlen on VARLEN_SPECS (Flash shapes, each
    sequence's cache drawn from its own seeded stream), timed from a restored snapshot with the L2 flushed."""
    import torch
    cfg = csa_synth.CONFIGS[5]
    B = len(VARLEN_SPECS)
    lens = [t for _, t in VARLEN_SPECS]
    N, T_max = sum(lens), max(lens)
    cap = max(c + t for c, t in VARLEN_SPECS) // cfg.ratio + 8
    parts = [csa_synth.synth_cache(cfg.replace(cid=cfg.cid + 300 + b), cap, B=1, ctx=c)
             for b, (c, _) in enumerate(VARLEN_SPECS)]
    d = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    snap = {k: d(torch.cat([getattr(p, k) for p in parts]))
            for k in ("pool", "ikeys", "window", "front_attn", "front_index", "n_rows", "pos")}
    del parts
    L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                  topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps)

    def comp(c):
        return csa.Compressor(wkv=d(c.wkv), wgate=d(c.wgate), ape=d(c.ape), norm_w=d(c.norm_w), d=c.d)
    ca, ci = comp(csa_synth.compressor(cfg, "attn")), comp(csa_synth.compressor(cfg, "index"))
    chunks = [csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 400 + b), t) for b, t in enumerate(lens)]
    x = d(torch.cat([ch.x[0] for ch in chunks]))
    q, kv, iq, iw = (d(torch.cat([getattr(ch, f) for ch in chunks])) for f in ("q", "kv", "iq", "iw"))
    cu = torch.tensor([0] + [sum(lens[:i + 1]) for i in range(B)], dtype=torch.int32, device=dev)
    sink, invf = d(csa_synth.sinks(cfg)), d(csa_synth.inv_freq(cfg))
    st = {k: v.clone() for k, v in snap.items()}
    n_i = st["n_rows"].clone()
    out = torch.empty(N, cfg.H, cfg.D, dtype=cfg.storage, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    u8 = lambda n: torch.empty(max(n, 256), dtype=torch.uint8, device=dev)  # noqa: E731
    ws_c = u8(csa.workspace_size(L, csa.OP_COMPRESS_VARLEN, B, N, cap))
    ws_p = u8(csa.workspace_size(L, csa.OP_ATTEND_PREFILL_VARLEN, B, N, cap))
    times = []
    for r in range(repeats + 1):
        for k in st:
            st[k].copy_(snap[k])
        n_i.copy_(snap["n_rows"])
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        csa.compress_append_varlen(L, ca, x, cu, T_max, st["pos"], st["front_attn"], st["pool"], st["n_rows"], invf,
                                   ws=ws_c, err=err)
        csa.compress_append_varlen(L, ci, x, cu, T_max, st["pos"], st["front_index"], st["ikeys"], n_i, invf,
                                   ws=ws_c, err=err)
        csa.attend_prefill_varlen(L, q, kv, iq, iw, sink, cu, T_max, st["pos"], st["window"], st["pool"],
                                  st["ikeys"], st["n_rows"], invf, out, ws=ws_p, err=err)
        e1.record()
        torch.cuda.synchronize()
        if r > 0:
            times.append(e0.elapsed_time(e1))
    assert err.item() == 0
    ms = statistics.median(times)
    flops = N * cfg.X * (2 * 2 * (cfg.D + cfg.Di)) * 2
    for c, t in VARLEN_SPECS:
        for i in range(t):
            nvis = min((c + t) // cfg.ratio, (c + i + 1) // cfg.ratio)
            flops += nvis * cfg.Hi * cfg.Di * 2 + (min(nvis, cfg.topk) + min(cfg.W, c + i + 1)) * cfg.H * cfg.D * 4
    _, tflops, _ = _peaks()
    return {"workload": "flash-prefill-varlen-b8-n4096", "requests": [{"context": c, "tokens": t}
                                                                      for c, t in VARLEN_SPECS],
            "tok_per_s": round(N / (ms / 1e3), 1), "ms_per_batch": round(ms, 4),
            "ms_per_batch_p10_p50_p90": [round(x, 4) for x in _percentiles(times)],
            "algorithmic_tflop": round(flops / 1e12, 4),
            "tensor_frac": round(flops / (ms / 1e3) / 1e12 / tflops, 4), "repeats": repeats,
            "calls": "csa_compress_append_varlen x 2 (attention and index pools), csa_attend_prefill_varlen"}


def cpu_baseline(cfg, budget_s: float) -> dict:
    """The float64 oracle on this host, on bounded samples of the headline workload: one core stepping one of the
    32 sequences (the primary figure, scaled x32 to a layer-step), and every core at once (one process per core,
    the 32 sequences split between them, whole layer-steps)."""
    info = cpu_info()
    one = run_oracle_processes(3, [[0]], 1, 400, budget_s)
    per_seq = statistics.mean(one["step_s"])
    P = max(1, min(info["nproc"] or 1, cfg.B))
    groups = [list(range(cfg.B))[k::P] for k in range(P)]
    allc = run_oracle_processes(3, groups, 1, 40, budget_s / 2)
    all_step = statistics.mean(allc["step_s"])
    return {"value": round(1.0 / (per_seq * cfg.B), 5), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"1 of {cfg.B} sequences x {one['steps']} decode steps of the same workload (after one "
                      f"untimed step), float64 numpy oracle, single-threaded BLAS; per-layer-step time = {cfg.B} x "
                      f"the per-sequence time ({1e3 * per_seq:.2f} ms)",
            "nproc": info["nproc"], "cpu_model": info["cpu_model"], "arch": info["arch"],
            "all_cores": {"value": round(1.0 / all_step, 5), "unit": UNIT, "cores": P,
                          "sample": f"all {cfg.B} sequences x {allc['steps']} layer-steps (after one untimed), "
                                    f"{P} processes of single-threaded BLAS, each stepping {cfg.B // P}-"
                                    f"{-(-cfg.B // P)} sequences; a layer-step = the slowest process's step",
                          "ms_per_layer_step": round(1e3 * all_step, 3)}}


# ----------------------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    """The reference arm: the float64 CPU oracle on the host cores, on the same workload (config 3, B = 32): W
    untimed and K timed layer-steps, each advancing all 32 sequences by one token, the sequences split over one
    single-threaded process per core (up to 32).  Under torchrun only rank 0 runs it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import csa_synth
    cfg = csa_synth.CONFIGS[3]
    info = cpu_info()
    P = max(1, min(info["nproc"] or 1, cfg.B))
    groups = [list(range(cfg.B))[k::P] for k in range(P)]
    r = run_oracle_processes(3, groups, args.warmup, args.steps, 3600.0)
    step_s = r["step_s"]
    ms = 1e3 * statistics.mean(step_s)
    value = 1e3 / ms
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
        "steps": r["steps"], "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "global_batch": cfg.B, "seq_len": cfg.ctx,
                   "step": f"one decode layer-step: all {cfg.B} sequences advance one token through the four calls",
                   "ms_per_step_p10_p50_p90": [round(1e3 * x, 3) for x in _percentiles(step_s)]},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": P, "kind": "oracle",
                         "sample": f"all {cfg.B} sequences x {r['steps']} layer-steps after {args.warmup} untimed, "
                                   f"float64 numpy oracle, {P} single-threaded processes (the sequences split "
                                   "between them); a layer-step = the slowest process's step",
                         "nproc": info["nproc"], "cpu_model": info["cpu_model"], "arch": info["arch"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _percentiles(xs, qs=(10, 50, 90)):
    v = sorted(xs)
    if not v:
        return [None for _ in qs]
    out = []
    for q in qs:
        k = (len(v) - 1) * q / 100.0
        lo, hi = int(k), min(int(k) + 1, len(v) - 1)
        out.append(v[lo] + (v[hi] - v[lo]) * (k - lo))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--prefill-repeats", type=int, default=3)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the config-2 (B = 1, 8K) and config-4 (ratio 128, B = 16, 256K) decode lines")
    ap.add_argument("--eager", action="store_true", help="launch kernels one by one instead of CUDA graphs")
    ap.add_argument("--index-fp8", action="store_true",
                    help="the headline workload with fp8 index rows (diagnostic and profiling; the default line and "
                         "its other_decode_workloads entry are unchanged)")
    ap.add_argument("--layers", type=int, default=8,
                    help="layers per model step (each its own weights and caches), one CUDA graph per step")
    ap.add_argument("--two-streams", action="store_true",
                    help="the two compress calls separately, the attention pool's on a side stream")
    ap.add_argument("--indexer", choices=["serial", "overlap"], default="serial",
                    help="after csa_compress_append_pair on the same stream: csa_index_topk (serial) or "
                         "csa_index_topk_overlapped without an event, whose scan runs beside the compress kernels")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--oracle-sample", nargs=5, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the 4096-token prefill chunk (for profiling its kernels); prints its record")
    ap.add_argument("--verify-only", action="store_true",
                    help="time only the verify-block model step (B 32, T 4; for profiling its kernels); prints its record")
    args = ap.parse_args()
    if args.verify_only:
        import torch
        import csa_synth
        import deepseek_v4_compressed_csa_gb300 as csa
        dev = torch.device("cuda", 0)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        print(json.dumps(verify_line(csa, csa_synth, dev, flush, args.steps, args.warmup, args.layers)))
        return
    if args.prefill_only:
        import torch
        import csa_synth
        import deepseek_v4_compressed_csa_gb300 as csa
        dev = torch.device("cuda", 0)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        print(json.dumps(run_prefill(csa, csa_synth, dev, flush, args.prefill_repeats)))
        print(json.dumps(run_prefill_varlen(csa, csa_synth, dev, flush, args.prefill_repeats)))
        print(json.dumps(run_prefill(csa, csa_synth, dev, flush, args.prefill_repeats, index_fp8=True)))
        return
    if args.oracle_sample:
        cid, seqs, warmup, steps, budget = args.oracle_sample
        print(json.dumps(oracle_sample(int(cid), [int(b) for b in seqs.split(",")], int(warmup), int(steps),
                                       float(budget))))
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
