#!/usr/bin/env python
"""Benchmark of the mixed sliding/global attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
    python bench.py --tp --workload 12b_decode      (tensor-parallel heads, one rank per GPU)

A step is one pass of the hot path over every layer of the workload: append of the new K/V
rows (owner layers), owner resolution, attention (decode: split-K partials + combine; prefill:
one pass) per layer. Steps are captured as CUDA graphs and replayed; the timed region is
bracketed by a barrier and device synchronisation, timed with CUDA events, max over ranks.

Default workload: batched ragged decode on 12B-shaped layers (batch 64, lengths uniform in
[128, 16384], 48 layer-steps), where the decode bandwidth the metric asks for is reachable;
the line also carries the prefill bucket (batch 4, 512 tokens onto a 3584-token prefix) as the
metric's second half, and the two batch-1 decode configurations.

Inputs are seeded synthetic N(0, 1) values drawn on the device (torch's CUDA generator), bf16.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "decode-attn HBM GB/s (% of 8 TB/s); prefill-attn bf16 TFLOP/s (% of peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
RAGGED_PHYS_LAYERS = 6   # distinct caches for 48 ragged layer-steps (one 5:1 period)
SOFTCAP_EXAMPLE = 50.0   # attention-logit soft-cap used to time the soft-capped entry point
BUCKET_REAL_EXAMPLE = [512, 384, 256, 128]   # real rows per sequence of the padded bucket timed
RING_EXAMPLE = 1024     # ring slots of the sliding layers' caches (the 12B window)
PAGE_EXAMPLE = 256      # keys per page of the paged pools

# dram bytes (read + write) per algorithmic byte of the decode row kernel, from one ncu capture
# of each launch kind (a batch-40 sliding layer in the unsplit launch configuration of the
# batch-64 one, and a batch-64 global layer); used only while the kernel sources hash to the
# recorded value
NCU_DECODE_TRAFFIC = {"source_sha1": "6045a0b6c038e3b758a6b23a20925842b6f34c5c",
                      "per_algorithmic_byte": {"sliding": 1.0153, "global": 1.0349}}
# dram bytes (read + write) per launch of the prefill pair kernels on the default prefill
# workload (batch 4, 512 tokens onto 3584), from one ncu capture of a sliding and a global
# layer; used only for that workload and while the kernel sources hash to the recorded value
NCU_PREFILL_TRAFFIC = {"source_sha1": "31b5a94eca65cdc6c26b052c2726d4b1edfad0c9", "batch": 4, "n_new": 512,
                       "ctx": 4096, "bytes_per_launch": {"sliding": 73969664 + 2414592,
                                                         "global": 50567936 + 282368}}


# ---------------------------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------------------------
def n_read(spec, ctx):
    return min(ctx, spec.window) if spec.kind == synth.SLIDING else ctx


def decode_bytes(w, l):
    """Bytes one decode launch of layer l must move: the K (and V) rows it attends, q, out."""
    s = w.layers[l]
    kv = sum(s.n_kv * n_read(s, c) * s.head_dim * 2 * (1 if s.k_eq_v else 2) for c in w.ctx_lens)
    return kv + 2 * w.batch * s.n_q * s.head_dim * 2


def append_bytes(w, l):
    s = w.layers[l]
    if not w.is_owner(l):
        return 0
    return 2 * w.batch * w.n_new * s.n_kv * s.head_dim * 2 * (1 if s.k_eq_v else 2)


def prefill_flops(w, l, n_real=None):
    """4 d n_q per attended (query, key) pair: QK^T and PV multiply-adds (real rows only for a
    padded bucket: they sit where the bucket's first n_real rows would)."""
    s = w.layers[l]
    pairs = 0
    for b, c in enumerate(w.ctx_lens):
        for i in range(w.n_new if n_real is None else n_real[b]):
            p = c - w.n_new + i
            pairs += min(p + 1, s.window) if s.kind == synth.SLIDING else p + 1
    return 4 * s.head_dim * s.n_q * pairs


def step_work(w, n_real=None):
    if w.n_new == 1:
        return sum(decode_bytes(w, l) + append_bytes(w, l) for l in range(w.n_layers))
    return sum(prefill_flops(w, l, n_real) for l in range(w.n_layers))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# the sources (and every header they include) of the kernels whose ncu traffic is recorded
DECODE_SOURCES = ("rows_attn.cu", "common.cuh", "tc.cuh", "tmap.h", "attn_internal.h")
PREFILL_SOURCES = ("prefill_pair.cu", "common.cuh", "tc.cuh", "tmap.h", "attn_internal.h")


def prefill_traffic(w, softcap=None, n_real=None):
    """DRAM bytes per attention launch of each layer kind from the recorded ncu capture, or
    None where it does not apply (another workload, the soft-capped or padded entry point, or
    kernel sources that no longer hash to the captured version)."""
    tr = NCU_PREFILL_TRAFFIC
    if (tr["source_sha1"] is None or softcap is not None or n_real is not None or
            tr["source_sha1"] != kernel_source_sha1(PREFILL_SOURCES) or
            (w.batch, w.n_new, max(w.ctx_lens)) != (tr["batch"], tr["n_new"], tr["ctx"])):
        return None
    return tr["bytes_per_launch"]


def kernel_source_sha1(names=DECODE_SOURCES):
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "mixed_sliding_global_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 20 ms; only those stamped inside [start(), stop()] count (the
    sampler is running, its first line read, before start() returns)."""
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.first = ""
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = self.proc.stdout.readline()   # sampling has begun
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.time()

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        t1 = time.time()
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in (self.first + out).strip().splitlines() if r.count(",") >= 9]
        mine = [r for r in rows if self.uuid and self.uuid.replace("GPU-", "") in r[1]] or rows
        inside = [r for r in mine if (lambda t: t is not None and self.t0 <= t <= t1)(self._stamp(r[0]))]
        use = inside or mine
        if not use:
            return None
        sm = [float(r[2]) for r in use if r[2].strip().replace(".", "").isdigit()]
        mx = [float(r[3]) for r in use if r[3].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[6:10]) if "Active" in v
                          and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "samples_around": len(mine)}


# ---------------------------------------------------------------------------------------------
# device state of a workload (seeded values drawn on the device)
# ---------------------------------------------------------------------------------------------
class DeviceState:
    def __init__(self, w, seed, device, phys_of_layer=None, softcap=None, n_real=None,
                 fused=False, ring=None, paged=None):
        import mixed_sliding_global_gb300 as g
        self.g, self.w, self.device = g, w, device
        self.softcap = softcap
        self.fused = fused  # decode: append inside the attention launch (one launch per layer)
        self.ring = ring    # sliding layers' caches: rings of this many slots (None: linear)
        # paged pools with pages of this many keys (None: one linear cache per sequence): a
        # global layer's pool holds the pages of positions [0, len), a sliding layer's only the
        # pages from its window start; pages are handed out in a seeded shuffled order
        self.paged = paged
        self.tables = {}
        # padded prefill bucket: real rows per sequence (the rest pad the bucket to n_new)
        self.n_real = None if n_real is None else torch.tensor(n_real, dtype=torch.int32,
                                                                device=device)
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        self.gen = gen
        n, B, cap = w.n_layers, w.batch, w.capacity
        phys = phys_of_layer or list(range(n))
        ctx = torch.tensor(w.ctx_lens, dtype=torch.int32)
        self.write_pos = (ctx - w.n_new).to(device)
        self.seq_lens = ctx.to(device) if n_real is None else \
            (ctx - w.n_new + torch.tensor(n_real, dtype=torch.int32)).to(device)
        kc_phys, vc_phys = {}, {}
        self.kc, self.vc = [None] * n, [None] * n
        self.q, self.k_new, self.v_new, self.out = [None] * n, [None] * n, [None] * n, [None] * n
        dt = synth.TORCH_DTYPE[w.dtype]
        for l, s in enumerate(w.layers):
            if w.is_owner(l):
                p = phys[l]
                if p not in kc_phys:
                    if paged:
                        kc_phys[p], vc_phys[p] = self._pools(s, B, dt)
                    elif ring and s.kind == synth.SLIDING:
                        # a ring holds the last `ring` tokens: every slot is a real past token
                        kc_phys[p] = self._randn((B, s.n_kv, ring, s.head_dim), dt)
                        vc_phys[p] = None if s.k_eq_v else self._randn((B, s.n_kv, ring, s.head_dim), dt)
                    else:
                        kc_phys[p] = self._cache(s, B, cap, dt)
                        vc_phys[p] = None if s.k_eq_v else self._cache(s, B, cap, dt)
                self.kc[l], self.vc[l] = kc_phys[p], vc_phys[p]
                self.k_new[l] = self._randn((B, w.n_new, s.n_kv, s.head_dim), dt)
                if not s.k_eq_v:
                    self.v_new[l] = self._randn((B, w.n_new, s.n_kv, s.head_dim), dt)
            self.q[l] = self._randn((B, w.n_new, s.n_q, s.head_dim), dt)
            self.out[l] = torch.empty_like(self.q[l])
        msl = max(w.ctx_lens)
        wsf = g.gemma_attn_workspace_size_paged if paged else g.gemma_attn_workspace_size
        ws = max(wsf(B, self.kind_of(s), s.window, s.n_q, s.n_kv, s.head_dim, msl, w.n_new)
                 for s in w.layers)
        self.ws = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
        self.max_seq_len = msl
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.cache_bytes = sum(t.numel() * t.element_size() for t in
                               list(kc_phys.values()) + [v for v in vc_phys.values() if v is not None])

    def _randn(self, shape, dt):
        return torch.randn(shape, generator=self.gen, device=self.device, dtype=torch.float32).to(dt)

    def _cache(self, s, B, cap, dt):
        """Cache with seeded values in the rows this step's attention reads; the other rows are
        never read and stay uninitialised."""
        c = torch.empty((B, s.n_kv, cap, s.head_dim), dtype=dt, device=self.device)
        for b, ctx in enumerate(self.w.ctx_lens):
            lo = synth.needed_row_lo(s, ctx, self.w.n_new)
            c[b, :, lo:ctx].copy_(self._randn((s.n_kv, ctx - lo, s.head_dim), dt))
        return c

    def _pools(self, s, B, dt):
        """K (and V) pools of one owner layer and the block table of its kind."""
        P, w = self.paged, self.w
        max_pages = -(-w.capacity // P)
        if s.kind not in self.tables:
            first = []
            for ctx in w.ctx_lens:
                lo = 0 if s.kind == synth.GLOBAL else max(0, ctx - s.window) & ~31
                first.append(lo // P)
            need = [-(-ctx // P) - f for ctx, f in zip(w.ctx_lens, first)]
            n_pages = sum(need)
            g = torch.Generator().manual_seed(4242 + s.kind)
            perm = torch.randperm(n_pages, generator=g)
            table = torch.zeros((B, max_pages), dtype=torch.int32)   # unread entries: page 0
            k = 0
            for b in range(B):
                table[b, first[b]:first[b] + need[b]] = perm[k:k + need[b]].to(torch.int32)
                k += need[b]
            self.tables[s.kind] = (table.to(self.device), n_pages)
        n_pages = self.tables[s.kind][1]
        kp = self._randn((n_pages, s.n_kv, P, s.head_dim), dt)
        vp = None if s.k_eq_v else self._randn((n_pages, s.n_kv, P, s.head_dim), dt)
        return kp, vp

    def kind_of(self, s):
        return self.g.GEMMA_SLIDING_RING if self.ring and s.kind == synth.SLIDING else s.kind

    def layer_call(self, l):
        w, s = self.w, self.w.layers[l]
        kw = dict(kind=self.kind_of(s), window=s.window, n_kv=s.n_kv, k_eq_v=s.k_eq_v, scale=w.scale(l),
                  workspace=self.ws, device_error=self.err)
        if self.softcap is not None:
            self.g.gemma_attn_softcap(self.out[l], self.q[l], self.kc, self.vc, w.owner_map, l,
                                      self.seq_lens, self.max_seq_len, softcap=self.softcap, **kw)
            return
        if self.n_real is not None:
            self.g.gemma_attn_prefill_bucket(self.out[l], self.q[l], self.kc, self.vc,
                                             w.owner_map, l, self.seq_lens, self.n_real,
                                             self.max_seq_len, **kw)
            return
        fn = self.g.gemma_attn_decode if w.n_new == 1 else self.g.gemma_attn_prefill
        fn(self.out[l], self.q[l], self.kc, self.vc, w.owner_map, l, self.seq_lens,
           self.max_seq_len, **kw)

    def append_call(self, l):
        s = self.w.layers[l]
        if self.ring and s.kind == synth.SLIDING:
            self.g.gemma_kv_append_ring(self.kc, self.vc, self.w.owner_map, l, self.k_new[l],
                                        self.v_new[l], self.write_pos, k_eq_v=s.k_eq_v,
                                        device_error=self.err)
            return
        if self.n_real is not None:
            self.g.gemma_kv_append_bucket(self.kc, self.vc, self.w.owner_map, l, self.k_new[l],
                                          self.v_new[l], self.write_pos, self.n_real,
                                          k_eq_v=s.k_eq_v, device_error=self.err)
            return
        self.g.gemma_kv_append(self.kc, self.vc, self.w.owner_map, l, self.k_new[l],
                               self.v_new[l], self.write_pos, k_eq_v=s.k_eq_v,
                               device_error=self.err)

    def fused_call(self, l):
        w, s = self.w, self.w.layers[l]
        o = w.owner_map[l]
        if self.paged:
            self.g.gemma_attn_paged(self.out[l], self.q[l], self.kc, self.vc, w.owner_map, l,
                                    self.seq_lens, self.tables[s.kind][0], self.max_seq_len,
                                    kind=s.kind, window=s.window, n_kv=s.n_kv, k_eq_v=s.k_eq_v,
                                    scale=w.scale(l), k_new=self.k_new[o], v_new=self.v_new[o],
                                    write_pos=self.write_pos, workspace=self.ws,
                                    device_error=self.err)
            return
        self.g.gemma_attn_decode_append(self.out[l], self.q[l], self.kc, self.vc, w.owner_map, l,
                                        self.k_new[o], self.v_new[o], self.write_pos,
                                        self.seq_lens, self.max_seq_len, kind=self.kind_of(s),
                                        window=s.window, n_kv=s.n_kv, k_eq_v=s.k_eq_v,
                                        scale=w.scale(l), workspace=self.ws,
                                        device_error=self.err)

    def layer_step(self, l):
        """Layer l's launches of a step (append and attention, or the fused launch)."""
        if self.fused:
            self.fused_call(l)
            return
        if self.w.is_owner(l):
            self.append_call(l)
        self.layer_call(l)

    def step(self, events=None):
        for l in range(self.w.n_layers):
            if self.fused:
                if events is not None:
                    events[l][0].record()
                self.fused_call(l)
                if events is not None:
                    events[l][1].record()
                continue
            if self.w.is_owner(l):
                self.append_call(l)
            if events is not None:
                events[l][0].record()
            self.layer_call(l)
            if events is not None:
                events[l][1].record()

    def launches_per_step(self):
        n = 0
        w = self.w
        for l, s in enumerate(w.layers):
            n += 1 if w.is_owner(l) and not self.fused else 0
            n += 1
            wsf = self.g.gemma_attn_workspace_size_paged if self.paged else \
                self.g.gemma_attn_workspace_size
            if w.n_new == 1 and wsf(w.batch, s.kind, s.window, s.n_q, s.n_kv, s.head_dim,
                                    self.max_seq_len, 1) > 0:
                n += 1  # split combine
        return n


def make_event(external):
    try:
        return torch.cuda.Event(enable_timing=True, external=external)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def capture(state, events=None):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        state.step(events)
    return g


# ---------------------------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The slowest rank's time: the job's step time (no data-path collective; only this)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_value(work_per_rank, world, ms_max, scale):
    """Whole-job throughput: every rank processes its own replica of the workload (weak
    scaling), so the job moves world x work in the slowest rank's time."""
    return world * work_per_rank / (ms_max * 1e-3) / scale


def build_library(world, local):
    from mixed_sliding_global_gb300 import _build
    if local == 0 and not _build.up_to_date():
        _build.build()
    barrier(world)
    import mixed_sliding_global_gb300 as g
    g.library(build_if_missing=False)


def _slice(w, offset, nl):
    """Layers [offset, offset + nl) of a model with its own caches (profiling captures)."""
    return synth.Workload(w.name, w.layers[offset:offset + nl], list(range(nl)), w.batch, w.dtype,
                          w.n_new, w.ctx_lens, w.capacity)


def workload(name, batch=None, layers=None, offset=0, max_len=None):
    if name == "ragged_decode":
        nl = layers or 48
        if max_len:   # shorter sequences and a smaller cache (profiling captures only)
            w = synth.ragged_decode(n_layers=offset + nl, batch=batch or 64,
                                    capacity=-(-(max_len + 1) // 64) * 64, max_len=max_len)
        else:
            w = synth.ragged_decode(n_layers=offset + nl, batch=batch or 64)
        if offset:
            w = _slice(w, offset, nl)
        return w, [(offset + l) % RAGGED_PHYS_LAYERS for l in range(nl)]
    if name == "e4b_decode":
        w = synth.e4b_decode()
    elif name == "12b_decode":
        w = synth.b12_decode()
    elif name == "prefill":
        w = synth.prefill_12b(batch=batch or 4)
    else:
        raise ValueError(name)
    if layers or offset:
        w = _slice(w, offset, layers or (w.n_layers - offset))
    return w, None


def timed_graph_run(w, phys, steps, warmup, device, world, per_launch=False, rotations=1,
                    softcap=None, n_real=None, fused=False, ring=None, paged=None, min_ms=None):
    """Capture one graph per input copy (rotating over `rotations` independent copies) and
    time `steps` replays after `warmup` replays; with min_ms, as many more steps as make the
    timed region last about min_ms (so that the clock samples fall inside it; the returned
    info holds the count). Returns step time and, with per_launch, the
    mean duration of each layer's attention launch, taken in a second pass of `steps` replays
    of graphs with an event pair around every launch (event nodes cost a few microseconds
    each and break the overlap of consecutive launches, so the step time is taken without
    them)."""
    states = [DeviceState(w, 1234 + 17 * r, device, phys, softcap, n_real, fused, ring, paged)
              for r in range(rotations)]
    for st in states:   # eager pass: sets kernel attributes, checks the error word
        st.step()
    torch.cuda.synchronize()
    for st in states:
        if st.err.item() != 0:
            raise RuntimeError(f"device error word {st.err.item()} in the eager pass")
    graphs = [capture(st) for st in states]
    steps_asked = steps
    torch.cuda.synchronize()
    for k in range(warmup):
        graphs[k % rotations].replay()
    if min_ms is not None:
        c0, c1 = make_event(False), make_event(False)
        c0.record()
        for k in range(rotations):
            graphs[k].replay()
        c1.record()
        torch.cuda.synchronize()
        steps = max(steps, int(min_ms / max(c0.elapsed_time(c1) / rotations, 1e-3)) + 1)
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0, t1 = make_event(False), make_event(False)
    t0.record()
    for k in range(steps):
        graphs[k % rotations].replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    del graphs
    launch_ms = None
    if per_launch:
        n_ev = steps_asked
        ev = [[(make_event(True), make_event(True)) for _ in range(w.n_layers)]
              for _ in range(n_ev)]
        eg = [capture(states[k % rotations], ev[k]) for k in range(n_ev)]
        for k in range(min(warmup, n_ev)):
            eg[k].replay()
        torch.cuda.synchronize()
        for k in range(n_ev):
            eg[k].replay()
        torch.cuda.synchronize()
        launch_ms = [sum(ev[k][l][0].elapsed_time(ev[k][l][1]) for k in range(n_ev)) / n_ev
                     for l in range(w.n_layers)]
        del eg
    for st in states:
        if st.err.item() != 0:
            raise RuntimeError(f"device error word {st.err.item()} after the timed region")
    info = {"launches_per_step": states[0].launches_per_step(),
            "cache_bytes": sum(s.cache_bytes for s in states), "steps": steps}
    del states
    torch.cuda.empty_cache()
    return ms, launch_ms, clk, info


def logit_run(steps, warmup, device, world, batch=64, rotations=4, min_ms=None):
    """The greedy step after the LM head: final-logit soft-cap (cap 30, written out) and argmax
    of [64][262144] bf16 logits, rotating over `rotations` input/output pairs (together larger
    than L2), each call captured in one graph. Returns time per call and launches per call."""
    import mixed_sliding_global_gb300 as gemma
    V = synth.VOCAB
    xs = [synth.logits(batch, V, seed=r).to(device) for r in range(rotations)]
    outs = [torch.empty_like(x) for x in xs]
    idx = torch.empty(batch, dtype=torch.int32, device=device)
    ws = torch.zeros(max(gemma.gemma_logit_workspace_size(batch, V), 16), dtype=torch.uint8,
                     device=device)

    def call(r):
        gemma.gemma_logit_softcap_argmax(xs[r], synth.LOGIT_SOFTCAP, idx, outs[r], ws)

    for r in range(rotations):
        call(r)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in range(rotations):
            call(r)
    for _ in range(warmup):
        g.replay()
    if min_ms is not None:
        # as many replays as make the timed region last about min_ms (clock samples inside)
        c0, c1 = make_event(False), make_event(False)
        c0.record()
        g.replay()
        c1.record()
        torch.cuda.synchronize()
        steps = max(steps, int(min_ms / max(c0.elapsed_time(c1), 1e-3)) + 1)
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0, t1 = make_event(False), make_event(False)
    t0.record()
    for _ in range(steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / (steps * rotations)
    n_split = -(-gemma.gemma_logit_workspace_size(batch, V) // (8 * batch))
    bytes_per_call = batch * V * 2 * 2 + batch * 4
    del g, xs, outs
    torch.cuda.empty_cache()
    return ms, bytes_per_call, 2 if n_split > 1 else 1, clk, steps


def e2e_run(w, phys, steps, warmup, device, fused=False):
    """Same step through the public API, eager, with this step's inputs copied from pinned host
    memory and the outputs read back every step (the caches stay resident: they are state).
    The copies run on two copy streams beside the attention launches: layer l's inputs are
    copied while earlier layers compute, and its output is read back once its launch is done.
    Events order each buffer's copy against its use, within a step and across steps."""
    st = DeviceState(w, 4321, device, phys, fused=fused)
    n = w.n_layers
    host_in = []
    for l in range(n):
        pairs = []
        for name in ("q", "k_new", "v_new"):
            t = getattr(st, name)[l]
            if t is not None:
                pairs.append((t.cpu().pin_memory(), t))
        host_in.append(pairs)
    meta = [(st.seq_lens.cpu().pin_memory(), st.seq_lens),
            (st.write_pos.cpu().pin_memory(), st.write_pos)]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in st.out]
    bi = sum(h.numel() * h.element_size() for pairs in host_in for h, _ in pairs) + \
        sum(h.numel() * h.element_size() for h, _ in meta)
    bo = sum(h.numel() * h.element_size() for h in host_out)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    used = [None] * n   # layer l's launches of the previous step are done (its inputs are free)
    read = [None] * n   # layer l's output of the previous step has been read back

    def record(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def one(after=None):
        if after is not None:
            s_in.wait_event(after)   # the timed region's start
        with torch.cuda.stream(s_in):
            if used[n - 1] is not None:
                s_in.wait_event(used[n - 1])   # every layer of the previous step read the lengths
            for h, d in meta:
                d.copy_(h, non_blocking=True)
            in_ev = []
            for l in range(n):
                if used[l] is not None:
                    s_in.wait_event(used[l])
                for h, d in host_in[l]:
                    d.copy_(h, non_blocking=True)
                in_ev.append(record(s_in))
        for l in range(n):
            comp.wait_event(in_ev[l])
            if read[l] is not None:
                comp.wait_event(read[l])
            st.layer_step(l)
            used[l] = record(comp)
        with torch.cuda.stream(s_out):
            for l in range(n):
                s_out.wait_event(used[l])
                host_out[l].copy_(st.out[l], non_blocking=True)
                read[l] = record(s_out)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    t0, t1 = make_event(False), make_event(False)
    t0.record()
    for k in range(steps):
        one(t0 if k == 0 else None)
    comp.wait_stream(s_out)   # the last outputs are back on the host
    t1.record()
    torch.cuda.synchronize()
    if st.err.item() != 0:
        raise RuntimeError(f"device error word {st.err.item()} in the end-to-end run")
    ms = t0.elapsed_time(t1) / steps
    del st
    torch.cuda.empty_cache()
    return ms, bi, bo


def host_cores():
    """Cores this process may run on (the affinity mask), not the machine's total."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_task(orc, w, l, seq):
    """Seeded inputs of one (layer, sequence) pair, and a callable that runs the oracle on them
    (the append of the step's rows, then the attention). Returns (work, callable)."""
    hb = synth.layer_batch(w, l, [seq])
    one = synth.Workload(w.name, w.layers, w.owner_map, 1, w.dtype, w.n_new, [w.ctx_lens[seq]],
                         w.capacity)
    work = (decode_bytes(one, l) + append_bytes(one, l)) if w.n_new == 1 else prefill_flops(one, l)

    def run():
        kcs = [None] * w.n_layers
        vcs = [None] * w.n_layers
        kcs[l] = hb.k_cache
        orc.kv_append(kcs[l], hb.k_new, hb.write_pos.tolist())
        if hb.v_cache is not None:
            vcs[l] = hb.v_cache
            orc.kv_append(vcs[l], hb.v_new, hb.write_pos.tolist())
        orc.attention(w.layers, w.owner_map, l, kcs, vcs, hb.q, hb.seq_lens.tolist(), w.scale(l))
    return work, run


def oracle_sample(w, budget_s, layers_pick=None, threads=1):
    """Time the fp64 oracle (as it stands) on (layer, sequence) pairs of a sliding and a global
    layer until about budget_s seconds of wall time in the oracle; returns (algorithmic work
    done, seconds, description, threads). With threads > 1 the unchanged oracle runs on that
    many pairs at once (one pair per thread; the C oracle releases the interpreter while it
    computes): inputs are generated first, untimed, then the oracle calls of the round are
    timed together, wall clock."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import load_oracle
    orc = load_oracle()
    pick = layers_pick or [next(l for l, s in enumerate(w.layers) if s.kind == synth.SLIDING),
                           next(l for l, s in enumerate(w.layers) if s.kind == synth.GLOBAL)]
    pairs = [(l, seq) for seq in range(w.batch) for l in pick]
    work, secs, n_done, i = 0, 0.0, 0, 0
    max_pairs = 4 * len(pairs)   # at most four passes over the workload's pairs
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while secs < budget_s and n_done < max_pairs:
            batch = [pairs[(i + k) % len(pairs)] for k in range(threads)]
            i += threads
            tasks = list(ex.map(lambda pr: _oracle_task(orc, w, *pr), batch))
            t = time.perf_counter()
            list(ex.map(lambda wr: wr[1](), tasks))
            secs += time.perf_counter() - t
            work += sum(wr[0] for wr in tasks)
            n_done += len(tasks)
            del tasks
    how = "single thread" if threads == 1 else f"{threads} threads, one pair each at a time"
    desc = (f"oracle on layers {pick} (one sliding, one global), {n_done} layer-sequence pairs "
            f"of the workload ({how})")
    return work, secs, desc, threads


# ---------------------------------------------------------------------------------------------
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w, _ = workload(args.workload)
    unit = "GB/s" if w.n_new == 1 else "TFLOP/s"
    scale = 1e9 if w.n_new == 1 else 1e12
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_sample(w, 1e-9, threads=cores)
    work, secs = 0, 0.0
    for _ in range(args.steps):
        wk, s, desc, _ = oracle_sample(w, args.ref_budget, threads=cores)
        work += wk
        secs += s
    value = work / secs / scale
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": w.batch, "layers": w.n_layers},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_logits(args):
    """The greedy step after the LM head alone (final-logit soft-cap + argmax of [64][262144]
    bf16 logits), one JSON line; the default run reports it under `also`."""
    world, rank, local = dist_setup()
    build_library(world, local)
    device = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    ms, nbytes, launches, clk, lsteps = logit_run(args.steps, args.warmup, device, world)
    ms = max_over_ranks(ms, world)
    v = world * nbytes / (ms * 1e-3) / 1e9
    line = {"metric": "logit soft-cap + argmax HBM GB/s", "value": v, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "logits", "batch": 64,
                                            "vocab": synth.VOCAB, "softcap": synth.LOGIT_SOFTCAP},
            "roofline": {"bound": "hbm", "achieved": v / world, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": v / world / peaks["hbm_gbs"],
                         "bytes_per_call": nbytes, "peak_source": peak_src},
            "gpu_launches": launches * 4 * args.steps, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_tp(args):
    """Tensor-parallel decode, one rank per GPU: every rank holds its head shard of each layer
    (tp.RankStep: query heads split over the ranks, a KV head replicated where a layer has
    fewer than the ranks) and runs append + attention of every layer on it; the ranks exchange
    nothing inside the step. Strong scaling: the model and batch are fixed, the heads split.
    `value` counts the bytes all ranks move (replicated KV heads once per rank that reads
    them); `unsharded_bytes_per_step` is the same step on one GPU."""
    import dataclasses
    from mixed_sliding_global_gb300.tp import RankStep
    world, rank, local = dist_setup()
    build_library(world, local)
    device = torch.device("cuda", local)
    if args.workload not in ("e4b_decode", "12b_decode"):
        raise SystemExit("--tp times the batch-1 decode workloads (e4b_decode, 12b_decode)")
    w, _ = workload(args.workload)
    st = DeviceState(w, 1234, device)   # the whole model's inputs: same seed on every rank
    rs = RankStep(w.layers, w.owner_map, rank, world, device)
    for l in range(w.n_layers):
        if w.is_owner(l):
            rs.load_cache(l, st.kc[l], st.vc[l])
    loc = rs.local_inputs([(st.q[l], st.k_new[l], st.v_new[l], st.write_pos, st.seq_lens)
                           for l in range(w.n_layers)])
    msl = st.max_seq_len
    del st
    torch.cuda.empty_cache()
    outs = [torch.empty_like(x[0]) for x in loc]
    scales = [w.scale(l) for l in range(w.n_layers)]
    rs.run(loc, outs, scales, msl)   # eager pass: workspaces, kernel attributes, error word
    torch.cuda.synchronize()
    if rs.err.item() != 0:
        raise RuntimeError(f"device error word {rs.err.item()} in the eager pass")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rs.run(loc, outs, scales, msl)
    for _ in range(args.warmup):
        g.replay()
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0, t1 = make_event(False), make_event(False)
    t0.record()
    for _ in range(args.steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if rs.err.item() != 0:
        raise RuntimeError(f"device error word {rs.err.item()} after the timed region")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)

    import mixed_sliding_global_gb300 as gemma

    def shard_workload(r):
        from mixed_sliding_global_gb300.tp import head_shard
        ls = [dataclasses.replace(s, n_q=sh.n_q, n_kv=sh.n_kv) for s, sh in
              zip(w.layers, (head_shard(s.n_q, s.n_kv, r, world) for s in w.layers))]
        return synth.Workload(w.name, ls, w.owner_map, w.batch, w.dtype, w.n_new, w.ctx_lens,
                              w.capacity)
    total = sum(step_work(shard_workload(r)) for r in range(world))
    mine = shard_workload(rank)
    launches = 0
    for l, s in enumerate(mine.layers):
        launches += (1 if mine.is_owner(l) else 0) + 1
        launches += gemma.gemma_attn_workspace_size(w.batch, s.kind, s.window, s.n_q, s.n_kv,
                                                    s.head_dim, msl, 1) > 0
    line = {"metric": METRIC, "mode": "tensor-parallel decode", "value":
            total / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) drawn on the device, stored as bf16)",
            "config": {"workload": args.workload, "batch": w.batch, "layers": w.n_layers,
                       "ctx": max(w.ctx_lens), "parallelism": f"tp{world}",
                       "append": "separate launch", "l2": "inputs larger than L2"},
            "bytes_per_step_all_ranks": total, "unsharded_bytes_per_step": step_work(w),
            "gpu_launches": launches * args.steps, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_native(args):
    world, rank, local = dist_setup()
    build_library(world, local)
    device = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    w, phys = workload(args.workload, args.batch, args.layers, args.layer_offset, args.max_len)
    decode = w.n_new == 1
    unit = "GB/s" if decode else "TFLOP/s"
    scale = 1e9 if decode else 1e12
    work = step_work(w)
    fused_main = w.n_new == 1 and not args.two_launch and args.softcap is None
    ms, launch_ms, clk, info = timed_graph_run(w, phys, args.steps, args.warmup, device, world,
                                               per_launch=True, softcap=args.softcap,
                                               fused=fused_main)
    ms = max_over_ranks(ms, world)
    value = job_value(work, world, ms, scale)

    # roofline of the dominant kernel: the attention launch of the layer kind with the largest
    # share of time (rows_attn_bf16_kernel plus its split combine)
    if decode:
        per_bytes = [decode_bytes(w, l) for l in range(w.n_layers)]
        peak = peaks["hbm_gbs"]
        kinds = {}
        for kind, name in ((synth.SLIDING, "sliding"), (synth.GLOBAL, "global")):
            ls = [l for l, s in enumerate(w.layers) if s.kind == kind]
            if ls:
                kinds[name] = (sum(per_bytes[l] for l in ls), sum(launch_ms[l] for l in ls), len(ls),
                               w.layers[ls[0]].head_dim)
        dom = max(kinds, key=lambda k: kinds[k][1])
        b, t, n, d = kinds[dom]
        achieved = b / (t * 1e-3) / 1e9
        traffic = None
        if NCU_DECODE_TRAFFIC["source_sha1"] == kernel_source_sha1():
            traffic = NCU_DECODE_TRAFFIC["per_algorithmic_byte"][dom] * b / n
        import mixed_sliding_global_gb300 as gemma
        sd = next(s for s in w.layers if (s.kind == synth.SLIDING) == (dom == "sliding"))
        split = gemma.gemma_attn_workspace_size(w.batch, sd.kind, sd.window, sd.n_q, sd.n_kv,
                                                sd.head_dim, max(w.ctx_lens), 1) > 0
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": f"rows_attn_bf16_kernel<{d}>" +
                          (" + split combine" if split else " (one CTA per sequence and KV head)") +
                          f" ({dom} layers)",
                "algorithmic_bytes_per_launch": b / n, "launch_us": 1e3 * t / n,
                "peak_source": peak_src}
        for name, (bk, tk, nk, dk) in kinds.items():
            roof[name] = {"bytes_per_launch": bk / nk, "launch_us": 1e3 * tk / nk,
                          "achieved_gbs": bk / (tk * 1e-3) / 1e9,
                          "frac": bk / (tk * 1e-3) / 1e9 / peak}
        roof["all_layers"] = {"achieved_gbs": sum(per_bytes) / (sum(launch_ms) * 1e-3) / 1e9,
                              "frac": sum(per_bytes) / (sum(launch_ms) * 1e-3) / 1e9 / peak}
    else:
        per_flops = [prefill_flops(w, l) for l in range(w.n_layers)]
        achieved = sum(per_flops) / (sum(launch_ms) * 1e-3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "kernel": "attention launch (prefill)", "peak_source": peak_src + " sustained"}
        tr = prefill_traffic(w, args.softcap)
        traffic_ok = tr is not None
        n_launch, traffic_sum = 0, 0.0
        for kind, name in ((synth.SLIDING, "sliding"), (synth.GLOBAL, "global")):
            ls = [l for l, s in enumerate(w.layers) if s.kind == kind]
            if ls:
                f = sum(per_flops[l] for l in ls)
                t = sum(launch_ms[l] for l in ls)
                roof[name] = {"tflops": f / (t * 1e-3) / 1e12, "launch_us": 1e3 * t / len(ls),
                              "traffic": tr[name] if traffic_ok else None}
                if traffic_ok:
                    n_launch += len(ls)
                    traffic_sum += len(ls) * tr[name]
        # per attention launch of the step, averaged over its launches
        roof["traffic"] = traffic_sum / n_launch if n_launch else None

    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) drawn on the device, stored as bf16)",
            "config": {"workload": args.workload, "batch": w.batch, "layers": w.n_layers,
                       "n_new": w.n_new, "ctx": (f"uniform[129,{16384 if not args.max_len else args.max_len}+1]"
                                                 if args.workload == "ragged_decode"
                                                 else max(w.ctx_lens)),
                       "parallelism": f"dp{world}" if world > 1 else "single",
                       "l2": "inputs larger than L2 (each layer-step reads > 129 MB)"
                       if args.workload == "ragged_decode" else "inputs larger than L2",
                       "phys_caches": len(set(phys)) if phys else w.n_layers,
                       **({"softcap": args.softcap} if args.softcap is not None else {}),
                       "append": "inside the attention launch" if fused_main else
                                 "separate launch",
                       "cache_gb": info["cache_bytes"] / 1e9},
            "roofline": roof,
            "gpu_launches": info["launches_per_step"] * args.steps,
            "clocks": clk}

    if not args.quick:
        e2e_ms, bi, bo = e2e_run(w, phys, max(3, args.steps // 4), 2, device, fused_main)
        e2e_ms = max_over_ranks(e2e_ms, world)
        line["e2e"] = {"value": world * work / (e2e_ms * 1e-3) / scale, "unit": unit,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms}
        if rank == 0:
            # the oracle on all of this host's cores, and on one core
            cores = host_cores()
            wk, secs, desc, _ = oracle_sample(w, args.cpu_budget, threads=cores)
            wk1, secs1, desc1, _ = oracle_sample(w, args.cpu_budget / 2, threads=1)
            line["cpu_baseline"] = {"value": wk / secs / scale, "unit": unit, "cores": cores,
                                    "kind": "oracle", "sample": desc,
                                    "single_core": {"value": wk1 / secs1 / scale, "unit": unit,
                                                    "cores": 1, "sample": desc1}}
        # the other benchmark configurations, same contract, reported alongside
        also = {}
        # prefill_softcap: the prefill bucket through the soft-capped entry point (cap 50, an
        # example value: the pages name an attention soft-cap without its value)
        # prefill_bucket: the prefill bucket padded, real lengths 512/384/256/128 of 512 (the
        # TFLOP/s count the real rows' work only)
        # *_two_launch: the batch-1 decodes with a separate append launch per owner layer (the
        # plain rows append inside the attention launch)
        # ragged_decode_ring: the headline workload with its sliding layers' caches as rings of
        # 1024 slots (the window) instead of 16448 rows
        # ragged_decode_paged: the headline workload over paged pools of 256-key pages holding
        # only the pages the step reads (global: [0, len); sliding: from the window start)
        for name in [n for n in ("prefill", "prefill_softcap", "prefill_bucket", "12b_decode",
                                 "12b_decode_two_launch", "e4b_decode", "e4b_decode_two_launch",
                                 "ragged_decode_ring", "ragged_decode_paged")
                     if n != args.workload]:
            cap2 = SOFTCAP_EXAMPLE if name == "prefill_softcap" else None
            real2 = BUCKET_REAL_EXAMPLE if name == "prefill_bucket" else None
            fused2 = not name.startswith("prefill") and not name.endswith("_two_launch")
            ring2 = RING_EXAMPLE if name == "ragged_decode_ring" else None
            paged2 = PAGE_EXAMPLE if name == "ragged_decode_paged" else None
            w2, phys2 = workload("prefill" if name.startswith("prefill") else
                                 name.replace("_two_launch", "").replace("_ring", "")
                                 .replace("_paged", ""))
            rot = 12 if name.startswith("e4b_decode") else 1   # e4b inputs rotate past L2
            ms2, lm2, clk2, info2 = timed_graph_run(w2, phys2, args.steps, args.warmup, device,
                                                    world, per_launch=(w2.n_new > 1),
                                                    rotations=rot, softcap=cap2, n_real=real2,
                                                    fused=fused2, ring=ring2, paged=paged2,
                                                    min_ms=60.0)
            ms2 = max_over_ranks(ms2, world)
            d2 = w2.n_new == 1
            u2, sc2 = ("GB/s", 1e9) if d2 else ("TFLOP/s", 1e12)
            v2 = world * step_work(w2, real2) / (ms2 * 1e-3) / sc2
            ent = {"value": v2, "unit": u2, "ms_per_step": ms2,
                   "frac": v2 / (peaks["hbm_gbs"] if d2 else peaks["bf16_tflops_sustained"]),
                   "us_per_layer_step": 1e3 * ms2 / w2.n_layers,
                   "gpu_launches_per_step": info2["launches_per_step"],
                   "steps": info2["steps"], "clocks": clk2}
            if lm2 is not None:
                ach = sum(prefill_flops(w2, l, real2) for l in range(w2.n_layers)) / \
                    (sum(lm2) * 1e-3) / 1e12
                ent["roofline"] = {"bound": "tensor", "achieved": ach,
                                   "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                                   "frac": ach / peaks["bf16_tflops_sustained"],
                                   "peak_source": peak_src + " sustained"}
                tr2 = prefill_traffic(w2, cap2, real2)
                n2, tsum2 = 0, 0.0
                for kind, nm in ((synth.SLIDING, "sliding"), (synth.GLOBAL, "global")):
                    ls = [l for l, s in enumerate(w2.layers) if s.kind == kind]
                    f = sum(prefill_flops(w2, l, real2) for l in ls)
                    t = sum(lm2[l] for l in ls)
                    ent["roofline"][nm] = {"tflops": f / (t * 1e-3) / 1e12,
                                           "launch_us": 1e3 * t / len(ls),
                                           "traffic": tr2[nm] if tr2 else None}
                    if tr2:
                        n2 += len(ls)
                        tsum2 += len(ls) * tr2[nm]
                # DRAM bytes per attention launch, averaged over the step's launches
                ent["roofline"]["traffic"] = tsum2 / n2 if n2 else None
            if rot > 1:
                ent["l2"] = f"{rot} rotating input copies"
            if cap2 is not None:
                ent["softcap"] = cap2
            if real2 is not None:
                ent["n_real"] = real2
            if ring2 is not None:
                ent["ring_slots"] = ring2
                ent["cache_gb"] = info2["cache_bytes"] / 1e9
            if paged2 is not None:
                ent["page_size"] = paged2
                ent["cache_gb"] = info2["cache_bytes"] / 1e9
            also[name] = ent
        # the greedy step after the LM head: final-logit soft-cap 30 (capped logits written)
        # and argmax over the pages' 262,144-token vocabulary, batch 64, bf16
        lms, lbytes, llaunch, lclk, lsteps = logit_run(args.steps, args.warmup, device, world,
                                                       min_ms=60.0)
        lms = max_over_ranks(lms, world)
        lv = world * lbytes / (lms * 1e-3) / 1e9
        also["logit_softcap_argmax"] = {
            "value": lv, "unit": "GB/s", "ms_per_step": lms, "frac": lv / peaks["hbm_gbs"],
            "config": {"batch": 64, "vocab": synth.VOCAB, "softcap": synth.LOGIT_SOFTCAP,
                       "dtype": "bf16", "capped_output": True},
            "bytes_per_call": lbytes, "gpu_launches_per_step": llaunch, "steps": lsteps,
            "l2": "4 rotating input/output pairs (268 MB)", "clocks": lclk}
        line["also"] = also
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="ragged_decode",
                    choices=["ragged_decode", "e4b_decode", "12b_decode", "prefill", "logits"])
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller ragged batch (profiling captures only; not a bench line)")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer ragged layer-steps (profiling captures only; not a bench line)")
    ap.add_argument("--max-len", type=int, default=None,
                    help="ragged lengths up to this (profiling captures only; not a bench line)")
    ap.add_argument("--layer-offset", type=int, default=0,
                    help="first ragged layer (profiling captures only; not a bench line)")
    ap.add_argument("--two-launch", action="store_true",
                    help="decode workloads: a separate append launch before each attention "
                         "launch (default: the append inside the attention launch)")
    ap.add_argument("--softcap", type=float, default=None,
                    help="time the workload through the soft-capped entry point with this cap")
    ap.add_argument("--tp", action="store_true",
                    help="batch-1 decode workloads: tensor-parallel heads, one rank per GPU")
    ap.add_argument("--quick", action="store_true",
                    help="main workload only (no e2e, CPU baseline or other configurations)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--ref-budget", type=float, default=4.0,
                    help="seconds of oracle work per reference step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "logits":
        run_logits(args)
    elif args.tp:
        run_tp(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
