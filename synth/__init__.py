"""Seeded synthetic workloads for the mixed sliding/global attention step.

This module is shared by the CUDA path's tests and benchmark and by the oracle
side. It holds shapes, layer patterns, owner maps, sequence lengths and seeded
random tensors only: no attention arithmetic lives here.

Workload shapes follow the Gemma-4 configurations described in "Porting Gemma-4
(2B / 4B / 12B) to AWS Inferentia2" (model family table: 8q/2kv heads and
head_dim 256 with sliding_window=512 on E4B; 16q/8kv at head_dim 256 with
sliding_window=1024, global layers with one KV head at head_dim 512 and
attention_k_eq_v on 12B) and the 12B model card ("48 layers ... 16 attention /
8 KV heads, head_dim 256 (global layers 512)").

Random values: every tensor is drawn as float32 N(0, 1) from a CPU
``torch.Generator`` seeded with ``BASE_SEED + tensor_id`` and then rounded to
the storage dtype (bf16 round-to-nearest-even through ``Tensor.to``), so the
GPU and the oracle see the same bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

SLIDING, GLOBAL = 0, 1
BF16, FP32 = 0, 1
BASE_SEED = 1234

TORCH_DTYPE = {BF16: torch.bfloat16, FP32: torch.float32}


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    kind: int          # SLIDING or GLOBAL
    window: int        # sliding window W (keys including the query's own position)
    n_q: int
    n_kv: int
    head_dim: int
    k_eq_v: bool       # the layer attends with V := K


@dataclasses.dataclass
class Workload:
    name: str
    layers: List[LayerSpec]
    owner_map: List[int]      # owner_map[l]: the layer whose cache layer l reads
    batch: int
    dtype: int                # BF16 or FP32 storage / IO dtype
    n_new: int                # tokens appended per sequence this step (1 = decode bucket)
    ctx_lens: List[int]       # valid cache tokens per sequence after the append
    capacity: int             # cache slots per (sequence, kv head)

    @property
    def mode(self) -> str:
        return "decode" if self.n_new == 1 else "prefill"

    @property
    def prefix_lens(self) -> List[int]:
        return [c - self.n_new for c in self.ctx_lens]

    @property
    def n_layers(self) -> int:
        return len(self.layers)

    def is_owner(self, layer: int) -> bool:
        return self.owner_map[layer] == layer

    def scale(self, layer: int) -> float:
        return 1.0 / math.sqrt(self.layers[layer].head_dim)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def pattern_5_to_1(n_layers: int) -> List[int]:
    """Five sliding layers then one global layer, repeated (global at l % 6 == 5)."""
    return [GLOBAL if l % 6 == 5 else SLIDING for l in range(n_layers)]


def _layers_12b(n_layers: int = 48) -> List[LayerSpec]:
    sliding = LayerSpec(SLIDING, 1024, 16, 8, 256, False)
    glob = LayerSpec(GLOBAL, 0, 16, 1, 512, True)
    return [glob if k == GLOBAL else sliding for k in pattern_5_to_1(n_layers)]


def tiny(mode: str = "decode", ctx: int = 64, n_new: Optional[int] = None) -> Workload:
    """2 layers (sliding W=16, global), batch 1, 4q/1kv, head_dim 64, fp32."""
    layers = [LayerSpec(SLIDING, 16, 4, 1, 64, False), LayerSpec(GLOBAL, 0, 4, 1, 64, False)]
    if n_new is None:
        n_new = 1 if mode == "decode" else 8
    return Workload("tiny", layers, [0, 1], 1, FP32, n_new, [ctx], _round_up(ctx, 8))


def e4b_decode(n_layers: int = 12, ctx: int = 2048, batch: int = 1) -> Workload:
    """E4B-shaped decode: 5 sliding (W=512) : 1 global, 8q/2kv, head_dim 256,
    the last 4 layers KV-shared with the most recent owner layer of the same kind."""
    kinds = pattern_5_to_1(n_layers)
    layers = [LayerSpec(k, 512 if k == SLIDING else 0, 8, 2, 256, False) for k in kinds]
    n_shared = 4 if n_layers >= 8 else 0
    owner = list(range(n_layers))
    for l in range(n_layers - n_shared, n_layers):
        cands = [o for o in range(n_layers - n_shared) if kinds[o] == kinds[l]]
        owner[l] = max(cands)
    return Workload("e4b_decode", layers, owner, batch, BF16, 1, [ctx] * batch, _round_up(ctx, 64))


def b12_decode(n_layers: int = 48, ctx: int = 8192, batch: int = 1) -> Workload:
    """12B-shaped decode: 48 layers, no KV sharing, batch 1, context 8192."""
    return Workload("12b_decode", _layers_12b(n_layers), list(range(n_layers)), batch, BF16, 1,
                    [ctx] * batch, _round_up(ctx, 64))


def ragged_lengths(batch: int = 64, lo: int = 128, hi: int = 16384) -> List[int]:
    """Per-sequence cached lengths before the append, uniform in [lo, hi], seeded."""
    g = torch.Generator().manual_seed(BASE_SEED + 7)
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


def ragged_decode(n_layers: int = 48, batch: int = 64, capacity: int = 16448,
                  max_len: int = 16384) -> Workload:
    """Batched ragged decode on 12B-shaped layers: one new token per sequence is
    appended at slot L_b, attention length L_b + 1 (L_b uniform in [128, max_len])."""
    pre = ragged_lengths(batch, hi=max_len)
    return Workload("ragged_decode", _layers_12b(n_layers), list(range(n_layers)), batch, BF16, 1,
                    [p + 1 for p in pre], capacity)


def prefill_12b(n_layers: int = 48, batch: int = 4, prefix: int = 3584, n_new: int = 512) -> Workload:
    """Prefill bucket on 12B-shaped layers: n_new new tokens onto a cached prefix."""
    ctx = prefix + n_new
    return Workload("prefill", _layers_12b(n_layers), list(range(n_layers)), batch, BF16, n_new,
                    [ctx] * batch, _round_up(ctx, 64))


WORKLOADS = {
    "tiny_decode": lambda: tiny("decode"),
    "tiny_prefill": lambda: tiny("prefill"),
    "e4b_decode": e4b_decode,
    "12b_decode": b12_decode,
    "ragged_decode": ragged_decode,
    "prefill": prefill_12b,
}


# ----------------------------------------------------------------------------------------------
# Seeded tensors
# ----------------------------------------------------------------------------------------------
Q, K_ROWS, V_ROWS, K_NEW, V_NEW = 0, 1, 2, 3, 4


def tensor_id(layer: int, what: int, seq: int) -> int:
    return ((layer * 8 + what) * 8192) + seq


def randn(shape, tid: int, dtype: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(BASE_SEED + tid)
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(TORCH_DTYPE[dtype])


# final logits of a greedy step: [batch][vocab], N(0, 8^2) (most values inside the cap of 30,
# a few beyond it), rounded to the dtype; seeded per call
LOGIT_SOFTCAP = 30.0
VOCAB = 262144


def logits(batch: int, vocab: int = VOCAB, seed: int = 0, dtype: int = BF16) -> torch.Tensor:
    g = torch.Generator().manual_seed(BASE_SEED + (1 << 30) + seed)  # apart from tensor ids
    x = torch.randn((batch, vocab), generator=g, dtype=torch.float32) * 8.0
    return x.to(torch.bfloat16 if dtype == BF16 else torch.float32)


def needed_row_lo(spec: LayerSpec, ctx: int, n_new: int) -> int:
    """First cache row any query of this step may attend: 0 for global layers; for sliding
    layers the oldest window start among the new queries. Rows below it are never read and
    are filled with a NaN sentinel in device caches."""
    if spec.kind == GLOBAL:
        return 0
    return max(0, ctx - n_new + 1 - spec.window)


@dataclasses.dataclass
class SeqLayerInputs:
    q: torch.Tensor                    # [n_new][n_q][d]
    row_lo: int                        # first generated cache row
    k_rows: Optional[torch.Tensor]     # [n_kv][prefix - row_lo][d] (owner layers only)
    v_rows: Optional[torch.Tensor]     # same, None when k_eq_v or not an owner
    k_new: Optional[torch.Tensor]      # [n_new][n_kv][d] (owner layers only)
    v_new: Optional[torch.Tensor]      # None when k_eq_v or not an owner


def seq_layer_inputs(w: Workload, layer: int, seq: int) -> SeqLayerInputs:
    """Seeded inputs of one sequence for one layer. Shared layers get only q: they read
    their owner's cache."""
    spec = w.layers[layer]
    d, ctx, n_new = spec.head_dim, w.ctx_lens[seq], w.n_new
    q = randn((n_new, spec.n_q, d), tensor_id(layer, Q, seq), w.dtype)
    if not w.is_owner(layer):
        return SeqLayerInputs(q, 0, None, None, None, None)
    lo = needed_row_lo(spec, ctx, n_new)
    pre = ctx - n_new
    n_rows = max(0, pre - lo)
    k_rows = randn((spec.n_kv, n_rows, d), tensor_id(layer, K_ROWS, seq), w.dtype)
    k_new = randn((n_new, spec.n_kv, d), tensor_id(layer, K_NEW, seq), w.dtype)
    v_rows = v_new = None
    if not spec.k_eq_v:
        v_rows = randn((spec.n_kv, n_rows, d), tensor_id(layer, V_ROWS, seq), w.dtype)
        v_new = randn((n_new, spec.n_kv, d), tensor_id(layer, V_NEW, seq), w.dtype)
    return SeqLayerInputs(q, lo, k_rows, v_rows, k_new, v_new)


@dataclasses.dataclass
class LayerBatch:
    """Batched host tensors of one layer, in the cache layout [B][n_kv][cap][d]."""
    q: torch.Tensor                    # [B][n_new][n_q][d]
    k_cache: Optional[torch.Tensor]    # [B][n_kv][cap][d], NaN outside generated rows
    v_cache: Optional[torch.Tensor]
    k_new: Optional[torch.Tensor]      # [B][n_new][n_kv][d]
    v_new: Optional[torch.Tensor]
    write_pos: torch.Tensor            # int32 [B]: slot of the first new token
    seq_lens: torch.Tensor             # int32 [B]: valid tokens after the append


def layer_batch(w: Workload, layer: int, seqs: Optional[List[int]] = None) -> LayerBatch:
    """Assemble the seeded inputs of the given sequences (default: all) for one layer."""
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    spec = w.layers[layer]
    dt = TORCH_DTYPE[w.dtype]
    B, d, cap = len(seqs), spec.head_dim, w.capacity
    per = [seq_layer_inputs(w, layer, s) for s in seqs]
    q = torch.stack([p.q for p in per])
    k_cache = v_cache = k_new = v_new = None
    if w.is_owner(layer):
        k_cache = torch.full((B, spec.n_kv, cap, d), float("nan"), dtype=dt)
        if not spec.k_eq_v:
            v_cache = torch.full((B, spec.n_kv, cap, d), float("nan"), dtype=dt)
        for i, (s, p) in enumerate(zip(seqs, per)):
            pre = w.ctx_lens[s] - w.n_new
            k_cache[i, :, p.row_lo:pre] = p.k_rows
            if v_cache is not None:
                v_cache[i, :, p.row_lo:pre] = p.v_rows
        k_new = torch.stack([p.k_new for p in per])
        if not spec.k_eq_v:
            v_new = torch.stack([p.v_new for p in per])
    ctx = torch.tensor([w.ctx_lens[s] for s in seqs], dtype=torch.int32)
    return LayerBatch(q, k_cache, v_cache, k_new, v_new, ctx - w.n_new, ctx)
