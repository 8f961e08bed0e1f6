"""Helpers for the parity tests: run a synthetic workload through the C ABI on the GPU, and
through the oracle on the CPU, from the same seeded host tensors.

The expected side calls only ``oracle``; the GPU side calls only the product binding.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import torch

import synth
from oracle import load_oracle

BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3   # bf16 outputs, fp32 accumulation
FP32_MAX_ABS = 1e-4                       # fp32 debug path


@dataclasses.dataclass
class HostLayer:
    batch: synth.LayerBatch
    seqs: List[int]


def host_inputs(w: synth.Workload, layers: Sequence[int], seqs: Optional[Sequence[int]] = None
                ) -> Dict[int, synth.LayerBatch]:
    """Seeded host inputs of the given layers and of the owner layers they read."""
    need = sorted(set(layers) | {w.owner_map[l] for l in layers})
    return {l: synth.layer_batch(w, l, seqs) for l in need}


def oracle_outputs(w: synth.Workload, hb: Dict[int, synth.LayerBatch], layers: Sequence[int],
                   q_range=None, softcap: float = 0.0) -> Dict[int, torch.Tensor]:
    """fp64 oracle outputs [B][n_tok][n_q][d] of each layer, after the oracle's own append of
    the new rows into copies of the owner caches. q_range=(i0, i1) restricts the queries to
    tokens [i0, i1) of the step (exactly: earlier keys are all a query may see)."""
    orc = load_oracle()
    n = w.n_layers
    kcs: List[Optional[torch.Tensor]] = [None] * n
    vcs: List[Optional[torch.Tensor]] = [None] * n
    for l, b in hb.items():
        if w.is_owner(l):
            kcs[l] = b.k_cache.clone()
            orc.kv_append(kcs[l], b.k_new, b.write_pos.tolist())
            if b.v_cache is not None:
                vcs[l] = b.v_cache.clone()
                orc.kv_append(vcs[l], b.v_new, b.write_pos.tolist())
    out = {}
    for l in layers:
        q = hb[l].q
        lens = hb[l].seq_lens.tolist()
        if q_range is not None:
            i0, i1 = q_range
            q = q[:, i0:i1].contiguous()
            lens = [x - w.n_new + i1 for x in lens]
        out[l] = orc.attention(w.layers, w.owner_map, l, kcs, vcs, q, lens, w.scale(l),
                               softcap=softcap)
    return out


class DeviceRun:
    """Device copies of a workload's host inputs and the C-ABI calls of one step."""

    def __init__(self, w: synth.Workload, hb: Dict[int, synth.LayerBatch], device="cuda"):
        import mixed_sliding_global_gb300 as g
        self.g = g
        self.w = w
        self.hb = hb
        n = w.n_layers
        self.kc: List[Optional[torch.Tensor]] = [None] * n
        self.vc: List[Optional[torch.Tensor]] = [None] * n
        self.dev = {}
        for l, b in hb.items():
            d = {"q": b.q.to(device), "seq_lens": b.seq_lens.to(device),
                 "write_pos": b.write_pos.to(device)}
            if w.is_owner(l):
                self.kc[l] = b.k_cache.to(device)
                d["k_new"] = b.k_new.to(device)
                if b.v_cache is not None:
                    self.vc[l] = b.v_cache.to(device)
                    d["v_new"] = b.v_new.to(device)
            self.dev[l] = d
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def append(self, l: int) -> None:
        d, spec = self.dev[self.w.owner_map[l]], self.w.layers[l]
        self.g.gemma_kv_append(self.kc, self.vc, self.w.owner_map, l, d["k_new"], d.get("v_new"),
                               d["write_pos"], k_eq_v=spec.k_eq_v, device_error=self.err)

    def attend(self, l: int, max_seq_len: Optional[int] = None,
               softcap: Optional[float] = None, prefill_entry: bool = False) -> torch.Tensor:
        w, spec, d = self.w, self.w.layers[l], self.dev[l]
        msl = max(w.ctx_lens) if max_seq_len is None else max_seq_len
        q = d["q"]
        out = torch.empty_like(q)
        B = q.shape[0]
        ws_n = self.g.gemma_attn_workspace_size(B, spec.kind, spec.window, spec.n_q, spec.n_kv,
                                                spec.head_dim, msl, w.n_new)
        ws = torch.zeros(max(ws_n, 1), dtype=torch.uint8, device=q.device)
        kw = dict(kind=spec.kind, window=spec.window, n_kv=spec.n_kv, k_eq_v=spec.k_eq_v,
                  scale=w.scale(l), workspace=ws, device_error=self.err)
        if softcap is not None:
            self.g.gemma_attn_softcap(out, q, self.kc, self.vc, w.owner_map, l, d["seq_lens"], msl,
                                      softcap=softcap, **kw)
        else:
            # prefill_entry: one new token through gemma_attn_prefill instead of the decode entry
            fn = self.g.gemma_attn_decode if w.n_new == 1 and not prefill_entry \
                else self.g.gemma_attn_prefill
            fn(out, q, self.kc, self.vc, w.owner_map, l, d["seq_lens"], msl, **kw)
        return out

    def step(self, layers: Sequence[int]) -> Dict[int, torch.Tensor]:
        outs = {}
        for l in layers:
            if self.w.is_owner(l):
                self.append(l)
            outs[l] = self.attend(l)
        torch.cuda.synchronize()
        return outs


def compare(got: torch.Tensor, ref: torch.Tensor, dtype: int):
    diff = (got.double().cpu() - ref).abs()
    assert torch.isfinite(got).all(), "non-finite output"
    mx, mean = diff.max().item(), diff.mean().item()
    if dtype == synth.FP32:
        assert mx <= FP32_MAX_ABS, f"max abs err {mx:.3e} > {FP32_MAX_ABS}"
    else:
        assert mx <= BF16_MAX_ABS, f"max abs err {mx:.3e} > {BF16_MAX_ABS}"
        assert mean <= BF16_MEAN_ABS, f"mean abs err {mean:.3e} > {BF16_MEAN_ABS}"
    return mx, mean
