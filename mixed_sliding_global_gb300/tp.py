"""Tensor-parallel head sharding of the attention step (one rank's slice of every layer).

"Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", section 2.2: under tensor parallelism the
query, key and value projections are column-parallel, so rank r holds a contiguous slice of the
query heads and the key/value heads they read ("head r -> rank r"); section 2.3 with the 12B
card: a global layer with fewer KV heads than ranks keeps its K (and V) replicated on every rank,
each rank's group size being (n_q / TP) / n_kv. The attention step itself exchanges nothing:
each rank attends its own heads over its own cache shard, and the sum over ranks happens after
the row-parallel output projection, outside this path. So a rank's step is the plain library
call on its slice; this module computes the slice and cuts the tensors. It does no arithmetic.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class HeadShard:
    q_lo: int        # query heads [q_lo, q_lo + n_q) of the layer
    n_q: int
    kv_lo: int       # key/value heads [kv_lo, kv_lo + n_kv) they read
    n_kv: int
    replicated: bool  # the KV heads are shared with another rank's query heads


def head_shard(n_q: int, n_kv: int, rank: int, world: int) -> HeadShard:
    """Rank `rank`'s heads of a layer with n_q query and n_kv key/value heads over `world` ranks.
    Query head h reads KV head h // (n_q / n_kv); a rank's query heads must read either whole
    groups (n_kv split across ranks) or part of one group (its KV head replicated)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank or world size")
    if n_q % n_kv != 0 or n_q % world != 0:
        raise ValueError(f"{n_q} query heads do not split over {world} ranks")
    g = n_q // n_kv
    nq = n_q // world
    q_lo = rank * nq
    kv_lo, kv_hi = q_lo // g, (q_lo + nq - 1) // g + 1
    n_kv_l = kv_hi - kv_lo
    if nq % n_kv_l != 0 or (n_kv_l > 1 and nq // n_kv_l != g):
        raise ValueError(f"query heads {q_lo}..{q_lo + nq - 1} straddle a group of {g}")
    return HeadShard(q_lo, nq, kv_lo, n_kv_l, replicated=nq < g)


def shard_heads(t: torch.Tensor, lo: int, n: int, dim: int) -> torch.Tensor:
    """A contiguous copy of heads [lo, lo + n) along `dim` (a rank holds its own shard)."""
    return t.narrow(dim, lo, n).contiguous()


def shard_q(q: torch.Tensor, s: HeadShard) -> torch.Tensor:
    """q or out [B][n_tok][n_q][d] -> this rank's query heads."""
    return shard_heads(q, s.q_lo, s.n_q, 2)


def shard_cache(cache: torch.Tensor, s: HeadShard) -> torch.Tensor:
    """cache [B][n_kv][cap][d] -> this rank's KV heads (all of them when replicated)."""
    return shard_heads(cache, s.kv_lo, s.n_kv, 1)


def shard_new_rows(rows: torch.Tensor, s: HeadShard) -> torch.Tensor:
    """new K/V rows [B][n_new][n_kv][d] -> this rank's KV heads."""
    return shard_heads(rows, s.kv_lo, s.n_kv, 2)


def tp_decode(out_local, q_local, k_local, v_local, owner_map, layer, seq_lens, max_seq_len, *,
              s: HeadShard, kind, window, k_eq_v, scale, workspace=None, device_error=None,
              stream=None):
    """One rank's decode step of a layer: the library's decode call on the rank's shard
    (k_local/v_local: per-layer lists of shard caches, None for shared layers)."""
    from .binding import gemma_attn_decode
    gemma_attn_decode(out_local, q_local, k_local, v_local, owner_map, layer, seq_lens,
                      max_seq_len, kind=kind, window=window, n_kv=s.n_kv, k_eq_v=k_eq_v,
                      scale=scale, workspace=workspace, device_error=device_error, stream=stream)


class RankStep:
    """One rank's share of a decode step over every layer of a model (one process per GPU).

    The rank holds its head shard of each owner layer's cache on its own device (the pages'
    "head r -> rank r", with a KV head replicated where a layer has fewer KV heads than ranks),
    appends the step's rows of its KV heads and attends its query heads of every layer. Ranks
    exchange nothing during the step; `gather` all-gathers the per-layer outputs along the query
    heads afterwards (the sum over ranks of the real model follows the row-parallel output
    projection, outside this path).

    `append(step, layer, k_new, v_new, write_pos, spec)` (into step.k / step.v) and
    `attend(step, out, q, layer, seq_lens, max_seq_len, spec, shard, scale)` default to this
    library's calls; they are parameters so that the same rank logic runs on CPU ranks with a
    stand-in for the kernels.
    """

    def __init__(self, layers, owner_map, rank: int, world: int, device, append=None,
                 attend=None):
        self.layers, self.owner_map = list(layers), list(owner_map)
        self.rank, self.world, self.device = rank, world, device
        self.shards = [head_shard(s.n_q, s.n_kv, rank, world) for s in self.layers]
        self.k = [None] * len(self.layers)
        self.v = [None] * len(self.layers)
        self._append = append or RankStep._lib_append
        self._attend = attend or RankStep._lib_attend
        self.err = None
        self._ws = {}   # per-layer split workspace, kept across steps

    # ---- the library's calls on this rank's device ----
    def _lib_append(self, layer, k_new, v_new, write_pos, spec):
        from .binding import gemma_kv_append
        if self.err is None:
            self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        gemma_kv_append(self.k, self.v, self.owner_map, layer, k_new, v_new, write_pos,
                        k_eq_v=spec.k_eq_v, device_error=self.err)

    def _lib_attend(self, out, q, layer, seq_lens, max_seq_len, spec, shard, scale):
        from .binding import gemma_attn_workspace_size
        if self.err is None:
            self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        ws_n = gemma_attn_workspace_size(q.shape[0], spec.kind, spec.window, shard.n_q, shard.n_kv,
                                         spec.head_dim, max_seq_len, 1)
        ws = self._ws.get(layer)
        if ws is None or ws.numel() < ws_n:
            ws = self._ws[layer] = torch.zeros(max(ws_n, 16), dtype=torch.uint8,
                                               device=self.device)
        tp_decode(out, q, self.k, self.v, self.owner_map, layer, seq_lens, max_seq_len, s=shard,
                  kind=spec.kind, window=spec.window, k_eq_v=spec.k_eq_v, scale=scale,
                  workspace=ws, device_error=self.err)

    # ---- the step ----
    def load_cache(self, layer: int, k_cache: torch.Tensor, v_cache=None) -> None:
        """This rank's shard of an owner layer's full cache [B][n_kv][cap][d], on its device."""
        sh = self.shards[layer]
        self.k[layer] = shard_cache(k_cache, sh).to(self.device)
        self.v[layer] = None if v_cache is None else shard_cache(v_cache, sh).to(self.device)

    def local_inputs(self, layer_inputs):
        """This rank's slice of every layer's inputs, on its device; layer_inputs[l] = (q, k_new,
        v_new, write_pos, seq_lens) with the full head dimension."""
        loc = []
        for l, (q, k_new, v_new, write_pos, seq_lens) in enumerate(layer_inputs):
            sh = self.shards[l]
            own = self.owner_map[l] == l
            loc.append((shard_q(q, sh).to(self.device),
                        shard_new_rows(k_new, sh).to(self.device) if own else None,
                        shard_new_rows(v_new, sh).to(self.device) if own and v_new is not None
                        else None,
                        write_pos.to(self.device), seq_lens.to(self.device)))
        return loc

    def run(self, local, outs, scales, max_seq_len: int) -> None:
        """The rank's step on inputs already sliced (local_inputs): append (owner layers) and
        attend every layer into outs[l] [B][1][n_q / world][d]. Library calls only, so the
        step can be captured in a CUDA graph."""
        for l, spec in enumerate(self.layers):
            q, k_new, v_new, write_pos, seq_lens = local[l]
            if self.owner_map[l] == l:
                self._append(self, l, k_new, v_new, write_pos, spec)
            self._attend(self, outs[l], q, l, seq_lens, max_seq_len, spec, self.shards[l],
                         scales[l])

    def step(self, layer_inputs, scales, max_seq_len: int):
        """local_inputs + run; returns this rank's output of every layer."""
        local = self.local_inputs(layer_inputs)
        outs = [torch.empty_like(x[0]) for x in local]
        self.run(local, outs, scales, max_seq_len)
        return outs

    def gather(self, outs, group=None):
        """All-gather each layer's output along the query heads (rank-major), outside the
        attention step; returns the full outputs [B][1][n_q][d] on every rank."""
        if self.world == 1:
            return list(outs)
        import torch.distributed as dist
        full = []
        for o in outs:
            parts = [torch.empty_like(o) for _ in range(self.world)]
            dist.all_gather(parts, o.contiguous(), group=group)
            full.append(torch.cat(parts, dim=2))
        return full
