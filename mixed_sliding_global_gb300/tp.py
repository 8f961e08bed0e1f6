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
