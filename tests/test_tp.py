"""Tensor-parallel head sharding on CPU: the shard rules for the pages' configurations, and gloo
ranks (world 2 and 4) that each attend their own heads over their own cache shards (the oracle
stands in for the kernels on CPU) and all-gather the outputs: the gathered result equals the
unsharded step exactly (every query head's arithmetic is the same; nothing is exchanged)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixed_sliding_global_gb300.tp import head_shard


@pytest.mark.parametrize("n_q,n_kv,world,expect", [
    (8, 2, 2, [(0, 4, 0, 1, False), (4, 4, 1, 1, False)]),          # E4B at TP=2
    (16, 8, 2, [(0, 8, 0, 4, False), (8, 8, 4, 4, False)]),         # 12B sliding at TP=2
    (16, 1, 2, [(0, 8, 0, 1, True), (8, 8, 0, 1, True)]),           # 12B global: K replicated
    (16, 2, 4, [(0, 4, 0, 1, True), (4, 4, 0, 1, True), (8, 4, 1, 1, True), (12, 4, 1, 1, True)]),
    (8, 2, 1, [(0, 8, 0, 2, False)]),
])
def test_head_shards(n_q, n_kv, world, expect):
    got = [head_shard(n_q, n_kv, r, world) for r in range(world)]
    assert [(s.q_lo, s.n_q, s.kv_lo, s.n_kv, s.replicated) for s in got] == expect


@pytest.mark.parametrize("n_q,n_kv,world", [(12, 3, 2), (8, 2, 3), (6, 4, 2)])
def test_unsplittable_heads_are_rejected(n_q, n_kv, world):
    with pytest.raises(ValueError):
        head_shard(n_q, n_kv, 0, world)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _sharded_outputs(wname, rank, world):
    """This rank's outputs of every layer, computed on its shards only."""
    import dataclasses
    import synth
    from harness import host_inputs
    from oracle import load_oracle
    from mixed_sliding_global_gb300 import tp
    w = {"e4b": lambda: synth.e4b_decode(ctx=300),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=700)}[wname]()
    layers = list(range(w.n_layers))
    hb = host_inputs(w, layers)
    orc = load_oracle()
    shards = [tp.head_shard(s.n_q, s.n_kv, rank, world) for s in w.layers]
    local = [dataclasses.replace(s, n_q=sh.n_q, n_kv=sh.n_kv) for s, sh in zip(w.layers, shards)]
    kcs, vcs = [None] * w.n_layers, [None] * w.n_layers
    for l in layers:
        if w.is_owner(l):
            b, sh = hb[l], shards[l]
            kcs[l] = tp.shard_cache(b.k_cache, sh)
            orc.kv_append(kcs[l], tp.shard_new_rows(b.k_new, sh), b.write_pos.tolist())
            if b.v_cache is not None:
                vcs[l] = tp.shard_cache(b.v_cache, sh)
                orc.kv_append(vcs[l], tp.shard_new_rows(b.v_new, sh), b.write_pos.tolist())
    return [orc.attention(local, w.owner_map, l, kcs, vcs, tp.shard_q(hb[l].q, shards[l]),
                          hb[l].seq_lens.tolist(), w.scale(l)) for l in layers]


def _worker(rank, world, port, wname, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = _sharded_outputs(wname, rank, world)
    gathered = []
    for o in mine:
        parts = [torch.empty_like(o) for _ in range(world)]
        dist.all_gather(parts, o.contiguous())
        gathered.append(torch.cat(parts, dim=2))        # query heads are rank-major
    if rank == 0:
        out["full"] = gathered
    dist.destroy_process_group()


@pytest.mark.parametrize("wname,world", [("e4b", 2), ("12b", 2), ("12b", 4)])
def test_gloo_ranks_gather_the_unsharded_step(wname, world):
    import synth
    from harness import host_inputs, oracle_outputs
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, wname, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        gathered = out["full"]
    w = {"e4b": lambda: synth.e4b_decode(ctx=300),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=700)}[wname]()
    layers = list(range(w.n_layers))
    ref = oracle_outputs(w, host_inputs(w, layers), layers)
    for l in layers:
        assert torch.equal(gathered[l], ref[l]), l


def _driver_worker(rank, world, port, wname, out):
    """The rank driver (tp.RankStep) on a CPU gloo rank, with the oracle standing in for the
    kernels: shards loaded, rows appended, every layer attended, outputs all-gathered."""
    import dataclasses
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import synth
    from harness import host_inputs
    from oracle import load_oracle
    from mixed_sliding_global_gb300.tp import RankStep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = {"e4b": lambda: synth.e4b_decode(ctx=300),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=700)}[wname]()
    layers = list(range(w.n_layers))
    hb = host_inputs(w, layers)
    orc = load_oracle()

    def append(step, l, k_new, v_new, write_pos, spec):
        orc.kv_append(step.k[l], k_new, write_pos.tolist())
        if v_new is not None:
            orc.kv_append(step.v[l], v_new, write_pos.tolist())

    def attend(step, out, q, l, seq_lens, max_seq_len, spec, sh, scale):
        local = [dataclasses.replace(s, n_q=x.n_q, n_kv=x.n_kv)
                 for s, x in zip(w.layers, step.shards)]
        out.copy_(orc.attention(local, w.owner_map, l, step.k, step.v, q, seq_lens.tolist(),
                                scale))

    step = RankStep(w.layers, w.owner_map, rank, world, "cpu", append=append, attend=attend)
    for l in layers:
        if w.is_owner(l):
            step.load_cache(l, hb[l].k_cache, hb[l].v_cache)
    inputs = [(hb[l].q, hb[l].k_new, hb[l].v_new, hb[l].write_pos, hb[l].seq_lens)
              for l in layers]
    outs = step.step(inputs, [w.scale(l) for l in layers], max(w.ctx_lens))
    full = step.gather(outs)
    if rank == 0:
        out["full"] = full
    dist.destroy_process_group()


@pytest.mark.parametrize("wname,world", [("e4b", 2), ("12b", 2)])
def test_rank_driver_on_gloo_ranks(wname, world):
    """tp.RankStep, one process per rank: the gathered outputs equal the unsharded step's,
    rounded to the step's dtype alike (every query head's arithmetic is the same)."""
    import synth
    from harness import host_inputs, oracle_outputs
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_driver_worker, args=(r, world, port, wname, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        gathered = out["full"]
    w = {"e4b": lambda: synth.e4b_decode(ctx=300),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=700)}[wname]()
    layers = list(range(w.n_layers))
    ref = oracle_outputs(w, host_inputs(w, layers), layers)
    for l in layers:
        assert torch.equal(gathered[l], ref[l].to(gathered[l].dtype)), l
