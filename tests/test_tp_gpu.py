"""GPU: the tensor-parallel rank slices of a decode step, run one after the other on one GPU
through the library (the ranks exchange nothing inside attention), concatenated over the
query heads, match the oracle's unsharded step."""
import dataclasses

import pytest
import torch

from harness import compare, host_inputs, oracle_outputs
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wname,world", [("e4b", 2), ("12b", 2), ("12b", 4)])
def test_rank_slices_match_the_oracle(wname, world):
    import mixed_sliding_global_gb300 as g
    from mixed_sliding_global_gb300 import tp
    w = {"e4b": lambda: synth.e4b_decode(ctx=900),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=3000)}[wname]()
    layers = list(range(w.n_layers))
    hb = host_inputs(w, layers)
    ref = oracle_outputs(w, hb, layers)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = {l: [] for l in layers}
    msl = max(w.ctx_lens)
    for rank in range(world):
        shards = [tp.head_shard(s.n_q, s.n_kv, rank, world) for s in w.layers]
        kc, vc = [None] * w.n_layers, [None] * w.n_layers
        for l in layers:           # this rank's cache shards, with this step's rows appended
            if w.is_owner(l):
                b, sh = hb[l], shards[l]
                kc[l] = tp.shard_cache(b.k_cache, sh).cuda()
                vc[l] = tp.shard_cache(b.v_cache, sh).cuda() if b.v_cache is not None else None
                g.gemma_kv_append(kc, vc, w.owner_map, l,
                                  tp.shard_new_rows(b.k_new, sh).cuda(),
                                  tp.shard_new_rows(b.v_new, sh).cuda() if b.v_new is not None
                                  else None, b.write_pos.cuda(), k_eq_v=w.layers[l].k_eq_v,
                                  device_error=err)
        for l in layers:
            s, sh = w.layers[l], shards[l]
            q = tp.shard_q(hb[l].q, sh).cuda()
            out = torch.empty_like(q)
            ws_n = g.gemma_attn_workspace_size(w.batch, s.kind, s.window, sh.n_q, sh.n_kv,
                                               s.head_dim, msl, 1)
            ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
            tp.tp_decode(out, q, kc, vc, w.owner_map, l, hb[l].seq_lens.cuda(), msl, s=sh,
                         kind=s.kind, window=s.window, k_eq_v=s.k_eq_v, scale=w.scale(l),
                         workspace=ws, device_error=err)
            outs[l].append(out)
    torch.cuda.synchronize()
    assert err.item() == 0
    for l in layers:
        compare(torch.cat(outs[l], dim=2), ref[l], w.dtype)


@pytest.mark.parametrize("wname,world", [("e4b", 1), ("e4b", 2), ("12b", 2)])
def test_rank_driver_with_the_library(wname, world):
    """tp.RankStep with the library's calls: each rank's step (load its shards, append, attend
    every layer) run in turn on one GPU, outputs concatenated over the query heads in rank
    order (what `gather` all-gathers), against the oracle's unsharded step. At world 1 the
    driver's own gather is used."""
    from mixed_sliding_global_gb300.tp import RankStep
    w = {"e4b": lambda: synth.e4b_decode(ctx=900),
         "12b": lambda: synth.b12_decode(n_layers=6, ctx=3000)}[wname]()
    layers = list(range(w.n_layers))
    hb = host_inputs(w, layers)
    ref = oracle_outputs(w, hb, layers)
    inputs = [(hb[l].q, hb[l].k_new, hb[l].v_new, hb[l].write_pos, hb[l].seq_lens)
              for l in layers]
    scales = [w.scale(l) for l in layers]
    parts = {l: [] for l in layers}
    for rank in range(world):
        rs = RankStep(w.layers, w.owner_map, rank, world, "cuda")
        for l in layers:
            if w.is_owner(l):
                rs.load_cache(l, hb[l].k_cache, hb[l].v_cache)
        outs = rs.step(inputs, scales, max(w.ctx_lens))
        if world == 1:
            outs = rs.gather(outs)
        torch.cuda.synchronize()
        assert rs.err.item() == 0
        for l in layers:
            parts[l].append(outs[l])
    for l in layers:
        compare(torch.cat(parts[l], dim=2).cpu(), ref[l], w.dtype)
