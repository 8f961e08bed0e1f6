"""GPU parity in the launch configurations the benchmark times.

The benchmark's headline is the batch-64 ragged decode over 12B-shaped layers; its other lines
time the same decode over ring caches and paged pools, and the prefill bucket at batch 4. The
launch configuration (split plan, grid) depends on the batch, the lengths and max_seq_len, so
these tests run each timed configuration at its full size, through the entry point the
benchmark calls, and compare sampled outputs element by element with the fp64 oracle (the
oracle runs on the sampled sequences or query tokens only; their seeded inputs equal the full
workload's). Each test first checks that the plan equals the benchmark's (the workspace size
for these arguments, which fixes the number and size of key chunks).
"""
import pytest
import torch

import synth
from harness import DeviceRun, compare, host_inputs, oracle_outputs
from synth import BF16, GLOBAL, SLIDING, Workload  # noqa: F401

pytestmark = pytest.mark.gpu

PAGE = 256    # keys per page of the benchmark's paged pools
RING = 1024   # ring slots of the benchmark's sliding caches


def _sampled(w):
    lens = w.ctx_lens
    return sorted({lens.index(min(lens)), lens.index(max(lens)), 7, 33, 63})


def _oracle_on(w, layer, seqs):
    sub = Workload(w.name, w.layers, w.owner_map, len(seqs), w.dtype, 1,
                   [w.ctx_lens[s] for s in seqs], w.capacity)
    return oracle_outputs(sub, host_inputs(w, [layer], seqs), [layer])[layer]


def _fused_decode(gr, w, layer, kc, vc, kind, ws):
    """The benchmark's decode call: the step's K/V rows appended inside the attention launch."""
    g, spec, d = gr.g, w.layers[layer], gr.dev[layer]
    out = torch.empty_like(d["q"])
    g.gemma_attn_decode_append(out, d["q"], kc, vc, w.owner_map, layer, d["k_new"],
                               d.get("v_new"), d["write_pos"], d["seq_lens"], max(w.ctx_lens),
                               kind=kind, window=spec.window, n_kv=spec.n_kv,
                               k_eq_v=spec.k_eq_v, scale=w.scale(layer), workspace=ws,
                               device_error=gr.err)
    return out


def test_ragged_decode_full_batch_global_layer():
    """The batch-64 global layer (16 q / 1 kv head, head_dim 512, K as V) over all 64 ragged
    sequences in the benchmark's plan: 19 chunks of 864 keys per sequence, merged by the
    combine pass."""
    import mixed_sliding_global_gb300 as g
    w = synth.ragged_decode(n_layers=6)
    spec, msl = w.layers[5], max(w.ctx_lens)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    ws_n = g.gemma_attn_workspace_size(64, GLOBAL, 0, 16, 1, 512, msl, 1)
    if n_sm == 152:
        # 64 x 16385 keys over eight chunks per SM: 864-key chunks, 19 per sequence; scratch of
        # 64 sequences x 16 heads x 19 chunks x (512 + 2) floats, each part 256-byte aligned
        rows = 64 * 16 * 19
        assert -(-msl // 864) == 19
        assert ws_n == -(-rows * 512 * 4 // 256) * 256 + -(-rows * 2 * 4 // 256) * 256, ws_n
    assert ws_n > 0
    hb = host_inputs(w, [5])
    gr = DeviceRun(w, hb)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device="cuda")
    got = _fused_decode(gr, w, 5, gr.kc, gr.vc, GLOBAL, ws)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    seqs = _sampled(w)
    compare(got[seqs].cpu(), _oracle_on(w, 5, seqs), BF16)


def _ring_from_linear(lin, write_pos, R):
    """[B][H][cap][d] linear cache -> [B][H][R][d] ring holding positions [wp - R, wp) at p % R
    (zeros before position 0)."""
    B, H, cap, d = lin.shape
    ring = torch.zeros((B, H, R, d), dtype=lin.dtype, device=lin.device)
    for b in range(B):
        wp = int(write_pos[b])
        lo = max(0, wp - R)
        pos = torch.arange(lo, wp, device=lin.device)
        ring[b, :, pos % R] = lin[b, :, lo:wp]
    return torch.nan_to_num(ring, nan=0.0)


def test_ragged_decode_full_batch_ring_sliding_layer():
    """The benchmark's ring variant: the batch-64 sliding layer on rings of 1024 slots (one
    CTA per (sequence, KV head), no split), appended inside the launch."""
    import mixed_sliding_global_gb300 as g
    w = synth.ragged_decode(n_layers=6)
    spec, msl = w.layers[0], max(w.ctx_lens)
    assert g.gemma_attn_workspace_size(64, g.GEMMA_SLIDING_RING, 1024, 16, 8, 256, msl, 1) == 0
    hb = host_inputs(w, [0])
    gr = DeviceRun(w, hb)
    wp = hb[0].write_pos
    kr = [_ring_from_linear(gr.kc[0], wp, RING)]
    vr = [_ring_from_linear(gr.vc[0], wp, RING)]
    gr.kc[0] = gr.vc[0] = None   # the linear caches are not needed on the device any more
    torch.cuda.empty_cache()
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    d = gr.dev[0]
    out = torch.empty_like(d["q"])
    g.gemma_attn_decode_append(out, d["q"], kr, vr, w.owner_map, 0, d["k_new"], d["v_new"],
                               d["write_pos"], d["seq_lens"], msl, kind=g.GEMMA_SLIDING_RING,
                               window=spec.window, n_kv=spec.n_kv, k_eq_v=False,
                               kv_capacity=RING, scale=w.scale(0), workspace=ws,
                               device_error=gr.err)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    seqs = _sampled(w)
    compare(out[seqs].cpu(), _oracle_on(w, 0, seqs), BF16)


def _pool(cache, B, cap, seed):
    """The cache as a pool of PAGE-key pages through a shuffled block table."""
    max_pages = -(-cap // PAGE)
    n_pages = B * max_pages + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    table = perm[:B * max_pages].view(B, max_pages).to(torch.int32)
    n_kv, d = cache.shape[1], cache.shape[3]
    # rows the generator did not write stay NaN, in the pages and the spare pages alike
    pool = torch.full((n_pages, n_kv, PAGE, d), float("nan"), dtype=cache.dtype, device=cache.device)
    padded = torch.full((B, n_kv, max_pages * PAGE, d), float("nan"), dtype=cache.dtype,
                        device=cache.device)
    padded[:, :, :cap] = cache
    blocks = padded.view(B, n_kv, max_pages, PAGE, d).permute(0, 2, 1, 3, 4)
    pool[table.long().view(-1).to(cache.device)] = blocks.reshape(B * max_pages, n_kv, PAGE, d)
    return pool, table.to(cache.device), max_pages, n_pages


@pytest.mark.parametrize("layer", [0, 5])
def test_ragged_decode_full_batch_paged(layer):
    """The benchmark's paged variant at batch 64 (pages of 256 keys), both layer kinds, with
    the append inside the launch: the sliding layer unsplit, the global layer split."""
    import mixed_sliding_global_gb300 as g
    w = synth.ragged_decode(n_layers=6)
    spec, msl = w.layers[layer], max(w.ctx_lens)
    ws_n = g.gemma_attn_workspace_size_paged(64, spec.kind, spec.window, spec.n_q, spec.n_kv,
                                             spec.head_dim, msl, 1)
    assert (ws_n == 0) == (spec.kind == SLIDING)
    hb = host_inputs(w, [layer])
    gr = DeviceRun(w, hb)
    kp, table, max_pages, n_pages = _pool(gr.kc[layer], 64, w.capacity, seed=11 + layer)
    vp = None
    if gr.vc[layer] is not None:
        vp = _pool(gr.vc[layer], 64, w.capacity, seed=11 + layer)[0]
    gr.kc[layer] = gr.vc[layer] = None
    torch.cuda.empty_cache()
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    d = gr.dev[layer]
    out = torch.empty_like(d["q"])
    g.gemma_attn_paged(out, d["q"], [kp], [vp], [0], 0, d["seq_lens"], table, msl,
                       kind=spec.kind, window=spec.window, n_kv=spec.n_kv, k_eq_v=spec.k_eq_v,
                       scale=w.scale(layer), k_new=d["k_new"], v_new=d.get("v_new"),
                       write_pos=d["write_pos"], workspace=ws, device_error=gr.err)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    seqs = _sampled(w)
    compare(out[seqs].cpu(), _oracle_on(w, layer, seqs), BF16)


def test_prefill_bucket_full_batch_middle_tiles():
    """The benchmark's prefill bucket (batch 4, 512 tokens onto 3584) on both layer kinds,
    checked on query tokens that include middle 128-row tiles of both kinds (tokens 192-255:
    sliding tile 3, global tiles 24-31) and the first and last tokens."""
    import mixed_sliding_global_gb300 as g
    w = synth.prefill_12b(n_layers=6, batch=4)
    for l in (0, 5):
        s = w.layers[l]
        assert g.gemma_attn_workspace_size(4, s.kind, s.window, s.n_q, s.n_kv, s.head_dim,
                                           max(w.ctx_lens), w.n_new) == 0
    hb = host_inputs(w, [0, 5])
    gr = DeviceRun(w, hb)
    got = {}
    for l in (0, 5):
        gr.append(l)
        got[l] = gr.attend(l)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    for qr in ((0, 4), (192, 256), (508, 512)):
        ref = oracle_outputs(w, hb, [0, 5], q_range=qr)
        for l in (0, 5):
            compare(got[l][:, qr[0]:qr[1]].cpu(), ref[l], BF16)
