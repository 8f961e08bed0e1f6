"""GPU: the paged KV pool. The logical cache of each owner layer is scattered into a shared
pool of pages through a shuffled block table (with spare pages the table never names); the
paged entry points must give the oracle's outputs on the logical cache, and the paged append
must place the new rows exactly where the plain append does (gathered back, bit for bit)."""
import pytest
import torch

from harness import DeviceRun, compare, host_inputs, oracle_outputs
import synth
from synth import BF16, FP32, GLOBAL, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu


def one_layer(spec, n_new, ctx_lens, cap, dtype=BF16):
    return Workload("paged", [spec], [0], len(ctx_lens), dtype, n_new, list(ctx_lens), cap)


def make_table(B, cap, page, seed, spare=5):
    max_pages = -(-cap // page)
    n_pages = B * max_pages + spare
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    table = perm[:B * max_pages].view(B, max_pages).to(torch.int32).contiguous()
    return table, n_pages


def to_pool(cache, table, n_pages, page):
    """[B][n_kv][cap][d] -> [n_pages][n_kv][page][d] through the block table (spare pages NaN)."""
    B, n_kv, cap, d = cache.shape
    max_pages = table.shape[1]
    padded = torch.full((B, n_kv, max_pages * page, d), float("nan"), dtype=cache.dtype,
                        device=cache.device)
    padded[:, :, :cap] = cache
    pool = torch.full((n_pages, n_kv, page, d), float("nan"), dtype=cache.dtype,
                      device=cache.device)
    blocks = padded.view(B, n_kv, max_pages, page, d).permute(0, 2, 1, 3, 4)
    pool[table.long().view(-1).to(cache.device)] = blocks.reshape(B * max_pages, n_kv, page, d)
    return pool


def from_pool(pool, table, cap):
    B, max_pages = table.shape
    n_pages, n_kv, page, d = pool.shape
    blocks = pool[table.long().view(-1).to(pool.device)].view(B, max_pages, n_kv, page, d)
    return blocks.permute(0, 2, 1, 3, 4).reshape(B, n_kv, max_pages * page, d)[:, :, :cap]


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def run_paged(w, page, seed, fused=False, softcap=None):
    import mixed_sliding_global_gb300 as g
    hb = host_inputs(w, [0])
    ref = oracle_outputs(w, hb, [0])[0]
    gr = DeviceRun(w, hb)
    spec, d = w.layers[0], gr.dev[0]
    B = len(w.ctx_lens)
    table, n_pages = make_table(B, w.capacity, page, seed)
    tdev = table.cuda()
    # pools from the caches before this step's append
    kp = [to_pool(gr.kc[0], table, n_pages, page)]
    vp = [to_pool(gr.vc[0], table, n_pages, page) if gr.vc[0] is not None else None]
    # the plain append gives the expected cache contents
    gr.append(0)
    msl = max(w.ctx_lens)
    ws_n = g.gemma_attn_workspace_size_paged(B, spec.kind, spec.window, spec.n_q, spec.n_kv,
                                             spec.head_dim, msl, w.n_new)
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    kw = dict(kind=spec.kind, window=spec.window, n_kv=spec.n_kv, k_eq_v=spec.k_eq_v,
              scale=w.scale(0), workspace=ws, device_error=gr.err)
    if fused:
        g.gemma_attn_paged(out, d["q"], kp, vp, [0], 0, d["seq_lens"], tdev, msl,
                           k_new=d["k_new"], v_new=d.get("v_new"), write_pos=d["write_pos"], **kw)
    else:
        g.gemma_kv_append_paged(kp, vp, [0], 0, d["k_new"], d.get("v_new"), d["write_pos"], tdev,
                                k_eq_v=spec.k_eq_v, device_error=gr.err)
        g.gemma_attn_paged(out, d["q"], kp, vp, [0], 0, d["seq_lens"], tdev, msl, **kw)
    torch.cuda.synchronize()
    assert gr.err.item() == 0, gr.err.item()
    compare(out, ref, w.dtype)
    # every cache row the step can read or wrote, bit for bit (rows never written stay NaN on
    # both sides, so compare bit patterns)
    assert torch.equal(bits(from_pool(kp[0], table, w.capacity)), bits(gr.kc[0]))
    if vp[0] is not None:
        assert torch.equal(bits(from_pool(vp[0], table, w.capacity)), bits(gr.vc[0]))


CASES = [
    # spec, n_new, ctx_lens, cap, page
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 1, [1, 129, 1000, 4097], 4224, 128),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 1, [5, 1025, 3000], 3072, 256),
    (LayerSpec(SLIDING, 512, 8, 2, 256, False), 1, [2048, 700], 2048, 128),
    (LayerSpec(GLOBAL, 0, 8, 2, 256, False), 1, [2048, 33], 2048, 384),
    (LayerSpec(SLIDING, 37, 8, 1, 128, False), 1, [5, 37, 38, 300], 384, 128),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 40, [40, 333], 384, 128),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 200, [1500, 200], 1536, 256),
    (LayerSpec(GLOBAL, 0, 16, 4, 128, True), 100, [100, 700], 768, 128),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_paged_matches_oracle(case):
    spec, n_new, lens, cap, page = CASES[case]
    run_paged(one_layer(spec, n_new, lens, cap), page, seed=case)


@pytest.mark.parametrize("case", [0, 1, 2, 3, 4])
def test_paged_fused_append_decode(case):
    spec, n_new, lens, cap, page = CASES[case]
    run_paged(one_layer(spec, n_new, lens, cap), page, seed=100 + case, fused=True)


@pytest.mark.parametrize("case", [0, 1, 5])
def test_paged_fp32_debug_path(case):
    spec, n_new, lens, cap, page = CASES[case]
    run_paged(one_layer(spec, n_new, lens, cap, FP32), page, seed=200 + case)


def test_ragged_batch_sampled_sequences():
    """The ragged batch-64 decode's global layer at full size, pages of 256 keys, on the
    shortest and longest sequences and two more (the oracle runs on those only)."""
    w = synth.ragged_decode(n_layers=6)
    lens = w.ctx_lens
    pick = sorted({lens.index(min(lens)), lens.index(max(lens)), 7, 40})
    spec = w.layers[5]
    sub = Workload("ragged-paged", [spec], [0], len(pick), BF16, 1, [lens[i] for i in pick],
                   w.capacity)
    run_paged(sub, 256, seed=300)


def test_bad_page_index_is_reported_not_read():
    """A block-table entry outside the pool sets GEMMA_DEVERR_PAGE; its rows read as zeros and
    nothing is written through it (the rest of the pool is unchanged)."""
    import mixed_sliding_global_gb300 as g
    spec = LayerSpec(GLOBAL, 0, 16, 1, 512, True)
    w = one_layer(spec, 1, [300, 500], 512)
    hb = host_inputs(w, [0])
    gr = DeviceRun(w, hb)
    d = gr.dev[0]
    table, n_pages = make_table(2, 512, 128, seed=7)
    kp = [to_pool(gr.kc[0], table, n_pages, 128)]
    before = kp[0].clone()
    table[1, 3] = n_pages + 4   # holds positions 384..511 of sequence 1, including its new row
    tdev = table.cuda()
    ws = torch.zeros(max(g.gemma_attn_workspace_size_paged(2, GLOBAL, 0, 16, 1, 512, 500, 1),
                         16), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    g.gemma_attn_paged(out, d["q"], kp, [None], [0], 0, d["seq_lens"], tdev, 500, kind=GLOBAL,
                       window=0, n_kv=1, k_eq_v=True, scale=w.scale(0), k_new=d["k_new"],
                       write_pos=d["write_pos"], workspace=ws, device_error=gr.err)
    torch.cuda.synchronize()
    assert gr.err.item() & g.GEMMA_DEVERR_PAGE
    # sequence 0's new row went to its own page; nothing else in the pool changed
    changed = (bits(kp[0]) != bits(before)).any(dim=-1).nonzero().tolist()
    p0 = int(table[0, 299 // 128])
    assert all(pg == p0 for pg, _, _ in changed) and len(changed) == 1
