"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element.

Tolerances (stated by the method's target): bf16 outputs with fp32 accumulation must be within
max |err| <= 2e-2 and mean |err| <= 2e-3 of the oracle; the fp32 debug path within 1e-4.
Every cache is NaN outside the rows the generator wrote, so any read outside the window or
past a sequence's length poisons the output and fails the comparison.
"""
import pytest
import torch

import synth
from synth import GLOBAL, SLIDING, BF16, FP32, LayerSpec, Workload
from harness import DeviceRun, compare, host_inputs, oracle_outputs

pytestmark = pytest.mark.gpu


def run_and_compare(w, layers, seqs=None, q_range=None, max_seq_len=None, prefill_entry=False):
    hb = host_inputs(w, layers, seqs)
    ref = oracle_outputs(w, hb, layers, q_range)
    gr = DeviceRun(w, hb)
    got = {}
    for l in layers:
        if w.is_owner(l):
            gr.append(l)
        got[l] = gr.attend(l, max_seq_len, prefill_entry=prefill_entry)
    torch.cuda.synchronize()
    assert gr.err.item() == 0, f"device error word {gr.err.item()}"
    errs = {}
    for l in layers:
        g = got[l]
        if q_range is not None:
            g = g[:, q_range[0]:q_range[1]]
        errs[l] = compare(g, ref[l], w.dtype)
    return errs


# ------------------------------------------------------------------------------------------
# the tiny case, fp32 debug path (<= 1e-4)
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("mode,ctx", [("decode", 64), ("prefill", 64), ("prefill", 72)])
def test_tiny_fp32(mode, ctx):
    run_and_compare(synth.tiny(mode, ctx=ctx), [0, 1])


def test_tiny_bf16():
    w = synth.tiny("decode")
    w.dtype = BF16
    run_and_compare(w, [0, 1])
    w = synth.tiny("prefill")
    w.dtype = BF16
    run_and_compare(w, [0, 1])


# ------------------------------------------------------------------------------------------
# shape sweep: several tiles, ragged tails, every head_dim and group size, both kinds
# ------------------------------------------------------------------------------------------
def one_layer(spec, n_new, ctx_lens, cap, dtype=BF16):
    return Workload("sweep", [spec], [0], len(ctx_lens), dtype, n_new, list(ctx_lens), cap)


DECODE_SHAPES = [
    # spec, ctx_lens, cap
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [8192], 8192),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), [8192], 8192),
    (LayerSpec(SLIDING, 512, 8, 2, 256, False), [2048], 2048),
    (LayerSpec(GLOBAL, 0, 8, 2, 256, False), [2048], 2048),
    (LayerSpec(GLOBAL, 0, 4, 4, 64, False), [1, 2, 33, 100, 1000], 1024),
    (LayerSpec(SLIDING, 37, 8, 1, 128, False), [5, 37, 38, 300], 320),
    (LayerSpec(GLOBAL, 0, 16, 4, 128, True), [777, 31, 4097], 4160),
    (LayerSpec(SLIDING, 100, 16, 16, 64, True), [3, 250], 256),
    (LayerSpec(SLIDING, 1, 2, 1, 256, False), [1, 9], 16),
    (LayerSpec(GLOBAL, 0, 8, 1, 512, False), [63, 64, 65, 3000], 3008),
]


@pytest.mark.parametrize("case", range(len(DECODE_SHAPES)))
def test_decode_shapes(case):
    spec, lens, cap = DECODE_SHAPES[case]
    run_and_compare(one_layer(spec, 1, lens, cap), [0])


@pytest.mark.parametrize("case", [0, 4, 5, 8])
def test_decode_shapes_fp32(case):
    spec, lens, cap = DECODE_SHAPES[case]
    run_and_compare(one_layer(spec, 1, lens, cap, FP32), [0])


PREFILL_SHAPES = [
    # spec, n_new, ctx_lens, cap, q_range
    (LayerSpec(SLIDING, 7, 4, 2, 64, False), 13, [13, 20, 50], 64, None),
    (LayerSpec(GLOBAL, 0, 2, 1, 128, True), 9, [9, 100], 128, None),
    (LayerSpec(SLIDING, 64, 8, 8, 512, False), 33, [40, 200], 200, None),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 40, [40, 333], 352, None),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 512, [4096], 4096, (0, 24)),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 512, [4096], 4096, (488, 512)),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 512, [4096], 4096, (0, 8)),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 512, [4096], 4096, (504, 512)),
    # several 128-row tiles on the tensor-memory path (head_dim <= 256)
    (LayerSpec(GLOBAL, 0, 16, 1, 256, True), 100, [100, 700], 704, None),
    (LayerSpec(SLIDING, 130, 8, 2, 128, False), 300, [300, 1000], 1024, None),
    (LayerSpec(GLOBAL, 0, 1, 1, 64, False), 200, [333, 200], 352, None),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 160, [4096, 1500], 4096, None),
    (LayerSpec(SLIDING, 5, 4, 4, 256, True), 70, [90, 71], 96, None),
    # head_dim 256 runs on CTA pairs: 96 units of 256 rows, more than there are pairs, so a pair
    # walks several units (each a few 128-key tiles); every output compared
    (LayerSpec(SLIDING, 256, 4, 2, 256, False), 768, [868, 800, 900, 768, 1000, 850, 790, 880],
     1024, None),
    # groups of 4 and 8 query heads on the pair kernels (Q and output boxes of G heads x 128 / G
    # tokens)
    (LayerSpec(SLIDING, 100, 16, 4, 256, False), 70, [200, 90], 256, None),
    (LayerSpec(GLOBAL, 0, 8, 1, 512, True), 50, [120, 50], 128, None),
    # head_dim 512 runs on clusters of two pairs: 40 units, more than there are clusters
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 64, [164, 67, 314, 128, 64, 244, 97, 264, 192, 141],
     320, None),
    # a window of one key on the pair kernels: every query attends only itself (the output is
    # its own V row), so most of each 128-key tile is masked for every row, and at head_dim 512
    # the partners swap partial scores that are mostly masked
    (LayerSpec(SLIDING, 1, 4, 2, 256, False), 40, [40, 300], 320, None),
    (LayerSpec(SLIDING, 1, 4, 1, 512, True), 20, [20, 150], 160, None),
]


@pytest.mark.parametrize("case", range(len(PREFILL_SHAPES)))
def test_prefill_shapes(case):
    spec, n_new, lens, cap, qr = PREFILL_SHAPES[case]
    run_and_compare(one_layer(spec, n_new, lens, cap), [0], q_range=qr)


# One new token through the prefill entry (served by the decode kernels, split over key chunks
# with the workspace), with a sequence of length 1 whose token attends only itself.
@pytest.mark.parametrize("spec", [LayerSpec(GLOBAL, 0, 2, 1, 256, False),
                                  LayerSpec(SLIDING, 3, 16, 1, 512, True)])
def test_prefill_entry_with_one_new_token(spec):
    run_and_compare(one_layer(spec, 1, [1, 77, 130], 160), [0], prefill_entry=True)


@pytest.mark.parametrize("case", [0, 1, 3])
def test_prefill_shapes_fp32(case):
    spec, n_new, lens, cap, qr = PREFILL_SHAPES[case]
    run_and_compare(one_layer(spec, n_new, lens, cap, FP32), [0], q_range=qr)


# ------------------------------------------------------------------------------------------
# the workload configurations at full size
# ------------------------------------------------------------------------------------------
def test_e4b_decode_all_layers():
    """12 layers, 5:1 sliding/global, last four layers KV-shared, batch 1, context 2048."""
    w = synth.e4b_decode()
    run_and_compare(w, list(range(w.n_layers)))


def test_12b_decode_sliding_and_global():
    w = synth.b12_decode()
    run_and_compare(w, [0, 5])


def test_ragged_decode_sampled_sequences():
    """Batch 64 ragged lengths: sequences with the shortest, the longest and two more."""
    w = synth.ragged_decode(n_layers=6)
    lens = w.ctx_lens
    seqs = sorted({lens.index(min(lens)), lens.index(max(lens)), 7, 33})
    hb_w = Workload(w.name, w.layers, w.owner_map, len(seqs), w.dtype, 1,
                    [lens[s] for s in seqs], w.capacity)
    # the sampled sequences keep their own seeded inputs (seeds depend on the sequence index)
    hb = host_inputs(w, [0, 5], seqs)
    ref = oracle_outputs(hb_w, hb, [0, 5])
    gr = DeviceRun(hb_w, hb)
    for l in (0, 5):
        gr.append(l)
        got = gr.attend(l, max_seq_len=max(lens))
        torch.cuda.synchronize()
        compare(got, ref[l], w.dtype)
    assert gr.err.item() == 0


def test_prefill_bucket_sampled_queries():
    w = synth.prefill_12b(n_layers=6, batch=2)
    for qr in ((0, 8), (255, 263), (504, 512)):
        run_and_compare(w, [0, 5], q_range=qr)


# ------------------------------------------------------------------------------------------
# properties that hold at any size
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("spec", [LayerSpec(GLOBAL, 0, 16, 1, 512, True),
                                  LayerSpec(SLIDING, 1024, 16, 8, 256, False)])
def test_split_plan_does_not_change_the_result(spec):
    """A larger max_seq_len hint changes the split over keys; outputs agree within tolerance."""
    w = one_layer(spec, 1, [3000, 5000], 16448)
    hb = host_inputs(w, [0])
    ref = oracle_outputs(w, hb, [0])[0]
    outs = []
    for msl in (5000, 16448):
        gr = DeviceRun(w, hb)
        gr.append(0)
        outs.append(gr.attend(0, max_seq_len=msl))
        torch.cuda.synchronize()
        compare(outs[-1], ref, BF16)
    assert (outs[0].float() - outs[1].float()).abs().max().item() <= 2e-2


def test_workspace_is_reusable_across_calls():
    """The workspace holds no state between calls: consecutive decode calls with different batch
    and split plans on one workspace match calls on fresh workspaces bit for bit."""
    import mixed_sliding_global_gb300 as g
    cases = [(LayerSpec(GLOBAL, 0, 16, 1, 512, True), [3000, 5000, 777], 5056),
             (LayerSpec(SLIDING, 1024, 16, 8, 256, False), [4000, 1500], 4032),
             (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [9000], 9024)]
    shared = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for spec, lens, cap in cases:
            w = one_layer(spec, 1, lens, cap)
            hb = host_inputs(w, [0])
            gr = DeviceRun(w, hb)
            gr.append(0)
            fresh = gr.attend(0)
            d = gr.dev[0]
            out = torch.empty_like(fresh)
            g.gemma_attn_decode(out, d["q"], gr.kc, gr.vc, [0], 0, d["seq_lens"], max(lens),
                                kind=spec.kind, window=spec.window, n_kv=spec.n_kv,
                                k_eq_v=spec.k_eq_v, scale=w.scale(0), workspace=shared,
                                device_error=gr.err)
            torch.cuda.synchronize()
            assert gr.err.item() == 0
            assert torch.equal(out, fresh), (rep, spec)


def test_ragged_decode_full_batch_sliding_layer():
    """The batch-64 ragged decode's sliding layer in the launch configuration the benchmark
    times (512 (sequence, KV head) units fill the GPU: one CTA each, no split), checked on
    sampled sequences; their seeded inputs equal those of the full batch."""
    w = synth.ragged_decode(n_layers=6)
    lens = w.ctx_lens
    seqs = sorted({lens.index(min(lens)), lens.index(max(lens)), 7, 33, 63})
    hb = host_inputs(w, [0])
    gr = DeviceRun(w, hb)
    gr.append(0)
    got = gr.attend(0, max_seq_len=max(lens))
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    sub = Workload(w.name, w.layers, w.owner_map, len(seqs), w.dtype, 1, [lens[s] for s in seqs],
                   w.capacity)
    ref = oracle_outputs(sub, host_inputs(w, [0], seqs), [0])[0]
    compare(got[seqs].cpu(), ref, w.dtype)


def test_split_plan_of_the_benchmark_shapes():
    """The planner leaves the batch-64 sliding layers unsplit (their 512 units fill the GPU over
    1024-key windows: no scratch, no combine), splits the batch-1 sliding layers into at most
    eight chunks merged inside their cluster (no scratch), and splits the global layers over
    keys with a combine pass (scratch needed)."""
    import mixed_sliding_global_gb300 as g
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert 64 * 8 >= 2 * n_sm
    assert g.gemma_attn_workspace_size(64, SLIDING, 1024, 16, 8, 256, 16385, 1) == 0
    assert g.gemma_attn_workspace_size(64, g.GEMMA_SLIDING_RING, 1024, 16, 8, 256, 16385, 1) == 0
    assert g.gemma_attn_workspace_size_paged(64, SLIDING, 1024, 16, 8, 256, 16385, 1) == 0
    assert g.gemma_attn_workspace_size(64, GLOBAL, 0, 16, 1, 512, 16385, 1) > 0
    assert g.gemma_attn_workspace_size(1, SLIDING, 1024, 16, 8, 256, 8192, 1) == 0
    assert g.gemma_attn_workspace_size(1, GLOBAL, 0, 16, 1, 512, 8192, 1) > 0


# ------------------------------------------------------------------------------------------
# small grids whose split merges inside one thread-block cluster of 9 to 16 chunks (above the
# portable cluster size): every head_dim, K and V or K as V, both kinds, fused append included
# ------------------------------------------------------------------------------------------
BIG_CLUSTER_SHAPES = [
    # (spec, lens after the append, capacity); chunks = ceil(max len / 32) <= 16 and
    # batch x n_kv x chunks <= 152, so the plan keeps every chunk and merges in the cluster
    (LayerSpec(GLOBAL, 0, 8, 2, 64, False), [300, 450], 512),
    (LayerSpec(GLOBAL, 0, 16, 4, 128, True), [500], 512),
    (LayerSpec(SLIDING, 512, 16, 8, 256, False), [2000], 2048),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [350, 500, 129], 512),
    (LayerSpec(SLIDING, 300, 8, 1, 512, False), [1000, 290], 1024),
]


# latency-bound splits finer than a cluster holds (more than 16 chunks of 32 or 64 keys) whose
# keys fit 16 chunks of at most 128: coarsened to one 16-chunk cluster, no scratch, no combine
COARSENED_SHAPES = [
    (LayerSpec(GLOBAL, 0, 8, 2, 256, False), [2048], 2048),        # E4B's global layers
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [1500, 900], 1536),
    (LayerSpec(SLIDING, 1500, 8, 4, 128, True), [3000], 3008),
]


@pytest.mark.parametrize("case", range(len(COARSENED_SHAPES)))
def test_decode_coarsened_to_one_cluster(case):
    import mixed_sliding_global_gb300 as g
    spec, lens, cap = COARSENED_SHAPES[case]
    msl = max(lens)
    assert g.gemma_attn_workspace_size(len(lens), spec.kind, spec.window, spec.n_q, spec.n_kv,
                                       spec.head_dim, msl, 1) == 0
    run_and_compare(one_layer(spec, 1, lens, cap), [0])


@pytest.mark.parametrize("case", range(len(BIG_CLUSTER_SHAPES)))
def test_decode_in_big_clusters(case):
    import mixed_sliding_global_gb300 as g
    spec, lens, cap = BIG_CLUSTER_SHAPES[case]
    w = one_layer(spec, 1, lens, cap)
    msl = max(lens)
    n_read = min(spec.window, msl) if spec.kind == SLIDING else msl
    chunks = -(-n_read // 32)
    assert 8 < chunks <= 16 and len(lens) * spec.n_kv * chunks <= 152
    # a cluster plan needs no scratch
    assert g.gemma_attn_workspace_size(len(lens), spec.kind, spec.window, spec.n_q, spec.n_kv,
                                       spec.head_dim, msl, 1) == 0
    run_and_compare(w, [0])
    # the same launch with the step's K/V row written inside it
    hb = host_inputs(w, [0])
    ref = oracle_outputs(w, hb, [0])
    gr = DeviceRun(w, hb)
    d = gr.dev[0]
    out = torch.empty_like(d["q"])
    g.gemma_attn_decode_append(out, d["q"], gr.kc, gr.vc, w.owner_map, 0, d["k_new"],
                               d.get("v_new"), d["write_pos"], d["seq_lens"], msl,
                               kind=spec.kind, window=spec.window, n_kv=spec.n_kv,
                               k_eq_v=spec.k_eq_v, scale=w.scale(0),
                               workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"),
                               device_error=gr.err)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    compare(out.cpu(), ref[0], BF16)
