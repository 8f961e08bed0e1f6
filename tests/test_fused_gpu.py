"""GPU: gemma_attn_decode_append (the append inside the decode launch) equals the two-launch
append + decode bit for bit (outputs and caches), and matches the oracle."""
import pytest
import torch

import mixed_sliding_global_gb300 as g
from harness import DeviceRun, compare, host_inputs, oracle_outputs
from synth import BF16, FP32, GLOBAL, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu


def one_layer(spec, ctx_lens, cap, dtype=BF16):
    return Workload("fused", [spec], [0], len(ctx_lens), dtype, 1, list(ctx_lens), cap)


def bits(t):
    """Bitwise view (the synthetic caches hold NaN outside the rows they generate)."""
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def fused(gr, w, l=0, write_pos=None):
    spec, d = w.layers[l], gr.dev[w.owner_map[l]]
    q = gr.dev[l]["q"]
    out = torch.empty_like(q)
    msl = max(w.ctx_lens)
    ws_n = g.gemma_attn_workspace_size(q.shape[0], spec.kind, spec.window, spec.n_q, spec.n_kv,
                                       spec.head_dim, msl, 1)
    ws = torch.zeros(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    g.gemma_attn_decode_append(out, q, gr.kc, gr.vc, w.owner_map, l, d.get("k_new"),
                               d.get("v_new"), d["write_pos"] if write_pos is None else write_pos,
                               gr.dev[l]["seq_lens"], msl, kind=spec.kind, window=spec.window,
                               n_kv=spec.n_kv, k_eq_v=spec.k_eq_v, scale=w.scale(l), workspace=ws,
                               device_error=gr.err)
    torch.cuda.synchronize()
    return out


SHAPES = [
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [8192, 100, 3000], 8192),     # split keys
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), [5000, 700], 5056),
    (LayerSpec(SLIDING, 512, 8, 2, 256, False), [2048], 2048),
    (LayerSpec(GLOBAL, 0, 4, 4, 64, False), [1, 2, 33, 1000], 1024),
    (LayerSpec(SLIDING, 37, 8, 1, 128, False), [5, 37, 38, 300], 320),
]


@pytest.mark.parametrize("dtype", [BF16, FP32])
@pytest.mark.parametrize("spec,ctx,cap", SHAPES)
def test_fused_equals_append_then_decode(spec, ctx, cap, dtype):
    w = one_layer(spec, ctx, cap, dtype)
    hb = host_inputs(w, [0])
    two = DeviceRun(w, hb)
    two.append(0)
    ref = two.attend(0)
    torch.cuda.synchronize()
    one = DeviceRun(w, hb)
    got = fused(one, w)
    assert one.err.item() == 0 and two.err.item() == 0
    assert torch.equal(got, ref)
    assert torch.equal(bits(one.kc[0]), bits(two.kc[0]))
    if one.vc[0] is not None:
        assert torch.equal(bits(one.vc[0]), bits(two.vc[0]))
    compare(got, oracle_outputs(w, hb, [0])[0], dtype)


def test_fused_slot_before_the_last_position_and_outside_the_window():
    """The new row may go to any slot: one inside the attended range (written by the CTA whose
    chunk holds it, before it reads the chunk) or one outside it (written, not read)."""
    spec = LayerSpec(SLIDING, 64, 8, 2, 256, False)
    w = one_layer(spec, [3000, 3000], 3008)
    hb = host_inputs(w, [0])
    for wp in ([2995, 100], [2999, 2990]):
        pos = torch.tensor(wp, dtype=torch.int32)
        two, one = DeviceRun(w, hb), DeviceRun(w, hb)
        for gr in (two, one):   # the last slot holds finite data when the new row goes elsewhere
            gr.kc[0][:, :, 2999] = 0.25
            gr.vc[0][:, :, 2999] = -0.5
        two.dev[0]["write_pos"] = pos.cuda()
        two.append(0)
        ref = two.attend(0)
        got = fused(one, w, write_pos=pos.cuda())
        assert one.err.item() == 0
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)
        assert torch.equal(bits(one.kc[0]), bits(two.kc[0]))
        assert torch.equal(bits(one.vc[0]), bits(two.vc[0]))


def test_fused_on_a_shared_layer_is_plain_decode():
    layers = [LayerSpec(GLOBAL, 0, 8, 2, 256, False)] * 2
    w = Workload("fused_shared", layers, [0, 0], 2, BF16, 1, [900, 2000], 2048)
    hb = host_inputs(w, [0, 1])
    gr = DeviceRun(w, hb)
    gr.append(0)
    ref = gr.attend(1)
    before = gr.kc[0].clone()
    got = fused(gr, w, l=1)
    assert torch.equal(got, ref)
    assert torch.equal(bits(gr.kc[0]), bits(before))


def test_fused_write_pos_out_of_range_is_reported():
    spec = LayerSpec(GLOBAL, 0, 4, 1, 64, True)
    w = one_layer(spec, [60, 60], 64)
    hb = host_inputs(w, [0])
    gr = DeviceRun(w, hb)
    before = gr.kc[0].clone()
    fused(gr, w, write_pos=torch.tensor([64, 59], dtype=torch.int32, device="cuda"))
    assert gr.err.item() & g.GEMMA_DEVERR_WRITE_POS
    after = gr.kc[0]
    assert torch.equal(after[0].view(torch.int16), before[0].view(torch.int16))  # nothing written
    assert torch.equal(after[1, :, 59].cpu(), hb[0].k_new[1, 0])
