"""GPU: sliding layers whose cache is a ring of R slots (GEMMA_SLIDING_RING: position p at slot
p % R). The oracle runs on the ordinary linear cache; the GPU on a ring built from it, with
contexts several times longer than the ring."""
import pytest
import torch

import mixed_sliding_global_gb300 as g
from harness import compare, host_inputs, oracle_outputs
from synth import BF16, FP32, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu


def one_layer(spec, n_new, ctx_lens, dtype=BF16):
    cap = max(ctx_lens) + 64
    return Workload("ring", [spec], [0], len(ctx_lens), dtype, n_new, list(ctx_lens), cap)


def to_ring(lin, write_pos, R):
    """ring[b, :, p % R] = lin[b, :, p] for the last R positions before write_pos[b]; every
    slot holds finite data (a ring holds real past tokens)."""
    B, H, _, d = lin.shape
    lin = torch.nan_to_num(lin, nan=0.0)
    ring = torch.zeros((B, H, R, d), dtype=lin.dtype)
    for b in range(B):
        pre = int(write_pos[b])
        for p in range(max(0, pre - R), pre):
            ring[b, :, p % R] = lin[b, :, p]
    return ring


def expected_ring(lin_appended, lens, R):
    B, H, _, d = lin_appended.shape
    ring = torch.zeros((B, H, R, d), dtype=lin_appended.dtype)
    for b in range(B):
        for p in range(max(0, lens[b] - R), lens[b]):
            ring[b, :, p % R] = lin_appended[b, :, p]
    return ring


def run_ring(w, R, fused=False, ring_in=None, softcap=None, q_gain=1.0):
    spec = w.layers[0]
    hb = host_inputs(w, [0])
    b0 = hb[0]
    b0.q.mul_(q_gain)  # (a power of two: exact in bf16)
    dev = "cuda"
    kr = to_ring(b0.k_cache, b0.write_pos, R).to(dev)
    vr = to_ring(b0.v_cache, b0.write_pos, R).to(dev) if b0.v_cache is not None else None
    q = b0.q.to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    msl = max(w.ctx_lens)
    ws_n = g.gemma_attn_workspace_size(w.batch, g.GEMMA_SLIDING_RING, spec.window, spec.n_q,
                                       spec.n_kv, spec.head_dim, msl, w.n_new)
    ws = torch.zeros(max(ws_n, 1), dtype=torch.uint8, device=dev)
    kw = dict(kind=g.GEMMA_SLIDING_RING, window=spec.window, n_kv=spec.n_kv,
              k_eq_v=spec.k_eq_v, scale=w.scale(0), workspace=ws, device_error=err)
    kn = b0.k_new.to(dev)
    vn = b0.v_new.to(dev) if b0.v_new is not None else None
    wp, lens = b0.write_pos.to(dev), b0.seq_lens.to(dev)
    if fused:
        g.gemma_attn_decode_append(out, q, [kr], [vr], [0], 0, kn, vn, wp, lens, msl, **kw)
    else:
        g.gemma_kv_append_ring([kr], [vr], [0], 0, kn, vn, wp, k_eq_v=spec.k_eq_v,
                               device_error=err)
        if softcap is not None:
            g.gemma_attn_softcap(out, q, [kr], [vr], [0], 0, lens, msl, softcap=softcap, **kw)
        else:
            fn = g.gemma_attn_decode if w.n_new == 1 else g.gemma_attn_prefill
            fn(out, q, [kr], [vr], [0], 0, lens, msl, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0
    return hb, out, kr, vr


CASES = [
    # spec, n_new, ctx_lens, R
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 1, [8192, 1500, 900, 1025], 1024),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 1, [5000, 3333], 1280),
    (LayerSpec(SLIDING, 512, 8, 2, 256, False), 1, [2048, 700], 512),
    (LayerSpec(SLIDING, 37, 8, 1, 128, False), 1, [5, 37, 38, 300], 128),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 128, [3000, 1500], 1152),   # tcgen05 prefill
    (LayerSpec(SLIDING, 37, 8, 1, 64, False), 40, [300, 45], 128),
]


@pytest.mark.parametrize("dtype", [BF16, FP32])
@pytest.mark.parametrize("spec,n_new,ctx,R", CASES)
def test_ring_matches_oracle(spec, n_new, ctx, R, dtype):
    w = one_layer(spec, n_new, ctx, dtype)
    hb, out, kr, vr = run_ring(w, R)
    compare(out, oracle_outputs(w, hb, [0])[0], dtype)
    # the ring after the append: the last R tokens of every sequence at their slots
    b0 = hb[0]
    lin = torch.nan_to_num(b0.k_cache, nan=0.0).clone()
    linv = torch.nan_to_num(b0.v_cache, nan=0.0).clone()
    for b in range(w.batch):
        wp = int(b0.write_pos[b])
        lin[b, :, wp:wp + n_new] = b0.k_new[b].transpose(0, 1)
        linv[b, :, wp:wp + n_new] = b0.v_new[b].transpose(0, 1)
    lens = [int(x) for x in b0.seq_lens]
    assert torch.equal(kr.cpu(), expected_ring(lin, lens, R))
    assert torch.equal(vr.cpu(), expected_ring(linv, lens, R))


# the soft-capped entry point on ring caches: decode (split keys), the CTA-pair prefill, and the
# one-SM prefill at head_dim 64; queries scaled so that the cap bites
@pytest.mark.parametrize("case", [0, 4, 5])
def test_ring_softcap_matches_oracle(case):
    spec, n_new, ctx, R = CASES[case]
    w = one_layer(spec, n_new, ctx, BF16)
    hb, out, _, _ = run_ring(w, R, softcap=30.0, q_gain=2.0)
    compare(out, oracle_outputs(w, hb, [0], softcap=30.0)[0], BF16)


def test_ring_fused_decode_equals_append_then_decode():
    spec = LayerSpec(SLIDING, 1024, 16, 8, 256, False)
    w = one_layer(spec, 1, [9000, 1200, 50], BF16)
    _, out_two, kr_two, vr_two = run_ring(w, 1152)
    hb, out_one, kr_one, vr_one = run_ring(w, 1152, fused=True)
    assert torch.equal(out_one, out_two)
    assert torch.equal(kr_one, kr_two) and torch.equal(vr_one, vr_two)
    compare(out_one, oracle_outputs(w, hb, [0])[0], BF16)
