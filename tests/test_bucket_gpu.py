"""GPU: padded prefill buckets. Each sequence brings n_new rows of which the first n_real[b]
are real: the real rows must match the oracle run on those rows alone, the pad rows' outputs
must be exactly zero, and the pad rows must never reach the cache."""
import pytest
import torch

import mixed_sliding_global_gb300 as g
from harness import BF16_MAX_ABS, compare, host_inputs
from oracle import load_oracle
from synth import BF16, FP32, GLOBAL, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu


def one_layer(spec, n_new, prefixes, cap, dtype=BF16):
    ctx = [p + n_new for p in prefixes]
    return Workload("bucket", [spec], [0], len(ctx), dtype, n_new, ctx, cap)


def oracle_bucket(w, hb, n_real):
    """Oracle: append only the real rows of each sequence, then attend with those rows alone;
    pad rows are zero. Returns (out [B][n_new][n_q][d] fp64, K cache, V cache)."""
    orc = load_oracle()
    b0 = hb[0]
    spec = w.layers[0]
    kc = b0.k_cache.clone()
    vc = b0.v_cache.clone() if b0.v_cache is not None else None
    out = torch.zeros(b0.q.shape, dtype=torch.float64)
    for b, nr in enumerate(n_real):
        wp = int(b0.write_pos[b])
        if nr == 0:
            continue
        orc.kv_append(kc[b:b + 1], b0.k_new[b:b + 1, :nr].contiguous(), [wp])
        if vc is not None:
            orc.kv_append(vc[b:b + 1], b0.v_new[b:b + 1, :nr].contiguous(), [wp])
        q = b0.q[b:b + 1, :nr].contiguous()
        o = orc.attention(w.layers, w.owner_map, 0, [kc[b:b + 1].contiguous()],
                          [vc[b:b + 1].contiguous() if vc is not None else None], q, [wp + nr],
                          w.scale(0))
        out[b, :nr] = o[0]
    return out, kc, vc


def gpu_bucket(w, hb, n_real, err=None):
    spec, b0 = w.layers[0], hb[0]
    dev = "cuda"
    kc = [b0.k_cache.to(dev)]
    vc = [b0.v_cache.to(dev) if b0.v_cache is not None else None]
    nr = torch.tensor(n_real, dtype=torch.int32, device=dev)
    wp = b0.write_pos.to(dev)
    lens = (b0.write_pos + torch.tensor(n_real, dtype=torch.int32).clamp(min=0)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev) if err is None else err
    g.gemma_kv_append_bucket(kc, vc, [0], 0, b0.k_new.to(dev),
                             b0.v_new.to(dev) if b0.v_new is not None else None, wp, nr,
                             k_eq_v=spec.k_eq_v, device_error=err)
    q = b0.q.to(dev)
    out = torch.full_like(q, 7.0)
    msl = max(w.ctx_lens)
    ws_n = g.gemma_attn_workspace_size(w.batch, spec.kind, spec.window, spec.n_q, spec.n_kv,
                                       spec.head_dim, msl, w.n_new)
    ws = torch.zeros(max(ws_n, 1), dtype=torch.uint8, device=dev)
    g.gemma_attn_prefill_bucket(out, q, kc, vc, [0], 0, lens, nr, msl, kind=spec.kind,
                                window=spec.window, n_kv=spec.n_kv, k_eq_v=spec.k_eq_v,
                                scale=w.scale(0), workspace=ws, device_error=err)
    torch.cuda.synchronize()
    return out, kc[0], vc[0], err


def same_with_nan(a, b):
    a, b = a.cpu(), b.cpu()
    na, nb = torch.isnan(a.float()), torch.isnan(b.float())
    return torch.equal(na, nb) and torch.equal(a[~na], b[~nb])


CASES = [
    # spec, n_new, prefixes, cap, n_real
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 64, [1200, 40, 300], 1280, [64, 21, 0]),
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 64, [500, 7, 130], 576, [1, 64, 37]),
    (LayerSpec(SLIDING, 37, 8, 1, 64, False), 128, [90, 0], 256, [100, 128]),
    (LayerSpec(GLOBAL, 0, 8, 2, 128, False), 16, [33, 250], 272, [16, 5]),
]


@pytest.mark.parametrize("dtype", [BF16, FP32])
@pytest.mark.parametrize("spec,n_new,prefixes,cap,n_real", CASES)
def test_bucket_matches_oracle(spec, n_new, prefixes, cap, n_real, dtype):
    w = one_layer(spec, n_new, prefixes, cap, dtype)
    hb = host_inputs(w, [0])
    ref, kref, vref = oracle_bucket(w, hb, n_real)
    out, kc, vc, err = gpu_bucket(w, hb, n_real)
    assert err.item() == 0
    for b, nr in enumerate(n_real):
        assert out[b, nr:].abs().sum().item() == 0, "pad rows must be zero"
        if nr:
            compare(out[b:b + 1, :nr], ref[b:b + 1, :nr], dtype)
    # pad rows never reach the cache: it equals the oracle's real-rows-only append (NaN where
    # nothing was written)
    assert same_with_nan(kc, kref)
    if vc is not None:
        assert same_with_nan(vc, vref)


def test_full_bucket_is_the_plain_prefill():
    spec = LayerSpec(GLOBAL, 0, 16, 1, 512, True)
    w = one_layer(spec, 96, [400, 900], 1024)
    hb = host_inputs(w, [0])
    out, kc, _, err = gpu_bucket(w, hb, [96, 96])
    b0 = hb[0]
    kc2 = [b0.k_cache.cuda()]
    g.gemma_kv_append(kc2, [None], [0], 0, b0.k_new.cuda(), None, b0.write_pos.cuda(), k_eq_v=True)
    q = b0.q.cuda()
    plain = torch.empty_like(q)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    g.gemma_attn_prefill(plain, q, kc2, [None], [0], 0, b0.seq_lens.cuda(), max(w.ctx_lens),
                         kind=spec.kind, window=0, n_kv=1, k_eq_v=True, scale=w.scale(0),
                         workspace=ws)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out, plain)


def test_bad_n_real_is_reported_and_zeroed():
    spec = LayerSpec(SLIDING, 1024, 16, 8, 256, False)
    w = one_layer(spec, 32, [100, 100], 192)
    hb = host_inputs(w, [0])
    n_real = [33, 10]   # 33 > n_new
    out, _, _, err = gpu_bucket(w, hb, n_real)
    assert err.item() & g.GEMMA_DEVERR_N_REAL
    assert out[0].abs().sum().item() == 0
    assert out[1, :10].abs().sum().item() > 0 and out[1, 10:].abs().sum().item() == 0


@pytest.mark.parametrize("d,kind,n_q,n_kv,keqv", [(256, SLIDING, 16, 8, False),
                                                  (512, GLOBAL, 16, 1, True)])
def test_prefill_bad_seq_len_is_reported_and_zeroed(d, kind, n_q, n_kv, keqv):
    """A sequence whose length is below its new tokens: reported, its rows zeros; the other
    sequence is unaffected (both CTA-pair kernels)."""
    B, n_new, cap = 2, 40, 256
    gen = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, n_new, n_q, d, device="cuda", generator=gen).bfloat16()
    kc = torch.randn(B, n_kv, cap, d, device="cuda", generator=gen).bfloat16()
    vc = None if keqv else torch.randn(B, n_kv, cap, d, device="cuda", generator=gen).bfloat16()
    lens = torch.tensor([100, 20], dtype=torch.int32, device="cuda")   # 20 < n_new
    out = torch.full_like(q, 7.0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g.gemma_attn_prefill(out, q, [kc], [vc], [0], 0, lens, 100, kind=kind,
                         window=64 if kind == SLIDING else 0, n_kv=n_kv, k_eq_v=keqv,
                         scale=d ** -0.5, device_error=err)
    torch.cuda.synchronize()
    assert err.item() & g.GEMMA_DEVERR_SEQ_LEN
    assert out[1].float().abs().sum().item() == 0
    assert torch.isfinite(out[0].float()).all() and out[0].float().abs().sum().item() > 0
