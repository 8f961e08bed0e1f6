"""GPU: the append kernel is a bit-exact placed copy; device-side range errors are reported."""
import pytest
import torch

import mixed_sliding_global_gb300 as g
from oracle import load_oracle

pytestmark = pytest.mark.gpu


def _rand(shape, seed, dtype):
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed)).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n_new,d,k_eq_v", [(1, 256, False), (512, 512, True), (7, 64, False),
                                            (3, 128, True)])
def test_append_matches_oracle_bit_exactly(dtype, n_new, d, k_eq_v):
    B, n_kv, cap = 3, 2, 600
    pos = [0, 17, cap - n_new]
    kc = _rand((B, n_kv, cap, d), 1, dtype)
    vc = None if k_eq_v else _rand((B, n_kv, cap, d), 2, dtype)
    kn = _rand((B, n_new, n_kv, d), 3, dtype)
    vn = None if k_eq_v else _rand((B, n_new, n_kv, d), 4, dtype)
    ref_k = kc.clone()
    load_oracle().kv_append(ref_k, kn, pos)
    dk = kc.cuda()
    dv = vc.cuda() if vc is not None else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g.gemma_kv_append([dk], [dv], [0], 0, kn.cuda(), vn.cuda() if vn is not None else None,
                      torch.tensor(pos, dtype=torch.int32, device="cuda"), k_eq_v=k_eq_v,
                      device_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(dk.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       ref_k.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    if vc is not None:
        ref_v = vc.clone()
        load_oracle().kv_append(ref_v, vn, pos)
        assert torch.equal(dv.cpu(), ref_v)


def test_shared_layer_append_is_a_no_op():
    kc = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    kn = torch.ones(1, 1, 1, 64, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    # layer 1 reads layer 0: nothing is written, not even into layer 0's cache
    g.gemma_kv_append([kc, None], [None, None], [0, 0], 1, kn, None, pos, k_eq_v=True)
    torch.cuda.synchronize()
    assert kc.abs().sum().item() == 0


def test_write_pos_out_of_range_is_reported_and_skipped():
    kc = torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    kn = torch.ones(2, 3, 1, 64, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([6, 2], dtype=torch.int32, device="cuda")   # 6 + 3 > 8
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g.gemma_kv_append([kc], None, [0], 0, kn, None, pos, k_eq_v=True, device_error=err)
    torch.cuda.synchronize()
    assert err.item() & g.GEMMA_DEVERR_WRITE_POS
    assert kc[0].abs().sum().item() == 0             # the bad sequence was skipped
    assert kc[1, 0, 2:5].float().eq(1).all()         # the good one was written


def test_seq_len_beyond_hint_is_reported_and_zeroed():
    B, n_q, d, cap = 2, 4, 128, 256
    q = torch.randn(B, 1, n_q, d, device="cuda").bfloat16()
    kc = torch.randn(B, 1, cap, d, device="cuda").bfloat16()
    lens = torch.tensor([100, 200], dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    g.gemma_attn_decode(out, q, [kc], None, [0], 0, lens, 150, kind=g.GEMMA_GLOBAL, window=0,
                        n_kv=1, k_eq_v=True, scale=0.1, workspace=ws, device_error=err)
    torch.cuda.synchronize()
    assert err.item() & g.GEMMA_DEVERR_SEQ_LEN
    assert out[1].float().abs().sum().item() == 0     # seq_len 200 > max_seq_len 150
    assert torch.isfinite(out[0].float()).all() and out[0].float().abs().sum().item() > 0
