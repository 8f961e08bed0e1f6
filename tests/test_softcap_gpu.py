"""GPU: the soft-capped attention entry point (each scaled score s becomes c * tanh(s / c))
matches the oracle's soft-capped definition, on decode and prefill, bf16 and the fp32 debug
path. Queries are scaled by powers of two (exact in bf16) so that the cap saturates."""
import pytest
import torch

from harness import DeviceRun, compare, host_inputs, oracle_outputs
from synth import BF16, FP32, GLOBAL, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu


def one_layer(spec, n_new, ctx_lens, cap, dtype=BF16):
    return Workload("softcap", [spec], [0], len(ctx_lens), dtype, n_new, list(ctx_lens), cap)


def run(w, softcap, q_gain):
    hb = host_inputs(w, [0])
    hb[0].q.mul_(q_gain)
    ref = oracle_outputs(w, hb, [0], softcap=softcap)[0]
    gr = DeviceRun(w, hb)
    gr.append(0)
    got = gr.attend(0, softcap=softcap)
    torch.cuda.synchronize()
    assert gr.err.item() == 0
    return compare(got, ref, w.dtype)


CASES = [
    # spec, n_new, ctx_lens, cap
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 1, [3000, 777], 3008),       # decode, split keys
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 1, [4000, 1500], 4032),
    (LayerSpec(GLOBAL, 0, 8, 2, 128, False), 1, [5, 300], 320),
    (LayerSpec(SLIDING, 1024, 16, 8, 256, False), 128, [1300, 300], 1344),  # prefill, tcgen05
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), 96, [700, 200], 704),         # two CTA pairs
    (LayerSpec(SLIDING, 37, 8, 1, 64, False), 40, [100, 45], 128),
]


@pytest.mark.parametrize("softcap,q_gain", [(2.0, 4.0), (30.0, 2.0)])
@pytest.mark.parametrize("spec,n_new,ctx,cap", CASES)
def test_softcap_matches_oracle(spec, n_new, ctx, cap, softcap, q_gain):
    run(one_layer(spec, n_new, ctx, cap), softcap, q_gain)


def test_softcap_fp32_debug_path():
    for n_new in (1, 8):
        w = one_layer(LayerSpec(SLIDING, 16, 4, 1, 64, False), n_new, [64], 64, dtype=FP32)
        run(w, 3.0, 4.0)


def test_softcap_zero_is_the_plain_call():
    w = one_layer(LayerSpec(GLOBAL, 0, 16, 1, 512, True), 64, [500, 128], 512)
    hb = host_inputs(w, [0])
    gr = DeviceRun(w, hb)
    gr.append(0)
    plain = gr.attend(0)
    zero = gr.attend(0, softcap=0.0)
    torch.cuda.synchronize()
    assert torch.equal(plain, zero)
