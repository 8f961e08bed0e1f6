"""GPU: the final-logit soft-cap and greedy argmax against the oracle's definition.

The greedy index is compared exactly (it is decided on the raw logits by exact comparisons on
both sides). The capped logits are compared within a relative bound derived from the
arithmetic: bf16 output is one rounding to 8 significant bits (2^-8 relative) after the hardware
tanh approximation (relative error below 2^-10.9) and fp32 multiplies, so |got - ref| <=
(2^-8 + 2^-10) |ref|; fp32 output uses the library tanhf (a few ulp) and fp32 multiplies, so
|got - ref| <= 2^-20 |ref|; both plus 1e-6 absolute for the logits nearest zero."""
import pytest
import torch

import mixed_sliding_global_gb300 as g
import synth

pytestmark = pytest.mark.gpu

REL = {synth.BF16: 2.0 ** -8 + 2.0 ** -10, synth.FP32: 2.0 ** -20}


def run(x_host, softcap, capped=True, in_place=False):
    x = x_host.cuda()
    B, V = x.shape
    out_idx = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    ws_n = g.gemma_logit_workspace_size(B, V)
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    cap_out = (x if in_place else torch.empty_like(x)) if capped else None
    g.gemma_logit_softcap_argmax(x, softcap, out_idx, cap_out, ws)
    torch.cuda.synchronize()
    return (cap_out.cpu() if capped else None), out_idx.cpu()


def check(orc, x_host, softcap, **kw):
    ref_cap, ref_idx = orc.logit_softcap_argmax(x_host, softcap)
    got_cap, got_idx = run(x_host.clone(), softcap, **kw)
    assert torch.equal(got_idx, ref_idx), (got_idx[:8], ref_idx[:8])
    if got_cap is not None:
        dt = synth.BF16 if x_host.dtype == torch.bfloat16 else synth.FP32
        gc = got_cap.double()
        fin = torch.isfinite(ref_cap)
        err = (gc - ref_cap).abs()
        assert (err[fin] <= REL[dt] * ref_cap[fin].abs() + 1e-6).all(), err[fin].max().item()
        assert torch.equal(torch.isnan(gc), torch.isnan(ref_cap))


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
@pytest.mark.parametrize("batch,vocab", [(1, 1), (3, 7), (2, 8), (4, 9), (5, 1000), (3, 4099),
                                         (2, 70001), (1, synth.VOCAB)])
@pytest.mark.parametrize("softcap", [30.0, 0.0])
def test_shapes(orc, dtype, batch, vocab, softcap):
    """Vocabularies that are not multiples of the vector width start rows at unaligned
    elements (scalar head and tail paths); several splits per row for the larger ones."""
    check(orc, synth.logits(batch, vocab, seed=batch * 7 + vocab, dtype=dtype), softcap)


def test_full_size_batch_64(orc):
    """The greedy step of the pages' vocabulary at batch 64 (bf16, cap 30), every row: each
    row's CTAs reduce its index in one launch (a cluster per row, no workspace)."""
    assert g.gemma_logit_workspace_size(64, synth.VOCAB) == 0
    check(orc, synth.logits(64, synth.VOCAB, seed=1), synth.LOGIT_SOFTCAP)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_one_long_row_two_launches(orc, dtype):
    """A single row too long for one cluster of CTAs: the pieces meet in the workspace and a
    second launch reduces them."""
    assert g.gemma_logit_workspace_size(1, 1 << 23) > 0
    x = synth.logits(1, 1 << 23, seed=11, dtype=dtype)
    x[0, (1 << 23) - 5] = x[0].float().max().item() + 1.0  # the maximum late in the row
    check(orc, x, 30.0)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.FP32])
def test_equal_maxima_take_the_first(orc, dtype):
    x = synth.logits(6, 50000, seed=3, dtype=dtype)
    for b, (i, j) in enumerate([(3, 49999), (0, 1), (25000, 25001), (7, 40000), (49998, 49999),
                                (12345, 12346)]):
        top = x[b].float().max().item() + 4.0
        x[b, i] = top
        x[b, j] = top
    check(orc, x, 30.0)


def test_nan_and_infinities(orc):
    nan, inf = float("nan"), float("inf")
    rows = [[nan, -inf, -inf, -inf], [nan, nan, nan, nan], [1.0, nan, 2.0, 2.0],
            [-inf, 5.0, inf, inf], [-2.0, -1.0, -1.0, -3.0]]
    x = torch.tensor(rows, dtype=torch.float32)
    _, idx = run(x, 30.0)
    assert idx.tolist() == [1, 0, 2, 2, 1]
    check(orc, x, 30.0)


def test_in_place_and_without_capped_output(orc):
    x = synth.logits(4, 30000, seed=5)
    check(orc, x, 30.0, in_place=True)
    check(orc, x, 30.0, capped=False)


def test_argmax_does_not_depend_on_the_cap():
    x = synth.logits(8, 100000, seed=9)
    _, a = run(x.clone(), 30.0)
    _, b = run(x.clone(), 0.0)
    _, c = run(x.clone(), 2.0)
    assert torch.equal(a, b) and torch.equal(a, c)
