"""GPU: the allocation-free decode entry point gives the results of the workspace one.

gemma_attn_decode_static serves callers that cannot allocate device memory: it takes its split
scratch from an array built into the library. Two calls in a row with different inputs and
split plans (so the shared scratch carries the first call's data into the second) must each
match gemma_attn_decode with a caller workspace, within the bf16 tolerance of the parity tests.
The file is named to be collected last.
"""
import pytest
import torch

import synth
from synth import GLOBAL, SLIDING, LayerSpec, Workload

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _inputs(spec, lens, cap, seed):
    w = Workload("no_alloc", [spec], [0], len(lens), synth.BF16, 1, list(lens), cap)
    hb = synth.layer_batch(w, 0)
    for b, n in enumerate(lens):      # this step's token goes to slot n - 1 of each sequence
        hb.k_cache[b, :, n - 1] = hb.k_new[b, 0]
        if hb.v_cache is not None:
            hb.v_cache[b, :, n - 1] = hb.v_new[b, 0]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(hb.q.shape, generator=g).bfloat16()   # a fresh query per call
    dev = lambda t: None if t is None else t.cuda()       # noqa: E731
    return w, dev(q), dev(hb.k_cache), dev(hb.v_cache), dev(hb.seq_lens)


def _caches(kc, vc):
    # the cache rows beyond the generated ones are NaN; the decode reads only rows < len
    return [kc], [vc]


# Two calls in a row per layer kind: the first with a large split plan (more sequences, longer
# contexts, more chunks), the second with a smaller plan whose chunks fall elsewhere in the
# shared array, so partial results the first call left behind would be read by the second if
# the kernels did not write every partial before reading it.
@pytest.mark.parametrize("spec,calls,cap", [
    (LayerSpec(GLOBAL, 0, 16, 1, 512, True), [([3000, 5000, 777, 4100], 11), ([2500], 12)], 5056),
    (LayerSpec(SLIDING, 8192, 16, 8, 256, False), [([9000, 8500], 11), ([5000], 12)], 9024),
])
def test_static_scratch_decode_matches_workspace_decode(spec, calls, cap):
    import mixed_sliding_global_gb300 as g
    outs, plans = [], []
    for call, (lens, seed) in enumerate(calls):
        w, q, kc, vc, sl = _inputs(spec, lens, cap, seed)
        msl = max(lens)
        kcs, vcs = _caches(kc, vc)
        kw = dict(kind=spec.kind, window=spec.window, n_kv=spec.n_kv, k_eq_v=spec.k_eq_v,
                  scale=w.scale(0))
        ws_n = g.gemma_attn_workspace_size(len(lens), spec.kind, spec.window, spec.n_q,
                                           spec.n_kv, spec.head_dim, msl, 1)
        assert ws_n > 0, "the case must use split scratch"
        plans.append(ws_n)
        # the workspace decode reads only what it wrote: a NaN-filled workspace must not matter
        ws = torch.full((ws_n // 4,), float("nan"), dtype=torch.float32, device="cuda")
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        g.gemma_attn_decode(ref, q, kcs, vcs, [0], 0, sl, msl, workspace=ws, device_error=err, **kw)
        g.gemma_attn_decode_static(got, q, kcs, vcs, [0], 0, sl, msl, device_error=err, **kw)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.isfinite(ref.float()).all() and torch.isfinite(got.float()).all()
        diff = (got.float() - ref.float()).abs()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS, (call, diff.max())
        outs.append(got)
    assert plans[0] > plans[1], "the first call's plan must be the larger one"


def test_static_scratch_rejects_oversized_plans():
    """A plan whose split scratch exceeds the built-in 32 MiB is refused before any launch."""
    import mixed_sliding_global_gb300 as g
    n_q, d, cap = 16, 512, 16448
    B = next((b for b in range(32, 129, 4)
              if g.gemma_attn_workspace_size(b, GLOBAL, 0, n_q, 1, d, cap, 1) > (32 << 20)), None)
    assert B is not None, "no batch in range needs more than 32 MiB of split scratch"
    q = torch.zeros(B, 1, n_q, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(8, dtype=torch.bfloat16, device="cuda")        # never read
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(g.GemmaError) as e:
        g.gemma_attn_decode_static(q, q, [kc], None, [0], 0, sl, cap, kind=GLOBAL, window=0,
                                   n_kv=1, k_eq_v=True, scale=0.05, kv_capacity=cap)
    assert e.value.status == -4
