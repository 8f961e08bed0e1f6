"""Pins of the fp64 oracle against facts outside itself.

Each ``pin_*`` function takes a loaded oracle and raises AssertionError (or OracleError) when
the oracle disagrees with:
  * a library routine: torch fp64 ``scaled_dot_product_attention`` with an explicit mask;
  * closed forms: uniform weights when K = 0, one-hot values, a window of one key, two keys;
  * invariants: window >= context equals global, K-as-V equals passing K as V, a shared layer
    equals a private copy of its owner's cache, one KV head broadcast equals replicated heads,
    key permutation, a common shift of every key, a common shift of every value;
  * hand-derived fixtures under tests/golden/.
The same functions run against deliberately broken oracle builds (test_oracle_mutants.py) to
show that every planted mistake is caught by at least one pin.
"""
from __future__ import annotations

import json
import math
import os
import types

import torch
import torch.nn.functional as F

from oracle import OracleError  # noqa: F401  (re-exported for the mutant test)

SLIDING, GLOBAL = 0, 1
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def L(kind, window, n_q, n_kv, d, k_eq_v=False):
    return types.SimpleNamespace(kind=kind, window=window, n_q=n_q, n_kv=n_kv, head_dim=d,
                                 k_eq_v=k_eq_v)


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _rand(shape, seed, dtype=torch.float32):
    return torch.randn(shape, generator=_gen(seed), dtype=torch.float32).to(dtype)


def _cache(B, n_kv, cap, d, seed, dtype=torch.float32):
    return _rand((B, n_kv, cap, d), seed, dtype)


def _dyadic(x):
    """Round to multiples of 1/256 so that sums of such values stay exact in fp32."""
    return (torch.round(x * 256.0) / 256.0).contiguous()


def single(orc, spec, q, kc, vc, lens, scale=None):
    """Run the oracle on a one-layer model (the layer owns its cache)."""
    scale = 1.0 / math.sqrt(spec.head_dim) if scale is None else scale
    return orc.attention([spec], [0], 0, [kc], [vc], q, lens, scale)


# ---------------------------------------------------------------------------------------------
# library routine: torch SDPA (fp64) with an explicit boolean mask
# ---------------------------------------------------------------------------------------------
def sdpa_reference(spec, q, kc, vc, lens, scale):
    """Per sequence: repeat each KV head over its group with repeat_interleave and call
    torch's scaled_dot_product_attention with a boolean mask (True = attend)."""
    B, n_tok, n_q, d = q.shape
    G = n_q // spec.n_kv
    outs = []
    for b in range(B):
        n = int(lens[b])
        k = kc[b, :, :n].double().repeat_interleave(G, dim=0)            # [n_q][n][d]
        v = (kc if spec.k_eq_v else vc)[b, :, :n].double().repeat_interleave(G, dim=0)
        pos = torch.arange(n - n_tok, n).view(n_tok, 1)
        key = torch.arange(n).view(1, n)
        mask = key <= pos
        if spec.kind == SLIDING:
            mask = mask & (pos - key < spec.window)
        qq = q[b].double().permute(1, 0, 2)                                 # [n_q][n_tok][d]
        o = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=scale)
        outs.append(o.permute(1, 0, 2))
    return torch.stack(outs)


SDPA_CASES = [
    # kind, W, n_q, n_kv, d, k_eq_v, n_tok, lens, cap
    (SLIDING, 16, 4, 1, 64, False, 1, [64], 64),        # tiny decode shape
    (SLIDING, 16, 4, 1, 64, False, 8, [64], 64),        # tiny prefill shape
    (GLOBAL, 0, 4, 1, 64, False, 8, [64], 72),
    (SLIDING, 5, 8, 2, 16, False, 1, [3, 9, 17], 20),   # window larger / smaller than context
    (SLIDING, 7, 8, 4, 32, False, 6, [6, 11, 30], 32),
    (GLOBAL, 0, 6, 3, 8, False, 3, [3, 5, 12], 12),
    (GLOBAL, 0, 16, 1, 32, True, 4, [9, 33], 40),       # k_eq_v, one KV head
    (SLIDING, 3, 2, 2, 8, True, 5, [5, 13], 16),
]


def pin_sdpa_random(orc):
    for ci, (kind, W, n_q, n_kv, d, kev, n_tok, lens, cap) in enumerate(SDPA_CASES):
        spec = L(kind, W, n_q, n_kv, d, kev)
        B = len(lens)
        q = _rand((B, n_tok, n_q, d), 100 + ci)
        kc = _cache(B, n_kv, cap, d, 200 + ci)
        vc = None if kev else _cache(B, n_kv, cap, d, 300 + ci)
        scale = 0.7 / math.sqrt(d)
        got = single(orc, spec, q, kc, vc, lens, scale)
        ref = sdpa_reference(spec, q, kc, vc, lens, scale)
        err = (got - ref).abs().max().item()
        assert err < 1e-12, f"SDPA case {ci}: max abs diff {err}"


def pin_sdpa_shared_layer(orc):
    """A 4-layer model whose layers 2 and 3 read layers 0 and 1: compare with SDPA on the
    owner's cache."""
    layers = [L(SLIDING, 6, 4, 2, 16), L(GLOBAL, 0, 4, 1, 32, True),
              L(SLIDING, 6, 4, 2, 16), L(GLOBAL, 0, 4, 1, 32, True)]
    owner = [0, 1, 0, 1]
    B, cap, n_tok, lens = 2, 24, 3, [10, 24]
    kcs = [_cache(B, 2, cap, 16, 11), _cache(B, 1, cap, 32, 12), None, None]
    vcs = [_cache(B, 2, cap, 16, 13), None, None, None]
    for layer in (2, 3):
        spec = layers[layer]
        q = _rand((B, n_tok, spec.n_q, spec.head_dim), 14 + layer)
        got = orc.attention(layers, owner, layer, kcs, vcs, q, lens, 0.25)
        o = owner[layer]
        ref = sdpa_reference(spec, q, kcs[o], vcs[o], lens, 0.25)
        assert (got - ref).abs().max().item() < 1e-12, f"shared layer {layer}"


def pin_bf16_decoding(orc):
    """bf16 inputs give exactly the result of the same values widened to fp32 by torch."""
    spec = L(SLIDING, 9, 8, 2, 32)
    lens, cap = [20, 31], 32
    q = _rand((2, 2, 8, 32), 21, torch.bfloat16)
    kc = _cache(2, 2, cap, 32, 22, torch.bfloat16)
    vc = _cache(2, 2, cap, 32, 23, torch.bfloat16)
    a = single(orc, spec, q, kc, vc, lens)
    b = single(orc, spec, q.float(), kc.float(), vc.float(), lens)
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------------------------
def _attended(kind, W, p, n):
    lo = 0 if kind == GLOBAL else max(0, p - W + 1)
    return list(range(lo, min(p, n - 1) + 1))


def pin_uniform_when_k_zero(orc):
    """K = 0 makes every score equal: the output is the mean of the attended values."""
    for kind, W in ((SLIDING, 16), (GLOBAL, 0), (SLIDING, 5)):
        spec = L(kind, W, 4, 1, 64)
        n, n_tok = 64, 8
        q = _rand((1, n_tok, 4, 64), 31)
        kc = torch.zeros((1, 1, n, 64))
        vc = _cache(1, 1, n, 64, 32)
        got = single(orc, spec, q, kc, vc, [n])
        for i in range(n_tok):
            p = n - n_tok + i
            js = _attended(kind, W, p, n)
            mean = vc[0, 0, js].double().mean(dim=0)
            for h in range(4):
                assert (got[0, i, h] - mean).abs().max().item() < 1e-13, (kind, W, i, h)


def pin_one_hot_values(orc):
    """V[j] = e_j with K = 0: output coordinate j is 1/|attended| exactly on the attended keys
    and 0 elsewhere, which pins the causal and window edges."""
    for kind, W, n_tok in ((SLIDING, 16, 1), (SLIDING, 16, 8), (GLOBAL, 0, 8), (SLIDING, 1, 4),
                           (SLIDING, 64, 8), (SLIDING, 70, 3)):
        n = d = 64
        spec = L(kind, W, 4, 1, d)
        q = _rand((1, n_tok, 4, d), 41)
        kc = torch.zeros((1, 1, n, d))
        vc = torch.eye(n, d).view(1, 1, n, d).contiguous()
        got = single(orc, spec, q, kc, vc, [n])
        for i in range(n_tok):
            p = n - n_tok + i
            js = set(_attended(kind, W, p, n))
            expect = torch.tensor([1.0 / len(js) if j in js else 0.0 for j in range(d)],
                                  dtype=torch.float64)
            for h in range(4):
                assert (got[0, i, h] - expect).abs().max().item() < 1e-14, (kind, W, n_tok, i)


def pin_window_of_one(orc):
    """W = 1: each query sees only its own position, so the output is V[p] exactly."""
    spec = L(SLIDING, 1, 4, 2, 16)
    n, n_tok = 12, 5
    q = _rand((2, n_tok, 4, 16), 51)
    kc = _cache(2, 2, n, 16, 52)
    vc = _cache(2, 2, n, 16, 53)
    got = single(orc, spec, q, kc, vc, [n, n - 3])
    for b, nb in enumerate((n, n - 3)):
        for i in range(n_tok):
            p = nb - n_tok + i
            for h in range(4):
                assert torch.equal(got[b, i, h], vc[b, h // 2, p].double()), (b, i, h)


def pin_two_keys(orc):
    """Two attended keys: weights are the logistic of the score difference."""
    d, scale = 16, 0.37
    spec = L(GLOBAL, 0, 2, 1, d)
    q = _rand((1, 1, 2, d), 61)
    kc = _cache(1, 1, 2, d, 62)
    vc = _cache(1, 1, 2, d, 63)
    got = single(orc, spec, q, kc, vc, [2], scale)
    k0, k1 = kc[0, 0, 0].double(), kc[0, 0, 1].double()
    v0, v1 = vc[0, 0, 0].double(), vc[0, 0, 1].double()
    for h in range(2):
        qh = q[0, 0, h].double()
        delta = scale * float(qh @ (k0 - k1))
        w0 = 1.0 / (1.0 + math.exp(-delta))
        expect = w0 * v0 + (1.0 - w0) * v1
        assert (got[0, 0, h] - expect).abs().max().item() < 1e-14, h


# ---------------------------------------------------------------------------------------------
# the optional attention-logit soft-cap: c * tanh(s / c) of the scaled score s
# ---------------------------------------------------------------------------------------------
def pin_softcap_far_above_scores_changes_nothing(orc):
    """A cap far above every score leaves the result unchanged: c tanh(s / c) differs from s
    by about s^3 / (3 c^2), here below 1e-10 for |s| < 10."""
    d = 32
    spec = L(SLIDING, 5, 4, 2, d)
    q = _rand((2, 3, 4, d), 71)
    kc = _cache(2, 2, 12, d, 72)
    vc = _cache(2, 2, 12, d, 73)
    lens, scale = [12, 9], 1.0 / math.sqrt(d)
    plain = orc.attention([spec], [0], 0, [kc], [vc], q, lens, scale)
    capped = orc.attention([spec], [0], 0, [kc], [vc], q, lens, scale, softcap=1.0e6)
    assert (plain - capped).abs().max().item() < 1e-9


def pin_softcap_saturated_scores(orc):
    """Scaled scores of +-L with L far above the cap become exactly +-c (tanh of +-5000 is +-1
    in double precision), so with one-hot value rows the output is the weight vector
    e^(+-c) / (n_plus e^c + n_minus e^-c). The scale is applied before the cap: scale 0.5 and
    q . k = +-2e4 give s = +-1e4."""
    d, c, scale = 8, 2.0, 0.5
    signs = [1, -1, 1, 1, -1, 1]
    n = len(signs)
    spec = L(GLOBAL, 0, 1, 1, d)
    q = torch.zeros(1, 1, 1, d)
    q[0, 0, 0, 0] = 1.0
    kc = torch.zeros(1, 1, n, d)
    vc = torch.zeros(1, 1, n, d)
    for j, sg in enumerate(signs):
        kc[0, 0, j, 0] = 2.0e4 * sg
        vc[0, 0, j, j] = 1.0
    got = orc.attention([spec], [0], 0, [kc], [vc], q, [n], scale, softcap=c)
    n_plus, n_minus = signs.count(1), signs.count(-1)
    den = n_plus * math.exp(c) + n_minus * math.exp(-c)
    for j, sg in enumerate(signs):
        assert abs(got[0, 0, 0, j].item() - math.exp(c * sg) / den) < 1e-15, j
    assert got[0, 0, 0, n:].abs().max().item() == 0.0


# ---------------------------------------------------------------------------------------------
# the final-logit soft-cap c * tanh(x / c) and the greedy argmax of the raw logits
# ---------------------------------------------------------------------------------------------
def pin_logit_cap_closed_forms(orc):
    """A cap far above the logits changes them by at most |x|^3 / (3 c^2); logits far above the
    cap become exactly +-c; x = c * atanh(1/2) becomes c / 2; the cap is odd in x."""
    x = _rand((3, 257), 81) * 4.0
    capped, _ = orc.logit_softcap_argmax(x, 1.0e6)
    xd = x.double()
    assert ((capped - xd).abs() <= xd.abs() ** 3 / (3.0e12) + 1e-15 * (1.0 + xd.abs())).all()
    c = 30.0
    sat = torch.tensor([[1.0e4, -1.0e4, 0.0, c * math.atanh(0.5)]], dtype=torch.float32)
    capped, _ = orc.logit_softcap_argmax(sat, c)
    assert capped[0, 0].item() == c and capped[0, 1].item() == -c and capped[0, 2].item() == 0.0
    assert abs(capped[0, 3].item() - c / 2) < 1e-5   # atanh argument rounded to fp32
    pos, _ = orc.logit_softcap_argmax(x, c)
    neg, _ = orc.logit_softcap_argmax((-x).contiguous(), c)
    assert (pos + neg).abs().max().item() < 1e-14
    plain, _ = orc.logit_softcap_argmax(x, 0.0)
    assert torch.equal(plain, xd)


def pin_logit_argmax_is_first_maximum(orc):
    """The greedy index equals numpy's argmax (first occurrence of the maximum) on rows with
    planted equal maxima, in bf16 and fp32."""
    import numpy as np
    for dtype in (torch.float32, torch.bfloat16):
        x = _rand((6, 1000), 82, dtype)
        for b, (i, j) in enumerate([(3, 900), (0, 999), (500, 501), (7, 8), (998, 999), (1, 2)]):
            top = x[b].float().max().item() + 1.0
            x[b, i] = top
            x[b, j] = top
        _, idx = orc.logit_softcap_argmax(x, 30.0)
        ref = np.argmax(x.float().numpy(), axis=1)
        assert idx.tolist() == ref.tolist()


def pin_logit_argmax_ignores_the_cap(orc):
    """The page's statement: the argmax of the capped logits (fp64, distinct values) is the
    argmax of the raw logits."""
    x = _rand((8, 4096), 83) * 6.0
    capped, idx = orc.logit_softcap_argmax(x, 30.0)
    assert idx.tolist() == torch.argmax(capped, dim=1).to(torch.int32).tolist()
    assert idx.tolist() == torch.argmax(x, dim=1).to(torch.int32).tolist()


def pin_logit_argmax_nan_and_infinities(orc):
    """Hand-derived: NaN is never selected; -inf rows pick their first entry; +inf wins."""
    nan, inf = float("nan"), float("inf")
    rows = [[nan, -inf, -inf, -inf], [nan, nan, nan, nan], [1.0, nan, 2.0, 2.0],
            [-inf, 5.0, inf, inf], [-2.0, -1.0, -1.0, -3.0]]
    _, idx = orc.logit_softcap_argmax(torch.tensor(rows, dtype=torch.float32), 30.0)
    assert idx.tolist() == [1, 0, 2, 2, 1]


# ---------------------------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------------------------
def pin_window_covering_context_is_global(orc):
    n, n_tok = 40, 6
    q = _rand((2, n_tok, 8, 32), 71)
    kc = _cache(2, 2, n, 32, 72)
    vc = _cache(2, 2, n, 32, 73)
    g = single(orc, L(GLOBAL, 0, 8, 2, 32), q, kc, vc, [n, 25])
    for W in (n, n + 1, 1000):
        s = single(orc, L(SLIDING, W, 8, 2, 32), q, kc, vc, [n, 25])
        assert torch.equal(g, s), W
    s = single(orc, L(SLIDING, n - 1, 8, 2, 32), q, kc, vc, [n, 25])
    assert not torch.equal(g, s), "a window shorter than the context must change the result"


def pin_k_eq_v_is_k_as_v(orc):
    for kind, W in ((GLOBAL, 0), (SLIDING, 9)):
        q = _rand((2, 3, 16, 32), 81)
        kc = _cache(2, 1, 30, 32, 82)
        a = single(orc, L(kind, W, 16, 1, 32, True), q, kc, None, [30, 17])
        b = single(orc, L(kind, W, 16, 1, 32, False), q, kc, kc.clone(), [30, 17])
        assert torch.equal(a, b)


def pin_shared_layer_is_owner_copy(orc):
    layers = [L(SLIDING, 8, 8, 2, 16), L(SLIDING, 8, 8, 2, 16), L(SLIDING, 8, 8, 2, 16)]
    kc0, vc0 = _cache(1, 2, 20, 16, 91), _cache(1, 2, 20, 16, 92)
    kc1, vc1 = _cache(1, 2, 20, 16, 93), _cache(1, 2, 20, 16, 94)
    q = _rand((1, 2, 8, 16), 95)
    shared = orc.attention(layers, [0, 1, 0], 2, [kc0, kc1, None], [vc0, vc1, None], q, [20], 0.3)
    private = orc.attention(layers, [0, 1, 2], 2, [kc0, kc1, kc0.clone()],
                            [vc0, vc1, vc0.clone()], q, [20], 0.3)
    assert torch.equal(shared, private)
    other = orc.attention(layers, [0, 1, 1], 2, [kc0, kc1, None], [vc0, vc1, None], q, [20], 0.3)
    assert not torch.equal(shared, other), "reading another owner must change the result"


def pin_broadcast_is_replication(orc):
    n_q, d, n = 8, 16, 21
    q = _rand((2, 4, n_q, d), 101)
    kc = _cache(2, 1, n, d, 102)
    vc = _cache(2, 1, n, d, 103)
    a = single(orc, L(SLIDING, 6, n_q, 1, d), q, kc, vc, [n, 13])
    b = single(orc, L(SLIDING, 6, n_q, n_q, d), q, kc.expand(2, n_q, n, d).contiguous(),
               vc.expand(2, n_q, n, d).contiguous(), [n, 13])
    assert torch.equal(a, b)


def pin_key_permutation(orc):
    """Decode on a global layer attends every cached key: permuting them changes nothing."""
    n, d = 33, 32
    q = _rand((1, 1, 4, d), 111)
    kc = _cache(1, 2, n, d, 112)
    vc = _cache(1, 2, n, d, 113)
    perm = torch.randperm(n, generator=_gen(114))
    a = single(orc, L(GLOBAL, 0, 4, 2, d), q, kc, vc, [n])
    b = single(orc, L(GLOBAL, 0, 4, 2, d), q, kc[:, :, perm].contiguous(),
               vc[:, :, perm].contiguous(), [n])
    assert (a - b).abs().max().item() < 1e-13


def pin_key_shift(orc):
    """Adding the same vector u to every key adds q.u to every score of a row: no change."""
    n, d = 26, 16
    spec = L(SLIDING, 10, 4, 2, d)
    q = _rand((1, 3, 4, d), 121)
    kc = _dyadic(_cache(1, 2, n, d, 122))
    vc = _cache(1, 2, n, d, 123)
    u = _dyadic(_rand((1, 2, 1, d), 124))      # k + u is exact in fp32
    a = single(orc, spec, q, kc, vc, [n])
    b = single(orc, spec, q, (kc + u).contiguous(), vc, [n])
    assert (a - b).abs().max().item() < 1e-12


def pin_value_shift(orc):
    """Weights sum to one: adding c to every value adds c to the output."""
    n, d = 26, 16
    spec = L(SLIDING, 10, 4, 2, d)
    q = _rand((1, 3, 4, d), 131)
    kc = _cache(1, 2, n, d, 132)
    vc = _dyadic(_cache(1, 2, n, d, 133))       # v + 3 is exact in fp32
    a = single(orc, spec, q, kc, vc, [n])
    b = single(orc, spec, q, kc, (vc + 3.0).contiguous(), [n])
    assert (b - a - 3.0).abs().max().item() < 1e-12


# ---------------------------------------------------------------------------------------------
# hand-derived fixtures
# ---------------------------------------------------------------------------------------------
def golden_cases():
    out = []
    for name in sorted(os.listdir(GOLDEN)):
        if name.endswith(".json"):
            with open(os.path.join(GOLDEN, name)) as f:
                out.append((name, json.load(f)))
    return out


def run_golden(orc, case):
    layers = [types.SimpleNamespace(**l) for l in case["layers"]]
    n_layers = len(layers)
    t = lambda x: torch.tensor(x, dtype=torch.float32).contiguous()  # noqa: E731
    kcs = [t(case["k_cache"][str(o)]) if str(o) in case["k_cache"] else None
           for o in range(n_layers)]
    vcs = [t(case["v_cache"][str(o)]) if str(o) in case.get("v_cache", {}) else None
           for o in range(n_layers)]
    got = orc.attention(layers, case["owner_map"], case["layer"], kcs, vcs, t(case["q"]),
                        case["seq_lens"], case["scale"])
    expect = torch.tensor(case["expected"], dtype=torch.float64)
    return got, expect


def pin_golden(orc):
    cases = golden_cases()
    assert cases, "no golden fixtures found"
    for name, case in cases:
        got, expect = run_golden(orc, case)
        assert got.shape == expect.shape, name
        assert (got - expect).abs().max().item() < case.get("tol", 1e-15), name


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
