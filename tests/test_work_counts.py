"""The benchmark's algorithmic work per launch (the roofline numerators) against a brute-force
count from the mask definition: query p attends key j iff j <= p and, on a sliding layer,
p - j < W. Decode bytes are the K (and V) rows attended by each sequence's single query, plus q
and out; prefill flops are 4 * head_dim * n_q per attended (query, key) pair."""
import numpy as np

import bench
import synth


def attended_keys(kind, window, p):
    j = np.arange(p + 1)
    ok = j <= p
    if kind == synth.SLIDING:
        ok &= (p - j) < window
    return int(ok.sum())


def brute_decode_bytes(w, l):
    s = w.layers[l]
    kv = 0
    for ln in w.ctx_lens:
        kv += s.n_kv * attended_keys(s.kind, s.window, ln - 1) * s.head_dim * 2 * \
            (1 if s.k_eq_v else 2)
    return kv + 2 * w.batch * s.n_q * s.head_dim * 2


def brute_prefill_flops(w, l):
    s = w.layers[l]
    pairs = 0
    for ln in w.ctx_lens:
        q = np.arange(ln - w.n_new, ln)[:, None]
        j = np.arange(ln)[None, :]
        m = j <= q
        if s.kind == synth.SLIDING:
            m &= (q - j) < s.window
        pairs += int(m.sum())
    return 4 * s.head_dim * s.n_q * pairs


def test_ragged_decode_bytes_per_launch():
    w = synth.ragged_decode(n_layers=6)
    for l in (0, 5):
        assert bench.decode_bytes(w, l) == brute_decode_bytes(w, l)
    assert bench.decode_bytes(w, 0) == 520847360     # sliding layer, as reported
    assert bench.decode_bytes(w, 5) == 481910784     # global layer (K as V), as reported


def test_batch1_decode_bytes():
    for w in (synth.b12_decode(n_layers=6), synth.e4b_decode()):
        for l in range(w.n_layers):
            assert bench.decode_bytes(w, l) == brute_decode_bytes(w, l)


def test_prefill_flops_per_launch():
    w = synth.prefill_12b(n_layers=6)
    for l in (0, 5):
        assert bench.prefill_flops(w, l) == brute_prefill_flops(w, l)
    assert abs(bench.prefill_flops(w, 0) / 1e9 - 34.36) < 0.01
    assert abs(bench.prefill_flops(w, 5) / 1e9 - 257.73) < 0.01
