"""Argument checks of the oracle (host logic only)."""
import pytest
import torch

from oracle import OracleError
from oracle_pins import L, GLOBAL, SLIDING


def test_owner_rules(orc):
    layers = [L(SLIDING, 4, 4, 2, 8), L(GLOBAL, 0, 4, 1, 8), L(SLIDING, 4, 4, 2, 8)]
    assert orc.resolve_owner(layers, [0, 1, 0], 2) == 0
    assert orc.resolve_owner(layers, [0, 1, 1], 2) < 0      # different kind / n_kv
    assert orc.resolve_owner(layers, [0, 1, 2], 1) == 1     # a layer may own its cache
    chain = layers + [L(SLIDING, 4, 4, 2, 8)]
    assert orc.resolve_owner(chain, [0, 1, 0, 2], 3) < 0    # owner that is itself shared
    assert orc.resolve_owner(layers, [0, 0, 2], 1) < 0      # kind mismatch
    assert orc.resolve_owner(layers, [2, 1, 2], 0) < 0      # owner later than the layer
    assert orc.resolve_owner(layers, [0, 1, 0], 3) < 0      # layer out of range


def test_bad_lengths(orc):
    spec = L(GLOBAL, 0, 4, 1, 8)
    q = torch.zeros(1, 2, 4, 8)
    kc = torch.zeros(1, 1, 8, 8)
    vc = torch.zeros(1, 1, 8, 8)
    with pytest.raises(OracleError):
        orc.attention([spec], [0], 0, [kc], [vc], q, [1], 1.0)   # fewer cached than queries
    with pytest.raises(OracleError):
        orc.attention([spec], [0], 0, [kc], [vc], q, [9], 1.0)   # beyond capacity
    with pytest.raises(OracleError):
        orc.attention([L(GLOBAL, 0, 3, 2, 8)], [0], 0, [kc], [vc], q[:, :, :3], [4], 1.0)
    with pytest.raises(OracleError):
        orc.attention([L(SLIDING, 0, 4, 1, 8)], [0], 0, [kc], [vc], q, [4], 1.0)  # W < 1


def test_append_is_a_placed_copy(orc):
    cache = torch.arange(2 * 3 * 6 * 4, dtype=torch.float32).view(2, 3, 6, 4).contiguous()
    rows = -torch.arange(2 * 2 * 3 * 4, dtype=torch.float32).view(2, 2, 3, 4).contiguous() - 1
    before = cache.clone()
    orc.kv_append(cache, rows, [1, 4])
    for b, pos in enumerate((1, 4)):
        for t in range(2):
            for h in range(3):
                assert torch.equal(cache[b, h, pos + t], rows[b, t, h])
        keep = [j for j in range(6) if not pos <= j < pos + 2]
        assert torch.equal(cache[b, :, keep], before[b, :, keep])
    with pytest.raises(OracleError):
        orc.kv_append(cache, rows, [5, 0])                      # would run past capacity
    with pytest.raises(OracleError):
        orc.kv_append(cache, rows, [-1, 0])
