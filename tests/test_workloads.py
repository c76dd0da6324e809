"""Host-side checks of the seeded input generator (shapes, determinism, routing recipe)."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name", ["tiny", "qwen3", "dsv3", "mixtral", "dsv3_static"])
def test_routing_shapes_distinct_and_normalised(name):
    cfg = W.CONFIGS[name]
    cfg = W.scaled(cfg, T=min(cfg.T, 512))
    ids, p = W.make_routing(cfg)
    assert ids.shape == (cfg.T, cfg.K) and ids.dtype == np.int32
    assert p.shape == (cfg.T, cfg.K) and p.dtype == np.float32
    assert ((ids >= 0) & (ids < cfg.E)).all()
    assert all(len(set(r)) == cfg.K for r in ids.tolist())
    assert np.allclose(p.sum(1), 1.0, atol=1e-6) and (p > 0).all()
    ids2, p2 = W.make_routing(cfg)
    assert np.array_equal(ids, ids2) and np.array_equal(p, p2)


def test_zipf_skew_and_hot_experts():
    ids, _ = W.make_routing(W.scaled(W.CONFIGS["mixtral"], T=4096))
    share = np.bincount(ids.ravel(), minlength=8) / ids.size
    assert share[0] > 0.25 and share[7] < 0.08 and (np.diff(share) < 0.02).all()
    ids, _ = W.make_routing(W.scaled(W.CONFIGS["dsv3_large"], T=1024))
    hot = np.isin(ids, [0, 1, 2, 3]).sum(1)
    # nearly every token reaches partition 0 (experts 0..31), which holds the hot experts
    assert (hot >= 1).mean() > 0.99 and hot.mean() > 2.5


def test_x_structure():
    cfg = W.scaled(W.CONFIGS["qwen3"], T=1000, H=64)
    x = W.f32_from_bf16_bits(W.make_x(cfg))
    big = np.abs(x).max(1) > 20
    assert big.sum() == 10
    cfg = W.scaled(W.CONFIGS["dsv3_large"], T=5000, H=32)
    x = W.f32_from_bf16_bits(W.make_x(cfg))
    assert ((x == 0).all(1)).sum() == 5


def test_bf16_rounding_of_generator():
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -0.0, 3.0e38], np.float32)
    assert W.bf16_bits_from_f32(v).tolist() == [0x3F80, 0x3F80, 0x3F82, 0x8000, 0x7F62]


def test_static_routing_is_balanced_and_fills_its_capacity():
    import oracle
    cfg = W.CONFIGS["dsv3_static"]
    ids, p = W.make_routing(cfg)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert (counts == cfg.T * cfg.K // cfg.E).all()
    assert (p == np.float32(1.0 / cfg.K)).all()
    L = oracle.layout(ids[:512], cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S, pad_multiple=16,
                      num_permuted_tokens=512 * cfg.K + 512)
    assert L.status == 0 and L.R == L.R_max          # every group a multiple of 16: no padding
    assert (L.part_tokens == 512 // cfg.P).all()     # each token's 8 experts share a partition
