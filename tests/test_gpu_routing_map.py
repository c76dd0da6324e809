"""GPU vs oracle parity of the routing-map conversions and of the layout made from a dense
routing map (fused_a2a page, HybridEPDispatch.forward: the map takes precedence over compact
ids; token_dispatcher page, _indices_to_multihot).  Everything bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import CANARY32, check_layout, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


@pytest.mark.parametrize("T,E,K,density", [(1, 1, 1, 1.0), (100, 8, 2, 0.2), (777, 256, 8, 0.03),
                                           (300, 1000, 32, 0.02), (64, 33, 4, 0.5),
                                           (200, 1024, 32, 0.02), (300, 16, 4, 0.3),
                                           (129, 128, 8, 0.06), (50, 512, 16, 0.03)])
def test_map_to_topk(ep, T, E, K, density):
    rng = np.random.default_rng(T + E)
    m = (rng.random((T, E)) < density).astype(np.uint8)
    m[0, : min(E, K)] = 1                 # a row with exactly K
    if E > K:
        m[-1, : K + 1] = 1                # a row with more than K
    d = rng.random((T, E)).astype(np.float32)
    ids, probs = ep.routing_map_to_topk(dev(m), dev(d), K)
    rids, rprobs = oracle.routing_map_to_topk(m, d, K)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.array_equal(probs.cpu().numpy(), rprobs)
    ids2, p2 = ep.routing_map_to_topk(dev(m).bool(), None, K)
    assert np.array_equal(ids2.cpu().numpy(), rids) and p2 is None


@pytest.mark.parametrize("T,E,K", [(1, 1, 1), (500, 8, 2), (640, 256, 8), (90, 1000, 32)])
def test_indices_to_multihot(ep, T, E, K):
    rng = np.random.default_rng(T * K)
    ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    ids[0, :] = ids[0, 0]                 # a repeated expert
    if T > 2:
        ids[1, 0] = E + 5                 # out of range: skipped
        ids[2, :] = -1
    p = rng.random((T, K)).astype(np.float32)
    m, d = ep.indices_to_multihot(dev(ids), dev(p), E)
    rm, rd = oracle.indices_to_multihot(ids, p, E)
    assert np.array_equal(m.cpu().numpy(), rm)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), rd.view(np.uint32))


@pytest.mark.parametrize("name,T", [("dsv3", 900), ("qwen3", 1000), ("mixtral", 1500)])
def test_layout_from_routing_map_takes_precedence(ep, name, T):
    cfg = W.scaled(W.CONFIGS[name], T=T)
    ids, probs = W.make_routing(cfg)
    m, d = oracle.indices_to_multihot(ids, probs, cfg.E)
    rids, rprobs = oracle.routing_map_to_topk(m, d, cfg.K)
    ref = oracle.layout(rids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    L = ep.Layout(cfg.T, cfg.K, cfg.E, cfg.P, bool(cfg.S))
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    decoy = torch.zeros(cfg.T, cfg.K, dtype=torch.int32, device="cuda")   # ignored: the map wins
    _, gids, gprobs = ep.dispatch_layout_routed(cfg.E, topk_ids=decoy, routing_map=dev(m),
                                                dense_probs=dev(d), n_parts=cfg.P,
                                                capacity=cfg.capacity, fused_shared=bool(cfg.S), out=L)
    assert np.array_equal(gids.cpu().numpy(), rids)
    assert np.array_equal(gprobs.cpu().numpy(), rprobs)
    check_layout(L, ref, ep)
    # the dense gradient layout: grad_probs [T, K] scattered back through the ids
    gp = np.random.default_rng(1).standard_normal((cfg.T, cfg.K)).astype(np.float32)
    gm, gd = ep.indices_to_multihot(gids, dev(gp), cfg.E)
    _, rd = oracle.indices_to_multihot(rids, gp, cfg.E)
    assert np.array_equal(gd.cpu().numpy(), rd)


def test_too_dense_map_is_reported_by_the_layout(ep):
    m = np.zeros((50, 16), np.uint8)
    m[:, 3] = 1
    m[7, :6] = 1                          # 6 experts with K = 4
    L = ep.Layout(50, 4, 16)
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    _, ids, _ = ep.dispatch_layout_routed(16, routing_map=dev(m), K=4, out=L)
    assert ep.read_status(L) == ep.STATUS_BAD_EXPERT
    assert ids.cpu().numpy()[7].tolist() == [16] * 4
    ref = oracle.layout(oracle.routing_map_to_topk(m, None, 4)[0], 16)
    check_layout(L, ref, ep)
