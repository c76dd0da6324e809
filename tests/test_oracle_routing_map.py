"""Pins of the oracle's conversions between a dense routing map and compact top-k ids.

Hand-worked cases are in tests/golden/routing_map_example.txt.  Beyond them: brute force over
every map of tiny sizes, round trips in both directions, and the layout of a map matching the
layout of the compact ids it came from (same groups, same tokens in the same order).
"""
import itertools

import numpy as np

import oracle
import workloads as W
from conftest import read_golden


def test_golden():
    recs = {g["name"]: g for g in read_golden("routing_map_example.txt")}
    g = recs["map"]
    T, E = int(g["T"][0]), int(g["E"][0])
    m = np.array([int(v) for v in g["map"]], np.uint8).reshape(T, E)
    d = np.array([float(v) for v in g["dense"]], np.float32).reshape(T, E)
    for K in (3, 2):
        ids, probs = oracle.routing_map_to_topk(m, d, K)
        assert ids.reshape(-1).tolist() == [int(v) for v in g[f"ids_K{K}"]]
        assert probs.reshape(-1).tolist() == [float(v) for v in g[f"probs_K{K}"]]
    h = recs["multihot"]
    T, E = int(h["T"][0]), int(h["E"][0])
    ids = np.array([int(v) for v in h["ids"]], np.int32).reshape(T, -1)
    p = np.array([float(v) for v in h["probs"]], np.float32).reshape(T, -1)
    m, d = oracle.indices_to_multihot(ids, p, E)
    assert m.reshape(-1).tolist() == [int(v) for v in h["map"]]
    assert d.reshape(-1).tolist() == [float(v) for v in h["dense"]]


def test_brute_force_every_map():
    T, E = 2, 3
    for flat in itertools.product((0, 1), repeat=T * E):
        m = np.array(flat, np.uint8).reshape(T, E)
        d = np.arange(T * E, dtype=np.float32).reshape(T, E) + 1
        for K in (1, 2, 3, 4):
            ids, probs = oracle.routing_map_to_topk(m, d, K)
            for t in range(T):
                sel = [e for e in range(E) if m[t, e]]
                if len(sel) > K:
                    assert ids[t].tolist() == [E] * K and (probs[t] == 0).all()
                else:
                    assert ids[t].tolist() == sel + [-1] * (K - len(sel))
                    assert probs[t].tolist() == [float(d[t, e]) for e in sel] + [0.0] * (K - len(sel))
            back, dense = oracle.indices_to_multihot(ids, probs, E)
            fits = m.sum(axis=1) <= K
            assert np.array_equal(back[fits], m[fits])
            assert np.array_equal(dense[fits], np.where(m[fits] == 1, d[fits], 0))
            assert (back[~fits] == 0).all()      # the marker id E routes nowhere


def test_round_trip_from_compact_ids():
    cfg = W.scaled(W.CONFIGS["qwen3"], T=200)
    ids, probs = W.make_routing(cfg)
    m, d = oracle.indices_to_multihot(ids, probs, cfg.E)
    assert (m.sum(axis=1) == cfg.K).all()
    ids2, probs2 = oracle.routing_map_to_topk(m, d, cfg.K)
    order = np.argsort(ids, axis=1, kind="stable")
    assert np.array_equal(ids2, np.take_along_axis(ids, order, axis=1))
    assert np.array_equal(probs2, np.take_along_axis(probs, order, axis=1))
    # -1 slots and a row of fewer experts
    ids[3, 2:] = -1
    m, d = oracle.indices_to_multihot(ids, probs, cfg.E)
    assert m[3].sum() == 2
    ids3, _ = oracle.routing_map_to_topk(m, d, cfg.K)
    assert ids3[3, 2:].tolist() == [-1] * (cfg.K - 2)


def test_layout_of_a_map_groups_the_same_tokens():
    cfg = W.scaled(W.CONFIGS["dsv3"], T=150)
    ids, probs = W.make_routing(cfg)
    m, d = oracle.indices_to_multihot(ids, probs, cfg.E)
    ids2, _ = oracle.routing_map_to_topk(m, d, cfg.K)
    A = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    B = oracle.layout(ids2, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    assert np.array_equal(A.row_offsets, B.row_offsets)
    assert np.array_equal(A.expert_ids, B.expert_ids)
    assert np.array_equal(A.src_info[:, 0], B.src_info[:, 0])   # same token in every row
    assert np.array_equal(A.part_tokens, B.part_tokens)


def test_too_many_experts_reaches_the_layout_as_bad_ids():
    m = np.zeros((4, 8), np.uint8)
    m[1, :5] = 1
    m[2, 3] = 1
    ids, _ = oracle.routing_map_to_topk(m, None, 4)
    assert ids[1].tolist() == [8] * 4
    L = oracle.layout(ids, 8)
    assert L.status & oracle.BAD_EXPERT and (L.row_of[1] == -1).all()
    assert L.R == 1
