"""Pins of the oracle's dispatch layout.

The layout has a plain definition: rows grouped by expert in ascending expert order, and inside
an expert the (token, slot) pairs in ascending flat order.  That makes it the unique permutation
that satisfies the invariants checked below, so brute force over every routing of tiny problems
pins it completely.  A hand-worked example is kept in tests/golden/layout_example.txt.
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import read_golden


def check_layout_invariants(ids, E, P, C, S, L):
    T, K = ids.shape
    valid = [(t, k) for t in range(T) for k in range(K) if 0 <= ids[t, k] < E]
    R = len(valid) + S * T
    G = E + S
    assert L.R == R
    ro = L.row_offsets
    # group sizes
    for e in range(E):
        assert ro[e + 1] - ro[e] == sum(1 for t, k in valid if ids[t, k] == e)
    if S:
        assert ro[G] - ro[E] == T
    assert ro[0] == 0 and ro[G] == R
    # every valid (t,k) appears exactly once and row_of / src_info are inverse
    seen = set()
    for t in range(T):
        for k in range(K):
            r = L.row_of[t, k]
            if (t, k) in valid:
                assert 0 <= r < ro[E]
                assert tuple(L.src_info[r]) == (t, k)
                e = ids[t, k]
                assert ro[e] <= r < ro[e + 1] and L.expert_ids[r] == e
                seen.add(r)
            else:
                assert r == -1
    assert len(seen) == len(valid)
    # stable inside every group: flat index strictly increasing along the rows
    for e in range(E):
        flat = [L.src_info[r][0] * K + L.src_info[r][1] for r in range(ro[e], ro[e + 1])]
        assert flat == sorted(flat) and len(set(flat)) == len(flat)
    # shared group: one row per token in token order, slot K
    if S:
        for t in range(T):
            r = ro[E] + t
            assert tuple(L.src_info[r]) == (t, K) and L.expert_ids[r] == E
    # per-partition received tokens and the overflow bit
    per = E // P
    for p in range(P):
        n = sum(1 for t in range(T) if any(0 <= ids[t, k] < E and ids[t, k] // per == p
                                           for k in range(K)))
        assert L.part_tokens[p] == n
    over = any(L.part_tokens[p] > C for p in range(P))
    assert bool(L.status & oracle.OVERFLOW) == over


def test_golden_example():
    g = read_golden("layout_example.txt")[0]
    T, K, E, S, P = (int(g[k][0]) for k in ("T", "K", "E", "S", "P"))
    ids = np.array([int(v) for v in g["topk_ids"]], np.int32).reshape(T, K)
    for C, key in ((2, "status_C2"), (3, "status_C3")):
        L = oracle.layout(ids, E, P=P, C=C, S=S)
        assert L.status == int(g[key][0])
        assert L.row_offsets.tolist() == [int(v) for v in g["row_offsets"]]
        assert L.expert_ids[:L.R].tolist() == [int(v) for v in g["expert_ids"]]
        assert L.src_info[:L.R].reshape(-1).tolist() == [int(v) for v in g["src_info"]]
        assert L.row_of.reshape(-1).tolist() == [int(v) for v in g["row_of"]]
        assert L.part_tokens.tolist() == [int(v) for v in g["part_tokens"]]


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (1, 2, 3), (2, 1, 3), (2, 2, 2), (3, 1, 3),
                                   (1, 4, 2), (4, 1, 2), (2, 2, 3)])
def test_brute_force_all_routings(T, K, E):
    """Every assignment of ids in {-1, .., E-1} to the T*K slots, with and without a shared
    expert, every partition count that divides E and capacities around the overflow edge."""
    parts = [p for p in range(1, E + 1) if E % p == 0]
    for flat in itertools.product(range(-1, E), repeat=T * K):
        ids = np.array(flat, np.int32).reshape(T, K)
        for S in (0, 1):
            for P in parts:
                for C in (0, 1, T):
                    L = oracle.layout(ids, E, P=P, C=C, S=S)
                    check_layout_invariants(ids, E, P, C, S, L)


def test_random_larger_cases():
    rng = np.random.default_rng(11)
    for trial in range(12):
        T = int(rng.integers(1, 90))
        K = int(rng.integers(1, 7))
        E = int(rng.choice([4, 8, 12, 16]))
        P = int(rng.choice([p for p in (1, 2, 4) if E % p == 0]))
        S = int(rng.integers(0, 2))
        ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
        C = int(rng.integers(0, T + 1))
        L = oracle.layout(ids, E, P=P, C=C, S=S)
        check_layout_invariants(ids, E, P, C, S, L)


def test_bad_expert_ids_are_flagged_and_masked():
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 8, size=(40, 3)).astype(np.int32)
    bad = ids.copy()
    bad[3, 1] = 8
    bad[17, 0] = -5
    bad[39, 2] = 1 << 30
    L = oracle.layout(bad, 8, P=2, C=40, S=1)
    assert L.status & oracle.BAD_EXPERT
    masked = bad.copy()
    masked[(masked < -1) | (masked >= 8)] = -1
    M = oracle.layout(masked, 8, P=2, C=40, S=1)
    assert M.status == 0
    for k in ("row_offsets", "row_of", "part_tokens"):
        assert np.array_equal(L[k], M[k])
    assert np.array_equal(L.src_info[:L.R], M.src_info[:M.R])
    assert np.array_equal(L.expert_ids[:L.R], M.expert_ids[:M.R])


def test_empty_and_all_unused():
    ids = np.full((5, 3), -1, np.int32)
    L = oracle.layout(ids, 4, P=2, C=0, S=0)
    assert L.R == 0 and L.status == 0 and (L.row_of == -1).all()
    assert L.row_offsets.tolist() == [0] * 5
    L = oracle.layout(ids, 4, P=2, C=0, S=1)
    assert L.R == 5 and L.row_offsets.tolist() == [0, 0, 0, 0, 0, 5]
