"""Pins of the oracle's padded layout and row capacity, and of the padding rows it dispatches.

Padding has a plain definition: each group's rows, then as many padding rows as bring the group
to a multiple of pad_multiple (token_dispatcher page, TokenDispatcherConfig.
moe_router_expert_pad_multiple and _align_up).  The brute force below builds the padded row list
by concatenation, group by group, with no scan; the hand-worked examples are in
tests/golden/layout_padded_example.txt.
"""
import itertools

import numpy as np
import pytest

import oracle
import workloads as W
from conftest import read_golden


def concat_rows(ids, E, S, pad):
    """Rows of the padded layout built by appending: a list of (token, slot, group)."""
    T, K = ids.shape
    rows = []
    for g in range(E + S):
        start = len(rows)
        if g < E:
            rows += [(t, k, g) for t in range(T) for k in range(K) if ids[t, k] == g]
        else:
            rows += [(t, K, g) for t in range(T)]
        while (len(rows) - start) % pad:
            rows.append((-1, -1, g))
    return rows


def check_against_concat(ids, E, S, pad, cap, L):
    T, K = ids.shape
    rows = concat_rows(ids, E, S, pad)
    R_max = cap if cap else T * K + S * T + (E + S) * (pad - 1)
    assert L.R_max == R_max and L.R == len(rows)
    assert bool(L.status & oracle.OVERFLOW) == (len(rows) > R_max)
    # group extents: multiples of pad
    for g in range(E + S):
        ext = L.row_offsets[g + 1] - L.row_offsets[g]
        assert ext % pad == 0 and [r[2] for r in rows].count(g) == ext
    row_of = np.full((T, K), -1)
    for r, (t, k, g) in enumerate(rows):
        if r >= R_max:
            continue
        assert tuple(L.src_info[r]) == (t, k) and L.expert_ids[r] == g
        if t >= 0 and k < K:
            row_of[t, k] = r
    assert np.array_equal(L.row_of, row_of)
    # rows past the recorded ones stay untouched
    assert (L.expert_ids[min(len(rows), R_max):] == -7).all()


def test_golden_examples():
    ids = np.array([[2, 0], [1, -1], [0, 2], [2, 1]], np.int32)
    for g in read_golden("layout_padded_example.txt"):
        S, pad, cap, C = (int(g[k][0]) for k in ("S", "pad", "cap", "C"))
        L = oracle.layout(ids, 3, P=3, C=C, S=S, pad_multiple=pad, num_permuted_tokens=cap or None)
        n = len(g["expert_ids"])
        assert L.R_max == int(g["R_max"][0]), g["name"]
        assert L.status == int(g["status"][0]), g["name"]
        assert L.row_offsets.tolist() == [int(v) for v in g["row_offsets"]], g["name"]
        assert L.expert_ids[:n].tolist() == [int(v) for v in g["expert_ids"]], g["name"]
        assert L.src_info[:n].reshape(-1).tolist() == [int(v) for v in g["src_info"]], g["name"]
        assert L.row_of.reshape(-1).tolist() == [int(v) for v in g["row_of"]], g["name"]


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (2, 1, 3), (2, 2, 2), (1, 3, 2), (3, 1, 2)])
def test_brute_force_all_routings(T, K, E):
    for flat in itertools.product(range(-1, E), repeat=T * K):
        ids = np.array(flat, np.int32).reshape(T, K)
        for S in (0, 1):
            for pad in (1, 2, 3, 4):
                n = len(concat_rows(ids, E, S, pad))
                for cap in (None, n, n - 1, 1):
                    if cap is not None and cap < 1:
                        continue
                    L = oracle.layout(ids, E, P=1, C=T, S=S, pad_multiple=pad,
                                      num_permuted_tokens=cap)
                    check_against_concat(ids, E, S, pad, cap, L)


def test_random_larger_cases():
    rng = np.random.default_rng(21)
    for trial in range(10):
        T = int(rng.integers(1, 70))
        K = int(rng.integers(1, 6))
        E = int(rng.choice([4, 8, 12]))
        S = int(rng.integers(0, 2))
        pad = int(rng.choice([1, 2, 4, 16, 128]))
        ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
        n = len(concat_rows(ids, E, S, pad))
        cap = [None, n, n - 1, max(1, n // 2)][trial % 4]
        L = oracle.layout(ids, E, P=2 if E % 2 == 0 else 1, C=T, S=S, pad_multiple=pad,
                          num_permuted_tokens=cap)
        check_against_concat(ids, E, S, pad, cap, L)


def test_pad_one_is_the_plain_layout():
    cfg = W.scaled(W.CONFIGS["dsv3"], T=300)
    ids, _ = W.make_routing(cfg)
    A = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    B = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S, pad_multiple=1,
                      num_permuted_tokens=A.R_max)
    for k in ("row_offsets", "row_of", "part_tokens", "expert_ids", "src_info"):
        assert np.array_equal(A[k], B[k])
    assert A.status == B.status == 0


def _remap(L0, L1):
    """Row of the padded layout L1 holding each row of the unpadded layout L0."""
    m = np.full(L0.R, -1)
    for r0 in range(L0.R):
        t, k = L0.src_info[r0]
        m[r0] = L1.row_offsets[L0.E] + t if k == L0.K else L1.row_of[t, k]
    return m


@pytest.mark.parametrize("pad", [2, 16, 128])
def test_padded_dispatch_moves_rows_and_zero_fills_padding(pad):
    """Every padded dispatch equals the unpadded one with its rows moved to the padded
    positions, and every padding row holds what an all-zero token dispatches to."""
    cfg = W.scaled(W.CONFIGS["qwen3"], T=40, H=256, S=1, E=16, K=4)
    inp = W.make_inputs(W.scaled(cfg, router="softmax"))
    x, ids, probs = inp["x"], inp["topk_ids"], inp["probs"]
    L0 = oracle.layout(ids, cfg.E, S=1)
    L1 = oracle.layout(ids, cfg.E, S=1, pad_multiple=pad)
    assert L1.R > L0.R and L1.status == 0
    m = _remap(L0, L1)
    pad_rows = np.array([r for r in range(L1.R) if L1.src_info[r][0] < 0])
    assert len(pad_rows) == L1.R - L0.R
    zero = np.zeros((1, cfg.H), np.uint16)

    f0, s0, i0, _ = oracle.dispatch_nvfp4(x, L0)
    f1, s1, i1, _ = oracle.dispatch_nvfp4(x, L1)
    zf, zs, zi = oracle.nvfp4_quantize_row(zero[0])
    assert (zf == 0).all() and (zs == 0).all() and zi == 0x3F80   # bf16 1.0: g = 1 for a zero row
    assert np.array_equal(f1[m], f0[:L0.R]) and np.array_equal(s1[m], s0[:L0.R])
    assert np.array_equal(i1[m], i0[:L0.R])
    assert (f1[pad_rows] == 0).all() and (s1[pad_rows] == 0).all() and (i1[pad_rows] == zi).all()
    assert (f1[L1.R:] == 0xA5).all()

    b0 = oracle.dispatch_bf16(x, L0)
    b1 = oracle.dispatch_bf16(x, L1)
    assert np.array_equal(b1[m], b0[:L0.R]) and (b1[pad_rows] == 0).all()

    c0, q0 = oracle.dispatch_fp8(x, L0)
    c1, q1 = oracle.dispatch_fp8(x, L1)
    assert np.array_equal(c1[m], c0[:L0.R]) and np.array_equal(q1[m], q0[:L0.R])
    assert (c1[pad_rows] == 0).all() and (q1[pad_rows] == 1.0).all()

    # combine ignores padding rows whatever they hold; combine_bwd zeroes their gradient
    y0 = W.make_expert_out(W.scaled(cfg, router="softmax"))[:L0.R_max]
    y1 = np.full((L1.R_max, cfg.H), 0x7FC0, np.uint16)   # NaN everywhere but the real rows
    y1[m] = y0[:L0.R]
    assert np.array_equal(oracle.combine(y1, probs, L1), oracle.combine(y0, probs, L0))
    g = W.make_grad_out(W.scaled(cfg, router="softmax"))
    gy0, gp0 = oracle.combine_bwd(g, y0, probs, L0)
    gy1, gp1 = oracle.combine_bwd(g, y1, probs, L1)
    assert np.array_equal(gy1[m], gy0[:L0.R]) and (gy1[pad_rows] == 0).all()
    assert np.array_equal(gp1, gp0)
    assert np.array_equal(oracle.dispatch_bwd(y1, L1), oracle.dispatch_bwd(y0, L0))


def test_row_capacity_overflow_writes_no_payload():
    cfg = W.scaled(W.CONFIGS["tiny"], T=50)
    inp = W.make_inputs(cfg)
    L = oracle.layout(inp["topk_ids"], cfg.E, pad_multiple=8, num_permuted_tokens=60)
    assert L.status == oracle.OVERFLOW and L.R > 60
    f, s, i, so = oracle.dispatch_nvfp4(inp["x"], L)
    assert (f == 0xA5).all() and (so == -7).all()
    assert (oracle.dispatch_bf16(inp["x"], L) == 0xA5A5).all()
    assert (oracle.dispatch_fp8(inp["x"], L)[0] == 0xA5).all()
