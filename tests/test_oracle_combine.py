"""Pins of the oracle's combine and both backward passes.

Against: round trips with identity experts and probabilities summing to one (combine of
dispatch returns x), the Tiny workload's closed form out[t] = sum_k p_k (1 + e_k/8) deq(x_t),
and adjoint identities that the mathematics fixes:
  <combine(y), g> = <y, combine_bwd_y(g)>,   grad_p[t,k] = d<combine(y), g>/dp[t,k],
  <dispatch(x), gd> = <x, dispatch_bwd(gd)>.
A dropped term, a wrong row index, a missing shared row or a transposed operand breaks one of
them.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return W.bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32) * scale)


def f(b):
    return W.f32_from_bf16_bits(b).astype(np.float64)


def routing(T, K, E, seed, unused=0.1):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < unused] = -1
    p = rng.random((T, K)) + 0.05
    p[ids < 0] = 0.0
    p = (p / np.maximum(p.sum(1, keepdims=True), 1e-30)).astype(np.float32)
    return ids, p


@pytest.mark.parametrize("S", [0, 1])
def test_bf16_round_trip_identity_experts(S):
    T, H, E, K = 50, 48, 7, 3
    ids, p = routing(T, K, E, 3)
    ids[:, 0] = np.where(ids[:, 0] < 0, 0, ids[:, 0])   # at least one slot per token
    x = rand_bf16((T, H), 4)
    L = oracle.layout(ids, E, S=S)
    y = oracle.dispatch_bf16(x, L)
    if S:
        # identity experts with the shared row zeroed: sum_k p_k x = x (sum p = 1)
        y[L.row_offsets[E]:L.R] = 0
    pr = p.copy()
    s = pr.sum(1)
    pr = (pr / np.where(s > 0, s, 1)[:, None]).astype(np.float32)
    out = oracle.combine(y, pr, L)
    xf, of = f(x), f(out)
    assert np.all(np.abs(of - xf) <= 2.0 ** -8 * np.abs(xf) + 1e-30)


def test_nvfp4_round_trip_identity_experts():
    T, H, E, K = 40, 64, 5, 2
    ids, _ = routing(T, K, E, 7, unused=0.0)
    p = np.full((T, K), 0.5, np.float32)
    x = rand_bf16((T, H), 8)
    L = oracle.layout(ids, E, S=0)
    fp4, sc, inv, _ = oracle.dispatch_nvfp4(x, L)
    R = L.R
    xf = f(x)
    g = np.float32(2688.0) / np.abs(W.f32_from_bf16_bits(x)).max(1)
    ginv_rows = 1.0 / g[L.src_info[:R, 0]].astype(np.float64)
    deq = oracle.dequantize_rows(fp4[:R], sc[:R], ginv_rows)
    y = np.zeros((L.R_max, H), np.uint16)
    y[:R] = np.array([[oracle.bf16_from_double(v) for v in row] for row in deq], np.uint16)
    out = f(oracle.combine(y, p, L))
    # per-element bound: half an E2M1 step (<= 1) times the block scale / g, plus two bf16 roundings
    sd = np.array([[oracle.e4m3_decode(int(s)) for s in row] for row in sc[:R]])
    blk = np.repeat(sd, 16, axis=1) / g[L.src_info[:R, 0]][:, None]
    bound_rows = 1.0 * blk
    bound = np.zeros((T, H))
    for t in range(T):
        bound[t] = bound_rows[L.row_of[t]].max(0)
    assert np.all(np.abs(out - xf) <= bound + 2.0 ** -7 * np.abs(xf) + 1e-30)


def test_tiny_closed_form():
    cfg = W.CONFIGS["tiny"]
    inp = W.make_inputs(cfg)
    L = oracle.layout(inp["topk_ids"], cfg.E)
    fp4, sc, inv, _ = oracle.dispatch_nvfp4(inp["x"], L)
    y = oracle.tiny_expert_outputs(fp4, sc, inv, L)
    out64 = oracle.combine(y, inp["probs"], L, want64=True)[1]
    # closed form from the dequantised token (same for all its copies)
    for t in range(cfg.T):
        c, s, i = oracle.nvfp4_quantize_row(inp["x"][t])
        d = oracle.dequantize_rows(c[None], s[None], np.array([oracle.bf16_to_double(i)]))[0]
        expect = sum(float(inp["probs"][t, k]) * (1 + inp["topk_ids"][t, k] / 8.0) * d
                     for k in range(cfg.K))
        # y rows were rounded to bf16 once: relative 2^-8 per term
        tol = sum(abs(float(inp["probs"][t, k])) * (1 + inp["topk_ids"][t, k] / 8.0) * np.abs(d)
                  for k in range(cfg.K)) * 2.0 ** -8
        assert np.all(np.abs(out64[t] - expect) <= tol + 1e-30)


@pytest.mark.parametrize("S", [0, 1])
def test_combine_bwd_adjoint_identities(S):
    T, H, E, K = 23, 32, 6, 3
    ids, p = routing(T, K, E, 12, unused=0.2)
    L = oracle.layout(ids, E, S=S)
    y = rand_bf16((L.R_max, H), 13)
    g = rand_bf16((T, H), 14)
    out, out64 = oracle.combine(y, p, L, want64=True)
    gy, gp, gy64 = oracle.combine_bwd(g, y, p, L, want64=True)
    R = L.R
    lhs = float(np.sum(out64 * f(g)))
    rhs = float(np.sum(f(y[:R]) * gy64[:R]))
    assert abs(lhs - rhs) <= 1e-12 * (np.sum(np.abs(out64 * f(g))) + 1)
    # grad_p = derivative of <combine(y), g> along each probability (combine is linear in p)
    base = float(np.sum(oracle.combine(y, np.zeros_like(p), L, want64=True)[1] * f(g)))
    for t in range(T):
        for k in range(K):
            e = np.zeros_like(p)
            e[t, k] = 1.0
            val = float(np.sum(oracle.combine(y, e, L, want64=True)[1] * f(g))) - base
            assert abs(gp[t, k] - val) <= 1e-9 * (abs(val) + 1)
            if ids[t, k] < 0:
                assert gp[t, k] == 0.0
    # bf16 rows are the single rounding of the binary64 products; shared rows copy g exactly
    for r in range(R):
        assert all(oracle.bf16_from_double(v) == b for v, b in zip(gy64[r][:4], gy[r][:4]))
    if S:
        assert np.array_equal(gy[L.row_offsets[E]:R], g)


@pytest.mark.parametrize("S", [0, 1])
def test_dispatch_bwd_adjoint(S):
    T, H, E, K = 31, 48, 5, 2
    ids, _ = routing(T, K, E, 21, unused=0.15)
    L = oracle.layout(ids, E, S=S)
    x = rand_bf16((T, H), 22)
    gd = rand_bf16((L.R_max, H), 23)
    disp = oracle.dispatch_bf16(x, L)
    gx, gx64 = oracle.dispatch_bwd(gd, L, want64=True)
    lhs = float(np.sum(f(disp[:L.R]) * f(gd[:L.R])))
    rhs = float(np.sum(f(x) * gx64))
    assert abs(lhs - rhs) <= 1e-12 * (np.sum(np.abs(f(disp[:L.R]) * f(gd[:L.R]))) + 1)


def test_nothing_written_on_bad_status():
    ids = np.array([[0, 9]], np.int32)
    L = oracle.layout(ids, 4)
    assert L.status == oracle.BAD_EXPERT
    y = rand_bf16((L.R_max, 16), 1)
    assert (oracle.combine(y, np.ones((1, 2), np.float32), L) == 0xA5A5).all()
    gy, gp = oracle.combine_bwd(rand_bf16((1, 16), 2), y, np.ones((1, 2), np.float32), L)
    assert (gy == 0xA5A5).all()


def test_shared_row_alone_when_probs_are_zero():
    """With every probability zero, combine returns the shared expert's row exactly (weight 1),
    and with no shared expert it returns zeros."""
    T, H, E, K = 9, 32, 4, 2
    ids, _ = routing(T, K, E, 30, unused=0.0)
    z = np.zeros((T, K), np.float32)
    L = oracle.layout(ids, E, S=1)
    y = rand_bf16((L.R_max, H), 31)
    out = oracle.combine(y, z, L)
    assert np.array_equal(out, y[L.row_offsets[E]:L.R])
    L0 = oracle.layout(ids, E, S=0)
    out0 = oracle.combine(y[:L0.R_max], z, L0)
    assert (W.f32_from_bf16_bits(out0) == 0).all()
    # dispatch backward of a single one-hot row returns it at its source token only
    gd = np.zeros((L.R_max, H), np.uint16)
    r = int(L.row_of[4, 1])
    gd[r] = y[r]
    gx = oracle.dispatch_bwd(gd, L)
    assert np.array_equal(gx[4], y[r]) and (W.f32_from_bf16_bits(np.delete(gx, 4, 0)) == 0).all()
