"""Pins of the oracle's NVFP4 quantisation and dispatch.

Against: hand-worked rows (tests/golden/nvfp4_rows.txt), the closed form 2688 = 6 * 448
(largest E2M1 times largest E4M3: the block holding the row maximum gets scale 448 and the
maximum element code +-6), the all-zero row, the dequantisation error bound, and the copy
structure of the dispatch (K routed copies plus the shared copy, rows past R untouched).
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from conftest import read_golden


def bf16_bits(v):
    return W.bf16_bits_from_f32(np.asarray(v, np.float32))


def unpack_codes(codes):
    out = np.empty(codes.size * 2, np.uint8)
    out[0::2] = codes & 0xF
    out[1::2] = codes >> 4
    return out


@pytest.mark.parametrize("rec", read_golden("nvfp4_rows.txt"), ids=lambda r: r["name"])
def test_golden_rows(rec):
    x = bf16_bits([float(v) for v in rec["x"]])
    assert np.array_equal(W.f32_from_bf16_bits(x), np.array([float(v) for v in rec["x"]], np.float32))
    codes, scales, inv = oracle.nvfp4_quantize_row(x)
    assert unpack_codes(codes).tolist() == [int(c, 16) for c in rec["codes"]]
    assert scales.tolist() == [int(c, 16) for c in rec["scales"]]
    assert inv == int(rec["inv"][0], 16)


def _random_rows(n, H, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal((n, H)).astype(np.float32) * scale)


@pytest.mark.parametrize("H,scale", [(16, 1.0), (256, 1.0), (2048, 50.0), (7168, 1.0), (64, 1e-30)])
def test_rowmax_block_gets_448_and_code_6(H, scale):
    """2688 = 6 * 448: the block holding max|x| gets E4M3 0x7E and that element code +-6."""
    xs = _random_rows(6, H, seed=H, scale=scale)
    for x in xs:
        xf = W.f32_from_bf16_bits(x)
        codes, scales, inv = oracle.nvfp4_quantize_row(x)
        q = unpack_codes(codes)
        i = int(np.argmax(np.abs(xf)))
        assert scales[i // 16] == 0x7E
        assert q[i] == (0xF if xf[i] < 0 else 0x7)
        assert scales.max() == 0x7E


def test_zero_row():
    x = np.zeros(64, np.uint16)
    codes, scales, inv = oracle.nvfp4_quantize_row(x)
    assert inv == 0x3F80 and not codes.any() and not scales.any()
    x[5] = 0x8000   # -0.0 keeps the row all-zero
    codes, scales, inv = oracle.nvfp4_quantize_row(x)
    assert inv == 0x3F80 and not codes.any() and not scales.any()


def test_inverse_scale_is_bf16_of_reciprocal():
    # rowmax = 2^k: g = 2688 * 2^-k exactly; 1/g = 2^k / 2688 = 2^(k-7) / 21
    for k in (-3, 0, 4, 9):
        x = np.zeros(32, np.float32)
        x[7] = -(2.0 ** k)
        x[20] = 2.0 ** (k - 1)
        _, _, inv = oracle.nvfp4_quantize_row(bf16_bits(x))
        exact = 2.0 ** (k - 7) / 21.0
        got = oracle.bf16_to_double(inv)
        assert abs(got - exact) <= 2.0 ** -9 * exact
        assert oracle.bf16_from_double(np.float32(1.0) / np.float32(2688.0 * 2.0 ** -k)) == inv


def _dequant_row(codes, scales, g):
    q = unpack_codes(codes)
    vals = np.array([oracle.e2m1_decode(int(c)) for c in q], np.float64)
    sd = np.repeat([oracle.e4m3_decode(int(s)) for s in scales], 16)
    return vals * sd / g, q, sd


@pytest.mark.parametrize("H,scale,seed", [(256, 1.0, 1), (2048, 1.0, 2), (7168, 1.0, 3), (512, 50.0, 4)])
def test_dequant_error_bound(H, scale, seed):
    """|code * sd / g - x| <= 1/2 * step(code) * sd / g for blocks with a normal E4M3 scale,
    where step is the E2M1 spacing at the code (step(6) = 2 also covers saturation)."""
    step = {0: 0.5, 1: 0.5, 2: 0.5, 3: 0.5, 4: 1.0, 5: 1.0, 6: 2.0, 7: 2.0}
    for x in _random_rows(4, H, seed, scale):
        xf = W.f32_from_bf16_bits(x).astype(np.float64)
        codes, scales, inv = oracle.nvfp4_quantize_row(x)
        a = np.abs(xf).max()
        g = np.float32(2688.0) / np.float32(a)
        deq, q, sd = _dequant_row(codes, scales, float(g))
        normal = np.repeat(scales >= 0x08, 16)
        st = np.array([step[int(c) & 7] for c in q])
        err = np.abs(deq - xf)
        bound = 0.5 * st * sd / float(g) * (1 + 1e-6)
        assert (err[normal] <= bound[normal]).all()
        # every element keeps its sign (or becomes zero)
        assert (np.sign(deq) * np.sign(xf) >= 0).all()


def test_subnormal_rows_no_nan_and_saturate():
    # rowmax far below 2688 / FLT_MAX: g clamps to FLT_MAX, every code stays finite
    x = np.zeros(32, np.uint16)
    x[0] = 0x0001           # smallest bf16 subnormal
    x[17] = 0x8003
    codes, scales, inv = oracle.nvfp4_quantize_row(x)
    q = unpack_codes(codes)
    assert inv == oracle.bf16_from_double(np.float32(1.0) / np.float32(np.finfo(np.float32).max))
    assert set(q.tolist()) <= set(range(16))


def test_dispatch_copies_and_untouched_rows():
    rng = np.random.default_rng(9)
    T, H, E, K = 37, 64, 6, 3
    ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    x = _random_rows(T, H, 21)
    for S in (0, 1):
        L = oracle.layout(ids, E, P=3, C=T, S=S)
        fp4, sc, inv, so = oracle.dispatch_nvfp4(x, L, fill=0x5A)
        assert so.tolist() == L.row_offsets.tolist()
        for t in range(T):
            c, s, i = oracle.nvfp4_quantize_row(x[t])
            rows = [r for r in L.row_of[t] if r >= 0] + ([L.row_offsets[E] + t] if S else [])
            for r in rows:
                assert np.array_equal(fp4[r], c) and np.array_equal(sc[r], s) and inv[r] == i
        assert (fp4[L.R:] == 0x5A).all() and (sc[L.R:] == 0x5A).all()
        bf = oracle.dispatch_bf16(x, L, fill=0x1234)
        for r in range(L.R):
            t = L.src_info[r][0]
            assert np.array_equal(bf[r], x[t])
        assert (bf[L.R:] == 0x1234).all()


def test_dispatch_writes_nothing_on_overflow():
    ids = np.array([[0, 1], [0, 1], [1, 0]], np.int32)
    L = oracle.layout(ids, 2, P=2, C=2, S=0)
    assert L.status == oracle.OVERFLOW
    x = _random_rows(3, 32, 1)
    fp4, sc, inv, so = oracle.dispatch_nvfp4(x, L, fill=0x77)
    assert (fp4 == 0x77).all() and (sc == 0x77).all() and (inv == 0x7777).all()
    assert (oracle.dispatch_bf16(x, L, fill=0x4321) == 0x4321).all()
