"""Pins of the oracle's FP8 (E4M3, one scale per 128-element block) quantisation and dispatch.

Hand-worked blocks are in tests/golden/fp8_blocks.txt.  Beyond them: exact power-of-two scaling
(a block multiplied by 2^j keeps its codes and its scale is multiplied by 2^j), the block's
largest magnitude landing on E4M3's largest finite value, block independence, the E4M3
rounding error bound of the dequantised values, and the dispatch copying each token's encoding
to exactly its rows.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from conftest import read_golden

B = oracle.FP8_BLOCK


def e4m3_values():
    return np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)


def test_golden_blocks():
    recs = {g["name"]: g for g in read_golden("fp8_blocks.txt")}
    x = np.zeros(4 * B, np.uint16)
    want = np.zeros(4 * B, np.uint8)
    for b, name in enumerate("ABCD"):
        for item in recs[name].get("x", []):
            i, v = item.split(":")
            x[b * B + int(i)] = int(v, 16)
        for item in recs[name].get("codes", []):
            i, v = item.split(":")
            want[b * B + int(i)] = int(v, 16)
    codes, scales = oracle.fp8_quantize_row(x)
    assert codes.tolist() == want.tolist()
    assert scales[:3].tolist() == [float(recs[n]["scale"][0]) for n in "ABC"]
    assert int(scales[3:].view(np.uint32)[0]) == int(recs["D"]["scale_bits"][0], 16)


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(3)
    x = W.bf16_bits_from_f32(rng.standard_normal(8 * B).astype(np.float32))
    c0, s0 = oracle.fp8_quantize_row(x)
    xf = W.f32_from_bf16_bits(x)
    for j in (-20, -3, 1, 7, 30):
        xj = W.bf16_bits_from_f32(xf * np.float32(2.0 ** j))   # exact: bf16 keeps its 8 bits
        cj, sj = oracle.fp8_quantize_row(xj)
        assert np.array_equal(cj, c0)
        assert np.array_equal(sj, (s0 * np.float32(2.0 ** j)).astype(np.float32))


def test_block_max_maps_to_largest_finite_and_blocks_are_independent():
    rng = np.random.default_rng(4)
    x = W.bf16_bits_from_f32((rng.standard_normal(6 * B) * 3).astype(np.float32))
    codes, scales = oracle.fp8_quantize_row(x)
    xf = W.f32_from_bf16_bits(x).reshape(-1, B)
    for b in range(6):
        i = int(np.argmax(np.abs(xf[b])))
        assert codes[b * B + i] == (0xFE if xf[b, i] < 0 else 0x7E)
    y = x.copy()
    y[2 * B:3 * B] = W.bf16_bits_from_f32(rng.standard_normal(B).astype(np.float32) * 100)
    c2, s2 = oracle.fp8_quantize_row(y)
    keep = np.ones(6 * B, bool)
    keep[2 * B:3 * B] = False
    assert np.array_equal(c2[keep], codes[keep])
    assert np.array_equal(np.delete(s2, 2), np.delete(scales, 2)) and s2[2] != scales[2]


def test_dequantisation_error_bound():
    """|code * scale - x| <= 2^-4 |x| (half a unit of E4M3's 3-bit mantissa) plus the binary32
    roundings of x*s and 1/s, or half the subnormal step 2^-9 times the scale below E4M3's
    normal range."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal(64 * B) * np.exp(rng.uniform(-8, 8, 64 * B))
    x = W.bf16_bits_from_f32(v.astype(np.float32))
    codes, scales = oracle.fp8_quantize_row(x)
    xf = W.f32_from_bf16_bits(x).astype(np.float64)
    deq = e4m3_values()[codes] * np.repeat(scales.astype(np.float64), B)
    bound = (2.0 ** -4 + 2.0 ** -20) * np.abs(xf) + 2.0 ** -10 * np.repeat(scales, B) * 1.0001
    assert (np.abs(deq - xf) <= bound).all()


def test_zero_and_negative_zero():
    x = np.zeros(2 * B, np.uint16)
    x[B:] = 0x8000
    codes, scales = oracle.fp8_quantize_row(x)
    assert (codes[:B] == 0x00).all() and (codes[B:] == 0x80).all()
    assert scales.tolist() == [1.0, 1.0]


def test_dispatch_copies_each_token_to_its_rows():
    cfg = W.scaled(W.CONFIGS["dsv3"], T=37, H=512)
    inp = W.make_inputs(cfg)
    L = oracle.layout(inp["topk_ids"], cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    codes, scales = oracle.dispatch_fp8(inp["x"], L)
    for t in range(cfg.T):
        c, s = oracle.fp8_quantize_row(inp["x"][t])
        rows = [r for r in L.row_of[t] if r >= 0] + [L.row_offsets[cfg.E] + t]
        for r in rows:
            assert np.array_equal(codes[r], c) and np.array_equal(scales[r], s)
    assert (codes[L.R:] == 0xA5).all()
    L.status = oracle.OVERFLOW
    assert (oracle.dispatch_fp8(inp["x"], L)[0] == 0xA5).all()
