"""Helpers shared by the GPU parity tests: host <-> device marshalling and comparisons against
the oracle.  Tolerances (stated once, used everywhere):

* layout, permutation, NVFP4 codes, E4M3 scales, bf16 inverse scales, bf16 dispatch: bit-exact;
* bf16 results of combine / combine_bwd / dispatch_bwd: |gpu - ref| <= max(2^-7 |ref|, 1e-3)
  element-wise, ref = the oracle's binary64 value before rounding;
* grad_probs (fp32 dot products over H): |gpu - ref| <= 2^-7 |ref| + 1e-3 + 2^-16 sum_i |g_i y_i|
  (the last term bounds fp32 accumulation of a sum that may cancel).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL = 2.0 ** -7
ABS = 1e-3
CANARY32 = -7


def dev_bf16(a_u16: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).to(device).view(torch.bfloat16)


def host_bf16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close_bf16(got_bits: np.ndarray, ref64: np.ndarray, what: str):
    got = f64(got_bits)
    err = np.abs(got - ref64)
    tol = np.maximum(REL * np.abs(ref64), ABS)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements outside tolerance, first at {tuple(i)}: "
                             f"gpu {got[tuple(i)]} ref {ref64[tuple(i)]}")


def assert_close_gradp(got: np.ndarray, ref: np.ndarray, abs_dot: np.ndarray, what: str):
    tol = REL * np.abs(ref) + ABS + 2.0 ** -16 * abs_dot
    bad = np.abs(got.astype(np.float64) - ref) > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outside tolerance, first {tuple(i)}: "
                             f"gpu {got[tuple(i)]} ref {ref[tuple(i)]}")


def new_layout(ep, T, K, E, P, S, device="cuda"):
    L = ep.Layout(T, K, E, P, bool(S), device=device)
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    return L


def check_layout(L, ref, ep):
    """Bit-exact layout parity; rows past R keep their canaries."""
    R = ref.R
    st = ep.read_status(L)
    assert st == ref.status, (st, ref.status)
    assert np.array_equal(L.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(L.part_tokens.cpu().numpy(), ref.part_tokens)
    T = ref.T
    if T:
        assert np.array_equal(L.row_of.cpu().numpy()[:T], ref.row_of)
    ei = L.expert_ids.cpu().numpy()
    si = L.src_info.cpu().numpy()
    assert np.array_equal(ei[:R], ref.expert_ids[:R])
    assert np.array_equal(si[:R], ref.src_info[:R])
    assert (ei[R:ref.R_max] == CANARY32).all() and (si[R:ref.R_max] == CANARY32).all()


def abs_dots(g_bits, y_bits, row_of):
    """sum_i |g[t,i] * y[row,i]| for every (t, k) (0 for an unused slot)."""
    g = np.abs(f64(g_bits))
    T, K = row_of.shape
    out = np.zeros((T, K))
    for k in range(K):
        r = row_of[:, k]
        ok = r >= 0
        out[ok, k] = np.sum(g[ok] * np.abs(f64(y_bits[r[ok]])), axis=1)
    return out


def mini_layout_for_token(ref, t, topk_row, E, S):
    """Oracle layout of token t alone, and the map from its rows to the full layout's rows."""
    L1 = oracle.layout(topk_row[None, :], E, S=S)
    K = topk_row.size
    src = np.full(L1.R_max, -1, np.int64)
    for k in range(K):
        if L1.row_of[0, k] >= 0:
            src[L1.row_of[0, k]] = ref.row_of[t, k]
    if S:
        src[L1.row_offsets[E]] = ref.row_offsets[E] + t
    return L1, src
