"""The hardware E2M1 / E4M3 conversions the NVFP4 kernel uses, checked against the oracle's
encoders (written from the format definitions) on every bf16 bit pattern, on windows of
binary32 patterns around every rounding midpoint, on random binary32 patterns, and on the
special values (signed zeros, infinities, saturation, subnormals).  NaN is excluded: the
dispatch never produces one from finite inputs."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def finite_bf16_patterns():
    b = np.arange(1 << 16, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return f[~np.isnan(f)]


def windows(mids, width=4096):
    out = []
    for m in mids:
        u = np.array([m], np.float32).view(np.uint32)[0].astype(np.int64)
        pats = np.arange(max(0, u - width), u + width + 1).astype(np.uint32)
        v = pats.view(np.float32)
        out += [v, -v]
    return np.concatenate(out)


def random_patterns(n, max_exp, seed):
    rng = np.random.default_rng(seed)
    sign = rng.integers(0, 2, n, dtype=np.uint32) << 31
    ex = rng.integers(0, 127 + max_exp + 1, n, dtype=np.uint32) << 23
    man = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    return (sign | ex | man).view(np.float32)


SPECIALS = np.array([0.0, -0.0, np.inf, -np.inf, np.finfo(np.float32).max, -np.finfo(np.float32).max,
                     np.finfo(np.float32).tiny, 1e-45, -1e-45, 6.0, -6.0, 448.0, -448.0, 464.0,
                     480.0, 1e30], np.float32)


def compare(ep, v, gpu_fn, ref_fn, what):
    v = np.ascontiguousarray(v, np.float32)
    got = gpu_fn(torch.from_numpy(v).cuda()).cpu().numpy()
    ref = ref_fn(v)
    bad = got != ref
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {bad.sum()} mismatches, first v={v[i]!r} "
                             f"(bits {v.view(np.uint32)[i]:#010x}) gpu {got[i]:#x} ref {ref[i]:#x}")


def test_e2m1_matches_definition(ep):
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]
    v = np.concatenate([finite_bf16_patterns(), windows(mids), random_patterns(1 << 22, 3, 1),
                        random_patterns(1 << 20, 127, 2), SPECIALS])
    compare(ep, v, ep.cvt_e2m1, oracle.e2m1_encode_array, "E2M1")


def test_e4m3_matches_definition(ep):
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    mids = [0.5 * (a + b) for a, b in zip(vals, vals[1:])] + [448.0, 464.0]
    v = np.concatenate([finite_bf16_patterns(), windows(mids, 1024), random_patterns(1 << 22, 9, 3),
                        random_patterns(1 << 20, 127, 4), SPECIALS])
    compare(ep, v, ep.cvt_e4m3, oracle.e4m3_encode_array, "E4M3")


def test_nibble_order_of_packed_codes(ep):
    """The dispatch puts element 2j in the low nibble of byte j: checked on a row whose even and
    odd elements have different codes."""
    from gpu_helpers import dev_bf16
    import workloads as W
    x = np.zeros((1, 32), np.float32)
    x[0, 0::2] = 6.0      # code 7
    x[0, 1::2] = 1.0      # code 2 after scaling by g/s = 1 (rowmax 6 -> g = 448, s = 448)
    xb = W.bf16_bits_from_f32(x)
    L = ep.dispatch_layout(torch.zeros(1, 1, dtype=torch.int32, device="cuda"), 1)
    fp4, sc, inv, so = ep.dispatch_nvfp4(dev_bf16(xb), L)
    codes = fp4.cpu().numpy()[0]
    assert (codes == 0x27).all(), codes
    assert (sc.cpu().numpy()[0] == 0x7E).all()
