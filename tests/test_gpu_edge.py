"""Edge cases and device-side error handling, GPU vs oracle.  None of these cases faults: bad
expert ids and capacity overflow are recorded in the layout's status word, after which every
data kernel writes nothing (checked with canary-filled outputs)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (assert_close_bf16, check_layout, dev, dev_bf16, host_bf16, new_layout)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def full_check(ep, ids, x, probs, y, E, P=1, C=None, S=0):
    T, K = ids.shape
    H = x.shape[1]
    C = T if C is None else C
    ref = oracle.layout(ids, E, P=P, C=C, S=S)
    L = new_layout(ep, T, K, E, P, S)
    ep.dispatch_layout(dev(ids) if T else torch.empty(0, K, dtype=torch.int32, device="cuda"),
                       E, P, C, bool(S), out=L)
    check_layout(L, ref, ep)
    R_max = max(ref.R_max, 1)
    fp4 = torch.full((R_max, H // 2), 0x5A, dtype=torch.uint8, device="cuda")
    sc = torch.full((R_max, H // 16), 0x5A, dtype=torch.uint8, device="cuda")
    inv = torch.full((R_max,), 0x1357, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    so = torch.full((E + S + 1,), -7, dtype=torch.int32, device="cuda")
    xd = dev_bf16(x) if T else torch.empty(0, H, dtype=torch.bfloat16, device="cuda")
    ep.dispatch_nvfp4(xd, L, out=(fp4, sc, inv, so))
    rfp4, rsc, rinv, rso = oracle.dispatch_nvfp4(x, ref, fill=0x5A)
    if ref.R_max:
        assert np.array_equal(fp4.cpu().numpy()[:ref.R_max], rfp4)
        assert np.array_equal(sc.cpu().numpy()[:ref.R_max], rsc)
        gi = host_bf16(inv)[:ref.R_max]
        if ref.status:
            assert (gi == 0x1357).all()
        else:
            assert np.array_equal(gi[:ref.R], rinv[:ref.R])
    if not ref.status:
        assert np.array_equal(so.cpu().numpy(), rso)
    if T:
        yd = dev_bf16(y)
        out = torch.full((T, H), 0x2468, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        ep.combine(yd, dev(probs), L, out=out)
        got = host_bf16(out)
        if ref.status:
            assert (got == 0x2468).all()
        else:
            _, r64 = oracle.combine(y, probs, ref, want64=True)
            assert_close_bf16(got, r64, "combine")
    return ref


def rand_case(T, K, E, H, seed, unused=0.0, dup=False):
    rng = np.random.default_rng(seed)
    if dup:
        ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32) if T else \
            np.zeros((0, K), np.int32)
    if unused:
        ids[rng.random((T, K)) < unused] = -1
    x = W.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    p = rng.random((T, K)).astype(np.float32)
    y = W.bf16_bits_from_f32(rng.standard_normal((max(T * K + T, 1), H)).astype(np.float32))
    return ids, x, p, y


def test_empty_input(ep):
    ids, x, p, y = rand_case(0, 4, 16, 64, 1)
    ref = full_check(ep, ids, x, p, y, 16, P=4, S=1)
    assert ref.R == 0


def test_all_slots_unused(ep):
    T, K, E, H = 300, 3, 8, 64
    ids = np.full((T, K), -1, np.int32)
    _, x, p, y = rand_case(T, K, E, H, 2)
    for S in (0, 1):
        ref = full_check(ep, ids, x, p, y, E, P=2, S=S)
        assert ref.R == S * T


@pytest.mark.parametrize("H", [16, 48, 96, 32768])
def test_hidden_sizes(ep, H):
    T = 40 if H == 32768 else 333
    ids, x, p, y = rand_case(T, 2, 6, H, H, unused=0.1)
    full_check(ep, ids, x, p, y, 6, P=3, S=1)


def test_largest_k_and_e(ep):
    ids, x, p, y = rand_case(300, 32, 1024, 64, 7, unused=0.05)
    full_check(ep, ids, x, p, y, 1024, P=16, S=1)


def test_largest_k_and_e_two_kernel_layout(ep):
    """K = 32 and E = 1024 with more ids (160,000) than one thread-block cluster holds, so the
    two-kernel layout runs at its widest count table."""
    ids, x, p, y = rand_case(5000, 32, 1024, 32, 17, unused=0.05)
    full_check(ep, ids, x, p, y, 1024, P=8, S=1)


def test_largest_token_count(ep):
    """T at the limit the entry points accept (2^24 tokens, 50,331,648 rows with the shared
    copies): every grid and every row index at the top of its range.  Ids include -1 and
    repeats within a token."""
    T, K, E, H = 1 << 24, 2, 8, 16
    rng = np.random.default_rng(16)
    ids = rng.integers(-1, E, size=(T, K), dtype=np.int32)
    x = W.bf16_bits_from_f32(rng.standard_normal((T, H), dtype=np.float32))
    p = rng.random((T, K), dtype=np.float32)
    y = np.resize(W.bf16_bits_from_f32(rng.standard_normal((65537, H), dtype=np.float32)),
                  (T * K + T, H))
    ref = full_check(ep, ids, x, p, y, E, P=4, S=1)
    assert ref.status == 0 and ref.R > T


def test_single_expert_single_slot(ep):
    ids, x, p, y = rand_case(129, 1, 1, 32, 8)
    full_check(ep, ids, x, p, y, 1)


def test_duplicate_ids_within_a_token(ep):
    ids, x, p, y = rand_case(517, 4, 3, 64, 9, dup=True)
    full_check(ep, ids, x, p, y, 3, S=1)


def test_ragged_last_tile_of_one_token(ep):
    ids, x, p, y = rand_case(4097, 2, 64, 32, 10, unused=0.02)
    full_check(ep, ids, x, p, y, 64, P=8)


@pytest.mark.parametrize("T", [17000, 34000])
def test_layout_beyond_one_cluster(ep, T):
    """17,000 tokens (136,000 ids): the single-cluster layout with more than 8192 ids per CTA,
    each lane's ids loaded in two batches.  34,000 tokens (272,000 ids): above what one
    thread-block cluster holds, so the two-kernel layout (tile histograms, scan by the last CTA,
    ranks) runs instead."""
    ids, x, p, y = rand_case(T, 8, 64, 16, 15, unused=0.03)
    ids[5, 3] = 64                     # one bad id: flagged, then nothing written
    ref = full_check(ep, ids, x, p, y, 64, P=4, S=1)
    assert ref.status == oracle.BAD_EXPERT
    ids[5, 3] = 7
    full_check(ep, ids, x, p, y, 64, P=4, C=T - 2000, S=1)


def test_bad_expert_ids_write_nothing(ep):
    ids, x, p, y = rand_case(200, 4, 16, 64, 11)
    ids[17, 2] = 16
    ids[150, 0] = -3
    ref = full_check(ep, ids, x, p, y, 16, P=4, S=1)
    assert ref.status == oracle.BAD_EXPERT


def test_overflow_writes_nothing_then_clears(ep):
    ids, x, p, y = rand_case(256, 4, 16, 64, 12)
    ids[:, 0] = 0                     # every token reaches partition 0
    ref = full_check(ep, ids, x, p, y, 16, P=4, C=255)
    assert ref.status == oracle.OVERFLOW
    ref = full_check(ep, ids, x, p, y, 16, P=4, C=256)
    assert ref.status == 0


def test_rows_with_zeros_subnormals_and_outliers(ep):
    T, K, E, H = 64, 2, 4, 128
    ids, x, p, y = rand_case(T, K, E, H, 13)
    x[3] = 0
    x[4] = 0x8000                     # all -0.0
    x[5, :] = 0
    x[5, 7] = 0x0001                  # smallest subnormal bf16
    x[5, 100] = 0x8002
    x[6] = W.bf16_bits_from_f32(W.f32_from_bf16_bits(x[6]) * np.float32(7.5e37))   # near the top
    x[7] = W.bf16_bits_from_f32(W.f32_from_bf16_bits(x[7]) * np.float32(1e-36))    # g clamps
    assert np.isfinite(W.f32_from_bf16_bits(x)).all()
    x[8, ::16] = 0                    # blocks with a zero element
    x[9, 16:32] = 0x0003              # a block of subnormals next to normal blocks
    full_check(ep, ids, x, p, y, E)


@pytest.mark.parametrize("H", [256, 512])
def test_fused_call_rows_with_zeros_subnormals_and_outliers(ep, H):
    """The same special rows through the fused layout + NVFP4 call, whose staged kernel (H a
    multiple of 256) takes the row and block maxima on packed bf16 patterns."""
    T, K, E = 600, 3, 16
    ids, x, p, y = rand_case(T, K, E, H, 14)
    x[3] = 0
    x[4] = 0x8000
    x[5, :] = 0
    x[5, 7] = 0x0001
    x[5, H - 3] = 0x8002
    x[6] = W.bf16_bits_from_f32(W.f32_from_bf16_bits(x[6]) * np.float32(7.5e37))
    x[7] = W.bf16_bits_from_f32(W.f32_from_bf16_bits(x[7]) * np.float32(1e-36))
    x[8, ::16] = 0
    x[9, 16:32] = 0x0003
    x[10, 32:48] = 0x807F                               # largest negative subnormal block
    x[11] = W.bf16_bits_from_f32(-np.abs(W.f32_from_bf16_bits(x[11])))   # all negative
    x[12, :] = 0x0001
    x[12, 200] = 0x7F7F                                 # largest finite bf16 beside subnormals
    assert np.isfinite(W.f32_from_bf16_bits(x)).all()
    ref = oracle.layout(ids, E, P=4, C=T, S=1)
    L = new_layout(ep, T, K, E, 4, 1)
    R_max = ref.R_max
    out = (torch.full((R_max, H // 2), 0x5A, dtype=torch.uint8, device="cuda"),
           torch.full((R_max, H // 16), 0x5A, dtype=torch.uint8, device="cuda"),
           torch.full((R_max,), 0x1357, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           torch.full((E + 2,), -7, dtype=torch.int32, device="cuda"))
    ep.dispatch_layout_nvfp4(dev(ids), dev_bf16(x), E, 4, T, True, out_layout=L, out=out)
    check_layout(L, ref, ep)
    rfp4, rsc, rinv, rso = oracle.dispatch_nvfp4(x, ref, fill=0x5A)
    assert np.array_equal(out[0].cpu().numpy(), rfp4)
    assert np.array_equal(out[1].cpu().numpy(), rsc)
    assert np.array_equal(host_bf16(out[2])[:ref.R], rinv[:ref.R])
    assert np.array_equal(out[3].cpu().numpy(), rso)


def _every_scale_code_rows(T, rng):
    """Rows of 128 blocks (H = 2048) whose block scales take every finite E4M3 code.  Element
    0 of each row is 2688, so g = 2688 / 2688 = 1 and sf = blockmax / 6; block c (c = 1..126)
    has the maximum 6 * value(c), so sf is exactly the value of code c, and the other 15
    elements are random fractions of that maximum.  Block 127 is all zero (code 0)."""
    H = 2048
    codes = np.arange(1, 127)
    vals = np.array([oracle.e4m3_decode(int(c)) for c in codes], np.float64)
    x = np.zeros((T, H), np.float32)
    for t in range(T):
        perm = rng.permutation(126)                       # which block gets which code
        for b in range(126):
            bm = 6.0 * vals[perm[b]]
            blk = bm * rng.uniform(-1, 1, 16)
            blk[rng.integers(16)] = bm * (1 if rng.random() < 0.5 else -1)
            x[t, 16 * b:16 * b + 16] = blk
        x[t, 126 * 16:127 * 16] = 0
        x[t, 127 * 16:] = 0
        x[t, 126 * 16] = 2688.0                           # the row maximum (block 126: code 0x7E)
    bits = W.bf16_bits_from_f32(x)
    # the block maxima and 2688 are bf16 values, so rounding to bf16 keeps them
    assert np.abs(W.f32_from_bf16_bits(bits)).max() == 2688.0
    return bits


def test_every_block_scale_code(ep):
    """Every E4M3 block-scale code (and with it every g / s quotient of the element scaling)
    through both NVFP4 kernels: the per-token dispatch and the fused call's staged one."""
    T, K, E = 300, 2, 8
    rng = np.random.default_rng(21)
    x = _every_scale_code_rows(T, rng)
    ids, _, p, y = rand_case(T, K, E, 16, 22)
    ref = oracle.layout(ids, E, P=1, C=T, S=1)
    rfp4, rsc, rinv, rso = oracle.dispatch_nvfp4(x, ref, fill=0x5A)
    assert set(np.unique(rsc[:ref.R])) >= set(range(0, 127)), "the rows cover every code"
    for fused in (False, True):
        L = new_layout(ep, T, K, E, 1, 1)
        out = (torch.full((ref.R_max, 1024), 0x5A, dtype=torch.uint8, device="cuda"),
               torch.full((ref.R_max, 128), 0x5A, dtype=torch.uint8, device="cuda"),
               torch.full((ref.R_max,), 0x1357, dtype=torch.int16, device="cuda").view(torch.bfloat16),
               torch.full((E + 2,), -7, dtype=torch.int32, device="cuda"))
        if fused:
            ep.dispatch_layout_nvfp4(dev(ids), dev_bf16(x), E, 1, T, True, out_layout=L, out=out)
        else:
            ep.dispatch_layout(dev(ids), E, 1, T, True, out=L)
            ep.dispatch_nvfp4(dev_bf16(x), L, out=out)
        check_layout(L, ref, ep)
        assert np.array_equal(out[0].cpu().numpy(), rfp4), f"codes (fused={fused})"
        assert np.array_equal(out[1].cpu().numpy(), rsc), f"scales (fused={fused})"
        assert np.array_equal(host_bf16(out[2])[:ref.R], rinv[:ref.R])


def test_status_word_and_read_status(ep):
    ids = dev(np.array([[0, 1], [2, 99]], np.int32))
    L = ep.dispatch_layout(ids, 4, n_parts=2)
    assert ep.read_status(L) == ep.STATUS_BAD_EXPERT
    with pytest.raises(ValueError):     # buffers sized for P = 2 cannot take P = 4
        ep.dispatch_layout(ids, 4, n_parts=4, out=L)
    L2 = ep.dispatch_layout(dev(np.array([[0, 1], [2, 3]], np.int32)), 4, n_parts=2, capacity=0, out=L)
    assert ep.read_status(L2) == ep.STATUS_OVERFLOW
    ep.dispatch_layout(dev(np.array([[0, 1], [2, 3]], np.int32)), 4, n_parts=2, capacity=2, out=L)
    assert ep.read_status(L) == 0


def test_invalid_arguments_raise(ep):
    ids = dev(np.zeros((4, 2), np.int32))
    with pytest.raises(ep.EPError):
        ep.dispatch_layout(ids, 8, n_parts=3)
    L = ep.dispatch_layout(ids, 8)
    x = torch.zeros(4, 40, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError):
        ep.dispatch_nvfp4(x, L)
