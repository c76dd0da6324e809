"""The benchmark's algorithmic byte counts (the numerators of every roofline fraction) against
a brute-force count: on small oracle layouts with unused slots and a shared expert, walk what
each operation must read and write by its definition, every distinct byte once."""
import numpy as np
import pytest

import bench
import oracle
import workloads as W


def brute_force(cfg, ids):
    T, K, E, S, H = cfg.T, cfg.K, cfg.E, cfg.S, cfg.H
    ref = oracle.layout(ids, E, P=1, C=T, S=S)
    valid = ids >= 0
    routed_rows = {int(r) for r in ref.row_of[valid]}
    shared_rows = {int(ref.row_offsets[E]) + t for t in range(T)} if S else set()
    rows = routed_rows | shared_rows                    # every row of the layout in use
    assert len(rows) == ref.R
    x, out = 2 * T * H, 2 * T * H                       # one token-major bf16 matrix
    ids_b = row_of_b = probs_b = 4 * T * K              # int32 / fp32 [T, K]
    meta = 12 * len(rows)                               # src_info (2 x int32) + expert_ids per row
    nvfp4_row = H // 2 + H // 16 + 2                    # codes, E4M3 block scales, bf16 inverse
    fp8_row = H + 4 * (H // 128)                        # codes, fp32 block scales
    y_row = 2 * H
    return ref.R, {
        "layout": ids_b + meta + row_of_b,
        "dispatch_nvfp4": x + len(rows) * nvfp4_row,
        "combine": len(rows) * y_row + probs_b + row_of_b + out,
        "dispatch_bf16": x + len(rows) * y_row + row_of_b,
        # g read once; y read for the routed rows (their dot products with g); grad_y written
        # for every row; probs, row_of read and grad_probs written
        "combine_bwd": x + len(routed_rows) * y_row + len(rows) * y_row + probs_b + row_of_b + 4 * T * K,
        "dispatch_bwd": len(rows) * y_row + row_of_b + out,
        "dispatch_fp8": x + len(rows) * fp8_row,
        "routing_map_layout": T * E + 4 * T * E + 4 * T * K + 4 * T * K + (ids_b + meta + row_of_b),
        "indices_to_multihot": ids_b + probs_b + T * E + 4 * T * E,
    }


@pytest.mark.parametrize("S,unused", [(0, 0.0), (1, 0.0), (1, 0.2), (0, 0.35)])
def test_algorithmic_bytes_match_a_brute_force_count(S, unused):
    rng = np.random.default_rng(40 + S)
    T, K, E, H = 61, 3, 8, 256
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < unused] = -1
    cfg = W.Config(950, "accounting", T=T, H=H, E=E, K=K, S=S, P=1)
    R, want = brute_force(cfg, ids)
    got = bench.algorithmic_bytes(cfg, R)
    assert set(got) == set(want)
    for k in want:
        assert got[k] == want[k], k


def test_padded_bytes_count_every_row_below_the_padded_extent():
    rng = np.random.default_rng(44)
    T, K, E, H, pad = 70, 2, 6, 128, 16
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    cfg = W.Config(951, "accounting", T=T, H=H, E=E, K=K, S=1, P=1)
    ref = oracle.layout(ids, E, P=1, C=T, S=1, pad_multiple=pad)
    R_pad = int(ref.row_offsets[E + 1])
    assert R_pad == ref.R and R_pad % pad == 0 and R_pad > T * K + T   # padding rows included
    got = bench.padded_bytes(cfg, R_pad)
    assert got["dispatch_nvfp4"] == 2 * T * H + R_pad * (H // 2 + H // 16 + 2)
    assert got["layout"] == 4 * T * K + 12 * R_pad + 4 * T * K


def test_dsv3_step_bytes():
    """The DSv3-shaped step the headline number is quoted on: layout + NVFP4 dispatch +
    combine over 36,864 rows move 795,598,848 algorithmic bytes."""
    cfg = W.CONFIGS["dsv3"]
    R = cfg.T * cfg.K + cfg.T
    b = bench.algorithmic_bytes(cfg, R)
    assert b["layout"] + b["dispatch_nvfp4"] + b["combine"] == 795_598_848
    assert b["combine"] == 587_464_704 and b["dispatch_nvfp4"] == 207_429_632
