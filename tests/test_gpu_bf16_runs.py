"""BF16 dispatch in runs of consecutive tokens: every hidden size that changes the run length
(4 tokens at H <= 2048, 2 at H = 4096, 1 above), token counts that leave a ragged last run,
padded groups and a capped row count, compared bit for bit with the oracle (canary-filled
outputs, so a row written twice, too early or past the layout shows)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import dev, dev_bf16, host_bf16

pytestmark = pytest.mark.gpu

CANARY = 0xA5A5


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


# (T, H, K, E, S, pad, cap): T mod the run length is non-zero wherever the run is longer than one
CASES = [
    (1, 4096, 2, 8, 0, 1, None),       # one run of one token where runs hold two
    (3, 4096, 2, 8, 1, 1, None),
    (1001, 4096, 3, 16, 1, 1, None),
    (777, 3072, 4, 32, 0, 16, None),   # two tokens a run, padded groups
    (5, 2048, 8, 64, 1, 1, None),      # four tokens a run
    (1003, 2048, 8, 128, 0, 128, None),
    (514, 1024, 5, 8, 1, 1, 3000),     # a static row capacity above the rows in use
    (514, 1024, 5, 8, 1, 1, 2000),     # ... and below them: the status word stops every row
    (6, 256, 2, 8, 0, 3, None),
    (7, 16, 1, 1, 1, 1, None),         # the smallest hidden size
    (9, 8192, 4, 16, 1, 1, None),      # one token a run
    (3, 32768, 2, 4, 0, 2, None),      # one token, several chunks a thread
]


@pytest.mark.parametrize("T,H,K,E,S,pad,cap", CASES)
def test_bf16_runs_match_oracle(ep, T, H, K, E, S, pad, cap):
    rng = np.random.default_rng(T * 131 + H)
    ids = np.stack([rng.permutation(E)[:K] if K <= E else rng.integers(0, E, K)
                    for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < 0.1] = -1
    x = W.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    ref = oracle.layout(ids, E, P=1, C=T, S=S, pad_multiple=pad, num_permuted_tokens=cap)
    L = ep.Layout(T, K, E, 1, bool(S), pad_multiple=pad, num_permuted_tokens=cap)
    ep.dispatch_layout_routed(E, topk_ids=dev(ids), n_parts=1, capacity=T, fused_shared=bool(S),
                              pad_multiple=pad, num_permuted_tokens=cap, out=L)
    assert ep.read_status(L) == ref.status
    rows = torch.full((ref.R_max, H), CANARY - 65536, dtype=torch.int16, device="cuda")
    ep.dispatch_bf16(dev_bf16(x), L, out=rows.view(torch.bfloat16))
    got = host_bf16(rows.view(torch.bfloat16))
    want = oracle.dispatch_bf16(x, ref, fill=CANARY)
    if ref.status:
        assert (got == CANARY).all(), "rows written under a set status word"
    else:
        assert np.array_equal(got, want), f"T={T} H={H}: BF16 rows differ from the oracle"
