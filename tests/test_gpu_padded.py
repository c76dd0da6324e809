"""GPU vs oracle parity of padded layouts, static row capacities and the padding rows every
dispatch writes (token_dispatcher page, TokenDispatcherConfig.moe_router_expert_pad_multiple
and moe_benchmark_static_routing; fused_a2a page, HybridEPDispatch.forward pad_multiple and
num_permuted_tokens), through the separate calls and the fused padded layout + NVFP4 call.
Layout, codes, scales and bf16 rows are bit-exact; combine and the backward passes are within
the tolerances of gpu_helpers."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (CANARY32, abs_dots, assert_close_bf16, assert_close_gradp, dev, dev_bf16,
                         host_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def padded_layout(ep, cfg, ids, pad, cap):
    L = ep.Layout(cfg.T, cfg.K, cfg.E, cfg.P, bool(cfg.S), pad_multiple=pad, num_permuted_tokens=cap)
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    L2, ids_used, probs = ep.dispatch_layout_routed(cfg.E, topk_ids=dev(ids), n_parts=cfg.P,
                                                    capacity=cfg.capacity, fused_shared=bool(cfg.S),
                                                    pad_multiple=pad, num_permuted_tokens=cap, out=L)
    assert L2 is L and probs is None
    return L


def check_padded_layout(ep, L, ref):
    assert ep.read_status(L) == ref.status
    assert L.R_max == ref.R_max
    assert np.array_equal(L.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(L.part_tokens.cpu().numpy(), ref.part_tokens)
    if ref.T:
        assert np.array_equal(L.row_of.cpu().numpy()[:ref.T], ref.row_of)
    n = min(ref.R, ref.R_max)
    ei, si = L.expert_ids.cpu().numpy(), L.src_info.cpu().numpy()
    assert np.array_equal(ei[:n], ref.expert_ids[:n])
    assert np.array_equal(si[:n], ref.src_info[:n])
    assert (ei[n:ref.R_max] == CANARY32).all() and (si[n:ref.R_max] == CANARY32).all()


def check_fused_padded(ep, cfg, ids, xd, pad, cap, ref, ref_rows):
    """ep_dispatch_layout_padded_nvfp4 gives the layout and NVFP4 rows (padding rows included)
    of the two separate calls."""
    L = ep.Layout(cfg.T, cfg.K, cfg.E, cfg.P, bool(cfg.S), pad_multiple=pad, num_permuted_tokens=cap)
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    Rm, H = ref.R_max, xd.shape[1]
    out = (torch.full((Rm, H // 2), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm, H // 16), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm,), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           torch.full((cfg.E + cfg.S + 1,), -7, dtype=torch.int32, device="cuda"))
    ep.dispatch_layout_padded_nvfp4(dev(ids), xd, cfg.E, cfg.P, cfg.capacity, bool(cfg.S), pad, cap,
                                    out_layout=L, out=out)
    check_padded_layout(ep, L, ref)
    rfp4, rsc, rinv, rso = ref_rows
    assert np.array_equal(out[0].cpu().numpy(), rfp4), "fused call: NVFP4 codes"
    assert np.array_equal(out[1].cpu().numpy(), rsc), "fused call: E4M3 scales"
    assert np.array_equal(host_bf16(out[2]), rinv), "fused call: inverse scales"
    assert np.array_equal(out[3].cpu().numpy(), rso), "fused call: scales_offsets"


def run_all(ep, cfg, pad, cap, x=None, ids=None, probs=None, y=None):
    inp = W.make_inputs(cfg) if ids is None else None
    ids = inp["topk_ids"] if ids is None else ids
    probs = inp["probs"] if probs is None else probs
    x = inp["x"] if x is None else x
    H = x.shape[1]
    ref = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S, pad_multiple=pad,
                        num_permuted_tokens=cap)
    L = padded_layout(ep, cfg, ids, pad, cap)
    check_padded_layout(ep, L, ref)
    Rm, G = ref.R_max, cfg.E + cfg.S
    xd = dev_bf16(x)

    out = (torch.full((Rm, H // 2), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm, H // 16), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm,), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           torch.full((G + 1,), -7, dtype=torch.int32, device="cuda"))
    ep.dispatch_nvfp4(xd, L, out=out)
    rfp4, rsc, rinv, rso = oracle.dispatch_nvfp4(x, ref, fill=0xA5)
    assert np.array_equal(out[0].cpu().numpy(), rfp4), "NVFP4 codes"
    assert np.array_equal(out[1].cpu().numpy(), rsc), "E4M3 scales"
    assert np.array_equal(host_bf16(out[2]), rinv), "inverse scales"
    if not ref.status:
        assert np.array_equal(out[3].cpu().numpy(), rso)
    check_fused_padded(ep, cfg, ids, xd, pad, cap, ref, (rfp4, rsc, rinv, rso))

    rows = torch.full((Rm, H), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ep.dispatch_bf16(xd, L, out=rows)
    assert np.array_equal(host_bf16(rows), oracle.dispatch_bf16(x, ref, fill=0xA5A5)), "bf16 rows"

    if H % 128 == 0:
        c8 = torch.full((Rm, H), 0xA5, dtype=torch.uint8, device="cuda")
        s8 = torch.full((Rm, 4 * (H // 128)), 0xA5, dtype=torch.uint8, device="cuda").view(torch.float32)
        ep.dispatch_fp8(xd, L, out=(c8, s8))
        rc8, rs8 = oracle.dispatch_fp8(x, ref, fill=0xA5)
        assert np.array_equal(c8.cpu().numpy(), rc8), "FP8 codes"
        assert np.array_equal(s8.cpu().numpy().view(np.uint32), rs8.view(np.uint32)), "FP8 scales"

    if ref.status:
        return ref
    # expert outputs with NaN in every padding row: combine must never read them
    if y is None:
        y = W.make_expert_out(W.scaled(cfg, T=cfg.T))
    y = np.resize(y, (Rm, H)).astype(np.uint16)
    pad_rows = ref.src_info[:ref.R, 0] < 0
    y[:ref.R][pad_rows] = 0x7FC0
    yd = dev_bf16(y)
    got = ep.combine(yd, dev(probs), L)
    _, ref64 = oracle.combine(y, probs, ref, want64=True)
    assert_close_bf16(host_bf16(got), ref64, "combine")
    g = W.bf16_bits_from_f32(np.random.default_rng(cfg.T).standard_normal((cfg.T, H)).astype(np.float32))
    gy = torch.full((Rm, H), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    gp = torch.full((cfg.T, cfg.K), float("nan"), dtype=torch.float32, device="cuda")
    ep.combine_bwd(dev_bf16(g), yd, dev(probs), L, out=(gy, gp))
    rgy, rgp, rgy64 = oracle.combine_bwd(g, y, probs, ref, want64=True)
    got_gy = host_bf16(gy)
    assert (got_gy[:ref.R][pad_rows] == 0).all(), "padding rows of grad_expert_out"
    real = ~pad_rows
    assert_close_bf16(got_gy[:ref.R][real], rgy64[:ref.R][real], "grad_expert_out")
    assert (got_gy[ref.R:] == 0xA5A5).all()
    assert_close_gradp(gp.cpu().numpy(), rgp, abs_dots(g, y, ref.row_of), "grad_probs")
    gx = ep.dispatch_bwd(yd, L)
    _, rgx64 = oracle.dispatch_bwd(y, ref, want64=True)
    assert_close_bf16(host_bf16(gx), rgx64, "grad_input")
    return ref


CASES = [  # name, T, H, pad, capacity mode
    ("tiny", None, None, 4, None),
    ("qwen3", 1000, 2048, 16, None),
    ("dsv3", 600, 1024, 128, None),
    ("dsv3", 600, 1024, 128, "exact"),
    ("mixtral", 1500, 512, 8, "exact"),
    ("dsv3_large", 2000, 512, 32, None),
    ("tiny", 300, 48, 4, None),                 # 3-byte block-scale rows (odd)
    ("qwen3", 400, 272, 16, "exact"),           # 17-byte block-scale rows (odd)
]


@pytest.mark.parametrize("name,T,H,pad,capmode", CASES,
                         ids=[f"{c[0]}-T{c[1]}-pad{c[3]}-{c[4]}" for c in CASES])
def test_padded_parity(ep, name, T, H, pad, capmode):
    cfg = W.CONFIGS[name]
    kw = {}
    if T:
        kw["T"] = T
    if H:
        kw["H"] = H
    if name == "dsv3_large":
        kw["C"] = T
    cfg = W.scaled(cfg, **kw)
    cap = None
    if capmode == "exact":
        ids, _ = W.make_routing(cfg)
        cap = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S, pad_multiple=pad).R
    ref = run_all(ep, cfg, pad, cap)
    assert ref.status == 0 and (ref.src_info[:ref.R, 0] < 0).any()   # padding rows exercised


@pytest.mark.parametrize("T", [20000, 34000])
def test_padded_layout_beyond_one_cluster(ep, T):
    """160,000 ids: the single-cluster layout with two id batches per lane; 272,000 ids: more
    than one thread-block cluster holds, so the two-kernel layout runs."""
    cfg = W.scaled(W.CONFIGS["dsv3"], T=T, H=256, C=T)
    run_all(ep, cfg, 64, None)


@pytest.mark.parametrize("short", [1, 700])
def test_row_capacity_overflow_writes_nothing(ep, short):
    cfg = W.scaled(W.CONFIGS["qwen3"], T=900, H=256)
    ids, _ = W.make_routing(cfg)
    need = oracle.layout(ids, cfg.E, pad_multiple=4).R
    ref = run_all(ep, cfg, 4, need - short)
    assert ref.status == oracle.OVERFLOW


def test_static_routing_full_layer_layout(ep):
    """The balanced static-routing workload at its own sizes: 128 rows per expert, groups
    padded to 128 (so no padding rows) and a static row capacity of exactly T*K + T."""
    cfg = W.CONFIGS["dsv3_static"]
    ref = run_all(ep, W.scaled(cfg, H=256), cfg.pad_multiple, cfg.num_permuted_tokens)
    assert ref.status == 0 and ref.R == ref.R_max == cfg.num_permuted_tokens
    assert (np.diff(ref.row_offsets[:cfg.E + 1]) == 128).all()


def test_padded_reuse_and_zero_tokens(ep):
    """A padded layout object reused with several routings; T = 0."""
    rng = np.random.default_rng(9)
    cfg = W.scaled(W.CONFIGS["tiny"], T=300, E=12, K=3, S=1, P=3)
    L = ep.Layout(cfg.T, cfg.K, cfg.E, cfg.P, True, pad_multiple=8)
    for trial in range(4):
        ids = rng.integers(-1, cfg.E, size=(cfg.T, cfg.K)).astype(np.int32)
        L.expert_ids.fill_(CANARY32)
        L.src_info.fill_(CANARY32)
        ep.dispatch_layout_routed(cfg.E, topk_ids=dev(ids), n_parts=cfg.P, capacity=cfg.T,
                                  fused_shared=True, pad_multiple=8, out=L)
        check_padded_layout(ep, L, oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.T, S=1, pad_multiple=8))
    L0 = ep.Layout(0, 2, 8, 1, True, pad_multiple=4)
    ep.dispatch_layout_routed(8, topk_ids=torch.empty(0, 2, dtype=torch.int32, device="cuda"),
                              fused_shared=True, pad_multiple=4, out=L0)
    assert ep.read_status(L0) == 0 and L0.row_offsets.cpu().tolist() == [0] * 10
    # the padded layout + NVFP4 call with no tokens: an empty layout, scales_offsets all 0
    L1, (_, _, _, so) = ep.dispatch_layout_padded_nvfp4(
        torch.empty(0, 2, dtype=torch.int32, device="cuda"),
        torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), 8, fused_shared=True, pad_multiple=4)
    assert ep.read_status(L1) == 0 and L1.row_offsets.cpu().tolist() == [0] * 10
    assert so.cpu().tolist() == [0] * 10


EDGE = [  # T, K, E, S, P, pad, case
    (300, 32, 1024, 1, 16, 7, "largest K and E, odd pad"),
    (100, 2, 4, 1, 2, 65536, "largest pad multiple"),
    (129, 1, 1, 0, 1, 3, "one expert, one slot"),
    (200, 3, 8, 1, 2, 8, "every slot unused"),
    (257, 4, 3, 1, 1, 5, "duplicate ids"),
    (17000, 8, 64, 1, 4, 16, "a bad id, single-cluster layout, two id batches"),
    (34000, 8, 64, 1, 4, 16, "a bad id, two-kernel layout"),
]


@pytest.mark.parametrize("T,K,E,S,P,pad,case", EDGE, ids=[c[-1] for c in EDGE])
def test_padded_edge_cases(ep, T, K, E, S, P, pad, case):
    rng = np.random.default_rng(T + K + E)
    H = 256 if T < 10000 else 128
    if case == "duplicate ids":
        ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    elif case == "every slot unused":
        ids = np.full((T, K), -1, np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        ids[rng.random((T, K)) < 0.05] = -1
    if case.startswith("a bad id"):
        ids[5, 3] = E
    x = W.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    p = rng.random((T, K)).astype(np.float32)
    y = W.bf16_bits_from_f32(rng.standard_normal((T * K + T, H)).astype(np.float32))
    cfg = W.Config(900, "edge", T=T, H=H, E=E, K=K, S=S, P=P)
    ref = run_all(ep, cfg, pad, None, x=x, ids=ids, probs=p, y=y)
    if case.startswith("a bad id"):
        assert ref.status == oracle.BAD_EXPERT
    else:
        assert ref.status == 0
