"""Parity at the five workloads' full sizes, every element compared, in the launch configuration
the benchmark times.

Each output the oracle defines is compared in full against the oracle run on the same seeded
inputs:
* the layout (row_offsets, row_of, src_info, expert_ids, part_tokens, status);
* every NVFP4 row (codes, E4M3 block scales, bf16 inverse scales), from the separate layout +
  dispatch calls and from the fused layout + NVFP4 call the benchmark step makes, and the rows
  past R, which keep the oracle's fill value;
* every BF16 row;
* every combined token;
* at the Qwen3-like layer, both backward passes: every grad_y row, every grad_p entry and every
  token of the dispatch backward pass.

The oracle's binary64 combine sums are taken in token chunks, so host memory stays bounded.
The large DeepSeek-V3-like microbatch must raise the overflow flag at capacity 20000 with every
output untouched, then pass in full at capacity 40000.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (abs_dots, assert_close_bf16, assert_close_gradp, check_layout, dev, dev_bf16,
                         host_bf16, new_layout)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FILL8 = 0xA5            # the oracle's fill byte for rows it does not write
FILL16 = 0xA5A5         # ... and its 16-bit fill
CHUNK_T = 2048          # tokens per oracle combine chunk (binary64 sums: CHUNK_T * H * 8 bytes)
CHUNK_R = 16384         # rows per host comparison chunk
_CACHE = {}


def inputs(cfg):
    """Generated once per workload shape (the capacity does not change the data)."""
    key = (cfg.name, cfg.T, cfg.H)
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = (W.make_inputs(cfg), W.make_expert_out(cfg))
    return _CACHE[key]


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def new_layout_padded(ep, T, K, E, P, S, pad, cap):
    L = ep.Layout(T, K, E, P, bool(S), pad_multiple=pad, num_permuted_tokens=cap)
    L.expert_ids.fill_(-7)
    L.src_info.fill_(-7)
    return L


def filled(shape, bits, dtype):
    """A device buffer holding the oracle's fill pattern (16-bit fills as int16 bit patterns)."""
    if dtype == torch.uint8:
        return torch.full(shape, bits, dtype=torch.uint8, device="cuda")
    return torch.full(shape, bits - 65536 if bits >= 32768 else bits, dtype=torch.int16, device="cuda")


def nvfp4_buffers(R_max, H, E, S):
    return (filled((R_max, H // 2), FILL8, torch.uint8), filled((R_max, H // 16), FILL8, torch.uint8),
            filled((R_max,), FILL16, torch.int16).view(torch.bfloat16),
            torch.full((E + S + 1,), -7, dtype=torch.int32, device="cuda"))


def assert_rows_equal(got: torch.Tensor, ref: np.ndarray, what: str):
    """Bit-exact comparison of a device buffer with the oracle's, CHUNK_R rows at a time."""
    assert got.shape[0] == ref.shape[0], (what, got.shape, ref.shape)
    g = got.view(torch.int16) if got.dtype == torch.bfloat16 else got
    for a in range(0, ref.shape[0], CHUNK_R):
        b = min(ref.shape[0], a + CHUNK_R)
        h = g[a:b].cpu().numpy()
        r = ref[a:b]
        if h.dtype != r.dtype:
            h = h.view(r.dtype)
        if not np.array_equal(h, r):
            bad = np.argwhere(h != r)[0]
            raise AssertionError(f"{what}: first difference at row {a + bad[0]}, index {tuple(bad[1:])}: "
                                 f"gpu {h[tuple(bad)]} oracle {r[tuple(bad)]}")


def token_slice(ref, t0, t1):
    """The oracle layout restricted to tokens [t0, t1): the same rows, the shared row of token t
    still at row_offsets[E] + t (the oracle computes it from the chunk's first token)."""
    sub = oracle.Layout(ref)
    sub["row_of"] = np.ascontiguousarray(ref.row_of[t0:t1])
    ro = ref.row_offsets.copy()
    ro[ref.E] += t0
    sub["row_offsets"] = ro
    sub["T"] = t1 - t0
    return sub


def check_combine_full(out, y_host, probs, ref, what, weighted=True):
    """Every token of combine (probs given) or of the dispatch backward pass (weighted False)
    against the oracle's binary64 sums."""
    got = host_bf16(out)
    for t0 in range(0, ref.T, CHUNK_T):
        t1 = min(ref.T, t0 + CHUNK_T)
        sub = token_slice(ref, t0, t1)
        p = probs[t0:t1] if weighted else None
        _, r64 = oracle.combine(y_host, p, sub, want64=True)
        assert_close_bf16(got[t0:t1], r64, f"{what}, tokens {t0}..{t1}")


def check_nvfp4_full(bufs, ref_rows, what):
    fp4, sc, inv, so = bufs
    rfp4, rsc, rinv, rso = ref_rows
    assert np.array_equal(so.cpu().numpy(), rso), what
    assert_rows_equal(fp4, rfp4, f"{what}: E2M1 codes")
    assert_rows_equal(sc, rsc, f"{what}: E4M3 block scales")
    assert_rows_equal(inv, rinv, f"{what}: inverse scales")


def run_full(ep, cfg, C=None, backward=False, bf16=False):
    C = cfg.capacity if C is None else C
    T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
    inp, y_host = inputs(cfg)
    x, ids, probs = inp["x"], inp["topk_ids"], inp["probs"]
    ref = oracle.layout(ids, E, P=P, C=C, S=S)
    R_max = ref.R_max
    xd, idd, pd = dev_bf16(x), dev(ids), dev(probs)

    # separate calls: layout, NVFP4 dispatch, combine
    L = new_layout(ep, T, K, E, P, S)
    ep.dispatch_layout(idd, E, P, C, bool(S), out=L)
    check_layout(L, ref, ep)
    bufs = nvfp4_buffers(R_max, H, E, S)
    ep.dispatch_nvfp4(xd, L, out=bufs)
    yd = dev_bf16(y_host)
    out = filled((T, H), FILL16, torch.int16).view(torch.bfloat16)
    ep.combine(yd, pd, L, out=out)
    # the fused layout + NVFP4 call
    Lf = new_layout(ep, T, K, E, P, S)
    fbufs = nvfp4_buffers(R_max, H, E, S)
    ep.dispatch_layout_nvfp4(idd, xd, E, P, C, bool(S), out_layout=Lf, out=fbufs)
    torch.cuda.synchronize()
    check_layout(Lf, ref, ep)

    ref_rows = oracle.dispatch_nvfp4(x, ref, fill=FILL8)   # every row untouched on overflow
    check_nvfp4_full(bufs, ref_rows, f"{cfg.name} NVFP4 dispatch")
    check_nvfp4_full(fbufs, ref_rows, f"{cfg.name} fused layout + NVFP4")
    del ref_rows, fbufs
    if ref.status:
        assert (out.view(torch.int16) == FILL16 - 65536).all(), "combine wrote on overflow"
        return ref
    check_combine_full(out, y_host, probs, ref, f"{cfg.name} combine")
    assert torch.equal(ep.combine(yd, pd, L).view(torch.int16), out.view(torch.int16)), "combine rerun"
    if bf16:
        rows = filled((R_max, H), FILL16, torch.int16).view(torch.bfloat16)
        ep.dispatch_bf16(xd, L, out=rows)
        assert_rows_equal(rows, oracle.dispatch_bf16(x, ref, fill=FILL16), f"{cfg.name} BF16 dispatch")
        del rows
    if backward:
        g = W.make_grad_out(cfg)
        gy = filled((R_max, H), FILL16, torch.int16).view(torch.bfloat16)
        gp = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
        ep.combine_bwd(dev_bf16(g), yd, pd, L, out=(gy, gp))
        rgy, rgp, rgy64 = oracle.combine_bwd(g, y_host, probs, ref, want64=True, fill=FILL16)
        R = ref.R
        gyh = host_bf16(gy)
        for a in range(0, R, CHUNK_R):
            b = min(R, a + CHUNK_R)
            assert_close_bf16(gyh[a:b], rgy64[a:b], f"{cfg.name} grad_y rows {a}..{b}")
        assert np.array_equal(gyh[R:], rgy[R:]), "grad_y rows past R were written"
        assert_close_gradp(gp.cpu().numpy(), rgp, abs_dots(g, y_host, ref.row_of), f"{cfg.name} grad_p")
        # determinism: a second call gives the same bytes (grad_p's reduction order is fixed)
        gy2, gp2 = ep.combine_bwd(dev_bf16(g), yd, pd, L)
        assert torch.equal(gy2[:R].view(torch.int16), gy[:R].view(torch.int16))
        assert torch.equal(gp2.view(torch.int32), gp.view(torch.int32))
        del gyh, rgy, rgy64, gy2, gp2
        gr = W.make_grad_rows(cfg)
        gx = filled((T, H), FILL16, torch.int16).view(torch.bfloat16)
        grd = dev_bf16(gr)
        ep.dispatch_bwd(grd, L, out=gx)
        check_combine_full(gx, gr, probs, ref, f"{cfg.name} dispatch backward", weighted=False)
        assert torch.equal(ep.dispatch_bwd(grd, L).view(torch.int16), gx.view(torch.int16))
    return ref


@pytest.mark.parametrize("name", ["tiny", "qwen3", "dsv3", "mixtral"])
def test_full_size(ep, name):
    cfg = W.CONFIGS[name]
    ref = run_full(ep, cfg, backward=(name == "qwen3"), bf16=(name in ("tiny", "mixtral", "dsv3")))
    assert ref.status == 0


def test_full_size_overflow_then_rerun(ep):
    cfg = W.CONFIGS["dsv3_large"]
    ref = run_full(ep, cfg, C=cfg.C)
    assert ref.status == oracle.OVERFLOW
    ref = run_full(ep, cfg, C=cfg.rerun_C)
    assert ref.status == 0


def test_full_size_fp8(ep):
    cfg = W.CONFIGS["dsv3"]
    T, H, E, K, S, P, C = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    inp, _ = inputs(cfg)
    x, ids = inp["x"], inp["topk_ids"]
    ref = oracle.layout(ids, E, P=P, C=C, S=S)
    L = new_layout(ep, T, K, E, P, S)
    ep.dispatch_layout(dev(ids), E, P, C, bool(S), out=L)
    codes = filled((ref.R_max, H), FILL8, torch.uint8)
    scales = filled((ref.R_max, 4 * (H // 128)), FILL8, torch.uint8)
    ep.dispatch_fp8(dev_bf16(x), L, out=(codes, scales.view(torch.float32)))
    rc, rs = oracle.dispatch_fp8(x, ref, fill=FILL8)
    assert_rows_equal(codes, rc, "FP8 codes")
    assert_rows_equal(scales, rs.view(np.uint8).reshape(ref.R_max, -1), "FP8 block scales")


@pytest.mark.parametrize("name,pad,cap", [("dsv3", 128, None), ("dsv3_static", 128, 36864)])
def test_full_size_padded(ep, name, pad, cap):
    """Padded layout, every NVFP4 row (padding rows included) and every combined token."""
    cfg = W.CONFIGS[name]
    T, H, E, K, S, P, C = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    inp = W.make_inputs(cfg)
    x, ids, probs = inp["x"], inp["topk_ids"], inp["probs"]
    ref = oracle.layout(ids, E, P=P, C=C, S=S, pad_multiple=pad, num_permuted_tokens=cap)
    assert ref.status == 0
    L = ep.Layout(T, K, E, P, bool(S), pad_multiple=pad, num_permuted_tokens=cap)
    ep.dispatch_layout_routed(E, topk_ids=dev(ids), n_parts=P, capacity=C, fused_shared=bool(S),
                              pad_multiple=pad, num_permuted_tokens=cap, out=L)
    assert ep.read_status(L) == 0
    assert np.array_equal(L.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(L.row_of.cpu().numpy(), ref.row_of)
    assert np.array_equal(L.expert_ids.cpu().numpy()[:ref.R], ref.expert_ids[:ref.R])
    assert np.array_equal(L.src_info.cpu().numpy()[:ref.R], ref.src_info[:ref.R])
    bufs = nvfp4_buffers(ref.R_max, H, E, S)
    xd = dev_bf16(x)
    ep.dispatch_nvfp4(xd, L, out=bufs)
    ref_rows = oracle.dispatch_nvfp4(x, ref, fill=FILL8)
    check_nvfp4_full(bufs, ref_rows, f"{name} padded NVFP4")
    # the fused padded layout + NVFP4 call the static-routing benchmark step makes
    Lf = new_layout_padded(ep, T, K, E, P, S, pad, cap)
    fbufs = nvfp4_buffers(ref.R_max, H, E, S)
    ep.dispatch_layout_padded_nvfp4(dev(ids), xd, E, P, C, bool(S), pad, cap, out_layout=Lf, out=fbufs)
    assert ep.read_status(Lf) == 0
    assert np.array_equal(Lf.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(Lf.row_of.cpu().numpy(), ref.row_of)
    assert np.array_equal(Lf.expert_ids.cpu().numpy()[:ref.R], ref.expert_ids[:ref.R])
    assert np.array_equal(Lf.src_info.cpu().numpy()[:ref.R], ref.src_info[:ref.R])
    check_nvfp4_full(fbufs, ref_rows, f"{name} fused padded layout + NVFP4")
    del ref_rows, fbufs
    y_host = np.resize(W.make_expert_out(cfg), (ref.R_max, H)).astype(np.uint16)
    out = ep.combine(dev_bf16(y_host), dev(probs), L)
    check_combine_full(out, y_host, probs, ref, f"{name} padded combine")


def test_full_size_routing_map_layout(ep):
    cfg = W.CONFIGS["dsv3"]
    T, E, K, S, P, C = cfg.T, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    inp, _ = inputs(cfg)
    m, d = oracle.indices_to_multihot(inp["topk_ids"], inp["probs"], E)
    rids, rprobs = oracle.routing_map_to_topk(m, d, K)
    ref = oracle.layout(rids, E, P=P, C=C, S=S)
    L = new_layout(ep, T, K, E, P, S)
    _, ids, probs = ep.dispatch_layout_routed(E, routing_map=dev(m), dense_probs=dev(d), K=K,
                                              n_parts=P, capacity=C, fused_shared=bool(S), out=L)
    assert np.array_equal(ids.cpu().numpy(), rids) and np.array_equal(probs.cpu().numpy(), rprobs)
    check_layout(L, ref, ep)
