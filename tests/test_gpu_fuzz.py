"""Seeded random shapes within the ABI's limits, every entry point against the oracle.

Each case draws T, K, E, H, P, S, the capacity, a padding multiple and a static row capacity,
and random ids (with unused slots, duplicates and, sometimes, a bad id), then runs the padded /
capped layout, the NVFP4, BF16 and (when H % 128 == 0) FP8 dispatches, combine and both
backward passes, comparing with the oracle like the parity tests (bit-exact or within the
stated tolerances; nothing written when the status word is set)."""
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


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.choice([0, 1, 7, 33, 129, 500, 1500, 3000]))
    K = int(rng.choice([1, 2, 3, 8, 13, 32]))
    E = int(rng.choice([1, 2, 5, 8, 64, 128, 256, 1000, 1024]))
    P = int(rng.choice([p for p in (1, 2, 4, 5, 8, 16) if E % p == 0 and p <= E]))
    S = int(rng.integers(0, 2))
    H = int(rng.choice([16, 48, 128, 256, 272, 768, 2048]))
    pad = int(rng.choice([1, 1, 2, 3, 16, 128]))
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    ids[rng.random((T, K)) < 0.1] = -1
    bad = T > 0 and rng.random() < 0.15
    if bad:
        ids[rng.integers(0, T), rng.integers(0, K)] = E + int(rng.integers(0, 3))
    C = int(rng.integers(0, T + 1)) if rng.random() < 0.3 else T
    need = oracle.layout(ids, E, P=P, C=C, S=S, pad_multiple=pad).R
    cap = None
    if rng.random() < 0.4 and need > 0:
        cap = int(max(1, need + int(rng.integers(-3, 4))))
    x = W.bf16_bits_from_f32((rng.standard_normal((T, H)) * np.exp(rng.uniform(-3, 3, (T, 1))))
                             .astype(np.float32))
    probs = rng.random((T, K)).astype(np.float32)
    return dict(T=T, K=K, E=E, P=P, S=S, H=H, pad=pad, C=C, cap=cap, ids=ids, x=x, probs=probs,
                rng=rng)


@pytest.mark.parametrize("seed", range(48))
def test_random_case(ep, seed):
    c = draw_case(seed)
    T, K, E, P, S, H, pad, C, cap = (c[k] for k in ("T", "K", "E", "P", "S", "H", "pad", "C", "cap"))
    ids, x, probs, rng = c["ids"], c["x"], c["probs"], c["rng"]
    ref = oracle.layout(ids, E, P=P, C=C, S=S, pad_multiple=pad, num_permuted_tokens=cap)
    L = ep.Layout(T, K, E, P, bool(S), pad_multiple=pad, num_permuted_tokens=cap)
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    ids_d = dev(ids) if T else torch.empty(0, K, dtype=torch.int32, device="cuda")
    ep.dispatch_layout_routed(E, topk_ids=ids_d, n_parts=P, capacity=C, fused_shared=bool(S),
                              pad_multiple=pad, num_permuted_tokens=cap, out=L)
    assert ep.read_status(L) == ref.status
    assert np.array_equal(L.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(L.part_tokens.cpu().numpy(), ref.part_tokens)
    if T:
        assert np.array_equal(L.row_of.cpu().numpy()[:T], ref.row_of)
    n = min(ref.R, ref.R_max)
    assert np.array_equal(L.expert_ids.cpu().numpy()[:n], ref.expert_ids[:n])
    assert np.array_equal(L.src_info.cpu().numpy()[:n], ref.src_info[:n])
    if T == 0:
        return
    Rm = ref.R_max
    xd = dev_bf16(x)

    out = (torch.full((Rm, H // 2), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm, H // 16), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm,), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           torch.full((E + S + 1,), -7, dtype=torch.int32, device="cuda"))
    ep.dispatch_nvfp4(xd, L, out=out)
    rfp4, rsc, rinv, rso = oracle.dispatch_nvfp4(x, ref, fill=0xA5)
    assert np.array_equal(out[0].cpu().numpy(), rfp4)
    assert np.array_equal(out[1].cpu().numpy(), rsc)
    assert np.array_equal(host_bf16(out[2]), rinv)

    # the fused padded layout + NVFP4 call: the same layout and rows
    Lf = ep.Layout(T, K, E, P, bool(S), pad_multiple=pad, num_permuted_tokens=cap)
    outf = tuple(torch.full_like(o, f) for o, f in zip(out, (0xA5, 0xA5, 0, -7)))
    outf[2].view(torch.int16).fill_(-23131)
    ep.dispatch_layout_padded_nvfp4(ids_d, xd, E, P, C, bool(S), pad, cap, out_layout=Lf, out=outf)
    assert ep.read_status(Lf) == ref.status
    assert np.array_equal(Lf.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(Lf.row_of.cpu().numpy(), ref.row_of)
    assert np.array_equal(Lf.expert_ids.cpu().numpy()[:n], ref.expert_ids[:n])
    assert np.array_equal(Lf.src_info.cpu().numpy()[:n], ref.src_info[:n])
    assert np.array_equal(outf[0].cpu().numpy(), rfp4)
    assert np.array_equal(outf[1].cpu().numpy(), rsc)
    assert np.array_equal(host_bf16(outf[2]), rinv)
    assert np.array_equal(outf[3].cpu().numpy(), rso)

    rows = torch.full((Rm, H), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ep.dispatch_bf16(xd, L, out=rows)
    assert np.array_equal(host_bf16(rows), oracle.dispatch_bf16(x, ref, fill=0xA5A5))

    if H % 128 == 0:
        c8, s8 = ep.dispatch_fp8(xd, L, out=(
            torch.full((Rm, H), 0xA5, dtype=torch.uint8, device="cuda"),
            torch.full((Rm, 4 * (H // 128)), 0xA5, dtype=torch.uint8, device="cuda").view(torch.float32)))
        rc8, rs8 = oracle.dispatch_fp8(x, ref, fill=0xA5)
        assert np.array_equal(c8.cpu().numpy(), rc8)
        assert np.array_equal(s8.cpu().numpy().view(np.uint32), rs8.view(np.uint32))

    if ref.status:
        return
    y = W.bf16_bits_from_f32(rng.standard_normal((Rm, H)).astype(np.float32))
    pad_rows = ref.src_info[:ref.R, 0] < 0
    y[:ref.R][pad_rows] = 0x7FC0             # never read by combine or the backward passes
    yd = dev_bf16(y)
    got = ep.combine(yd, dev(probs), L)
    _, r64 = oracle.combine(y, probs, ref, want64=True)
    assert_close_bf16(host_bf16(got), r64, "combine")
    g = W.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    gy, gp = ep.combine_bwd(dev_bf16(g), yd, dev(probs), L)
    rgy, rgp, rgy64 = oracle.combine_bwd(g, y, probs, ref, want64=True)
    got_gy = host_bf16(gy)
    assert (got_gy[:ref.R][pad_rows] == 0).all()
    assert_close_bf16(got_gy[:ref.R][~pad_rows], rgy64[:ref.R][~pad_rows], "grad_expert_out")
    assert_close_gradp(gp.cpu().numpy(), rgp, abs_dots(g, y, ref.row_of), "grad_probs")
    gx = ep.dispatch_bwd(yd, L)
    _, rgx64 = oracle.dispatch_bwd(y, ref, want64=True)
    assert_close_bf16(host_bf16(gx), rgx64, "grad_input")


@pytest.mark.parametrize("seed", range(24))
def test_random_fused_call_and_routing_map(ep, seed):
    """The fused layout + NVFP4 call, and the layout of the same routing given as a dense map,
    on seeded random shapes (no padding: the fused call takes none)."""
    c = draw_case(100 + seed)
    T, K, E, P, S, H, C = (c[k] for k in ("T", "K", "E", "P", "S", "H", "C"))
    ids, x, probs = c["ids"], c["x"], c["probs"]
    if T == 0:
        return
    ref = oracle.layout(ids, E, P=P, C=C, S=S)
    L = ep.Layout(T, K, E, P, bool(S))
    L.expert_ids.fill_(CANARY32)
    L.src_info.fill_(CANARY32)
    Rm = ref.R_max
    out = (torch.full((Rm, H // 2), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm, H // 16), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((Rm,), -23131, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           torch.full((E + S + 1,), -7, dtype=torch.int32, device="cuda"))
    ep.dispatch_layout_nvfp4(dev(ids), dev_bf16(x), E, P, C, bool(S), out_layout=L, out=out)
    assert ep.read_status(L) == ref.status
    assert np.array_equal(L.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(L.part_tokens.cpu().numpy(), ref.part_tokens)
    assert np.array_equal(L.row_of.cpu().numpy(), ref.row_of)
    si, ei = L.src_info.cpu().numpy(), L.expert_ids.cpu().numpy()
    assert np.array_equal(si[:ref.R], ref.src_info[:ref.R])
    assert np.array_equal(ei[:ref.R], ref.expert_ids[:ref.R])
    assert (si[ref.R:Rm] == CANARY32).all() and (ei[ref.R:Rm] == CANARY32).all()
    rfp4, rsc, rinv, _ = oracle.dispatch_nvfp4(x, ref, fill=0xA5)
    assert np.array_equal(out[0].cpu().numpy(), rfp4)
    assert np.array_equal(out[1].cpu().numpy(), rsc)
    assert np.array_equal(host_bf16(out[2]), rinv)

    # the same routing as a dense map (a map holds each expert once per token)
    m, d = oracle.indices_to_multihot(ids, probs, E)
    rids, rprobs = oracle.routing_map_to_topk(m, d, K)
    ref2 = oracle.layout(rids, E, P=P, C=C, S=S)
    L2 = ep.Layout(T, K, E, P, bool(S))
    _, gids, gprobs = ep.dispatch_layout_routed(E, routing_map=dev(m), dense_probs=dev(d), K=K,
                                                n_parts=P, capacity=C, fused_shared=bool(S), out=L2)
    assert np.array_equal(gids.cpu().numpy(), rids)
    assert np.array_equal(gprobs.cpu().numpy(), rprobs)
    assert ep.read_status(L2) == ref2.status
    assert np.array_equal(L2.row_offsets.cpu().numpy(), ref2.row_offsets)
    assert np.array_equal(L2.row_of.cpu().numpy(), ref2.row_of)
    gm, gd = ep.indices_to_multihot(dev(ids), dev(probs), E)
    assert np.array_equal(gm.cpu().numpy(), m)
    assert np.array_equal(gd.cpu().numpy().view(np.uint32), d.view(np.uint32))
