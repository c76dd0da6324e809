"""The dispatch -> combine step captured in a CUDA graph and replayed: every call of the path
only enqueues work on the caller's stream (launches with programmatic dependent launch become
programmatic graph edges), so a captured step replays with new inputs copied into its static
buffers and gives the same bytes as the eager calls.  The first eager call sets up the
per-device launch configuration, as the API asks before any capture."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def _inputs(cfg, seed_shift):
    c = W.scaled(cfg, index=cfg.index + 100 * seed_shift)
    inp = W.make_inputs(c)
    return inp, W.make_expert_out(c)


@pytest.mark.parametrize("name,T", [("dsv3", 1024), ("qwen3", 2048)])
def test_captured_step_replays_like_eager(ep, name, T):
    cfg = W.scaled(W.CONFIGS[name], T=T)
    E, K, S, P, C, H = cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity, cfg.H
    R_max = W.r_max(cfg)
    inp0, y0 = _inputs(cfg, 0)
    # static buffers the graph reads and writes
    ids = dev(inp0["topk_ids"])
    x = dev_bf16(inp0["x"])
    probs = dev(inp0["probs"])
    y = dev_bf16(y0)
    L = ep.Layout(cfg.T, K, E, P, bool(S))
    out_rows = (torch.empty(R_max, H // 2, dtype=torch.uint8, device="cuda"),
                torch.empty(R_max, H // 16, dtype=torch.uint8, device="cuda"),
                torch.empty(R_max, dtype=torch.bfloat16, device="cuda"),
                torch.empty(E + S + 1, dtype=torch.int32, device="cuda"))
    out = torch.empty(cfg.T, H, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, out=out_rows, stream=stream)
        ep.combine(y, probs, L, out=out, stream=stream)

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()                                   # eager: sets up the launch configuration
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()

    for shift in (1, 2):
        inp, yh = _inputs(cfg, shift)
        ids.copy_(dev(inp["topk_ids"]))
        x.copy_(dev_bf16(inp["x"]))
        probs.copy_(dev(inp["probs"]))
        y.copy_(dev_bf16(yh))
        for t in out_rows:
            t.view(torch.uint8).fill_(0x5A)
        out.view(torch.int16).fill_(0x1234)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in out_rows] + [out.clone(), L.row_of.clone(), L.row_offsets.clone(),
                                                L.src_info.clone()]
        # the same inputs through eager calls on fresh buffers
        L2 = ep.Layout(cfg.T, K, E, P, bool(S))
        _, rows2 = ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L2)
        out2 = ep.combine(y, probs, L2)
        torch.cuda.synchronize()
        assert ep.read_status(L) == 0 and ep.read_status(L2) == 0
        R = int(L2.row_offsets[L2.G].item())
        ref = [rows2[0][:R], rows2[1][:R], rows2[2][:R], rows2[3], out2, L2.row_of, L2.row_offsets,
               L2.src_info[:R]]
        mine = [got[0][:R], got[1][:R], got[2][:R], got[3], got[4], got[5], got[6], got[7][:R]]
        for a, b in zip(mine, ref):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    del g
