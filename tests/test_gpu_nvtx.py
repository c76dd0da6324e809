"""The optional NVTX ranges (EP_GB300_NVTX=1) change nothing but the profiler's view: a child
process with them on runs the fused layout + NVFP4 call, combine and both backward passes on a
Qwen3-shaped layer and must produce the same bytes as this process, which runs with them off."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
from test_gpu_nvtx import run_ops
np.savez(sys.argv[2], **run_ops())
"""


def run_ops() -> dict:
    import combine_topk_ids_histogram_gb300 as ep
    import workloads as W
    cfg = W.scaled(W.CONFIGS["qwen3"], T=600)
    inp = W.make_inputs(cfg)
    ids = torch.from_numpy(inp["topk_ids"]).cuda()
    probs = torch.from_numpy(inp["probs"]).cuda()
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.from_numpy(W.make_expert_out(cfg).view(np.int16)).cuda().view(torch.bfloat16)
    L = ep.Layout(cfg.T, cfg.K, cfg.E, cfg.P, bool(cfg.S))
    _, (fp4, sc, inv, so) = ep.dispatch_layout_nvfp4(ids, x, cfg.E, cfg.P, cfg.capacity, bool(cfg.S),
                                                     out_layout=L)
    out = ep.combine(y, probs, L)
    gy, gp = ep.combine_bwd(x, y, probs, L)
    gx = ep.dispatch_bwd(y, L)
    torch.cuda.synchronize()
    as_np = lambda t: t.contiguous().view(torch.uint8).cpu().numpy()
    return {"row_of": L.row_of.cpu().numpy(), "fp4": as_np(fp4), "sc": as_np(sc), "inv": as_np(inv),
            "out": as_np(out), "gy": as_np(gy), "gp": as_np(gp), "gx": as_np(gx)}


def test_nvtx_ranges_change_no_result(tmp_path):
    if os.environ.get("EP_GB300_NVTX", "0") not in ("", "0"):
        pytest.skip("this process must run with the ranges off")
    want = run_ops()
    path = str(tmp_path / "nvtx.npz")
    env = dict(os.environ, EP_GB300_NVTX="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    got = np.load(path)
    for name, arr in want.items():
        assert np.array_equal(got[name], arr), f"{name} differs with the NVTX ranges on"
