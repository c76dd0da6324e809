"""Concurrent callers: host threads, each with its own CUDA stream and its own layouts (and so
its own workspace), run the whole path at once on different workloads, several times over.
Every result must equal, byte for byte, the same calls made one after another on one stream:
the library keeps no state between calls other than per-device launch settings looked up under
a lock (the no-allocation layout, whose shared array is documented as not to be used by
overlapping calls, is left out)."""
import threading

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import dev, dev_bf16

pytestmark = pytest.mark.gpu

# (workload, tokens, hidden size): the fused call's staged dispatch (qwen3, dsv3), top-2 routing
# over 8 experts (mixtral), and the two-kernel layout beyond one cluster (the large microbatch's
# routing at 40,000 tokens, 320,000 ids; a short hidden size keeps the host-side inputs small)
CASES = [("qwen3", 1500, None), ("dsv3", 600, None), ("mixtral", 3000, None), ("dsv3_large", 40000, 256)]
REPEATS = 3


def host_inputs(cfg) -> tuple:
    return W.make_inputs(cfg), W.make_expert_out(cfg)


def run_path(ep, cfg, host, stream, start=None) -> dict:
    T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
    C = cfg.rerun_C if cfg.rerun_C else cfg.capacity
    inp, y_h = host
    with torch.cuda.stream(stream):
        ids, probs, x, y = dev(inp["topk_ids"]), dev(inp["probs"]), dev_bf16(inp["x"]), dev_bf16(y_h)
        if start is not None:
            start.wait()          # every thread launches its work at the same time
        res = {}
        for rep in range(REPEATS):
            L = ep.Layout(T, K, E, P, bool(S))
            _, nv = ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, stream=stream)
            L2 = ep.dispatch_layout(ids, E, P, C, bool(S), stream=stream)
            bf = ep.dispatch_bf16(x, L2, stream=stream)
            f8 = ep.dispatch_fp8(x, L2, stream=stream)
            out = ep.combine(y, probs, L, stream=stream)
            gy, gp = ep.combine_bwd(x, y, probs, L2, stream=stream)
            gx = ep.dispatch_bwd(y, L2, stream=stream)
            stream.synchronize()
            got = {"row_of": L.row_of, "row_offsets": L.row_offsets, "expert_ids": L2.expert_ids,
                   "src_info": L2.src_info, "fp4": nv[0], "sc": nv[1], "inv": nv[2], "bf16": bf,
                   "fp8": f8[0], "fp8_scales": f8[1], "out": out, "gy": gy, "gp": gp, "gx": gx}
            got = {k: v.contiguous().view(torch.uint8).cpu().numpy() for k, v in got.items()}
            if rep == 0:
                res = got
            else:
                for k in res:
                    assert np.array_equal(res[k], got[k]), f"{cfg.name}: {k} changed between repeats"
    return res


def test_concurrent_streams_match_serial():
    import combine_topk_ids_histogram_gb300 as ep
    cfgs = [W.scaled(W.CONFIGS[n], T=T, H=H) for n, T, H in CASES]
    hosts = [host_inputs(c) for c in cfgs]
    serial = [run_path(ep, c, h, torch.cuda.current_stream()) for c, h in zip(cfgs, hosts)]

    results, errors = [None] * len(cfgs), []
    start = threading.Barrier(len(cfgs), timeout=300)

    def worker(i):
        try:
            results[i] = run_path(ep, cfgs[i], hosts[i], torch.cuda.Stream(), start)
        except Exception as e:   # reported below, from the main thread
            errors.append(f"{cfgs[i].name}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cfgs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not errors, "\n".join(errors)
    for cfg, want, got in zip(cfgs, serial, results):
        assert got is not None, f"{cfg.name}: no result"
        for k in want:
            assert np.array_equal(want[k], got[k]), f"{cfg.name}: {k} differs from the serial run"
