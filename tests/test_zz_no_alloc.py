"""ep_dispatch_layout_noalloc: the dispatch layout for callers that cannot allocate device memory.

Callers such as code under a framework whose allocator owns the device, latency-critical paths
that must not allocate, or runtimes that only hand a library its inputs and outputs cannot give
the layout a scratch workspace.  This entry point takes its scratch from a fixed array inside
the library.  Its result must equal ep_dispatch_layout's bit for bit (the layout's tolerance is
exact), on two calls in a row that share that array.  The file sorts last so that a run that
stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _routing(T, K, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < 0.05] = -1
    return torch.from_numpy(ids).cuda()


def _layout_bytes(L):
    R = int(L.row_offsets[L.G].item())
    return {"row_offsets": L.row_offsets.cpu(), "row_of": L.row_of.cpu(),
            "part_tokens": L.part_tokens.cpu(), "status": L.status[:1].cpu(),
            "expert_ids": L.expert_ids[:R].cpu(), "src_info": L.src_info[:R].cpu()}


def test_noalloc_layout_equals_allocating_layout_on_two_calls():
    import combine_topk_ids_histogram_gb300 as ep

    T, K, E, P, S, C = 4096, 8, 256, 8, True, 4096      # the DSv3-shaped layer
    out = ep.Layout(T, K, E, P, S)
    out.c.workspace = None                              # the no-allocation call ignores it
    out.c.workspace_bytes = 0
    for call, seed in enumerate((101, 202)):            # two calls in a row share the array
        ids = _routing(T, K, E, seed)
        ref = ep.dispatch_layout(ids, E, P, C, S)       # the existing entry point
        got = ep.dispatch_layout_noalloc(ids, E, P, C, S, out=out)
        torch.cuda.synchronize()
        a, b = _layout_bytes(ref), _layout_bytes(got)
        for name in a:
            assert torch.equal(a[name], b[name]), f"call {call}: {name} differs"
        assert ep.read_status(got) == 0


def test_noalloc_layout_rejects_sizes_beyond_its_array():
    import combine_topk_ids_histogram_gb300 as ep

    T, K, E = 600000, 8, 256
    assert ep.layout_workspace_bytes(T, K, E) > ep.NOALLOC_WORKSPACE_BYTES
    lay = ep._Layout(row_offsets=256, expert_ids=256, src_info=256, row_of=256,
                     part_tokens=256, status=256)
    rc = ep.lib().ep_dispatch_layout_noalloc(256, T, K, E, 1, T, 0, ctypes.byref(lay), None)
    assert rc == ep.EP_ERR_TOO_LARGE
    assert "no-allocation" in ep.strerror(rc)
