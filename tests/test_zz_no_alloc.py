"""ep_dispatch_layout_noalloc: the dispatch layout for callers that cannot allocate device memory.

Callers such as code under a framework whose allocator owns the device, latency-critical paths
that must not allocate, or runtimes that only hand a library its inputs and outputs cannot give
the layout a scratch workspace.  This entry point needs none: sizes that fit one thread-block
cluster run the single-cluster kernel, and larger sizes take their scratch from a fixed array
inside the library.  Its result must equal ep_dispatch_layout's and the oracle's bit for bit (the
layout's tolerance is exact), on calls in a row that share that array, including a call that
reports an error followed by a clean one.  The file sorts last so that a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _routing(T, K, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < 0.05] = -1
    return ids


def _layout_bytes(L):
    R = int(L.row_offsets[L.G].item())
    return {"row_offsets": L.row_offsets.cpu(), "row_of": L.row_of.cpu(),
            "part_tokens": L.part_tokens.cpu(), "status": L.status[:1].cpu(),
            "expert_ids": L.expert_ids[:R].cpu(), "src_info": L.src_info[:R].cpu()}


def _no_workspace_layout(ep, T, K, E, P, S):
    out = ep.Layout(T, K, E, P, S)
    out.c.workspace = None                              # the no-allocation call ignores it
    out.c.workspace_bytes = 0
    return out


def _check_against_oracle(got, ids, E, P, C, S):
    ref = oracle.layout(ids, E, P=P, C=C, S=int(S))
    R = ref.R
    assert int(got.status[0].item()) == ref.status
    assert np.array_equal(got.row_offsets.cpu().numpy(), ref.row_offsets)
    assert np.array_equal(got.row_of.cpu().numpy(), ref.row_of)
    assert np.array_equal(got.part_tokens.cpu().numpy(), ref.part_tokens)
    assert np.array_equal(got.expert_ids[:R].cpu().numpy(), ref.expert_ids[:R])
    assert np.array_equal(got.src_info[:R].cpu().numpy(), ref.src_info[:R])


@pytest.mark.parametrize("T,K,E,P,S,C", [
    (4096, 8, 256, 8, True, 4096),        # the DSv3-shaped layer: fits one cluster, no scratch
    (40001, 8, 256, 8, False, 40001),     # 320,008 ids: the fixed scratch array, ragged tiles
])
def test_noalloc_layout_equals_allocating_layout_on_two_calls(T, K, E, P, S, C):
    import combine_topk_ids_histogram_gb300 as ep

    out = _no_workspace_layout(ep, T, K, E, P, S)
    for call, seed in enumerate((101, 202)):            # two calls in a row share the array
        ids_h = _routing(T, K, E, seed + T)
        ids = torch.from_numpy(ids_h).cuda()
        ref = ep.dispatch_layout(ids, E, P, C, S)       # the existing entry point
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        got = ep.dispatch_layout_noalloc(ids, E, P, C, S, out=out)
        torch.cuda.synchronize()
        if call == 1:   # the first call on a device may load kernels; later ones allocate nothing
            assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
            assert torch.cuda.memory_allocated() == alloc0
        a, b = _layout_bytes(ref), _layout_bytes(got)
        for name in a:
            assert torch.equal(a[name], b[name]), f"call {call}: {name} differs"
        assert ep.read_status(got) == 0
        _check_against_oracle(got, ids_h, E, P, C, S)


def test_noalloc_layout_error_then_clean_call():
    """A call that reports a bad expert id, one that overflows a partition, then a clean call:
    the shared array is left ready for the next call whatever the status."""
    import combine_topk_ids_histogram_gb300 as ep

    T, K, E, P, S = 40000, 8, 256, 8, True              # 320,000 ids: the fixed scratch array
    out = _no_workspace_layout(ep, T, K, E, P, S)
    ids_h = _routing(T, K, E, 7)
    bad = ids_h.copy()
    bad[12345, 3] = E                                   # one id outside [-1, E)
    got = ep.dispatch_layout_noalloc(torch.from_numpy(bad).cuda(), E, P, T, S, out=out)
    assert ep.read_status(got) == ep.STATUS_BAD_EXPERT
    rc = ep.lib().ep_read_status(got.ref, None, ctypes.byref(ctypes.c_int32()))
    assert rc == ep.EP_ERR_BAD_EXPERT
    _check_against_oracle(got, bad, E, P, T, S)
    got = ep.dispatch_layout_noalloc(torch.from_numpy(ids_h).cuda(), E, P, 1000, S, out=out)
    assert ep.read_status(got) & ep.STATUS_OVERFLOW
    rc = ep.lib().ep_read_status(got.ref, None, ctypes.byref(ctypes.c_int32()))
    assert rc == ep.EP_ERR_OVERFLOW
    _check_against_oracle(got, ids_h, E, P, 1000, S)
    ids = torch.from_numpy(ids_h).cuda()
    got = ep.dispatch_layout_noalloc(ids, E, P, T, S, out=out)
    assert ep.read_status(got) == 0
    ref = ep.dispatch_layout(ids, E, P, T, S)
    torch.cuda.synchronize()
    a, b = _layout_bytes(ref), _layout_bytes(got)
    for name in a:
        assert torch.equal(a[name], b[name]), f"clean call after errors: {name} differs"
    _check_against_oracle(got, ids_h, E, P, T, S)


def test_noalloc_layout_rejects_sizes_beyond_its_array():
    import combine_topk_ids_histogram_gb300 as ep

    T, K, E = 600000, 8, 256
    assert ep.layout_workspace_bytes(T, K, E) > ep.NOALLOC_WORKSPACE_BYTES
    lay = ep._Layout(row_offsets=256, expert_ids=256, src_info=256, row_of=256,
                     part_tokens=256, status=256)
    rc = ep.lib().ep_dispatch_layout_noalloc(256, T, K, E, 1, T, 0, ctypes.byref(lay), None)
    assert rc == ep.EP_ERR_TOO_LARGE
    assert "no-allocation" in ep.strerror(rc)
