"""GPU vs oracle parity of the FP8 (E4M3, one fp32 scale per 128 elements) dispatch (fused_a2a
page, init_hybrid_ep_buffer, fp8_dispatch): codes and scales bit-exact on the workload recipes,
edge rows and sizes, and nothing written while the layout's status is set."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import dev, dev_bf16, new_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def fp8_check(ep, cfg, x=None, ids=None, C=None):
    inp = W.make_inputs(cfg)
    x = inp["x"] if x is None else x
    ids = inp["topk_ids"] if ids is None else ids
    T, H = x.shape
    C = cfg.capacity if C is None else C
    ref = oracle.layout(ids, cfg.E, P=cfg.P, C=C, S=cfg.S)
    L = new_layout(ep, T, cfg.K, cfg.E, cfg.P, cfg.S)
    ep.dispatch_layout(dev(ids), cfg.E, cfg.P, C, bool(cfg.S), out=L)
    Rm = max(ref.R_max, 1)
    c8 = torch.full((Rm, H), 0xA5, dtype=torch.uint8, device="cuda")
    s8 = torch.full((Rm, 4 * (H // 128)), 0xA5, dtype=torch.uint8, device="cuda").view(torch.float32)
    ep.dispatch_fp8(dev_bf16(x), L, out=(c8, s8))
    rc8, rs8 = oracle.dispatch_fp8(x, ref, fill=0xA5)
    assert np.array_equal(c8.cpu().numpy()[:ref.R_max], rc8), "FP8 codes"
    assert np.array_equal(s8.cpu().numpy()[:ref.R_max].view(np.uint32), rs8.view(np.uint32)), "scales"
    return ref


CASES = [("tiny", None, None), ("qwen3", 1000, None), ("dsv3", 600, None), ("mixtral", 1500, None),
         ("dsv3_large", 2000, 1220), ("dsv3_static", 700, None)]


@pytest.mark.parametrize("name,T,C", CASES, ids=[c[0] for c in CASES])
def test_fp8_parity(ep, name, T, C):
    cfg = W.CONFIGS[name]
    kw = {"T": T} if T else {}
    if C:
        kw["C"] = C
    cfg = W.scaled(cfg, **kw) if kw else cfg
    ref = fp8_check(ep, cfg)
    if name == "dsv3_large":
        assert ref.status == oracle.OVERFLOW   # overflow: nothing written (checked above)


@pytest.mark.parametrize("H", [128, 384, 8192, 32768])
def test_fp8_hidden_sizes(ep, H):
    fp8_check(ep, W.scaled(W.CONFIGS["qwen3"], T=37 if H < 32768 else 5, H=H))


def test_fp8_edge_rows(ep):
    """All-zero rows, negative zeros, huge and tiny magnitudes, single-spike blocks."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=64, H=512)
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 512)).astype(np.float32)
    v[0] = 0.0
    v[1] = -0.0
    v[2] *= np.float32(2.0 ** 100)
    v[3] *= np.float32(2.0 ** -124)       # 448 / max overflows: s clamps to FLT_MAX
    v[4] = 0.0
    v[4, 7] = 3.0
    v[5, ::2] = 0.0
    v[6] = np.float32(1.0)
    x = W.bf16_bits_from_f32(v)
    x[1] = 0x8000
    fp8_check(ep, cfg, x=x)


def test_fp8_rejects_bad_hidden_size(ep):
    cfg = W.scaled(W.CONFIGS["tiny"], T=8, H=272)
    inp = W.make_inputs(cfg)
    L = new_layout(ep, 8, cfg.K, cfg.E, 1, 0)
    ep.dispatch_layout(dev(inp["topk_ids"]), cfg.E, out=L)
    with pytest.raises(ValueError):
        ep.dispatch_fp8(dev_bf16(inp["x"]), L)
    rc = ep.lib().ep_dispatch_fp8(dev_bf16(inp["x"]).data_ptr(), 272, L.ref, 0, 0, None)
    assert rc == ep.EP_ERR_INVALID_ARG
