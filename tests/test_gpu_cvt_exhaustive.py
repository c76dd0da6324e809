"""Every binary32 bit pattern the quantiser can feed the hardware conversions, converted on the
GPU and compared with the oracle's encoders (written from the format definitions):

* E2M1: every pattern whose value lies in [-8, 8] (2^30 + 2 patterns of each sign, signed zeros
  included).  The kernel converts products x * (g / s) whose magnitude the block scale keeps at
  or below 6 up to rounding, so [-8, 8] covers every input with margin.
* E4M3: every pattern in [0, 512].  The block scale (max |x| * g) / 6 is non-negative and at
  most 448 up to rounding.

The patterns are generated on the device and on the host from the same integer ranges, in
chunks of 2^26, and the oracle runs on several host threads (its C loop releases the GIL)."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26
E2M1_LAST = 0x41000000   # 8.0
E4M3_LAST = 0x44000000   # 512.0


@pytest.fixture(scope="module")
def ep():
    import combine_topk_ids_histogram_gb300 as ep
    return ep


def _check(a: int, b: int, negate: bool, gpu_codes: np.ndarray, ref_fn, what: str):
    v = np.arange(a, b, dtype=np.uint32).view(np.float32)
    if negate:
        v = -v
    ref = ref_fn(v)
    bad = gpu_codes != ref
    if bad.any():
        i = int(np.argmax(bad))
        return (f"{what}: {int(bad.sum())} mismatches in [{a:#x}, {b:#x}){' negated' if negate else ''}, "
                f"first bits {v.view(np.uint32)[i]:#010x} value {v[i]!r}: gpu {gpu_codes[i]:#x} "
                f"ref {ref[i]:#x}")
    return None


def _sweep(gpu_fn, ref_fn, last: int, signs, what: str):
    errors = []
    with ThreadPoolExecutor(max_workers=8) as pool:
        pending = []
        for negate in signs:
            for a in range(0, last + 1, CHUNK):
                b = min(last + 1, a + CHUNK)
                v = torch.arange(a, b, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
                if negate:
                    v = -v
                codes = gpu_fn(v).cpu().numpy()
                pending.append(pool.submit(_check, a, b, negate, codes, ref_fn, what))
                if len(pending) >= 8:
                    errors += [r for r in (p.result() for p in pending) if r]
                    pending = []
        errors += [r for r in (p.result() for p in pending) if r]
    assert not errors, "\n".join(errors)


def test_e2m1_every_pattern_in_minus8_8(ep):
    _sweep(ep.cvt_e2m1, oracle.e2m1_encode_array, E2M1_LAST, (False, True), "E2M1")


def test_e4m3_every_pattern_in_0_512(ep):
    _sweep(ep.cvt_e4m3, oracle.e4m3_encode_array, E4M3_LAST, (False,), "E4M3")
