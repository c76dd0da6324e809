"""The C ABI library loads, exports every symbol include/ep.h declares, and rejects bad
arguments on the host (no GPU needed: these paths return before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

import __graft_entry__ as entry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def libpath():
    return entry._load_builder().build()


@pytest.fixture(scope="module")
def checked_libpath():
    return entry._load_builder().build(checked=True)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("ep_dispatch_layout", "ep_dispatch_nvfp4", "ep_dispatch_bf16", "ep_combine",
              "ep_combine_bwd", "ep_dispatch_bwd", "ep_layout_workspace_bytes", "ep_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (ep_[a-z0-9_]+)$", out, flags=re.M))
    missing = set(declared_functions()) - exported
    assert not missing, missing
    lib = ctypes.CDLL(libpath)
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_checked_build_exports_the_same_symbols(libpath, checked_libpath):
    """The bounds-checked debug build is the same ABI."""
    def exported(path):
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                             check=True).stdout
        return set(re.findall(r"\bT (ep_[a-z0-9_]+)$", out, flags=re.M))
    assert exported(checked_libpath) == exported(libpath)
    assert set(declared_functions()) <= exported(checked_libpath)
    lib = ctypes.CDLL(checked_libpath)
    lib.ep_strerror.restype = ctypes.c_char_p
    assert b"bounds" in lib.ep_strerror(7)


def test_binding_signatures_cover_the_header(libpath):
    import combine_topk_ids_histogram_gb300 as ep
    assert set(ep.SIGNATURES) == set(declared_functions())


def test_library_needs_no_cuda_shared_library(libpath):
    out = subprocess.run(["readelf", "-d", libpath], capture_output=True, text=True).stdout
    assert "libcudart" not in out


def test_host_validation_without_gpu(libpath):
    import combine_topk_ids_histogram_gb300 as ep
    L = ep.lib()
    bad = ep.EP_ERR_INVALID_ARG
    assert L.ep_layout_workspace_bytes(128, 0, 8, 0) == 0          # K = 0
    assert L.ep_layout_workspace_bytes(128, 33, 8, 0) == 0         # K above the limit
    assert L.ep_layout_workspace_bytes(128, 9, 8, 0) > 0           # K > E: duplicate ids
    assert L.ep_layout_workspace_bytes(128, 2, 2048, 0) == 0       # E above the limit
    assert L.ep_layout_workspace_bytes(-1, 2, 8, 0) == 0
    assert L.ep_layout_workspace_bytes(128, 2, 8, 1) > 0
    assert L.ep_layout_workspace_bytes(0, 2, 8, 0) > 0
    lay = ep._Layout()
    ref = ctypes.byref(lay)
    # null layout, zero experts, partitions that do not divide E, negative capacity, misaligned
    assert L.ep_dispatch_layout(None, 4, 2, 8, 1, 4, 0, None, None) == bad
    assert L.ep_dispatch_layout(None, 4, 2, 0, 1, 4, 0, ref, None) == bad
    lay.row_offsets = lay.expert_ids = lay.src_info = lay.row_of = 256
    lay.part_tokens = lay.status = lay.workspace = 256
    lay.workspace_bytes = 1 << 20
    assert L.ep_dispatch_layout(256, 4, 2, 8, 3, 4, 0, ref, None) == bad
    assert L.ep_dispatch_layout(256, 4, 2, 8, 1, -1, 0, ref, None) == bad
    assert L.ep_dispatch_layout(258, 4, 2, 8, 1, 4, 0, ref, None) == bad
    lay.workspace_bytes = 8
    assert L.ep_dispatch_layout(256, 4, 2, 8, 1, 4, 0, ref, None) == bad
    # a layout that was never filled (T = K = E = 0) is rejected by every data call
    empty = ctypes.byref(ep._Layout())
    assert L.ep_dispatch_nvfp4(256, 64, empty, 256, 256, 256, 256, None) == bad
    assert L.ep_dispatch_bf16(256, 64, empty, 256, None) == bad
    assert L.ep_combine(256, 256, 64, empty, 256, None) == bad
    assert L.ep_combine_bwd(256, 256, 256, 64, empty, 256, 256, None) == bad
    assert L.ep_dispatch_bwd(256, 64, empty, 256, None) == bad
    # hidden size not a multiple of 16, or too large
    lay2 = ep._Layout(row_offsets=256, expert_ids=256, src_info=256, row_of=256, part_tokens=256,
                      status=256, workspace=256, workspace_bytes=1 << 20, T=4, K=2, E=8, P=1,
                      capacity=4, fused_shared=0)
    r2 = ctypes.byref(lay2)
    assert L.ep_dispatch_nvfp4(256, 40, r2, 256, 256, 256, 256, None) == bad
    assert L.ep_dispatch_nvfp4(256, 65536, r2, 256, 256, 256, 256, None) == bad
    assert L.ep_combine(256, 256, 24, r2, 256, None) == bad
    assert L.ep_combine(264, 256, 64, r2, 256, None) == bad      # misaligned expert_out
    assert L.ep_cvt_e2m1(None, None, -1, None) == bad
    assert L.ep_read_status(None, None, None) == bad
    assert ep.strerror(ep.EP_ERR_OVERFLOW).startswith("a logical partition")


def test_padding_and_routing_host_validation_without_gpu(libpath):
    """Host checks of the padded / routed layout, FP8 dispatch and the routing conversions;
    every call here is rejected before any CUDA call."""
    import combine_topk_ids_histogram_gb300 as ep
    L = ep.lib()
    bad = ep.EP_ERR_INVALID_ARG
    # rows every buffer holds: T*K + S*T + G*(pad-1), or the static capacity
    assert L.ep_rows_max(4096, 8, 256, 1, 1, 0) == 4096 * 9
    assert L.ep_rows_max(4096, 8, 256, 1, 128, 0) == 4096 * 9 + 257 * 127
    assert L.ep_rows_max(4096, 8, 256, 0, 128, 36864) == 36864
    assert L.ep_rows_max(4096, 8, 256, 0, 0, 0) == 4096 * 8          # pad <= 1: none
    assert L.ep_rows_max(4096, 8, 256, 0, 1, -5) == 0
    assert L.ep_rows_max(4096, 8, 256, 0, 70000, 0) == 0              # pad above 65536
    assert ep.rows_max(4, 2, 3, True, 4) == 24
    lay = ep._Layout(row_offsets=256, expert_ids=256, src_info=256, row_of=256, part_tokens=256,
                     status=256, workspace=256, workspace_bytes=1 << 20)
    ref = ctypes.byref(lay)
    args = (4, 2, 8, 1, 4, 0)
    assert L.ep_dispatch_layout_routed(256, None, None, *args, 0, 0, None, None, ref, None) == bad
    assert L.ep_dispatch_layout_routed(256, None, None, *args, 1, -1, None, None, ref, None) == bad
    # a routing map without the buffer for its compact ids
    assert L.ep_dispatch_layout_routed(None, 256, None, *args, 1, 0, None, None, ref, None) == bad
    assert L.ep_dispatch_layout_routed(None, 264, None, *args, 1, 0, 256, None, ref, None) == bad
    assert L.ep_routing_map_to_topk(256, None, 4, 8, 0, 256, None, None) == bad      # K = 0
    assert L.ep_routing_map_to_topk(256, None, 4, 2000, 2, 256, None, None) == bad   # E too large
    assert L.ep_routing_map_to_topk(256, None, 4, 8, 2, None, None, None) == bad
    assert L.ep_indices_to_multihot(256, None, 4, 2, 8, None, None, None) == bad
    assert L.ep_indices_to_multihot(256, 260, 4, 2, 8, 256, None, None) == bad      # misaligned
    lay2 = ep._Layout(row_offsets=256, expert_ids=256, src_info=256, row_of=256, part_tokens=256,
                      status=256, workspace=256, workspace_bytes=1 << 20, T=4, K=2, E=8, P=1,
                      capacity=4, fused_shared=0, pad_multiple=1, row_capacity=0)
    r2 = ctypes.byref(lay2)
    assert L.ep_dispatch_fp8(256, 192, r2, 256, 256, None) == bad     # H % 128 != 0
    assert L.ep_dispatch_fp8(256, 256, r2, None, 256, None) == bad
    lay2.pad_multiple = -1
    assert L.ep_dispatch_fp8(256, 256, r2, 256, 256, None) == bad     # a corrupt layout
    assert "row capacity" in ep.strerror(ep.EP_ERR_OVERFLOW)
